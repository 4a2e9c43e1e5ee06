"""pa_decode_run_static: the entry point for callers that cannot allocate device memory
(code inside another runtime's memory budget, or loops where an allocation may
synchronise the device).  It must give the same output as pa_decode_run with a
caller-allocated workspace, call after call, and refuse problems whose workspace would
exceed its fixed maximum.  Kept in a file of its own that pytest collects last."""
import pytest
import torch

from paged_attention_decode_02_gb300 import ops, synth
from tests import util

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_attention_decode_02_gb300 import build
    build.build()
    ops.load_library()


def _args(p, out, **kw):
    q = p["query"]
    if q.dtype == torch.uint8:
        q = q.view(torch.float8_e4m3fn)
    return ops.make_args(q, p["key_cache"], p["value_cache"], p["block_tables"], p["context_lens"],
                         out, key_scale=p["key_scale"], value_scale=p["value_scale"],
                         q_scale=p["q_scale"], softmax_scale=p["case"].scale_qk(), **kw)


CASES = [
    synth.config3(qlen=4, batch=4, context_lens=(300, 3000), seed=4001),
    synth.config5(synth.KV_MXFP4, batch=4, context_lens=(20000, 40000), seed=4002),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_static_workspace_matches_allocated_workspace(case):
    p = synth.to_device(synth.make(case), "cuda")
    shape = tuple(p["query"].shape)
    ref_out = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    args = _args(p, ref_out, task_budget=48)
    ws = ops.alloc_workspace(args)
    ops.pa_decode_run(args, ws)
    torch.cuda.synchronize()
    ref = ref_out.float().cpu().numpy()
    for _ in range(2):  # two calls in a row share the fixed array
        out = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        sargs = _args(p, out, task_budget=48)
        ops.pa_decode_run_static(sargs)
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        util.assert_parity(got, ref, case.kv, "static vs allocated workspace")


def test_static_workspace_refuses_oversized_problem():
    p = synth.to_device(synth.make(CASES[0]), "cuda")
    out = torch.empty(tuple(p["query"].shape), dtype=torch.bfloat16, device="cuda")
    args = _args(p, out, task_budget=200000)
    assert ops.pa_decode_workspace_size(args) > ops.STATIC_WORKSPACE_BYTES
    with pytest.raises(ops.PaDecodeError) as e:
        ops.pa_decode_run_static(args)
    assert e.value.status == ops.PA_ERR_WORKSPACE
