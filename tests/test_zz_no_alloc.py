"""pa_decode_run_static: the entry point for callers that cannot allocate device memory
(code inside another runtime's memory budget, or loops where an allocation may
synchronise the device).  With the same arguments it runs the same plan and the same
kernels as pa_decode_run with a caller-allocated workspace, so the two outputs must agree
bit for bit, call after call; the output must also match the oracle, the status word of
the fixed array must read back as 0 after each call, and problems whose workspace would
exceed the fixed maximum must be refused.  Kept in a file of its own that pytest collects
last."""
import numpy as np
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
    host = synth.make(case)
    ref = util.oracle_decode(host)
    p = synth.to_device(host, "cuda")
    shape = tuple(p["query"].shape)
    alloc_out = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    args = _args(p, alloc_out, task_budget=48)
    ws = ops.alloc_workspace(args)
    ops.pa_decode_run(args, ws)
    torch.cuda.synchronize()
    assert ops.pa_decode_read_status(ws) == 0
    alloc_bits = alloc_out.view(torch.int16).cpu().numpy()
    for _ in range(2):  # two calls in a row share the fixed array
        out = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        sargs = _args(p, out, task_budget=48)
        ops.pa_decode_run_static(sargs)
        torch.cuda.synchronize()
        assert ops.pa_decode_read_status_static() == 0
        assert np.array_equal(out.view(torch.int16).cpu().numpy(), alloc_bits), \
            "static vs allocated workspace: same plan, same kernels, different bits"
        util.assert_parity(out.float().cpu().numpy(), ref, case.kv, "static workspace vs oracle")


def test_static_workspace_refuses_oversized_problem():
    p = synth.to_device(synth.make(CASES[0]), "cuda")
    out = torch.empty(tuple(p["query"].shape), dtype=torch.bfloat16, device="cuda")
    args = _args(p, out, task_budget=200000)
    assert ops.pa_decode_workspace_size(args) > ops.STATIC_WORKSPACE_BYTES
    with pytest.raises(ops.PaDecodeError) as e:
        ops.pa_decode_run_static(args)
    assert e.value.status == ops.PA_ERR_WORKSPACE


def test_static_status_reports_a_wait_that_ran_out():
    # a child process whose first decode call leaves one ring slot per CTA unloaded: the
    # timeout must be readable through the static status word, and the next static call on
    # the same context must be correct with a clean status
    from tests.test_wait_timeout import run_child
    res = run_child("static")
    assert res["status"] == [ops.PA_DEVICE_WAIT_TIMEOUT, 0], res
