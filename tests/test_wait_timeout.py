"""A pipeline wait that runs out: the kernel gives up after its time limit, records the
timeout in the device status word and returns, and the context stays usable.  The wait is
made to run out on the host's request (an environment hook that leaves the first ring slot
of each CTA's first warp unloaded); nothing faults, traps or hangs."""
import pytest
import torch

from paged_attention_decode_02_gb300 import ops, synth
from tests import util

pytestmark = pytest.mark.gpu


def test_a_wait_that_runs_out_reports_timeout_and_the_context_survives(monkeypatch):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_attention_decode_02_gb300 import build
    build.build()
    ops.load_library()
    case = synth.config5(synth.KV_FP8, batch=2, context_lens=(20000, 30000), seed=2901)
    p = synth.make(case)
    dev = synth.to_device(p, "cuda")
    shape = tuple(p["query"].shape)
    monkeypatch.setenv("PA_DECODE_TEST_DROP_SLICE", "1")
    _, _, ws = ops.decode(dev, torch.zeros(shape, dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert ops.pa_decode_read_status(ws) == ops.PA_DEVICE_WAIT_TIMEOUT
    monkeypatch.delenv("PA_DECODE_TEST_DROP_SLICE")
    out, _, ws = ops.decode(dev, torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda"))
    torch.cuda.synchronize()
    assert ops.pa_decode_read_status(ws) == 0
    util.assert_parity(out.float().cpu().numpy(), util.oracle_decode(p), case.kv, case.name)
