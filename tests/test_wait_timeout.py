"""A pipeline wait that runs out: the kernel gives up after its time limit, records the
timeout in the device status word and returns, and the context stays usable.  The wait is
made to run out on the host's request: a child process started with
PA_DECODE_TEST_DROP_SLICE=1 (read once per process by the library; it affects that
process's first decode call only) leaves one ring slot of each CTA unloaded (in the tile
kernel, the first slot of the first warp; in the MXFP4 tcgen05 kernel, the chunk's first
block); nothing faults, traps or hangs."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run_child(mode: str, kv: str = "fp8") -> dict:
    env = dict(os.environ, PA_DECODE_TEST_DROP_SLICE="1")
    r = subprocess.run([sys.executable, "-m", "tests.wait_timeout_child", mode, kv], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    return json.loads(r.stdout.strip().splitlines()[-1])


@pytest.mark.parametrize("kv", ["fp8", "mxfp4"])
def test_a_wait_that_runs_out_reports_timeout_and_the_context_survives(kv):
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_attention_decode_02_gb300 import build
    build.build()
    res = run_child("allocated", kv)
    from paged_attention_decode_02_gb300 import ops
    assert res["status"] == [ops.PA_DEVICE_WAIT_TIMEOUT, 0], res
