"""Child process of the wait-timeout tests (not collected by pytest): started with
PA_DECODE_TEST_DROP_SLICE=1, so that the library's first decode call leaves one ring slot
per CTA unloaded and that pipeline wait runs out.  It makes that call, then a normal one on
the same context, and prints one JSON line: both status words and the second call's parity
against the oracle.  Usage: python -m tests.wait_timeout_child allocated|static [fp8|mxfp4]
(fp8 per-token KV runs the tile kernel, MXFP4 KV the block-scaled tcgen05 kernel)."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from paged_attention_decode_02_gb300 import ops, synth  # noqa: E402
from tests import util  # noqa: E402


def main(mode: str, kv: str):
    assert os.environ.get("PA_DECODE_TEST_DROP_SLICE") == "1"
    ops.load_library()
    case = synth.config5(synth.KV_FP8 if kv == "fp8" else synth.KV_MXFP4, batch=2,
                         context_lens=(20000, 30000), seed=2901)
    p = synth.make(case)
    ref = util.oracle_decode(p)  # before the first GPU call
    dev = synth.to_device(p, "cuda")
    shape = tuple(p["query"].shape)
    status = []
    out = None
    for _ in range(2):
        out = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
        if mode == "static":
            args = ops.make_args(dev["query"], dev["key_cache"], dev["value_cache"],
                                 dev["block_tables"], dev["context_lens"], out,
                                 key_scale=dev["key_scale"], value_scale=dev["value_scale"],
                                 softmax_scale=case.scale_qk())
            ops.pa_decode_run_static(args)
            torch.cuda.synchronize()
            status.append(ops.pa_decode_read_status_static())
        else:
            _, _, ws = ops.decode(dev, out)
            torch.cuda.synchronize()
            status.append(ops.pa_decode_read_status(ws))
    got = out.float().cpu().numpy()
    r, m = util.assert_parity(got, ref, case.kv, case.name)
    print(json.dumps({"status": status, "rel_l2": r, "max_abs": m}))


if __name__ == "__main__":
    main(sys.argv[1], sys.argv[2] if len(sys.argv) > 2 else "fp8")
