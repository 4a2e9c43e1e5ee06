"""The unowned-row invariant on the GPU: NaN / Inf / random bytes (and e8m0 255) in
every row no sequence owns, and in their per-token scales, give output that is finite
and bit-identical to the zero-filled run ("[FlyDSL] pa_decode: zero V rows past the
context before PV", Tests).  Also: repeated runs and CUDA-graph replays are bitwise
stable."""
import numpy as np
import pytest
import torch

from paged_attention_decode_02_gb300 import ops, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_attention_decode_02_gb300 import build
    build.build()
    ops.load_library()


def gpu_bits(p, **kw):
    dev = synth.to_device(p, "cuda")
    out = torch.full(tuple(p["query"].shape), float("nan"), dtype=torch.bfloat16, device="cuda")
    out, _, ws = ops.decode(dev, out, **kw)
    torch.cuda.synchronize()
    assert ops.pa_decode_read_status(ws) == 0
    return out.view(torch.int16).cpu().numpy()


def _f32(bits16):
    return (bits16.view(np.uint16).astype(np.uint32) << 16).view(np.float32)


def _cases():
    lens = [1, 17, 255, 257, 1000]
    out = []
    for page in (16, 64, 128):
        out.append(synth.Case(f"bf16_p{page}", synth.KV_BF16, synth.SCALE_NONE, synth.Q_BF16,
                              batch=5, qlen=1, num_kv_heads=1, num_q_heads=8, head_dim=128,
                              page_size=page, context_lens=lens, seed=3000 + page))
        out.append(synth.Case(f"fp8t_p{page}", synth.KV_FP8, synth.SCALE_TENSOR, synth.Q_BF16,
                              batch=5, qlen=4, num_kv_heads=2, num_q_heads=16, head_dim=256,
                              page_size=page, context_lens=lens, seed=3100 + page, kv_std=20.0))
        out.append(synth.Case(f"fp8k_p{page}", synth.KV_FP8, synth.SCALE_TOKEN, synth.Q_BF16,
                              batch=5, qlen=4, num_kv_heads=1, num_q_heads=4, head_dim=128,
                              page_size=page, context_lens=lens, seed=3200 + page, kv_std=20.0))
    out.append(synth.Case("mxfp4_p128", synth.KV_MXFP4, synth.SCALE_E8M0, synth.Q_E4M3,
                          batch=5, qlen=1, num_kv_heads=1, num_q_heads=16, head_dim=128,
                          page_size=128, context_lens=lens, seed=3300))
    out.append(synth.Case("mxfp4_p16_bfq", synth.KV_MXFP4, synth.SCALE_E8M0, synth.Q_BF16,
                          batch=5, qlen=1, num_kv_heads=2, num_q_heads=16, head_dim=128,
                          page_size=16, context_lens=lens, seed=3301))
    return out


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c.name)
@pytest.mark.parametrize("mode", ["split", "direct", "fused", "split-tc", "direct-tc"])
def test_unowned_fill_is_bit_identical(case, mode):
    # "-tc": the tcgen05 kernel (head_dim 128 shapes; others fall back to mma.sync)
    kernel = None
    if mode.endswith("-tc"):
        kernel = "tc"
        mode = mode[:-3]
    kw = dict(max_partitions=1 if mode == "direct" else 0, task_budget=16,
              merge_in_decode=mode == "fused", kernel=kernel)
    p = synth.make(case)
    base = gpu_bits(synth.refill(p, synth.FILL_ZERO), **kw)
    assert np.isfinite(_f32(base)).all()
    fills = (synth.FILL_NAN, synth.FILL_INF, synth.FILL_RANDOM)
    for fill in fills:
        got = gpu_bits(synth.refill(p, fill), **kw)
        assert np.isfinite(_f32(got)).all(), fill
        assert np.array_equal(got, base), fill


def test_repeat_and_graph_replay_are_bitwise_stable():
    case = synth.config3(qlen=4, batch=4, context_lens=(300, 2000), seed=3400)
    p = synth.make(case)
    dev = synth.to_device(p, "cuda")
    out = torch.empty(tuple(p["query"].shape), dtype=torch.bfloat16, device="cuda")
    out, args, ws = ops.decode(dev, out, task_budget=24)
    torch.cuda.synchronize()
    first = out.clone()
    ops.pa_decode_run(args, ws)
    torch.cuda.synchronize()
    assert torch.equal(first.view(torch.int16), out.view(torch.int16))
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        out.zero_()
        with torch.cuda.graph(g, stream=s):
            ops.pa_decode_run(args, ws, stream=s)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(first.view(torch.int16), out.view(torch.int16))
