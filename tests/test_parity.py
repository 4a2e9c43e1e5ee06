"""GPU parity: the CUDA path through the C ABI against the fp64 oracle.

Tolerances (stated for this method): relative L2 <= 5e-3 for bf16 KV and <= 3e-3
for fp8 / MXFP4 KV, max abs <= 3e-2.  Outputs are pre-filled with NaN so that an
unwritten row fails.  Small cases compare every element; full-size cases compare
every row of a sample of sequences that the oracle computes one by one.
"""
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


def run_gpu(p, **kw):
    dev = synth.to_device(p, "cuda")
    out = torch.full(tuple(p["query"].shape), float("nan"), dtype=torch.bfloat16, device="cuda")
    out, args, ws = ops.decode(dev, out, **kw)
    torch.cuda.synchronize()
    assert ops.pa_decode_read_status(ws) == 0
    return out.float().cpu().numpy()


SMALL = [
    synth.config1(),
    synth.config1(context_lens=[1, 1000], seed=2001),
    synth.config2("a"),
    synth.config2("b", batch=6, seed=2002),
    synth.config3(qlen=1, batch=4, context_lens=(200, 1500), seed=2003),
    synth.config3(qlen=4, batch=3, context_lens=(200, 900), seed=2004),
    synth.config4(batch=8),
    synth.config4(batch=5, context_lens=[2048, 1, 129, 0, 3000], seed=2005),
    synth.config5(synth.KV_MXFP4, batch=3, context_lens=(3000, 9000), seed=2006),
    synth.config5(synth.KV_FP8, batch=3, context_lens=(3000, 9000), seed=2007),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: f"{c.name}-s{c.seed}")
@pytest.mark.parametrize("mode", ["split", "direct", "fused"])
def test_small_cases_match_oracle(case, mode):
    p = synth.make(case)
    ref = util.oracle_decode(p)
    got = run_gpu(p, max_partitions=1 if mode == "direct" else 0, task_budget=64,
                  merge_in_decode=mode == "fused")
    util.assert_parity(got, ref, case.kv, case.name)


RAMP = [
    synth.replace(synth.config1(context_lens=[3000, 700], seed=2301), ramp=14.0),
    synth.replace(synth.config5(synth.KV_FP8, batch=3, context_lens=(3000, 9000), seed=2302), ramp=14.0),
    synth.replace(synth.config5(synth.KV_MXFP4, batch=3, context_lens=(3000, 9000), seed=2303), ramp=14.0),
    synth.replace(synth.config4(batch=6, seed=2304), ramp=10.0),
]


KERNELS = [None, "mma", "tc"]  # the library's choice, the mma.sync tile kernel, tcgen05 (f16 / f8f6f4)


@pytest.mark.parametrize("case", RAMP, ids=lambda c: f"{c.name}-ramp")
@pytest.mark.parametrize("mode", ["split", "direct"])
@pytest.mark.parametrize("kernel", KERNELS, ids=lambda k: k or "default")
def test_rising_magnitudes_match_oracle(case, mode, kernel):
    # scores and V scales keep growing along each sequence: the running max and the V
    # references rise again and again, and every rise rescales the accumulated output
    p = synth.make(case)
    ref = util.oracle_decode(p)
    got = run_gpu(p, max_partitions=1 if mode == "direct" else 0, task_budget=16, kernel=kernel)
    util.assert_parity(got, ref, case.kv, f"{case.name} {kernel}")


TC_CASES = [c for c in SMALL if c.head_dim == 128] + [
    synth.config3(qlen=1, batch=4, head_dim=128, context_lens=(200, 1500), seed=2401),
    synth.config3(qlen=2, batch=3, head_dim=128, context_lens=(200, 900), seed=2402),
    synth.config2("b", batch=5, head_dim=128, seed=2403),
]


@pytest.mark.parametrize("case", TC_CASES, ids=lambda c: f"{c.name}-q{c.qlen}-s{c.seed}")
@pytest.mark.parametrize("mode", ["split", "direct"])
def test_tensor_core_kernel_matches_oracle(case, mode):
    # the tcgen05 kernel (kernel="tc") on every head_dim-128 shape: bf16, fp8 per tensor
    # and per token, MXFP4; 8 to 32 query rows per KV head; pages of 16 to 128
    p = synth.make(case)
    util.assert_parity(run_gpu(p, max_partitions=1 if mode == "direct" else 0, task_budget=64,
                               kernel="tc"),
                       util.oracle_decode(p), case.kv, case.name + " tcgen05")


HUGE_K = [
    synth.replace(synth.config4(batch=6, seed=2601), k_e8m0_range=(236, 249)),
    synth.replace(synth.config5(synth.KV_MXFP4, batch=3, context_lens=(3000, 9000), seed=2602),
                  k_e8m0_range=(236, 249)),
]


@pytest.mark.parametrize("case", HUGE_K, ids=lambda c: f"{c.name}-b{c.batch}")
@pytest.mark.parametrize("mode", ["split", "direct"])
@pytest.mark.parametrize("kernel", KERNELS, ids=lambda k: k or "default")
def test_mxfp4_huge_k_exponents(case, mode, kernel):
    # K block exponents up to byte 249 (P2: logits went to inf there): scores near 2^122
    # must stay finite, and the one-hot softmax must pick the oracle's token
    p = synth.make(case)
    got = run_gpu(p, max_partitions=1 if mode == "direct" else 0, task_budget=16, kernel=kernel)
    assert np.all(np.isfinite(got))
    util.assert_parity(got, util.oracle_decode(p), case.kv, f"{case.name} huge K {kernel}")


CAUSAL = [
    synth.Case("causal_fp8_token", synth.KV_FP8, synth.SCALE_TOKEN, synth.Q_BF16, batch=5,
               qlen=4, num_kv_heads=2, num_q_heads=16, head_dim=128, page_size=16,
               context_lens=[1, 3, 4, 257, 2000], seed=2701, kv_std=20.0, causal=True),
    synth.replace(synth.config3(qlen=4, batch=4, context_lens=(200, 900), seed=2702), causal=True),
    synth.replace(synth.config2("b", batch=5, seed=2703), causal=True),
    synth.Case("causal_bf16", synth.KV_BF16, synth.SCALE_NONE, synth.Q_BF16, batch=4, qlen=2,
               num_kv_heads=1, num_q_heads=8, head_dim=128, page_size=16,
               context_lens=[1, 2, 33, 300], seed=2704, causal=True),
]


@pytest.mark.parametrize("case", CAUSAL, ids=lambda c: f"{c.name}-q{c.qlen}")
@pytest.mark.parametrize("mode", ["split", "direct", "fused"])
def test_causal_matches_oracle(case, mode):
    # query position i sees tokens < L - qlen + 1 + i; contexts shorter than qlen leave the
    # first positions with nothing to see (zero rows)
    p = synth.make(case)
    got = run_gpu(p, max_partitions=1 if mode == "direct" else 0, task_budget=24,
                  merge_in_decode=mode == "fused")
    util.assert_parity(got, util.oracle_decode(p), case.kv, case.name)


def test_causal_runs_on_the_mma_kernel_when_tcgen05_is_requested():
    case = CAUSAL[0]
    p = synth.make(case)
    util.assert_parity(run_gpu(p, task_budget=24, kernel="tc"), util.oracle_decode(p), case.kv,
                       case.name)


WINDOW = [
    synth.Case("window_fp8_token", synth.KV_FP8, synth.SCALE_TOKEN, synth.Q_BF16, batch=5,
               qlen=1, num_kv_heads=2, num_q_heads=16, head_dim=128, page_size=16,
               context_lens=[1, 17, 300, 2000, 5000], seed=2901, kv_std=20.0, window=1000),
    synth.Case("window_fp8_token_q4", synth.KV_FP8, synth.SCALE_TOKEN, synth.Q_BF16, batch=4,
               qlen=4, num_kv_heads=2, num_q_heads=16, head_dim=128, page_size=16,
               context_lens=[2, 40, 257, 900], seed=2902, kv_std=20.0, window=37),
    synth.replace(synth.config2("b", batch=5, seed=2903), causal=True, window=500),
    synth.replace(synth.config1(context_lens=[17, 257, 3000], batch=3, seed=2904), window=100),
    synth.Case("window_bf16_d256_causal", synth.KV_BF16, synth.SCALE_NONE, synth.Q_BF16,
               batch=3, qlen=2, num_kv_heads=1, num_q_heads=8, head_dim=256, page_size=64,
               context_lens=[3, 500, 1500], seed=2905, causal=True, window=64),
    synth.replace(synth.config3(qlen=4, batch=3, context_lens=(200, 900), seed=2906),
                  window=333),
    synth.replace(synth.config4(batch=8, seed=2907), window=600),
    synth.replace(synth.config5(synth.KV_MXFP4, batch=3, context_lens=(3000, 9000), seed=2908),
                  window=2048),
    synth.Case("window_one", synth.KV_FP8, synth.SCALE_TENSOR, synth.Q_BF16, batch=3,
               qlen=3, num_kv_heads=1, num_q_heads=8, head_dim=128, page_size=16,
               context_lens=[1, 50, 700], fill=synth.FILL_INF, seed=2909, kv_std=20.0,
               causal=True, window=1),
]


@pytest.mark.parametrize("case", WINDOW, ids=lambda c: f"{c.name}-w{c.window}")
@pytest.mark.parametrize("mode", ["split", "direct", "fused"])
def test_sliding_window_matches_oracle(case, mode):
    # query position i sees tokens > L - qlen + i - W; rows before every window hold the
    # unowned fill (NaN, +-448, random bytes with e8m0 255) and must have no effect
    p = synth.make(case)
    got = run_gpu(p, max_partitions=1 if mode == "direct" else 0, task_budget=24,
                  merge_in_decode=mode == "fused")
    util.assert_parity(got, util.oracle_decode(p), case.kv, case.name + " window")


@pytest.mark.parametrize("case", [WINDOW[0], WINDOW[2], WINDOW[6]], ids=lambda c: c.name)
def test_window_wider_than_every_context_is_bitwise_no_window(case):
    # the same plan, the same slices on the same paths: the same bits
    p = synth.make(synth.replace(case, window=0))
    plain = run_gpu(p, task_budget=24)
    pw = dict(p)
    pw["case"] = synth.replace(case, window=int(p["context_lens"].max()) + case.qlen)
    assert np.array_equal(run_gpu(pw, task_budget=24), plain)


def test_window_on_the_long_context_workload_sampled():
    case = synth.replace(synth.config5(synth.KV_FP8, batch=4, seed=2910), window=32768)
    p = synth.make(case)
    got = run_gpu(p)
    seqs = [0, 3]
    util.assert_parity(got[seqs], util.oracle_decode(p, seqs=seqs), case.kv, case.name)
    assert np.isfinite(got).all()


SHAPES = [
    # head_dim 64 (64-byte e4m3 rows, 128-byte bf16 rows) and GQA 4 (4 query rows), the
    # head sizes and GQA ratios of the first page's probe
    synth.Case("d64_bf16_g4", synth.KV_BF16, synth.SCALE_NONE, synth.Q_BF16, batch=5, qlen=1,
               num_kv_heads=2, num_q_heads=8, head_dim=64, page_size=16,
               context_lens=[1, 17, 255, 257, 3000], seed=3001),
    synth.Case("d64_bf16_g8_q4_causal", synth.KV_BF16, synth.SCALE_NONE, synth.Q_BF16, batch=4,
               qlen=4, num_kv_heads=1, num_q_heads=8, head_dim=64, page_size=64,
               context_lens=[2, 70, 513, 2000], seed=3002, causal=True),
    synth.Case("d64_fp8_tensor_g4", synth.KV_FP8, synth.SCALE_TENSOR, synth.Q_BF16, batch=4,
               qlen=1, num_kv_heads=4, num_q_heads=16, head_dim=64, page_size=128,
               context_lens=[1, 129, 1000, 4097], fill=synth.FILL_INF, seed=3003, kv_std=20.0),
    synth.Case("d64_fp8_token_g16_q2", synth.KV_FP8, synth.SCALE_TOKEN, synth.Q_BF16, batch=4,
               qlen=2, num_kv_heads=2, num_q_heads=32, head_dim=64, page_size=32,
               context_lens=[3, 300, 1500, 2500], seed=3004, kv_std=20.0, window=700),
    synth.Case("d64_fp8_token_e4m3q", synth.KV_FP8, synth.SCALE_TOKEN, synth.Q_E4M3, batch=3,
               qlen=1, num_kv_heads=1, num_q_heads=16, head_dim=64, page_size=16,
               context_lens=[40, 900, 5000], seed=3005, kv_std=20.0),
    synth.Case("d64_bf16_e4m3q_g4_q2", synth.KV_BF16, synth.SCALE_NONE, synth.Q_E4M3, batch=3,
               qlen=2, num_kv_heads=2, num_q_heads=8, head_dim=64, page_size=16,
               context_lens=[5, 600, 2100], seed=3006),
    synth.Case("d128_fp8_token_g4", synth.KV_FP8, synth.SCALE_TOKEN, synth.Q_BF16, batch=4,
               qlen=1, num_kv_heads=2, num_q_heads=8, head_dim=128, page_size=16,
               context_lens=[1, 200, 1000, 3000], seed=3007, kv_std=20.0),
    synth.Case("d256_bf16_g4", synth.KV_BF16, synth.SCALE_NONE, synth.Q_BF16, batch=3, qlen=1,
               num_kv_heads=2, num_q_heads=8, head_dim=256, page_size=64,
               context_lens=[7, 800, 2500], seed=3008),
]


@pytest.mark.parametrize("case", SHAPES, ids=lambda c: c.name)
@pytest.mark.parametrize("mode", ["split", "direct", "fused"])
def test_head_sizes_and_gqa_ratios(case, mode):
    p = synth.make(case)
    got = run_gpu(p, max_partitions=1 if mode == "direct" else 0, task_budget=24,
                  merge_in_decode=mode == "fused")
    util.assert_parity(got, util.oracle_decode(p), case.kv, case.name)


@pytest.mark.parametrize("kv", [synth.KV_BF16, synth.KV_FP8])
def test_head_dim_64_fused_merge_of_128_partitions(kv):
    # one long unit cut into 128 partitions: the fused merge's [rows, partitions] weights
    # are wider than a head_dim-64 output row
    scale = synth.SCALE_NONE if kv == synth.KV_BF16 else synth.SCALE_TOKEN
    case = synth.Case("d64_parts128", kv, scale, synth.Q_BF16, batch=1, qlen=2,
                      num_kv_heads=1, num_q_heads=16, head_dim=64, page_size=128,
                      context_lens=[60000], seed=3009, kv_std=20.0 if kv == synth.KV_FP8 else 1.0)
    p = synth.make(case)
    got = run_gpu(p, max_partitions=128, task_budget=152, merge_in_decode=True)
    util.assert_parity(got, util.oracle_decode(p), case.kv, case.name)
    split = run_gpu(p, max_partitions=128, task_budget=152)
    util.assert_parity(split, util.oracle_decode(p), case.kv, case.name + " split")


TRANS_V = [
    # fp8 per-tensor with the value cache stored [NB, Hkv, D, S] (the first page's
    # trans_v layout): K rows read in the order that matches the transposed V fragments
    synth.Case("tv_d128_g8", synth.KV_FP8, synth.SCALE_TENSOR, synth.Q_BF16, batch=6, qlen=1,
               num_kv_heads=2, num_q_heads=16, head_dim=128, page_size=16,
               context_lens=[1, 17, 255, 257, 1000, 5000], fill=synth.FILL_INF, seed=3101,
               kv_std=20.0, trans_v=True),
    synth.replace(synth.config2("b", batch=6, seed=3102), trans_v=True),
    synth.Case("tv_d64_g4_q2_window", synth.KV_FP8, synth.SCALE_TENSOR, synth.Q_BF16, batch=4,
               qlen=2, num_kv_heads=2, num_q_heads=8, head_dim=64, page_size=128,
               context_lens=[2, 130, 900, 3000], fill=synth.FILL_INF, seed=3103, kv_std=20.0,
               causal=True, window=300, trans_v=True),
    synth.Case("tv_d128_g16_q2", synth.KV_FP8, synth.SCALE_TENSOR, synth.Q_BF16, batch=4,
               qlen=2, num_kv_heads=1, num_q_heads=16, head_dim=128, page_size=32,
               context_lens=[5, 33, 700, 2600], fill=synth.FILL_INF, seed=3104, kv_std=20.0,
               trans_v=True),
    synth.Case("tv_d256_g8_q2", synth.KV_FP8, synth.SCALE_TENSOR, synth.Q_E4M3, batch=3,
               qlen=2, num_kv_heads=2, num_q_heads=16, head_dim=256, page_size=16,
               context_lens=[9, 400, 1800], fill=synth.FILL_INF, seed=3105, kv_std=20.0,
               trans_v=True),
    synth.Case("tv_d64_g16_q2", synth.KV_FP8, synth.SCALE_TENSOR, synth.Q_BF16, batch=3,
               qlen=2, num_kv_heads=1, num_q_heads=16, head_dim=64, page_size=64,
               context_lens=[64, 65, 2000], fill=synth.FILL_INF, seed=3106, kv_std=20.0,
               trans_v=True),
]


@pytest.mark.parametrize("case", TRANS_V, ids=lambda c: c.name)
@pytest.mark.parametrize("mode", ["split", "direct", "fused"])
def test_transposed_value_cache_matches_oracle(case, mode):
    p = synth.make(case)
    got = run_gpu(p, max_partitions=1 if mode == "direct" else 0, task_budget=24,
                  merge_in_decode=mode == "fused")
    util.assert_parity(got, util.oracle_decode(p), case.kv, case.name + " trans_v")


def test_transposed_value_cache_agrees_with_plain():
    case = TRANS_V[0]
    p = synth.make(case)
    plain = synth.make(synth.replace(case, trans_v=False))
    a, b = run_gpu(p, task_budget=24), run_gpu(plain, task_budget=24)
    assert util.rel_l2(a, b) < 2e-3


ROWS64 = [
    # 33 to 64 query rows per KV head (four m-tiles): the first page's GQA 16 x qlen 4 and
    # GQA 8 x qlen 7 / 8 cases (64 and 56 rows)
    synth.Case("r64_bf16_d64", synth.KV_BF16, synth.SCALE_NONE, synth.Q_BF16, batch=3, qlen=4,
               num_kv_heads=2, num_q_heads=32, head_dim=64, page_size=16,
               context_lens=[4, 300, 2000], seed=3201),
    synth.Case("r56_bf16_d128_q7_causal", synth.KV_BF16, synth.SCALE_NONE, synth.Q_BF16,
               batch=3, qlen=7, num_kv_heads=1, num_q_heads=8, head_dim=128, page_size=64,
               context_lens=[3, 257, 1500], seed=3202, causal=True),
    synth.Case("r64_fp8_token_d128_window", synth.KV_FP8, synth.SCALE_TOKEN, synth.Q_BF16,
               batch=3, qlen=4, num_kv_heads=1, num_q_heads=16, head_dim=128, page_size=16,
               context_lens=[17, 800, 4000], seed=3203, kv_std=20.0, window=1000),
    synth.Case("r64_fp8_tensor_d64_trans_v", synth.KV_FP8, synth.SCALE_TENSOR, synth.Q_BF16,
               batch=3, qlen=4, num_kv_heads=2, num_q_heads=32, head_dim=64, page_size=32,
               context_lens=[1, 500, 2500], fill=synth.FILL_INF, seed=3204, kv_std=20.0,
               trans_v=True),
    synth.Case("r64_fp8_tensor_d128_q8_trans_v", synth.KV_FP8, synth.SCALE_TENSOR, synth.Q_E4M3,
               batch=3, qlen=8, num_kv_heads=1, num_q_heads=8, head_dim=128, page_size=128,
               context_lens=[9, 700, 3000], fill=synth.FILL_INF, seed=3205, kv_std=20.0,
               trans_v=True, causal=True),
    # head_dim 256: four warps split the head dim of a token group
    synth.Case("r64_bf16_d256_causal", synth.KV_BF16, synth.SCALE_NONE, synth.Q_BF16, batch=3,
               qlen=4, num_kv_heads=1, num_q_heads=16, head_dim=256, page_size=64,
               context_lens=[1, 300, 1500], seed=3206, causal=True),
    synth.Case("r64_fp8_token_d256_q8_window", synth.KV_FP8, synth.SCALE_TOKEN, synth.Q_BF16,
               batch=3, qlen=8, num_kv_heads=2, num_q_heads=16, head_dim=256, page_size=16,
               context_lens=[9, 777, 3000], seed=3207, kv_std=20.0, window=900),
    synth.Case("r64_fp8_tensor_d256_trans_v", synth.KV_FP8, synth.SCALE_TENSOR, synth.Q_BF16,
               batch=3, qlen=4, num_kv_heads=1, num_q_heads=16, head_dim=256, page_size=32,
               context_lens=[2, 600, 2200], fill=synth.FILL_INF, seed=3208, kv_std=20.0,
               trans_v=True),
]


@pytest.mark.parametrize("case", ROWS64, ids=lambda c: c.name)
@pytest.mark.parametrize("mode", ["split", "direct", "fused"])
def test_up_to_64_query_rows_per_kv_head(case, mode):
    p = synth.make(case)
    got = run_gpu(p, max_partitions=1 if mode == "direct" else 0, task_budget=24,
                  merge_in_decode=mode == "fused")
    util.assert_parity(got, util.oracle_decode(p), case.kv, case.name)


SINKS = [
    synth.Case("sinks_fp8_token", synth.KV_FP8, synth.SCALE_TOKEN, synth.Q_BF16, batch=4,
               qlen=1, num_kv_heads=2, num_q_heads=16, head_dim=128, page_size=16,
               context_lens=[1, 100, 1000, 4000], seed=3301, kv_std=20.0, sink_mean=2.0),
    synth.Case("sinks_bf16_q4_causal_window", synth.KV_BF16, synth.SCALE_NONE, synth.Q_BF16,
               batch=3, qlen=4, num_kv_heads=1, num_q_heads=8, head_dim=256, page_size=64,
               context_lens=[3, 300, 2000], seed=3302, causal=True, window=200, sink_mean=1.0),
    synth.replace(synth.config4(batch=8, seed=3303), sink_mean=40.0),
    synth.replace(synth.config5(synth.KV_MXFP4, batch=3, context_lens=(3000, 9000), seed=3304),
                  sink_mean=45.0),
    synth.replace(TRANS_V[0], sink_mean=2.0, seed=3305),
]


@pytest.mark.parametrize("case", SINKS, ids=lambda c: c.name)
@pytest.mark.parametrize("mode", ["split", "direct", "fused"])
def test_attention_sinks_match_oracle(case, mode):
    p = synth.make(case)
    got = run_gpu(p, max_partitions=1 if mode == "direct" else 0, task_budget=24,
                  merge_in_decode=mode == "fused")
    util.assert_parity(got, util.oracle_decode(p), case.kv, case.name + " sinks")


def test_sink_limits():
    # a sink at -1e30 weighs nothing: the bits of the call without sinks; a dominant sink
    # takes all the weight: zero rows
    case = SINKS[0]
    p = synth.make(synth.replace(case, sink_mean=None))
    for maxp in (0, 1):  # split partitions with the reduce; one partition written directly
        plain = run_gpu(p, max_partitions=maxp, task_budget=24)
        q = dict(p)
        q["sinks"] = torch.full((case.num_q_heads,), -1e30)
        assert np.array_equal(run_gpu(q, max_partitions=maxp, task_budget=24), plain), maxp
        q["sinks"] = torch.full((case.num_q_heads,), 600.0)
        assert np.all(run_gpu(q, max_partitions=maxp, task_budget=24) == 0.0), maxp


PLAN_FREE = [synth.config1(), synth.config4(batch=8),
             synth.config4(batch=5, context_lens=[2048, 1, 129, 0, 3000], seed=2005),
             synth.config3(qlen=4, batch=3, context_lens=(200, 900), seed=2004),
             WINDOW[1], TRANS_V[0], CAUSAL[0], ROWS64[2]]


@pytest.mark.parametrize("case", PLAN_FREE, ids=lambda c: f"{c.name}-b{c.batch}")
def test_one_partition_run_equals_its_steps(case):
    # one partition per unit (the pages' plan-free mode: each unit one task, rows written
    # directly, no reduce): pa_decode_run and plan + decode + reduce give the same bits
    p = synth.make(case)
    dev = synth.to_device(p, "cuda")
    free = run_gpu(p, max_partitions=1, task_budget=7)
    out = torch.full(tuple(p["query"].shape), float("nan"), dtype=torch.bfloat16, device="cuda")
    q = dev["query"].view(torch.float8_e4m3fn) if dev["query"].dtype == torch.uint8 else dev["query"]
    args = ops.make_args(q, dev["key_cache"], dev["value_cache"], dev["block_tables"],
                         dev["context_lens"], out, key_scale=dev["key_scale"],
                         value_scale=dev["value_scale"], q_scale=dev["q_scale"],
                         softmax_scale=case.scale_qk(), max_partitions=1, task_budget=7,
                         causal=case.causal, q_quant=case.q_quant, sliding_window=case.window,
                         trans_v=case.trans_v)
    ws = ops.alloc_workspace(args)
    ops.pa_decode_plan(args, ws)
    ops.pa_decode(args, ws)
    ops.pa_decode_reduce(args, ws)
    torch.cuda.synchronize()
    assert ops.pa_decode_read_status(ws) == 0
    assert np.array_equal(free, out.float().cpu().numpy(), equal_nan=False)
    util.assert_parity(free, util.oracle_decode(p), case.kv, case.name + " one partition")


@pytest.mark.parametrize("case", [SINKS[0], synth.config4(batch=5, seed=3401), WINDOW[1]],
                         ids=lambda c: c.name)
def test_one_call_tensor_wrapper(case):
    # ops.paged_attention_decode: tensors in, output out, on the current stream
    p = synth.make(case)
    dev = synth.to_device(p, "cuda")
    out = ops.paged_attention_decode(
        dev["query"], dev["key_cache"], dev["value_cache"], dev["block_tables"],
        dev["context_lens"], key_scale=dev["key_scale"], value_scale=dev["value_scale"],
        q_scale=dev["q_scale"], softmax_scale=case.scale_qk(), causal=case.causal,
        sliding_window=case.window, trans_v=case.trans_v, sinks=dev.get("sinks"),
        q_quant=case.q_quant)
    torch.cuda.synchronize()
    assert out.dtype == torch.bfloat16 and tuple(out.shape) == tuple(p["query"].shape)
    util.assert_parity(out.float().cpu().numpy(), util.oracle_decode(p), case.kv,
                       case.name + " wrapper")


QQUANT = [
    synth.replace(synth.config4(batch=6, seed=2801), q=synth.Q_BF16, q_quant=True),
    synth.replace(synth.config5(synth.KV_MXFP4, batch=3, context_lens=(3000, 9000), seed=2802),
                  q_quant=True),
]


@pytest.mark.parametrize("case", QQUANT, ids=lambda c: f"{c.name}-b{c.batch}")
@pytest.mark.parametrize("mode", ["split", "direct"])
def test_mxfp4_with_query_quantised_in_kernel(case, mode):
    # the MXFP4 page's query mode: each bf16 head row quantised to e4m3 (scale amax / 448)
    # in the kernel; the oracle quantises the same way, in the same precision
    p = synth.make(case)
    got = run_gpu(p, max_partitions=1 if mode == "direct" else 0, task_budget=16)
    util.assert_parity(got, util.oracle_decode(p), case.kv, case.name + " quantised query")


_LENS30 = [int(x) for x in np.random.default_rng(2504).integers(1, 800, 30)]
MANY_TASKS = [
    synth.config4(batch=64, seed=2501),
    synth.config3(qlen=1, batch=40, head_dim=128, context_lens=(200, 1500), seed=2502),
    synth.config3(qlen=4, batch=24, context_lens=(100, 900), seed=2503),
    synth.config1(batch=30, context_lens=_LENS30, seed=2504),
]


@pytest.mark.parametrize("case", MANY_TASKS, ids=lambda c: f"{c.name}-b{c.batch}")
@pytest.mark.parametrize("mode", ["split", "direct"])
def test_many_tasks_per_chunk(case, mode):
    # three CTAs, each walking 16 to 30 tasks: past the tasks staged in shared memory at
    # CTA start, so both the staged and the global-memory paths of a task switch run,
    # with bf16 and e4m3 queries staged for the next task
    p = synth.make(case)
    got = run_gpu(p, max_partitions=1 if mode == "direct" else 0, task_budget=3)
    util.assert_parity(got, util.oracle_decode(p), case.kv, case.name + " many tasks")


@pytest.mark.parametrize("lens", [[0, 0], [1, 2], [255, 256, 257], [511, 512, 513, 767]])
def test_ragged_edges(lens):
    case = synth.Case("edges", synth.KV_FP8, synth.SCALE_TOKEN, synth.Q_BF16, batch=len(lens),
                      qlen=1, num_kv_heads=2, num_q_heads=16, head_dim=128, page_size=16,
                      context_lens=lens, seed=2100 + len(lens), kv_std=20.0)
    p = synth.make(case)
    ref = util.oracle_decode(p)
    got = run_gpu(p, task_budget=8)
    if sum(lens) == 0:
        assert np.all(got == 0.0)
    else:
        util.assert_parity(got, ref, case.kv, "edges")


def _bf16_ulp(x: np.ndarray) -> np.ndarray:
    a = np.maximum(np.abs(x), np.finfo(np.float32).tiny)
    return np.exp2(np.floor(np.log2(a)) - 7)


@pytest.mark.parametrize("kv,scale", [(synth.KV_BF16, synth.SCALE_NONE),
                                      (synth.KV_FP8, synth.SCALE_TENSOR),
                                      (synth.KV_FP8, synth.SCALE_TOKEN),
                                      (synth.KV_MXFP4, synth.SCALE_E8M0)],
                         ids=["bf16", "fp8_tensor", "fp8_token", "mxfp4"])
def test_context_one_gives_that_v_row(kv, scale):
    # one token: its softmax weight is exactly 1, so the output is that token's V row --
    # bitwise for bf16 KV, within one bf16 ulp of the dequantised row otherwise
    D = 128
    case = synth.Case("ctx1", kv, scale, synth.Q_BF16, batch=3, qlen=1, num_kv_heads=2,
                      num_q_heads=16, head_dim=D, page_size=16 if kv != synth.KV_MXFP4 else 128,
                      context_lens=[1, 1, 1], seed=3501, kv_std=20.0)
    p = synth.make(case)
    got = run_gpu(p, task_budget=8)
    ref = util.oracle_decode(p)  # the dequantised V row of token 0 (closed form, pinned on CPU)
    if kv == synth.KV_BF16:
        vc = p["value_cache"]
        for s in range(3):
            blk = int(p["block_tables"][s, 0])
            for h in range(16):
                assert np.array_equal(got[s, 0, h], vc[blk, h // 8, 0].float().numpy()), (s, h)
    else:
        assert np.all(np.abs(got - ref) <= _bf16_ulp(ref)), float(np.abs(got - ref).max())


@pytest.mark.parametrize("kv", [synth.KV_MXFP4, synth.KV_FP8], ids=["5a_mxfp4", "5b_fp8_token"])
def test_long_context_full_size_sampled(kv):
    # the launch configuration bench.py times: default split, separate reduce
    case = synth.config5(kv)
    p = synth.make(case)
    got = run_gpu(p)
    seqs = [0, 7, 15]
    ref = util.oracle_decode(p, seqs=seqs)
    util.assert_parity(got[seqs], ref, case.kv, case.name)
    assert np.isfinite(got).all()


@pytest.mark.parametrize("case", [synth.config3(qlen=1), synth.config3(qlen=4), synth.config2("b")],
                         ids=lambda c: c.name)
@pytest.mark.parametrize("kernel", [None, "mma"], ids=lambda k: k or "default")
def test_stated_sizes_sampled(case, kernel):
    # the workloads at their stated sizes (batch 16, 2 KV heads, head_dim 256) in the launch
    # configuration the per-workload timings use; the oracle computes the shortest and the
    # longest sequence and two more
    p = synth.make(case)
    got = run_gpu(p, kernel=kernel)
    lens = p["context_lens"].tolist()
    order = sorted(range(case.batch), key=lambda i: lens[i])
    seqs = sorted({order[0], order[-1], order[case.batch // 2], 5})
    util.assert_parity(got[seqs], util.oracle_decode(p, seqs=seqs), case.kv, case.name)
    assert np.isfinite(got).all()


@pytest.mark.parametrize("kv", [synth.KV_MXFP4, synth.KV_FP8], ids=["5a_mxfp4", "5b_fp8_token"])
def test_long_context_fused_merge_sampled(kv):
    case = synth.config5(kv, batch=6, seed=2200)
    p = synth.make(case)
    got = run_gpu(p, merge_in_decode=True)
    seqs = [0, 5]
    util.assert_parity(got[seqs], util.oracle_decode(p, seqs=seqs), case.kv, case.name)


def test_mxfp4_batch_4096_sampled():
    case = synth.config4(batch=4096)
    p = synth.make(case)
    got = run_gpu(p)
    seqs = [0, 1, 2047, 4095]
    ref = util.oracle_decode(p, seqs=seqs)
    util.assert_parity(got[seqs], ref, case.kv, case.name)
    assert np.isfinite(got).all()


SINGLE_LAUNCH = [
    synth.config1(),                                    # 2 units, 2 CTAs a unit
    synth.config4(batch=8),                             # 8 units, 8-CTA clusters (MXFP4)
    synth.config2("a"),                                 # 32 units, 4 CTAs a unit, qlen 4
    synth.config4(batch=5, context_lens=[2048, 1, 129, 0, 3000], seed=3501),  # empty and 1-token units
    synth.replace(synth.config1(context_lens=[700, 300], seed=3502), window=200),
    synth.replace(synth.config3(qlen=1, batch=3, context_lens=(100, 700), seed=3503), sink_mean=1.5),
]


@pytest.mark.parametrize("case", SINGLE_LAUNCH, ids=lambda c: f"{c.name}-s{c.seed}")
def test_single_launch_and_planned_paths_match_oracle(case):
    # small problems: pa_decode_run is one launch (a cluster of CTAs per unit merging its
    # partials, no plan, no reduce kernel); the split API runs the planned path on the same
    # input; both must match the oracle, and the single launch must leave no plan behind
    # that a later pa_decode / pa_decode_reduce would act on
    p = synth.make(case)
    ref = util.oracle_decode(p)
    dev = synth.to_device(p, "cuda")
    shape = tuple(p["query"].shape)
    q = dev["query"].view(torch.float8_e4m3fn) if dev["query"].dtype == torch.uint8 else dev["query"]

    def args_for(out):
        return ops.make_args(q, dev["key_cache"], dev["value_cache"], dev["block_tables"],
                             dev["context_lens"], out, key_scale=dev["key_scale"],
                             value_scale=dev["value_scale"], q_scale=dev["q_scale"],
                             softmax_scale=case.scale_qk(), q_quant=case.q_quant,
                             sliding_window=case.window, sinks=dev.get("sinks"))

    one = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    a1 = args_for(one)
    ws = ops.alloc_workspace(a1)
    ops.pa_decode_run(a1, ws)
    torch.cuda.synchronize()
    assert ops.pa_decode_read_status(ws) == 0
    util.assert_parity(one.float().cpu().numpy(), ref, case.kv, case.name + " single launch")
    # nothing left to act on: a decode and a reduce without a new plan write no row
    stale = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    a_stale = args_for(stale)
    ops.pa_decode(a_stale, ws)
    ops.pa_decode_reduce(a_stale, ws)
    torch.cuda.synchronize()
    assert torch.isnan(stale.float()).all()

    split = torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    a2 = args_for(split)
    ws2 = ops.alloc_workspace(a2)
    ops.pa_decode_plan(a2, ws2)
    ops.pa_decode(a2, ws2)
    ops.pa_decode_reduce(a2, ws2)
    torch.cuda.synchronize()
    assert ops.pa_decode_read_status(ws2) == 0
    util.assert_parity(split.float().cpu().numpy(), ref, case.kv, case.name + " planned")
