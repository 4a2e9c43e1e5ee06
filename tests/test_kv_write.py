"""MXFP4 KV-cache write: the oracle's conversion against independent formulations (CPU),
and the CUDA write kernel against the oracle, byte for byte (GPU).

The pages name the format the decode reads (e2m1 values, one e8m0 scale per 32 along
head_dim, element 2j in the low nibble of byte j) and say its pages come from a KV write
kernel ("[FlyDSL] pa_decode: MXFP4 K/V ...", Dependencies); the conversion is the OCP MX
one: scale 2^(floor(log2 amax) - 2), values rounded to the nearest e2m1 value, ties to the
even code, saturating at 6.
"""
import math

import numpy as np
import pytest
import torch

from oracle import pa_oracle as orc

E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _brute_codes(y: np.ndarray) -> np.ndarray:
    """Nearest of all 16 e2m1 codes by exhaustive search; ties to the even code; the sign
    of the input is kept (a negative value that rounds to zero is -0)."""
    table = np.array(E2M1 + [-v for v in E2M1])
    out = np.zeros(y.shape, np.uint8)
    for idx, v in np.ndenumerate(y):
        dist = np.abs(table - v)
        best = [c for c in range(16) if dist[c] == dist.min()]
        sign = 8 if math.copysign(1.0, float(v)) < 0 else 0
        cands = [c for c in best if (c & 8) == sign] or best
        even = [c for c in cands if (c & 1) == 0]
        out[idx] = (even or cands)[0]
    return out


def _brute_quantize(x: np.ndarray):
    D = x.shape[-1]
    rows = x.reshape(-1, D).astype(np.float64)
    data = np.zeros((rows.shape[0], D // 2), np.uint8)
    scales = np.zeros((rows.shape[0], D // 32), np.uint8)
    for r in range(rows.shape[0]):
        codes = np.zeros(D, np.uint8)
        for b in range(D // 32):
            blk = rows[r, 32 * b:32 * b + 32]
            amax = float(np.max(np.abs(blk)))
            if not np.all(np.isfinite(blk)):
                scales[r, b] = 255
                continue
            if amax == 0.0:
                E = 0
            else:
                m, e = math.frexp(amax)      # amax = m * 2^e, m in [0.5, 1)
                E = min(127, max(-126, (e - 1) - 2))
            scales[r, b] = E + 127
            codes[32 * b:32 * b + 32] = _brute_codes(blk / 2.0 ** E)
        data[r] = codes[0::2] | (codes[1::2] << 4)
    return data.reshape(*x.shape[:-1], D // 2), scales.reshape(*x.shape[:-1], D // 32)


def _zero_sign(data: np.ndarray) -> np.ndarray:
    """Codes with -0 read as +0 (the same value; the format does not fix the sign of a
    zero result)."""
    lo, hi = data & 15, data >> 4
    lo = np.where(lo == 8, 0, lo)
    hi = np.where(hi == 8, 0, hi)
    return (lo | (hi << 4)).astype(np.uint8)


def _dequant(data: np.ndarray, scales: np.ndarray) -> np.ndarray:
    lo, hi = (data & 15).astype(np.int64), (data >> 4).astype(np.int64)
    codes = np.stack([lo, hi], axis=-1).reshape(*data.shape[:-1], data.shape[-1] * 2)
    table = np.array(E2M1 + [-v for v in E2M1])
    sc = np.where(scales == 255, np.nan, np.ldexp(1.0, scales.astype(np.int64) - 127))
    return table[codes] * np.repeat(sc, 32, axis=-1)


def _mixed_rows(rng, rows, D):
    """Rows whose 32-blocks span magnitudes 2^-20 .. 2^20, with exact grid midpoints
    (ties), zeros, negative zeros and all-zero blocks, rounded to bf16."""
    x = rng.standard_normal((rows, D)) * np.exp2(rng.integers(-20, 21, (rows, D // 32))).repeat(32, -1)
    for r in range(rows):
        b = rng.integers(0, D // 32)
        E = int(rng.integers(-10, 10))
        mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0])
        x[r, 32 * b:32 * b + 8] = rng.choice([-1, 1], 8) * mids * 2.0 ** E
        x[r, 32 * b + 8] = 7.9 * 2.0 ** E  # amax in [4, 8) * 2^E: the block's scale is 2^E
        x[r, 32 * b + 9] = -0.0
    x[0, :32] = 0.0
    return torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()


@pytest.mark.parametrize("D", [64, 128, 256])
def test_oracle_matches_exhaustive_search(D):
    rng = np.random.default_rng(70 + D)
    x = _mixed_rows(rng, 12, D)
    d0, s0 = orc.mxfp4_quantize(x)
    d1, s1 = _brute_quantize(x)
    assert np.array_equal(s0, s1)
    assert np.array_equal(d0, d1)


def test_ties_go_to_the_even_code():
    x = np.zeros((1, 32), np.float32)
    x[0, :9] = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, 6.0]
    d, s = orc.mxfp4_quantize(x)
    assert s[0, 0] == 127  # amax 7: floor(log2 7) - 2 = 0
    codes = np.stack([d[0] & 15, d[0] >> 4], -1).reshape(-1)[:9]
    assert [E2M1[c] for c in codes] == [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, 6.0]


def test_values_on_the_grid_round_trip_exactly():
    # blocks of e2m1 values times 2^E whose largest magnitude is 4 or 6: the scale is 2^E
    rng = np.random.default_rng(71)
    vals = np.array(E2M1 + [-v for v in E2M1])
    x = rng.choice(vals, (8, 128))
    for r in range(8):
        for b in range(4):
            x[r, 32 * b] = rng.choice([4.0, 6.0, -4.0, -6.0])
    x = x * np.exp2(rng.integers(-30, 30, (8, 4))).repeat(32, -1)
    x = x.astype(np.float32)
    d, s = orc.mxfp4_quantize(x)
    np.testing.assert_array_equal(_dequant(d, s), x.astype(np.float64))


def test_error_bound_and_saturation():
    # |q - x| <= X (half the widest gap, between 4 and 6) below 6 X; between 6 X and 8 X
    # the value saturates to 6 X
    rng = np.random.default_rng(72)
    x = _mixed_rows(rng, 16, 128)
    d, s = orc.mxfp4_quantize(x)
    q = _dequant(d, s)
    X = np.ldexp(1.0, s.astype(np.int64) - 127).repeat(32, -1)
    a = np.abs(x)
    ok = np.where(a <= 6 * X, np.abs(q - x) <= X, np.abs(q) == 6 * X)
    assert ok.all()
    assert np.all(np.abs(x) < 8 * X)  # the scale covers the block's largest value


def test_special_blocks():
    x = np.zeros((1, 128), np.float32)
    x[0, 32] = np.nan
    x[0, 64] = np.inf
    x[0, 96:128] = 1e-39  # a subnormal block: the exponent clamps at -126
    d, s = orc.mxfp4_quantize(x)
    assert list(s[0]) == [127, 255, 255, 1]
    assert np.all(d[0, :48] == 0)


def test_planted_mistakes_are_caught():
    rng = np.random.default_rng(73)
    x = _mixed_rows(rng, 6, 128)
    d, s = orc.mxfp4_quantize(x)
    # swapped nibbles
    assert not np.array_equal(((d >> 4) | (d << 4)).astype(np.uint8), _brute_quantize(x)[0])
    # scales one binade off (floor(log2 amax) - 1: the largest values would exceed 6)
    q = _dequant(d, (s.astype(np.int64) + 1).astype(np.uint8))
    assert np.abs(q - x).max() > 0


# ---- GPU: the write kernel through the C ABI ---------------------------------------

def _gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from paged_attention_decode_02_gb300 import build, ops
    build.build()
    ops.load_library()
    return ops


def _gpu_write(ops, key, value, slots, NB, S):
    T, Hkv, D = key.shape
    kc = torch.full((NB, Hkv, S, D // 2), 0xAB, dtype=torch.uint8, device="cuda")
    vc = torch.full_like(kc, 0xAB)
    ks = torch.full((NB, Hkv, S, D // 32), 0xAB, dtype=torch.uint8, device="cuda")
    vs = torch.full_like(ks, 0xAB)
    args = ops.mxfp4_write_args(key.cuda(), value.cuda(), slots.cuda(), kc, vc, ks, vs)
    ops.mxfp4_kv_write(args)
    torch.cuda.synchronize()
    return kc.cpu().numpy(), vc.cpu().numpy(), ks.cpu().numpy(), vs.cpu().numpy()


@pytest.mark.gpu
@pytest.mark.parametrize("D", [64, 128, 256])
def test_write_kernel_matches_oracle(D):
    ops = _gpu_lib()
    rng = np.random.default_rng(80 + D)
    T, Hkv, NB, S = 300, 3, 12, 32
    key = torch.from_numpy(_mixed_rows(rng, T * Hkv, D).reshape(T, Hkv, D)).to(torch.bfloat16)
    value = torch.from_numpy(_mixed_rows(rng, T * Hkv, D).reshape(T, Hkv, D)).to(torch.bfloat16)
    slots = torch.from_numpy(rng.permutation(NB * S)[:T].astype(np.int64))
    slots[5] = -1          # skipped
    slots[6] = NB * S + 3  # past the cache: skipped too
    kc, vc, ks, vs = _gpu_write(ops, key, value, slots, NB, S)
    for src, cache, sc in ((key, kc, ks), (value, vc, vs)):
        d_ref, s_ref = orc.mxfp4_quantize(src.float().numpy())
        written = np.zeros((NB, S), bool)
        for t in range(T):
            sl = int(slots[t])
            if sl < 0 or sl >= NB * S:
                continue
            b, o = divmod(sl, S)
            written[b, o] = True
            assert np.array_equal(sc[b, :, o], s_ref[t]), t
            assert np.array_equal(_zero_sign(cache[b, :, o]), _zero_sign(d_ref[t])), t
        # slots no token maps to keep their bytes ([NB, S, Hkv, ...] view for the mask)
        assert np.all(np.moveaxis(cache, 2, 1)[~written] == 0xAB)
        assert np.all(np.moveaxis(sc, 2, 1)[~written] == 0xAB)


@pytest.mark.gpu
def test_write_kernel_special_blocks():
    ops = _gpu_lib()
    x = np.zeros((4, 1, 128), np.float32)
    x[0, 0, 32] = np.nan
    x[0, 0, 64] = -np.inf
    x[1, 0, :32] = 1e-39          # subnormal bf16 values
    x[2, 0, :] = 3.0e38           # near the bf16 maximum
    x[3, 0, ::2] = -1e-6          # tiny negatives next to zeros
    key = torch.from_numpy(x).to(torch.bfloat16)
    slots = torch.arange(4, dtype=torch.int64)
    kc, _, ks, _ = _gpu_write(ops, key, key.clone(), slots, 1, 16)
    d_ref, s_ref = orc.mxfp4_quantize(key.float().numpy())
    assert np.array_equal(ks[0, 0, :4], s_ref[:, 0])
    assert np.array_equal(_zero_sign(kc[0, 0, :4]), _zero_sign(d_ref[:, 0]))


@pytest.mark.gpu
def test_written_cache_decodes_like_the_oracle():
    # bf16 K/V -> the GPU write -> the GPU decode, against the oracle decode of the same
    # rows quantised by the oracle (no oracle input comes from the CUDA path)
    ops = _gpu_lib()
    from paged_attention_decode_02_gb300 import synth
    from tests import util
    rng = np.random.default_rng(90)
    B, Hkv, G, D, S = 3, 2, 8, 128, 128
    lens = [300, 1000, 2049]
    pages = [(L + S - 1) // S for L in lens]
    NB = 1 + sum(pages)
    perm = rng.permutation(np.arange(1, NB))
    bt = np.zeros((B, max(pages) + 2), np.int32)
    pos = 0
    slots = []
    for s, (L, n) in enumerate(zip(lens, pages)):
        bt[s, :n] = perm[pos:pos + n]
        pos += n
        slots += [int(bt[s, t // S]) * S + t % S for t in range(L)]
    T = len(slots)
    kx = torch.from_numpy(rng.standard_normal((T, Hkv, D)) * 3).to(torch.bfloat16)
    vx = torch.from_numpy(rng.standard_normal((T, Hkv, D)) * 3).to(torch.bfloat16)
    kc, vc, ks, vs = _gpu_write(ops, kx, vx, torch.tensor(slots, dtype=torch.int64), NB, S)
    # the oracle's cache: the same rows, quantised by the oracle, unwritten rows zero
    okc, ovc = np.zeros_like(kc), np.zeros_like(vc)
    oks, ovs = np.full_like(ks, 127), np.full_like(vs, 127)
    for src, c, sc in ((kx, okc, oks), (vx, ovc, ovs)):
        d, e = orc.mxfp4_quantize(src.float().numpy())
        for t, sl in enumerate(slots):
            c[sl // S, :, sl % S] = d[t]
            sc[sl // S, :, sl % S] = e[t]
    q = torch.randn((B, 1, Hkv * G, D), generator=torch.Generator().manual_seed(91)).to(torch.bfloat16)
    case = synth.Case("written", synth.KV_MXFP4, synth.SCALE_E8M0, synth.Q_BF16, batch=B, qlen=1,
                      num_kv_heads=Hkv, num_q_heads=Hkv * G, head_dim=D, page_size=S,
                      context_lens=lens)
    ctx = torch.tensor(lens, dtype=torch.int32)
    ref = util.oracle_decode({"case": case, "query": q, "q_scale": None,
                              "key_cache": torch.from_numpy(okc), "value_cache": torch.from_numpy(ovc),
                              "key_scale": torch.from_numpy(oks), "value_scale": torch.from_numpy(ovs),
                              "block_tables": torch.from_numpy(bt), "context_lens": ctx,
                              "num_blocks": NB})
    dev = {"case": case, "query": q.cuda(), "q_scale": None,
           "key_cache": torch.from_numpy(kc).cuda(), "value_cache": torch.from_numpy(vc).cuda(),
           "key_scale": torch.from_numpy(ks).cuda(), "value_scale": torch.from_numpy(vs).cuda(),
           "block_tables": torch.from_numpy(bt).cuda(), "context_lens": ctx.cuda(), "num_blocks": NB}
    out = torch.full(tuple(q.shape), float("nan"), dtype=torch.bfloat16, device="cuda")
    out, _, ws = ops.decode(dev, out)
    torch.cuda.synchronize()
    util.assert_parity(out.float().cpu().numpy(), ref, case.kv, "written cache")
