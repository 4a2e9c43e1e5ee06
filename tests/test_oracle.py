"""Pins of the fp64 oracle against things other than itself (CPU only).

Each check is chosen so that a plausible slip in the oracle -- a wrong exponent
bias, a dropped scale, a swapped nibble, a transposed head mapping, a read of an
unowned row -- fails at least one of them:

* format decoders against library casts (torch float8_e4m3fn / float8_e8m0fnu /
  bfloat16) and, for e2m1, against the value table of the OCP MX format;
* closed forms: context 1 returns that V row; identical K rows return the mean
  of V; context 0 returns zero;
* a dense brute force on tiny inputs: K/V materialised by an independent
  gather and dequantisation, ``torch.softmax`` in float64;
* the partition merge identity over a split context;
* the unowned-row invariant: NaN/Inf fills leave the output bit-identical.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import pa_oracle as orc
from paged_attention_decode_02_gb300 import synth
from tests import util

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")

# OCP MX e2m1 code points (magnitudes for codes 0..7; bit 3 is the sign).
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


# ---- decoders ----------------------------------------------------------------

def test_e4m3_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([orc.decode_e4m3(b) for b in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.isnan(got[0x7F]) and np.isnan(got[0xFF])
    assert np.isfinite(got[ok]).all()  # no Inf code in e4m3fn


def test_e2m1_all_codes_match_format_table():
    for n in range(16):
        mag = E2M1_TABLE[n & 7]
        want = -mag if n & 8 else mag
        got = orc.decode_e2m1(n)
        assert got == want and math.copysign(1.0, got) == math.copysign(1.0, want), n


def test_e8m0_all_codes_match_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = np.array([orc.decode_e8m0(b) for b in range(256)])
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(got[:255], ref[:255])
    assert all(got[b] == math.ldexp(1.0, b - 127) for b in range(255))


def test_bf16_matches_torch():
    g = torch.Generator().manual_seed(3)
    bits = torch.randint(-32768, 32768, (4096,), generator=g, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([orc.decode_bf16(int(b) & 0xFFFF) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(got[~nan], ref[~nan])


def test_pages_facts_golden():
    """Values the pages state outright (tests/golden/pages_facts.json, each cited)."""
    with open(os.path.join(GOLDEN, "pages_facts.json")) as f:
        facts = json.load(f)
    # e4m3 has no Inf: its "inf" fill is the finite +-448.
    fill = facts["e4m3_inf_fill"]
    assert orc.decode_e4m3(fill["pos_byte"]) == fill["value"]
    assert orc.decode_e4m3(fill["neg_byte"]) == -fill["value"]
    # e8m0 byte 255 is not a number.
    assert math.isnan(orc.decode_e8m0(facts["e8m0_nan_byte"]["byte"]))
    # The plan emits ceil(context_len / 256) tiles per sequence.
    tl = facts["tiles_per_sequence"]
    for L, n in zip(tl["context_lens"], tl["tiles"]):
        assert (L + tl["tile"] - 1) // tl["tile"] == n
    # MXFP4 page layout.
    mx = facts["mxfp4_layout"]
    case = synth.config4(batch=2)
    p = synth.make(case)
    assert list(p["key_cache"].shape[1:]) == mx["data_shape_after_pages"]
    assert list(p["key_scale"].shape[1:]) == mx["scale_shape_after_pages"]
    assert case.head_dim // mx["values_per_scale"] == mx["scale_shape_after_pages"][-1]


# ---- an independent dense brute force ---------------------------------------

def _dequant_dense(p: dict, which: str) -> torch.Tensor:
    """Dequantised cache [NB, Hkv, S, D] in float64, via library casts and tables."""
    case = p["case"]
    c = p["key_cache" if which == "k" else "value_cache"].cpu()
    if which == "v" and case.trans_v:  # stored [NB, Hkv, D, S]: back to token rows
        c = c.transpose(-1, -2)
    sc = p["key_scale" if which == "k" else "value_scale"]
    sc = None if sc is None else sc.cpu()
    if case.kv == synth.KV_BF16:
        return c.view(torch.bfloat16).to(torch.float64)
    if case.kv == synth.KV_FP8:
        x = c.view(torch.float8_e4m3fn).to(torch.float64)
        if case.scale == synth.SCALE_TENSOR:
            return x * float(sc[0])
        return x * sc.to(torch.float64)[..., None]
    lo = (c & 15).long()
    hi = (c >> 4).long()
    nib = torch.stack([lo, hi], dim=-1).reshape(*c.shape[:-1], c.shape[-1] * 2)
    table = torch.tensor(E2M1_TABLE + [-v for v in E2M1_TABLE], dtype=torch.float64)
    vals = table[nib]
    scale = sc.view(torch.float8_e8m0fnu).to(torch.float64)
    return vals * scale.repeat_interleave(32, dim=-1)


def _query_dense(p: dict) -> torch.Tensor:
    case = p["case"]
    q = p["query"].cpu()
    if case.q == synth.Q_BF16:
        return q.to(torch.float64)
    return q.view(torch.float8_e4m3fn).to(torch.float64) * p["q_scale"].cpu().to(torch.float64)[..., None]


def brute_force(p: dict, head_map=None, window=None) -> np.ndarray:
    case = p["case"]
    W = case.window if window is None else window
    K = _dequant_dense(p, "k")
    V = _dequant_dense(p, "v")
    Q = _query_dense(p)
    B, qlen, Hq, D = Q.shape
    G = case.gqa
    S = case.page_size
    sinks = p.get("sinks")
    out = torch.zeros((B, qlen, Hq, D), dtype=torch.float64)
    for s in range(B):
        L = int(p["context_lens"][s])
        if L == 0:
            continue
        t = torch.arange(L)
        blk = p["block_tables"][s].long()[t // S]
        for h in range(Hq):
            hkv = h // G if head_map is None else head_map(h)
            k = K[blk, hkv, t % S]          # [L, D]
            v = V[blk, hkv, t % S]
            for i in range(qlen):
                x = (k @ Q[s, i, h]) * case.scale_qk()
                seen = torch.ones(L, dtype=torch.bool)
                if case.causal:  # position i sees the tokens before L - qlen + 1 + i
                    seen &= t < L - qlen + 1 + i
                if W > 0:  # and, in a window, the W tokens that end at its own place
                    seen &= t > (L - qlen + i) - W
                if not bool(seen.any()):
                    continue
                # unseen rows may hold NaN: select, never multiply
                x = torch.where(seen, x, torch.tensor(-math.inf, dtype=x.dtype))
                if sinks is not None:  # the sink: one more softmax column, with a zero value
                    xs = torch.cat([x, sinks[h].to(torch.float64).reshape(1)])
                    w = torch.softmax(xs, dim=0)[:-1]
                else:
                    w = torch.softmax(x, dim=0)
                out[s, i, h] = torch.where(seen[:, None], v, torch.zeros_like(v)).mul(w[:, None]).sum(0)
    return out.numpy()


def _tiny_cases():
    return [
        synth.config1(context_lens=[17, 40], seed=11),
        synth.Case("t_fp8_tensor", synth.KV_FP8, synth.SCALE_TENSOR, synth.Q_BF16, batch=3,
                   qlen=2, num_kv_heads=2, num_q_heads=4, head_dim=64, page_size=16,
                   context_lens=[1, 33, 50], fill=synth.FILL_INF, seed=12, kv_std=20.0),
        synth.Case("t_fp8_token", synth.KV_FP8, synth.SCALE_TOKEN, synth.Q_BF16, batch=2,
                   qlen=1, num_kv_heads=2, num_q_heads=6, head_dim=64, page_size=16,
                   context_lens=[31, 70], fill=synth.FILL_NAN, seed=13, kv_std=20.0),
        synth.Case("t_mxfp4", synth.KV_MXFP4, synth.SCALE_E8M0, synth.Q_E4M3, batch=2,
                   qlen=1, num_kv_heads=1, num_q_heads=4, head_dim=128, page_size=16,
                   context_lens=[20, 45], fill=synth.FILL_RANDOM, seed=14),
        synth.Case("t_mxfp4_bfq", synth.KV_MXFP4, synth.SCALE_E8M0, synth.Q_BF16, batch=2,
                   qlen=2, num_kv_heads=2, num_q_heads=4, head_dim=64, page_size=32,
                   context_lens=[33, 64], fill=synth.FILL_RANDOM, seed=15),
        synth.Case("t_fp8_causal", synth.KV_FP8, synth.SCALE_TOKEN, synth.Q_BF16, batch=4,
                   qlen=4, num_kv_heads=2, num_q_heads=8, head_dim=64, page_size=16,
                   context_lens=[2, 4, 17, 40], fill=synth.FILL_NAN, seed=17, kv_std=20.0,
                   causal=True),
        synth.Case("t_bf16_window", synth.KV_BF16, synth.SCALE_NONE, synth.Q_BF16, batch=3,
                   qlen=1, num_kv_heads=1, num_q_heads=4, head_dim=64, page_size=16,
                   context_lens=[3, 40, 77], fill=synth.FILL_NAN, seed=18, window=20),
        synth.Case("t_fp8_window_q4", synth.KV_FP8, synth.SCALE_TOKEN, synth.Q_BF16, batch=4,
                   qlen=4, num_kv_heads=2, num_q_heads=8, head_dim=64, page_size=16,
                   context_lens=[2, 9, 33, 70], fill=synth.FILL_NAN, seed=19, kv_std=20.0,
                   window=7),
        synth.Case("t_fp8_window_causal", synth.KV_FP8, synth.SCALE_TENSOR, synth.Q_BF16,
                   batch=4, qlen=3, num_kv_heads=1, num_q_heads=2, head_dim=64, page_size=16,
                   context_lens=[1, 5, 18, 60], fill=synth.FILL_INF, seed=20, kv_std=20.0,
                   causal=True, window=5),
        synth.Case("t_fp8_trans_v", synth.KV_FP8, synth.SCALE_TENSOR, synth.Q_BF16, batch=3,
                   qlen=2, num_kv_heads=2, num_q_heads=4, head_dim=64, page_size=16,
                   context_lens=[1, 30, 70], fill=synth.FILL_NAN, seed=25, kv_std=20.0,
                   trans_v=True),
        synth.Case("t_bf16_trans_v_window", synth.KV_BF16, synth.SCALE_NONE, synth.Q_BF16,
                   batch=2, qlen=1, num_kv_heads=1, num_q_heads=2, head_dim=64, page_size=32,
                   context_lens=[40, 90], fill=synth.FILL_NAN, seed=26, trans_v=True, window=33),
        synth.Case("t_fp8_sinks", synth.KV_FP8, synth.SCALE_TOKEN, synth.Q_BF16, batch=3,
                   qlen=2, num_kv_heads=2, num_q_heads=8, head_dim=64, page_size=16,
                   context_lens=[1, 20, 60], fill=synth.FILL_NAN, seed=27, kv_std=20.0,
                   sink_mean=2.0),
        synth.Case("t_bf16_sinks_causal_window", synth.KV_BF16, synth.SCALE_NONE, synth.Q_BF16,
                   batch=3, qlen=3, num_kv_heads=1, num_q_heads=4, head_dim=64, page_size=16,
                   context_lens=[2, 9, 50], fill=synth.FILL_NAN, seed=28, causal=True,
                   window=6, sink_mean=0.0),
        synth.Case("t_mxfp4_window", synth.KV_MXFP4, synth.SCALE_E8M0, synth.Q_E4M3, batch=2,
                   qlen=1, num_kv_heads=1, num_q_heads=4, head_dim=128, page_size=16,
                   context_lens=[20, 45], fill=synth.FILL_RANDOM, seed=24, window=17),
    ]


@pytest.mark.parametrize("case", _tiny_cases(), ids=lambda c: c.name)
def test_bruteforce_dense(case):
    p = synth.make(case)
    got = util.oracle_decode(p)
    ref = brute_force(p)
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-12)


def test_bruteforce_detects_planted_mistakes():
    """The brute-force pin is sensitive: planted slips on the oracle's side fail it."""
    case = [c for c in _tiny_cases() if c.name == "t_mxfp4"][0]
    p = synth.make(case)
    ref = brute_force(p)
    # (1) rolled e8m0 block scales (block/scale mix-up)
    q = dict(p)
    q["key_scale"] = torch.roll(p["key_scale"], 1, dims=-1)
    assert util.rel_l2(util.oracle_decode(q), ref) > 1e-2
    # (2) swapped nibbles (element order inside a byte)
    q = dict(p)
    q["value_cache"] = ((p["value_cache"] >> 4) | (p["value_cache"] << 4)).to(torch.uint8)
    assert util.rel_l2(util.oracle_decode(q), ref) > 1e-2
    # (3) a transposed GQA head mapping
    c2 = synth.Case("t_gqa", synth.KV_FP8, synth.SCALE_TENSOR, synth.Q_BF16, batch=1, qlen=1,
                    num_kv_heads=2, num_q_heads=4, head_dim=64, page_size=16,
                    context_lens=[40], seed=16, kv_std=20.0)
    p2 = synth.make(c2)
    wrong = brute_force(p2, head_map=lambda h: h % 2)
    assert util.rel_l2(util.oracle_decode(p2), wrong) > 1e-2
    # (4) a dropped per-tensor scale
    q = dict(p2)
    q["value_scale"] = torch.tensor([1.0])
    assert util.rel_l2(util.oracle_decode(q), brute_force(p2)) > 1e-2


# ---- closed forms -------------------------------------------------------------

@pytest.mark.parametrize("kv", [synth.KV_BF16, synth.KV_FP8, synth.KV_MXFP4])
def test_context_one_returns_that_v_row(kv):
    scale = {synth.KV_BF16: synth.SCALE_NONE, synth.KV_FP8: synth.SCALE_TOKEN,
             synth.KV_MXFP4: synth.SCALE_E8M0}[kv]
    case = synth.Case("ctx1", kv, scale, synth.Q_BF16, batch=2, qlen=1, num_kv_heads=2,
                      num_q_heads=4, head_dim=64, page_size=16, context_lens=[1, 1],
                      seed=21, kv_std=20.0)
    p = synth.make(case)
    got = util.oracle_decode(p)
    V = _dequant_dense(p, "v")
    for s in range(2):
        blk = int(p["block_tables"][s, 0])
        for h in range(4):
            assert np.array_equal(got[s, 0, h], V[blk, h // 2, 0].numpy())


def test_huge_k_exponents_select_the_top_token():
    # e8m0 K bytes up to 249 (P2: the byte that sent the logits to inf): the logits lie
    # ~2^120 apart, so the softmax is one-hot and each output row is exactly the V row of
    # the token with the largest q.k, found here on the dense dequantised cache
    case = synth.Case("k249", synth.KV_MXFP4, synth.SCALE_E8M0, synth.Q_BF16, batch=2, qlen=1,
                      num_kv_heads=1, num_q_heads=4, head_dim=128, page_size=16,
                      context_lens=[37, 70], seed=31, k_e8m0_range=(236, 249))
    p = synth.make(case)
    got = util.oracle_decode(p)
    K, V, Q = _dequant_dense(p, "k"), _dequant_dense(p, "v"), _query_dense(p)
    bt = p["block_tables"].cpu()
    for s, L in enumerate([37, 70]):
        rows = [(int(bt[s, t // 16]), t % 16) for t in range(L)]
        keys = torch.stack([K[b, 0, r] for b, r in rows])
        for h in range(4):
            top = int(torch.argmax(keys @ Q.reshape(2, 4, 128)[s, h]))
            b, r = rows[top]
            assert np.all(np.isfinite(got[s, 0, h]))
            assert np.array_equal(got[s, 0, h], V[b, 0, r].numpy())


def test_causal_with_one_query_position_is_the_plain_result():
    case = synth.Case("c1", synth.KV_BF16, synth.SCALE_NONE, synth.Q_BF16, batch=3, qlen=1,
                      num_kv_heads=2, num_q_heads=4, head_dim=64, page_size=16,
                      context_lens=[5, 16, 33], seed=41)
    p = synth.make(case)
    pc = dict(p)
    pc["case"] = synth.replace(case, causal=True)
    assert np.array_equal(util.oracle_decode(pc), util.oracle_decode(p))


def test_causal_position_sees_the_context_up_to_itself():
    # query position i of a causal call equals the plain call on the same cache with the
    # context cut to L - qlen + 1 + i (zeros when that is empty)
    qlen = 4
    case = synth.Case("ci", synth.KV_FP8, synth.SCALE_TOKEN, synth.Q_BF16, batch=3, qlen=qlen,
                      num_kv_heads=2, num_q_heads=4, head_dim=64, page_size=16,
                      context_lens=[2, 19, 48], fill=synth.FILL_NAN, seed=42, kv_std=20.0,
                      causal=True)
    p = synth.make(case)
    got = util.oracle_decode(p)
    plain = synth.replace(case, causal=False)
    for i in range(qlen):
        pi = dict(p)
        pi["case"] = plain
        pi["context_lens"] = (p["context_lens"] - (qlen - 1 - i)).clamp(min=0)
        ref = util.oracle_decode(pi)
        assert np.array_equal(got[:, i], ref[:, i]), i
    assert np.all(got[0, :2] == 0.0)  # L = 2 < qlen: the first two positions see nothing


def test_window_of_one_is_the_positions_own_v_row():
    # W = 1 with causal masking: every query position sees exactly the token at its own
    # place L - qlen + i; without it, position i sees [L - qlen + i, L), and only the last
    # one a single token
    qlen = 3
    for causal in (False, True):
        case = synth.Case("w1", synth.KV_FP8, synth.SCALE_TOKEN, synth.Q_BF16, batch=2,
                          qlen=qlen, num_kv_heads=1, num_q_heads=2, head_dim=64, page_size=16,
                          context_lens=[5, 33], fill=synth.FILL_NAN, seed=61, kv_std=20.0,
                          causal=causal, window=1)
        p = synth.make(case)
        got = util.oracle_decode(p)
        V = _dequant_dense(p, "v")
        for s, L in enumerate([5, 33]):
            for i in range(qlen) if causal else [qlen - 1]:
                t = L - qlen + i
                want = V[int(p["block_tables"][s, t // 16]), 0, t % 16].numpy()
                for h in range(2):
                    assert np.array_equal(got[s, i, h], want), (causal, s, i)


def test_window_wider_than_the_context_changes_nothing():
    for causal in (False, True):
        case = synth.Case("ww", synth.KV_BF16, synth.SCALE_NONE, synth.Q_BF16, batch=3, qlen=2,
                          num_kv_heads=2, num_q_heads=4, head_dim=64, page_size=16,
                          context_lens=[1, 17, 50], seed=62, causal=causal)
        p = synth.make(case)
        pw = dict(p)
        pw["case"] = synth.replace(case, window=51)  # = L_max + qlen - 1: holds every token
        assert np.array_equal(util.oracle_decode(pw), util.oracle_decode(p))


def test_window_equals_attention_over_its_token_range():
    # one query position: the window [L - W, L) through the range entry point of the same
    # cache without a window (a separate path of the oracle: an explicit token range)
    W = 23
    case = synth.Case("wr", synth.KV_FP8, synth.SCALE_TOKEN, synth.Q_BF16, batch=3, qlen=1,
                      num_kv_heads=2, num_q_heads=8, head_dim=64, page_size=16,
                      context_lens=[10, 40, 90], fill=synth.FILL_ZERO, seed=63, kv_std=20.0)
    p = synth.make(case)
    pw = dict(p)
    pw["case"] = synth.replace(case, window=W)
    got = util.oracle_decode(pw)
    plain = util.oracle_problem(p)
    for s, L in enumerate([10, 40, 90]):
        for hkv in range(2):
            _, _, o = plain.attend_range(s, hkv, max(0, L - W), L)
            np.testing.assert_array_equal(got[s, 0, 4 * hkv:4 * hkv + 4], o.reshape(4, 64))


def test_window_pins_catch_off_by_one():
    # a window one token wider or narrower is a different result on this data
    case = [c for c in _tiny_cases() if c.name == "t_fp8_window_q4"][0]
    p = synth.make(synth.replace(case, fill=synth.FILL_ZERO))
    got = util.oracle_decode(p)
    for w in (case.window - 1, case.window + 1):
        assert util.rel_l2(got, brute_force(p, window=w)) > 1e-3, w


@pytest.mark.parametrize("kv", [synth.KV_BF16, synth.KV_FP8])
def test_transposed_value_cache_gives_the_same_result(kv):
    # the same values stored [NB, Hkv, D, S] instead of [NB, Hkv, S, D]: the same bits
    scale = synth.SCALE_NONE if kv == synth.KV_BF16 else synth.SCALE_TENSOR
    case = synth.Case("tv", kv, scale, synth.Q_BF16, batch=3, qlen=2, num_kv_heads=2,
                      num_q_heads=8, head_dim=64, page_size=16, context_lens=[3, 40, 100],
                      fill=synth.FILL_ZERO, seed=64, kv_std=20.0)
    p = synth.make(case)
    pt = synth.make(synth.replace(case, trans_v=True))
    assert torch.equal(pt["value_cache"].transpose(-1, -2), p["value_cache"])
    assert np.array_equal(util.oracle_decode(pt), util.oracle_decode(p))
    # and the layout is not symmetric: the transposed bytes read as plain V differ
    wrong = dict(pt)
    wrong["case"] = synth.replace(case, trans_v=False)
    wrong["value_cache"] = pt["value_cache"].reshape(p["value_cache"].shape)
    assert util.rel_l2(util.oracle_decode(wrong), util.oracle_decode(p)) > 1e-2


def test_sinks_at_minus_infinity_change_nothing():
    case = synth.Case("sk0", synth.KV_FP8, synth.SCALE_TENSOR, synth.Q_BF16, batch=3, qlen=2,
                      num_kv_heads=2, num_q_heads=8, head_dim=64, page_size=16,
                      context_lens=[1, 30, 70], seed=65, kv_std=20.0)
    p = synth.make(case)
    ps = dict(p)
    ps["sinks"] = torch.full((8,), -1e30)
    assert np.array_equal(util.oracle_decode(ps), util.oracle_decode(p))


def test_sinks_with_identical_keys_closed_form():
    # every score equals c: out = mean(V) * L e^c / (L e^c + e^s)
    case = synth.Case("skc", synth.KV_BF16, synth.SCALE_NONE, synth.Q_BF16, batch=1, qlen=1,
                      num_kv_heads=1, num_q_heads=3, head_dim=64, page_size=16,
                      context_lens=[37], seed=66)
    p = synth.make(case)
    kc = p["key_cache"].clone()
    row = kc[int(p["block_tables"][0, 0]), 0, 0].clone()
    for t in range(37):
        kc[int(p["block_tables"][0, t // 16]), 0, t % 16] = row
    p["key_cache"] = kc
    p["sinks"] = torch.tensor([-1.0, 0.5, 4.0])
    got = util.oracle_decode(p)
    V = _dequant_dense(p, "v")
    t = torch.arange(37)
    mean = V[p["block_tables"][0].long()[t // 16], 0, t % 16].mean(dim=0).numpy()
    Q = _query_dense(p)
    for h in range(3):
        c = float(row.to(torch.float64) @ Q[0, 0, h]) * case.scale_qk()
        s_h = float(p["sinks"][h])
        want = mean * (37 * math.exp(c)) / (37 * math.exp(c) + math.exp(s_h))
        np.testing.assert_allclose(got[0, 0, h], want, rtol=1e-12, atol=1e-13)


def test_a_dominant_sink_drives_the_output_to_zero():
    case = synth.Case("skz", synth.KV_BF16, synth.SCALE_NONE, synth.Q_BF16, batch=2, qlen=1,
                      num_kv_heads=1, num_q_heads=2, head_dim=64, page_size=16,
                      context_lens=[5, 40], seed=67)
    p = synth.make(case)
    p["sinks"] = torch.tensor([600.0, 600.0])
    got = util.oracle_decode(p)
    assert np.all(np.isfinite(got)) and np.abs(got).max() < 1e-200


def test_e4m3_rounding_matches_torch():
    # every finite e4m3 value, every midpoint between neighbours (ties go to the even
    # code), and random floats, against torch's float32 -> float8_e4m3fn cast
    codes = [c for c in range(256) if (c & 0x7F) != 0x7F]
    vals = np.array(sorted({orc.decode_e4m3(c) for c in codes}), dtype=np.float64)
    pos = vals[vals >= 0]
    mids = (pos[1:] + pos[:-1]) / 2
    rng = np.random.default_rng(7)
    rnd = np.concatenate([rng.uniform(-448, 448, 4000), rng.uniform(-0.02, 0.02, 2000)])
    x = np.concatenate([vals, mids, -mids, rnd]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([orc.round_e4m3(float(v)) for v in x])
    assert np.array_equal(got, ref)
    assert orc.round_e4m3(500.0) == 448.0 and orc.round_e4m3(-1e6) == -448.0


def _quant_rows_torch(Q: torch.Tensor) -> torch.Tensor:
    """Per head row: s = amax / 448, y = q / s in float32, torch's e4m3 cast, times s."""
    q32 = Q.to(torch.float32)
    amax = q32.abs().amax(dim=-1, keepdim=True)
    s = amax / torch.tensor(448.0, dtype=torch.float32)
    y = torch.where(amax > 0, q32 / torch.where(amax > 0, s, torch.ones_like(s)), torch.zeros_like(q32))
    e = y.to(torch.float8_e4m3fn).to(torch.float64)
    return e * s.to(torch.float64)


def test_quantised_query_matches_dense_torch_path():
    case = synth.Case("qq", synth.KV_MXFP4, synth.SCALE_E8M0, synth.Q_BF16, batch=3, qlen=1,
                      num_kv_heads=2, num_q_heads=8, head_dim=128, page_size=16,
                      context_lens=[5, 40, 77], fill=synth.FILL_RANDOM, seed=51, q_quant=True)
    p = synth.make(case)
    got = util.oracle_decode(p)
    K, V = _dequant_dense(p, "k"), _dequant_dense(p, "v")
    Q = _quant_rows_torch(_query_dense(p).reshape(3, 8, 128))
    bt = p["block_tables"].cpu()
    for s, L in enumerate([5, 40, 77]):
        rows = [(int(bt[s, t // 16]), t % 16) for t in range(L)]
        for h in range(8):
            k = torch.stack([K[b, h // 4, r] for b, r in rows])
            v = torch.stack([V[b, h // 4, r] for b, r in rows])
            w = torch.softmax((k @ Q[s, h]) * case.scale_qk(), dim=0)
            np.testing.assert_allclose(got[s, 0, h], (w @ v).numpy(), rtol=1e-11, atol=1e-12)
    # and the quantisation is not a no-op on this data
    plain = dict(p)
    plain["case"] = synth.replace(case, q_quant=False)
    assert util.rel_l2(util.oracle_decode(plain), got) > 1e-4


def test_quantised_query_of_exact_rows_is_the_plain_query():
    # rows that are e4m3 codes times 2^-4 with |max| = 448 * 2^-4: s = 2^-4 exactly and
    # every y is already an e4m3 value, so the quantised query equals the stored one
    case = synth.Case("qx", synth.KV_MXFP4, synth.SCALE_E8M0, synth.Q_BF16, batch=2, qlen=1,
                      num_kv_heads=1, num_q_heads=4, head_dim=128, page_size=16,
                      context_lens=[9, 30], fill=synth.FILL_RANDOM, seed=52, q_quant=True)
    p = synth.make(case)
    rng = np.random.default_rng(53)
    finite = np.array([orc.decode_e4m3(c) for c in range(256) if (c & 0x7F) != 0x7F])
    q = rng.choice(finite, size=(2, 4, 128)) / 16.0
    q[..., 0] = 448.0 / 16.0
    p["query"] = torch.from_numpy(q).to(torch.bfloat16).reshape(p["query"].shape)
    assert torch.equal(torch.from_numpy(q).to(torch.bfloat16).to(torch.float64),
                       torch.from_numpy(q))  # bf16-exact
    plain = dict(p)
    plain["case"] = synth.replace(case, q_quant=False)
    assert np.array_equal(util.oracle_decode(p), util.oracle_decode(plain))


def test_identical_keys_give_mean_of_v():
    case = synth.Case("samek", synth.KV_FP8, synth.SCALE_TENSOR, synth.Q_BF16, batch=1,
                      qlen=1, num_kv_heads=1, num_q_heads=2, head_dim=64, page_size=16,
                      context_lens=[37], seed=22, kv_std=20.0)
    p = synth.make(case)
    kc = p["key_cache"].clone()
    row = kc[int(p["block_tables"][0, 0]), 0, 0].clone()
    for t in range(37):
        kc[int(p["block_tables"][0, t // 16]), 0, t % 16] = row
    p["key_cache"] = kc
    got = util.oracle_decode(p)
    V = _dequant_dense(p, "v")
    t = torch.arange(37)
    blk = p["block_tables"][0].long()[t // 16]
    mean = V[blk, 0, t % 16].mean(dim=0).numpy()
    for h in range(2):
        np.testing.assert_allclose(got[0, 0, h], mean, rtol=1e-13, atol=1e-13)


def test_context_zero_gives_zero():
    case = synth.config1(context_lens=[0, 17], seed=23)
    p = synth.make(case)
    got = util.oracle_decode(p)
    assert np.all(got[0] == 0.0)
    assert np.abs(got[1]).sum() > 0


def test_split_merge_identity():
    """Merging (m, l, o) of [0, a) and [a, L) reproduces the full softmax."""
    case = synth.config3(qlen=2, context_lens=(60, 90), batch=2, seed=24)
    p = synth.make(case)
    prob = util.oracle_problem(p)
    full = prob.decode()
    L = int(p["context_lens"][1])
    for a in (1, 17, L // 2, L - 1):
        m1, l1, o1 = prob.attend_range(1, 1, 0, a)
        m2, l2, o2 = prob.attend_range(1, 1, a, L)
        M = np.maximum(m1, m2)
        w1, w2 = l1 * np.exp(m1 - M), l2 * np.exp(m2 - M)
        merged = (w1[:, None] * o1 + w2[:, None] * o2) / (w1 + w2)[:, None]
        G = case.gqa
        for r in range(case.qlen * G):
            i, h = r // G, G + r % G
            np.testing.assert_allclose(merged[r], full[1, i, h], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("make_case", [
    lambda: synth.config1(seed=31),
    lambda: synth.config2("a", batch=5, context_lens=[1, 17, 255, 257, 1000], seed=32),
    lambda: synth.config3(qlen=1, batch=2, context_lens=(20, 300), seed=33),
    lambda: synth.config4(batch=2, context_lens=[2000, 77], seed=34),
], ids=["bf16", "fp8_tensor", "fp8_token", "mxfp4"])
def test_unowned_rows_do_not_reach_output(make_case):
    p = synth.make(make_case())
    base = util.oracle_decode(synth.refill(p, synth.FILL_ZERO))
    assert np.isfinite(base).all()
    for fill in (synth.FILL_NAN, synth.FILL_INF, synth.FILL_RANDOM):
        got = util.oracle_decode(synth.refill(p, fill))
        assert np.array_equal(got, base), fill


def test_oracle_refuses_bad_tables():
    p = synth.make(synth.config1(seed=41))
    bt = p["block_tables"].clone()
    bt[0, 0] = p["num_blocks"]  # out of range
    q = dict(p)
    q["block_tables"] = bt
    with pytest.raises(ValueError):
        util.oracle_decode(q)


def test_parity_checker_catches_planted_errors():
    """The comparison itself: an oracle-side perturbation of 0.05 at one element, a NaN,
    or a dropped V scale must fail it, while the bf16 rounding of the oracle passes."""
    p = synth.make(synth.config3(qlen=1, batch=2, context_lens=(40, 90), seed=51))
    ref = util.oracle_decode(p)
    rounded = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
    util.assert_parity(rounded, ref, synth.KV_FP8)
    bad = ref.copy()
    bad[1, 0, 3, 17] += 0.05
    with pytest.raises(AssertionError):
        util.assert_parity(bad, ref, synth.KV_FP8)
    bad = ref.copy()
    bad[0, 0, 0, 0] = np.nan
    with pytest.raises(AssertionError):
        util.assert_parity(bad, ref, synth.KV_FP8)
    q = dict(p)
    q["value_scale"] = p["value_scale"] * 1.05
    with pytest.raises(AssertionError):
        util.assert_parity(util.oracle_decode(q), ref, synth.KV_FP8)
