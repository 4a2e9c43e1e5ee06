"""Test helpers: hand the synthetic workload bytes to the oracle, and compare."""
from __future__ import annotations

import numpy as np
import torch

from oracle import pa_oracle as orc
from paged_attention_decode_02_gb300 import synth

_KV = {synth.KV_BF16: orc.KV_BF16, synth.KV_FP8: orc.KV_E4M3, synth.KV_MXFP4: orc.KV_MXFP4}
_SC = {synth.SCALE_NONE: orc.SCALE_NONE, synth.SCALE_TENSOR: orc.SCALE_TENSOR,
       synth.SCALE_TOKEN: orc.SCALE_TOKEN, synth.SCALE_E8M0: orc.SCALE_E8M0}
_Q = {synth.Q_BF16: orc.Q_BF16, synth.Q_E4M3: orc.Q_E4M3}


def cpu(t):
    return None if t is None else t.detach().cpu()


def oracle_problem(p: dict, seqs=None) -> orc.Problem:
    """Oracle view of a synthetic problem; ``seqs`` restricts it to some sequences."""
    case = p["case"]
    bt, cl = cpu(p["block_tables"]), cpu(p["context_lens"])
    q, qs = cpu(p["query"]), cpu(p["q_scale"])
    batch = case.batch
    if seqs is not None:
        idx = torch.as_tensor(list(seqs), dtype=torch.long)
        bt, cl, q = bt[idx], cl[idx], q[idx]
        qs = qs[idx] if (qs is not None and qs.numel() > 1) else qs
        batch = len(idx)
    return orc.Problem(
        batch=batch, qlen=case.qlen, num_q_heads=case.num_q_heads,
        num_kv_heads=case.num_kv_heads, head_dim=case.head_dim, page_size=case.page_size,
        num_blocks=p["num_blocks"], kv_format=_KV[case.kv], scale_kind=_SC[case.scale],
        q_format=orc.Q_BF16_TO_E4M3 if case.q_quant else _Q[case.q],
        softmax_scale=case.scale_qk(), query=q,
        key_cache=cpu(p["key_cache"]), value_cache=cpu(p["value_cache"]),
        key_scale=cpu(p["key_scale"]), value_scale=cpu(p["value_scale"]), q_scale=qs,
        block_tables=bt, context_lens=cl, causal=case.causal, window=case.window,
        trans_v=case.trans_v, sinks=cpu(p.get("sinks")))


def oracle_decode(p: dict, seqs=None, nthreads: int = 0) -> np.ndarray:
    return oracle_problem(p, seqs).decode(nthreads)


def rel_l2(got: np.ndarray, ref: np.ndarray) -> float:
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.linalg.norm(ref.ravel())
    num = np.linalg.norm((got - ref).ravel())
    return float(num / den) if den > 0 else float(num)


def max_abs(got, ref) -> float:
    d = np.abs(np.asarray(got, np.float64) - np.asarray(ref, np.float64))
    return float(d.max()) if d.size else 0.0


# Tolerances stated for the GPU path against the fp64 oracle.
TOL_REL_L2 = {synth.KV_BF16: 5e-3, synth.KV_FP8: 3e-3, synth.KV_MXFP4: 3e-3}
TOL_MAX_ABS = 3e-2
# The output is bf16: one unit in the last place is 2^-7 of the value's binade, at most
# 2^-7 |x| (the round-to-nearest error alone reaches 2^-9 |x|).  The absolute bound is
# applied beyond that quantum, since MXFP4 outputs reach |48| at the workloads' e8m0
# range, where a single bf16 rounding is 0.125.
def bf16_ulp(x) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits): 2^(floor(log2 |x|) - 7)."""
    ax = np.abs(np.asarray(x, np.float64))
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.exp2(e - 7), 0.0)


def excess_abs(got, ref) -> float:
    """max(|got - ref| - ulp_bf16(ref)): the output is bf16, so a result computed with any
    error at all may round to the neighbour of the correctly rounded value."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    d = np.abs(got - ref) - bf16_ulp(ref)
    return float(d.max()) if d.size else 0.0


def assert_parity(got, ref, kv: str, what: str = ""):
    r = rel_l2(got, ref)
    m = max_abs(got, ref)
    e = excess_abs(got, ref)
    assert np.isfinite(np.asarray(got, np.float64)).all(), f"{what}: non-finite output"
    assert r <= TOL_REL_L2[kv], f"{what}: rel-L2 {r:.3e} > {TOL_REL_L2[kv]:.1e}"
    assert e <= TOL_MAX_ABS, (f"{what}: max-abs beyond one bf16 ulp {e:.3e} > "
                              f"{TOL_MAX_ABS:.1e} (raw max-abs {m:.3e})")
    return r, m
