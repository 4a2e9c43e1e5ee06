"""Seeded synthetic decode workloads (inputs only; none of the decode arithmetic).

Both the CUDA path and the fp64 oracle read the bytes made here, so this module
must stay free of attention math.  Every tensor comes from a seeded
``torch.Generator``; the recipe for each workload follows the shapes, value
distributions and block-table structure of the pages' tests:

* block table: the owned pages of every sequence are a random permutation of
  blocks 1..NB-1, block 0 is owned by nobody, and every row carries 2 padded
  columns pointing at block 0 ("[FlyDSL] pa_decode: zero V rows past the
  context before PV", Tests);
* every row no sequence owns -- all of block 0 and the unwritten tail of each
  last page -- holds the chosen fill (NaN, the finite +-448 "inf" of e4m3,
  e8m0 255 and random bytes for MXFP4, or zero), together with its per-token
  scale when there is one.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

KV_BF16, KV_FP8, KV_MXFP4 = "bf16", "fp8", "mxfp4"
SCALE_NONE, SCALE_TENSOR, SCALE_TOKEN, SCALE_E8M0 = "none", "tensor", "token", "e8m0"
Q_BF16, Q_E4M3 = "bf16", "e4m3"
FILL_NAN, FILL_INF, FILL_ZERO, FILL_RANDOM = "nan", "inf", "zero", "random"


@dataclasses.dataclass
class Case:
    """One decode workload.  ``context_lens`` is a list, or a (lo, hi) range drawn uniformly."""
    name: str
    kv: str
    scale: str
    q: str
    batch: int
    qlen: int
    num_kv_heads: int
    num_q_heads: int
    head_dim: int
    page_size: int
    context_lens: object
    fill: str = FILL_NAN
    seed: int = 1000
    softmax_scale: Optional[float] = None
    kv_std: float = 1.0          # fp8: K/V bytes are e4m3(kv_std * N(0,1))
    tensor_scale: float = 0.05   # fp8 per-tensor k_scale = v_scale
    token_scale: tuple = (0.01, 0.1)
    e8m0_range: tuple = (120, 130)
    k_e8m0_range: Optional[tuple] = None  # MXFP4 K exponents, when they differ from V's
    causal: bool = False  # query length > 1: position i sees tokens < L - qlen + 1 + i
    q_quant: bool = False  # bf16 query quantised to e4m3 per head row by the kernel (MXFP4)
    # sliding window W > 0: query position i (place p = L - qlen + i) sees tokens t > p - W;
    # rows before every position's window hold the fill, like rows no sequence owns
    window: int = 0
    # value cache stored head-dim major per page, [NB, Hkv, D, S] (bf16 / fp8 only)
    trans_v: bool = False
    # attention sinks: one fp32 logit per query head (in the units of the softmax-scaled
    # scores), drawn N(sink_mean, 1); None: no sinks
    sink_mean: Optional[float] = None
    pad_columns: int = 2
    extra_blocks: int = 0
    # > 0: magnitudes grow along each sequence by 2^(ramp * position / length) -- bf16 K and
    # V rows, fp8 per-token scales, MXFP4 e8m0 exponents (rounded) -- so that later tokens
    # keep raising the running max and the V references
    ramp: float = 0.0

    @property
    def gqa(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def scale_qk(self) -> float:
        return self.softmax_scale if self.softmax_scale is not None else 1.0 / math.sqrt(self.head_dim)


def replace(case: Case, **kw) -> Case:
    return dataclasses.replace(case, **kw)


# ---- the five workloads ----------------------------------------------------

def config1(**kw) -> Case:
    """bf16 KV, batch 2, 1 KV head, GQA 8, head_dim 128, qlen 1, page 16, lengths {17, 257}."""
    c = Case("cfg1_bf16", KV_BF16, SCALE_NONE, Q_BF16, batch=2, qlen=1, num_kv_heads=1,
             num_q_heads=8, head_dim=128, page_size=16, context_lens=[17, 257],
             fill=FILL_NAN, seed=1001)
    return replace(c, **kw)


def config2(sub: str = "b", **kw) -> Case:
    """fp8 e4m3 per-tensor (0.05), batch 16, 2 KV heads, GQA 8, D 256, qlen 4, page 64.
    sub 'a': lengths cycle over {1, 17, 255, 257, 1000}; sub 'b': uniform [1, 4096]."""
    lens = ([1, 17, 255, 257, 1000] * 4)[:16] if sub == "a" else (1, 4096)
    c = Case(f"cfg2{sub}_fp8_tensor", KV_FP8, SCALE_TENSOR, Q_BF16, batch=16, qlen=4,
             num_kv_heads=2, num_q_heads=16, head_dim=256, page_size=64, context_lens=lens,
             fill=FILL_INF, seed=1002 + (0 if sub == "a" else 10), kv_std=20.0)
    return replace(c, **kw)


def config3(qlen: int = 1, **kw) -> Case:
    """fp8 e4m3 per-token scales U[0.01, 0.1], batch 16, 2 KV heads, 16 query heads, D 256,
    page 16, qlen 1 or 4, lengths uniform [2048, 8192]."""
    c = Case(f"cfg3_fp8_token_q{qlen}", KV_FP8, SCALE_TOKEN, Q_BF16, batch=16, qlen=qlen,
             num_kv_heads=2, num_q_heads=16, head_dim=256, page_size=16,
             context_lens=(2048, 8192), fill=FILL_NAN, seed=1003 + 10 * qlen, kv_std=20.0)
    return replace(c, **kw)


def config4(batch: int = 64, **kw) -> Case:
    """MXFP4 KV, page 128, D 128, 1 KV head, GQA 16, qlen 1, e4m3 Q (per-row scale), ctx 2048."""
    c = Case(f"cfg4_mxfp4_b{batch}", KV_MXFP4, SCALE_E8M0, Q_E4M3, batch=batch, qlen=1,
             num_kv_heads=1, num_q_heads=16, head_dim=128, page_size=128,
             context_lens=[2048] * batch, fill=FILL_RANDOM, seed=1004 + batch)
    return replace(c, **kw)


def config5(kv: str = KV_MXFP4, **kw) -> Case:
    """Long context: batch 16, 1 KV head, GQA 16, D 128, page 128, qlen 1, bf16 Q,
    lengths uniform [120000, 131072]; MXFP4 (5a) or fp8 per-token (5b)."""
    if kv == KV_MXFP4:
        c = Case("cfg5a_mxfp4_long", KV_MXFP4, SCALE_E8M0, Q_BF16, batch=16, qlen=1,
                 num_kv_heads=1, num_q_heads=16, head_dim=128, page_size=128,
                 context_lens=(120000, 131072), fill=FILL_RANDOM, seed=1005)
    else:
        c = Case("cfg5b_fp8_token_long", KV_FP8, SCALE_TOKEN, Q_BF16, batch=16, qlen=1,
                 num_kv_heads=1, num_q_heads=16, head_dim=128, page_size=128,
                 context_lens=(120000, 131072), fill=FILL_NAN, seed=1015, kv_std=20.0)
    return replace(c, **kw)


# ---- generation ------------------------------------------------------------

def _lens(case: Case, g: torch.Generator) -> torch.Tensor:
    if isinstance(case.context_lens, tuple):
        lo, hi = case.context_lens
        return torch.randint(lo, hi + 1, (case.batch,), generator=g, dtype=torch.int64).to(torch.int32)
    lens = list(case.context_lens)
    assert len(lens) == case.batch, "context_lens must have one entry per sequence"
    return torch.tensor(lens, dtype=torch.int32)


def row_bytes(case: Case) -> int:
    return {KV_BF16: 2 * case.head_dim, KV_FP8: case.head_dim, KV_MXFP4: case.head_dim // 2}[case.kv]


def _e4m3_bytes(x: torch.Tensor) -> torch.Tensor:
    """Round to the nearest e4m3 value, saturating at +-448 (the generator's quantizer)."""
    return x.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)


def make(case: Case, device: str | torch.device = "cpu") -> dict:
    """Build every input tensor of ``case`` on ``device`` (CPU generator, then copied).

    Returns a dict with: query, q_scale, key_cache, value_cache, key_scale,
    value_scale, block_tables, context_lens, owned (bool [NB, S] per KV head row
    ownership mask, CPU), plus 'case'.  bf16 caches are torch.bfloat16
    [NB, Hkv, S, D]; fp8 caches are torch.uint8 (e4m3 bytes) [NB, Hkv, S, D];
    MXFP4 caches are torch.uint8 [NB, Hkv, S, D/2] with uint8 e8m0 scales
    [NB, Hkv, S, D/32].
    """
    g = torch.Generator().manual_seed(case.seed)
    B, S, Hkv, D = case.batch, case.page_size, case.num_kv_heads, case.head_dim
    lens = _lens(case, g)
    pages = [(int(L) + S - 1) // S for L in lens]
    total_pages = sum(pages)
    NB = 1 + total_pages + case.extra_blocks
    width = max(pages + [0]) + case.pad_columns
    width = max(width, 1)
    perm = (torch.randperm(NB - 1, generator=g) + 1).to(torch.int32)
    bt = torch.zeros((B, width), dtype=torch.int32)
    owned = torch.zeros((NB, S), dtype=torch.bool)
    pos = 0
    for s in range(B):
        n = pages[s]
        if n:
            blks = perm[pos:pos + n]
            pos += n
            bt[s, :n] = blks
            L = int(lens[s])
            owned[blks[:-1].long()] = True
            tail = L - (n - 1) * S
            owned[int(blks[-1]), :tail] = True
            lo = max(0, L - case.qlen - case.window + 1) if case.window > 0 else 0
            if lo > 0:
                owned[blks[:lo // S].long()] = False
                owned[int(blks[lo // S]), :lo % S] = False
    own4 = owned[:, None, :].expand(NB, Hkv, S)
    frac = torch.zeros((NB, S), dtype=torch.float32)  # position / length of owned rows
    if case.ramp > 0:
        pos = 0
        for s in range(B):
            n, L = pages[s], int(lens[s])
            if n:
                blks = bt[s, :n].long()
                p_ = torch.arange(n * S, dtype=torch.float32).reshape(n, S) / max(L, 1)
                frac[blks] = p_
                pos += n

    # query
    Hq, qlen = case.num_q_heads, case.qlen
    qf = torch.randn((B, qlen, Hq, D), generator=g, dtype=torch.float32)
    q_scale = None
    if case.q == Q_BF16:
        query = qf.to(torch.bfloat16)
    else:
        amax = qf.abs().amax(dim=-1, keepdim=True).clamp_min(1e-12)
        q_scale = (amax / 448.0).to(torch.float32)
        query = _e4m3_bytes(qf / q_scale)
        q_scale = q_scale.reshape(B, qlen, Hq).contiguous()

    rb = row_bytes(case)
    key_scale = value_scale = None
    if case.kv == KV_BF16:
        kc = torch.randn((NB, Hkv, S, D), generator=g).to(torch.bfloat16)
        vc = torch.randn((NB, Hkv, S, D), generator=g).to(torch.bfloat16)
        caches = [kc.view(torch.int16), vc.view(torch.int16)]
    elif case.kv == KV_FP8:
        kc = _e4m3_bytes(case.kv_std * torch.randn((NB, Hkv, S, D), generator=g))
        vc = _e4m3_bytes(case.kv_std * torch.randn((NB, Hkv, S, D), generator=g))
        caches = [kc, vc]
        if case.scale == SCALE_TENSOR:
            key_scale = torch.tensor([case.tensor_scale], dtype=torch.float32)
            value_scale = torch.tensor([case.tensor_scale], dtype=torch.float32)
        else:
            lo, hi = case.token_scale
            key_scale = lo + (hi - lo) * torch.rand((NB, Hkv, S), generator=g)
            value_scale = lo + (hi - lo) * torch.rand((NB, Hkv, S), generator=g)
    else:
        kc = torch.randint(0, 256, (NB, Hkv, S, rb), generator=g, dtype=torch.int32).to(torch.uint8)
        vc = torch.randint(0, 256, (NB, Hkv, S, rb), generator=g, dtype=torch.int32).to(torch.uint8)
        caches = [kc, vc]
        lo, hi = case.k_e8m0_range or case.e8m0_range
        key_scale = torch.randint(lo, hi + 1, (NB, Hkv, S, D // 32), generator=g,
                                  dtype=torch.int32).to(torch.uint8)
        lo, hi = case.e8m0_range
        value_scale = torch.randint(lo, hi + 1, (NB, Hkv, S, D // 32), generator=g,
                                    dtype=torch.int32).to(torch.uint8)

    if case.ramp > 0:
        f = (case.ramp * frac)[:, None, :].expand(NB, Hkv, S)  # log2 growth per row
        if case.kv == KV_BF16:
            g2 = torch.exp2(f)[..., None]
            kc = (kc.float() * g2).to(torch.bfloat16)
            vc = (vc.float() * g2).to(torch.bfloat16)
            caches = [kc.view(torch.int16), vc.view(torch.int16)]
        elif case.kv == KV_FP8 and case.scale == SCALE_TOKEN:
            key_scale = key_scale * torch.exp2(f)
            value_scale = value_scale * torch.exp2(f)
        elif case.kv == KV_MXFP4:
            add = torch.round(f).to(torch.int32)[..., None]
            key_scale = (key_scale.to(torch.int32) + add).clamp(0, 254).to(torch.uint8)
            value_scale = (value_scale.to(torch.int32) + add).clamp(0, 254).to(torch.uint8)

    # fill every row that no sequence owns
    unowned = ~own4
    _fill(case, caches, key_scale, value_scale, unowned, g)

    sinks = None
    if case.sink_mean is not None:
        sinks = case.sink_mean + torch.randn((case.num_q_heads,), generator=g, dtype=torch.float32)
    vcache = caches[1].view(torch.bfloat16) if case.kv == KV_BF16 else caches[1]
    if case.trans_v:
        assert case.kv != KV_MXFP4, "trans_v is a bf16 / fp8 layout"
        vcache = vcache.transpose(-1, -2).contiguous()  # [NB, Hkv, D, S]
    out = {
        "case": case,
        "query": query,
        "q_scale": q_scale,
        "key_cache": caches[0].view(torch.bfloat16) if case.kv == KV_BF16 else caches[0],
        "value_cache": vcache,
        "key_scale": key_scale,
        "value_scale": value_scale,
        "block_tables": bt,
        "context_lens": lens,
        "sinks": sinks,
        "owned": owned,
        "num_blocks": NB,
    }
    if str(device) != "cpu":
        out = to_device(out, device)
    return out


def _fill(case, caches, key_scale, value_scale, unowned, g):
    n = int(unowned.sum())
    if n == 0:
        return
    for c in caches:
        rows = c[unowned]            # [n, row] in storage type
        if case.fill == FILL_ZERO:
            rows.zero_()
        elif case.kv == KV_BF16:
            if case.fill == FILL_NAN:
                rows.fill_(0x7FC0)
            elif case.fill == FILL_INF:
                sign = torch.randint(0, 2, rows.shape, generator=g, dtype=torch.int16)
                rows.copy_(torch.where(sign > 0, torch.tensor(0x7F80, dtype=torch.int16),
                                       torch.tensor(-128, dtype=torch.int16)))  # +inf / -inf
            else:
                rows.copy_(torch.randint(-32768, 32768, rows.shape, generator=g, dtype=torch.int32).to(torch.int16))
        elif case.kv == KV_FP8:
            if case.fill == FILL_NAN:
                rows.fill_(0x7F)
            elif case.fill == FILL_INF:
                sign = torch.randint(0, 2, rows.shape, generator=g, dtype=torch.int32).to(torch.uint8)
                rows.copy_(0x7E | (sign << 7))  # +-448
            else:
                rows.copy_(torch.randint(0, 256, rows.shape, generator=g, dtype=torch.int32).to(torch.uint8))
        else:  # MXFP4: any byte is a number; the hostile part is the e8m0 scale
            rows.copy_(torch.randint(0, 256, rows.shape, generator=g, dtype=torch.int32).to(torch.uint8))
        c[unowned] = rows
    if case.scale == SCALE_TOKEN:
        for sc in (key_scale, value_scale):
            if case.fill == FILL_ZERO:
                sc[unowned] = 0.0
            elif case.fill == FILL_INF:
                sc[unowned] = float("inf")
            else:
                sc[unowned] = float("nan")
    elif case.scale == SCALE_E8M0:
        for sc in (key_scale, value_scale):
            if case.fill == FILL_ZERO:
                sc[unowned] = 0
            else:
                sc[unowned] = 255


def refill(problem: dict, fill: str, seed: int = 7) -> dict:
    """Same owned bytes, a different fill of the unowned rows (a new dict of clones)."""
    case = replace(problem["case"], fill=fill)
    S, Hkv = case.page_size, case.num_kv_heads
    owned = problem["owned"]
    NB = owned.shape[0]
    unowned = ~owned[:, None, :].expand(NB, Hkv, S)
    out = dict(problem)
    out["case"] = case
    kc = problem["key_cache"].detach().cpu().clone()
    vc = problem["value_cache"].detach().cpu().clone()
    caches = [kc.view(torch.int16), vc.view(torch.int16)] if case.kv == KV_BF16 else [kc, vc]
    ks = problem["key_scale"].detach().cpu().clone() if problem["key_scale"] is not None else None
    vs = problem["value_scale"].detach().cpu().clone() if problem["value_scale"] is not None else None
    _fill(case, caches, ks, vs, unowned, torch.Generator().manual_seed(seed))
    out["key_cache"], out["value_cache"] = kc, vc
    out["key_scale"], out["value_scale"] = ks, vs
    dev = problem["query"].device
    if dev.type != "cpu":
        for k in ("key_cache", "value_cache", "key_scale", "value_scale"):
            if out[k] is not None:
                out[k] = out[k].to(dev)
    return out


def to_device(problem: dict, device) -> dict:
    out = dict(problem)
    for k, v in problem.items():
        if isinstance(v, torch.Tensor) and k != "owned":
            out[k] = v.to(device)
    return out


def kv_bytes_per_token(case: Case) -> int:
    """Algorithmic K+V(+scale) bytes of one owned token of one KV head."""
    rb = row_bytes(case)
    extra = {SCALE_NONE: 0, SCALE_TENSOR: 0, SCALE_TOKEN: 8, SCALE_E8M0: 2 * (case.head_dim // 32)}[case.scale]
    return 2 * rb + extra


def algorithmic_bytes(case: Case, context_lens: Sequence[int]) -> int:
    """KV + scale bytes of owned tokens, plus Q and O bytes, plus the table and lengths."""
    tokens = int(sum(int(x) for x in context_lens))
    kvb = tokens * case.num_kv_heads * kv_bytes_per_token(case)
    qb = case.batch * case.qlen * case.num_q_heads * case.head_dim * (2 if case.q == Q_BF16 else 1)
    ob = case.batch * case.qlen * case.num_q_heads * case.head_dim * 2
    pages = sum((int(L) + case.page_size - 1) // case.page_size for L in context_lens)
    return kvb + qb + ob + 4 * pages + 4 * case.batch
