// pa_tc.cuh -- the sm_103a tensor-core decode kernel (tcgen05, TMEM accumulators) for
// head_dim 128 and up to 32 query rows per KV head.
//
// Each CTA walks the tasks of its plan chunk in 128-token tiles (one TMEM lane per
// token).  Warp roles:
//   warp 0      gathers each tile's K / V pages (and per-token or e8m0 scales) through
//               the block table with TMA into a ring of raw stages;
//   warp 1      owns the tensor memory, converts each task's query rows into the MMA's
//               B operand, and issues every tcgen05.mma:  S^T = K Q^T (tokens on the
//               M dimension) and O^T += V^T P^T (head dims on the M dimension);
//   warps 2-9   the softmax group: two threads own each token of S (each half the query
//               rows); they keep the running max and sums, rescale O in TMEM when the
//               max rises, and write P;
//   warps 10-17 the widening group: V (and MXFP4 K) to f16 in double-buffered shared
//               memory, running ahead of the softmax group, so that tile k+1 is widened
//               while tile k's softmax runs and the tensor cores run its PV.
// Scores of tokens at or past the context length become -inf and their V rows are
// written as zeros (or zeroed in place for bf16), so unowned rows never reach the output
// ("[FlyDSL] pa_decode: zero V rows past the context before PV", Fix).  fp8 K feeds the
// tensor cores as stored (kind::f8f6f4) against the query split exactly into two e4m3
// terms; per-token scales fold into the scores and into P; MXFP4 block scales fold into
// the widened K (relative to the token's largest block) and V (relative to a running
// per-block reference).  The running max and V references rise lazily, by more than
// 2^8 and 8x; a rise rescales O in TMEM.
#pragma once

#include <cuda_fp8.h>

#include "pa_tile.cuh"

namespace pa {

// TcCfg<format, scale kind, padded query rows, raw stages>.
template <int KIND_, int SKT_, int RPAD_, int NS_>
struct TcCfg {
  static constexpr int KIND = KIND_, SKT = SKT_, RPAD = RPAD_, NS = NS_;
  static constexpr int D = 128, TT = 128;
  static constexpr int NSW = 8;                  // softmax warps: two per TMEM lane quarter
  static constexpr int NWW = 8;                  // widening warps
  static constexpr int NCW = NSW + NWW;
  static constexpr int NTHREADS = 64 + 32 * NCW;
  static constexpr int RH = RPAD / 2;            // query rows per softmax thread
  static constexpr bool TOK = SKT == SK_TOKEN;
  static constexpr bool SCALES = SKT == SK_TOKEN || SKT == SK_E8M0;
  static constexpr bool QK_F8 = KIND == KIND_FP8;  // e4m3 K as stored, query split hi + lo
  static constexpr bool KDQ = KIND == KIND_FP4;    // K widened to f16 by the consumers
  static constexpr bool VDQ = KIND != KIND_BF16;   // V widened to f16 by the consumers
  static constexpr int SUB = KIND == KIND_FP4 ? 64 : 128;  // TMA box row bytes
  static constexpr int NSUB = KIND == KIND_BF16 ? 2 : 1;   // boxes across a cache row
  static constexpr int RAW_T = NSUB * TT * SUB;             // one tensor's tile
  static constexpr int RAW_SC = SCALES ? 4 * TT : 0;        // one tensor's tile scales
  static constexpr int SLOT = (2 * RAW_T + 2 * RAW_SC + 1023) / 1024 * 1024;
  static constexpr int NSC = QK_F8 ? 2 * RPAD : RPAD;  // S columns per buffer
  static constexpr int SBUF = 2;                       // S buffers: QK runs a tile ahead
  static constexpr int Q_BYTES = QK_F8 ? NSC * 128 : RPAD * 256;
  static constexpr int NQB = SBUF + 1;                 // query buffers (task ordinal mod NQB)
  static constexpr int P_BYTES = RPAD * 256;           // [2 token atoms][RPAD rows][128 B]
  static constexpr int VF_BYTES = VDQ ? TT * 256 : 0;  // [2 dim atoms][128 tokens][128 B]
  static constexpr int KF_BYTES = KDQ ? TT * 256 : 0;
  static constexpr int BUF_BYTES = P_BYTES + VF_BYTES + KF_BYTES;  // one of two tile buffers
  static constexpr int RED_W = 2 * RH + 10;                         // exchange words per warp
  static constexpr int VINFO_W = 8;  // per tile buffer: MXFP4 V exponent drops [4], references [4]
  static constexpr int OFF_RING = 0;
  static constexpr int OFF_Q = OFF_RING + NS * SLOT;
  static constexpr int OFF_BUF = OFF_Q + NQB * Q_BYTES;
  static constexpr int OFF_QC = OFF_BUF + 2 * BUF_BYTES;
  static constexpr int OFF_RED = OFF_QC + NQB * RPAD * 4;
  static constexpr int OFF_VINFO = OFF_RED + NCW * RED_W * 4;
  static constexpr int OFF_BAR = (OFF_VINFO + 2 * VINFO_W * 4 + 7) / 8 * 8;
  static constexpr int B_RAW_FULL = 0, B_RAW_EMPTY = NS, B_S_FULL = 2 * NS;
  static constexpr int B_KF_FULL = B_S_FULL + SBUF, B_VINFO = B_KF_FULL + 2;
  static constexpr int B_PV_READY = B_VINFO + 2, B_PV_DONE = B_PV_READY + 2;
  static constexpr int B_SYNC_S = B_PV_DONE + 2, B_SYNC_W = B_SYNC_S + 1;
  static constexpr int B_MMA_DONE = B_SYNC_W + 1, NBAR = B_MMA_DONE + 1;
  static constexpr int RAW_EMPTY_COUNT = NCW + (KIND == KIND_FP4 ? 0 : 1);
  // arrival count of barrier i: TMA / MMA-commit signals 1, a group signals one per warp
  // (widening group NWW, softmax group NSW, both NCW), a raw stage one per consumer warp
  // (+ 1 commit when the tensor cores read the stage)
  static constexpr uint32_t bar_count(int i) {
    return i < B_RAW_EMPTY  ? 1u
           : i < B_S_FULL   ? (uint32_t)RAW_EMPTY_COUNT
           : i < B_KF_FULL  ? 1u
           : i < B_PV_READY ? (uint32_t)NWW
           : i < B_PV_DONE  ? (uint32_t)NCW
           : i < B_SYNC_S   ? 1u
           : i < B_SYNC_W   ? (uint32_t)NSW
           : i < B_MMA_DONE ? (uint32_t)NWW
                            : 1u;
  }
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 16 + 1024;  // + slack to align the base to 1 KiB
  static constexpr int COL_O = SBUF * NSC;           // TMEM columns: S buffers, then O
  static constexpr int TCOLS_NEED = SBUF * NSC + RPAD;
  static constexpr int TMEM_COLS = TCOLS_NEED <= 32    ? 32
                                   : TCOLS_NEED <= 64  ? 64
                                   : TCOLS_NEED <= 128 ? 128
                                                       : 256;
  static constexpr uint32_t FMT = KIND == KIND_BF16 ? 1u : 0u;  // bf16 : f16 (e4m3 for QK_F8)
  static constexpr uint32_t IDESC_QK = umma_idesc(FMT, FMT, 0, 0, NSC, 128);
  static constexpr uint32_t IDESC_PV = umma_idesc(FMT, FMT, 1, 0, RPAD, 128);
  static_assert(RPAD == 16 || RPAD == 32, "query rows padded to 16 or 32");
  static_assert(SLOT % 1024 == 0 && Q_BYTES % 1024 == 0 && BUF_BYTES % 1024 == 0,
                "128-byte-swizzled operands sit on 1 KiB boundaries");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static_assert(NS >= 2, "at least double-buffered pages");
};

// ---------------------------------------------------------------------------------------
struct TcTask {
  int s, hkv, part, L, t0, n, unit;
};

__device__ __forceinline__ TcTask tc_task(const DecodeParams& p, int task) {
  const PlanTask tk = p.tasks[task];
  TcTask r;
  r.s = tk.seq;
  r.hkv = tk.hkv_part & 0xFFFF;
  r.part = tk.hkv_part >> 16;
  r.L = clamped_context(p, r.s);
  r.t0 = tk.tile_begin * kTileTokens;
  int t1 = tk.tile_end * kTileTokens;
  t1 = t1 < r.L ? t1 : r.L;
  r.n = t1 > r.t0 ? (t1 - r.t0 + 127) >> 7 : 0;
  r.unit = r.s * p.Hkv + r.hkv;
  return r;
}

// A cursor over the non-empty tasks' 128-token tiles, in the order every role walks them.
struct TileCur {
  int task, te, i, k, ord;
  bool valid;
  TcTask T;
};

__device__ __forceinline__ void cur_next_task(TileCur& c, const DecodeParams& p) {
  for (;;) {
    if (++c.task >= c.te) {
      c.valid = false;
      return;
    }
    c.T = tc_task(p, c.task);
    if (c.T.n > 0) break;
  }
  c.i = 0;
  ++c.ord;
}
__device__ __forceinline__ void cur_init(TileCur& c, const DecodeParams& p, int tb, int te) {
  c.task = tb - 1;
  c.te = te;
  c.k = 0;
  c.ord = -1;
  c.valid = true;
  cur_next_task(c, p);
}
__device__ __forceinline__ void cur_advance(TileCur& c, const DecodeParams& p) {
  ++c.k;
  if (++c.i >= c.T.n) cur_next_task(c, p);
}

// Bounded wait that also stops every later wait once any role has given up.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                        int* status) {
  if (*abort_flag) return false;
  if (mbar_wait_bounded(bar, parity)) return true;
  *abort_flag = 1;
  atomicOr(status, ST_TIMEOUT);
  return false;
}

// Byte offset of (row, byte column) in a region of 128-byte rows swizzled in 1 KiB atoms.
__device__ __forceinline__ uint32_t sw128(int row, int bcol) {
  return (uint32_t)(row * 128 + ((((bcol >> 4) ^ (row & 7)) << 4) | (bcol & 15)));
}

// ---------------------------------------------------------------------------------------
// Warp 0: page gather.  Block-table entries arrive 32 boxes at a time, one per lane, the
// next 32 loaded while the current ones are used, so no TMA issue waits on a global load.
template <class C>
__device__ void tc_producer(const DecodeParams& p, const CUtensorMap* tmk, const CUtensorMap* tmv,
                            uint8_t* sm, uint64_t* bars, volatile int* abort_flag, int tb, int te,
                            int lane) {
  const int page_shift = __ffs(p.S) - 1, page_mask = p.S - 1;
  const int box = p.S < C::TT ? p.S : C::TT;
  const int box_shift = __ffs(box) - 1;
  const int bpt = C::TT >> box_shift;  // boxes per tile
  if (lane == 0) {
    tma_prefetch_desc(tmk);
    tma_prefetch_desc(tmv);
  }
  TileCur c;
  cur_init(c, p, tb, te);
  bool ok = true;
  int cur_task = -1, bbase = 0, bcur = 0, bnxt = 0;
  const int32_t* btrow = nullptr;
  auto bt_load = [&](int b) -> int {  // block of box b of the current task (0 past the context)
    const int tok = c.T.t0 + b * box;
    return tok < c.T.L ? btrow[tok >> page_shift] : 0;
  };
  for (; c.valid; cur_advance(c, p)) {
    if (c.task != cur_task) {
      cur_task = c.task;
      btrow = p.bt + (int64_t)c.T.s * p.bt_stride;
      bbase = 0;
      bcur = bt_load(lane);
      bnxt = bt_load(32 + lane);
    }
    const int b0 = c.i * bpt;  // first box of this tile
    if (b0 + bpt > bbase + 64) {  // cannot happen with bpt <= 32; kept as a guard
      ok = false;
      break;
    }
    if (b0 >= bbase + 32) {
      bbase += 32;
      bcur = bnxt;
      bnxt = bt_load(bbase + 32 + lane);
    }
    const int k = c.k, slot = k % C::NS, f = k / C::NS;
    if (f > 0 && !tc_wait(&bars[C::B_RAW_EMPTY + slot], (f - 1) & 1, abort_flag, p.status)) {
      ok = false;
      break;
    }
    const int c0 = c.T.t0 + c.i * C::TT;
    const int ntok = min(C::TT, c.T.L - c0);
    const int nbox = (ntok + box - 1) >> box_shift;
    uint8_t* dst = sm + C::OFF_RING + slot * C::SLOT;
    uint64_t* full = &bars[C::B_RAW_FULL + slot];
    // box j of this tile is box b0 + j of the task: lane (b0 + j - bbase) of bcur / bnxt
    const int idx = b0 + lane - bbase;
    const int from_cur = __shfl_sync(0xffffffffu, bcur, idx & 31);
    const int from_nxt = __shfl_sync(0xffffffffu, bnxt, idx & 31);
    int blk = idx < 32 ? from_cur : from_nxt;
    blk = blk < 0 ? 0 : (blk >= p.NB ? p.NB - 1 : blk);
    if (lane == 0)
      mbar_arrive_expect_tx(full, (uint32_t)(nbox * box * (2 * C::NSUB * C::SUB + (C::SCALES ? 8 : 0))));
    __syncwarp();
    if (lane < nbox) {  // nbox <= 128 / 8
      fence_proxy_async();  // the slot was last read through the generic proxy
      const int tok = c0 + lane * box;
      const int srow = tok & page_mask;
#pragma unroll
      for (int u = 0; u < C::NSUB; ++u) {
        const int off = u * (C::TT * C::SUB) + lane * box * C::SUB;
        tma_load_4d(dst + off, tmk, full, u * C::SUB, srow, c.T.hkv, blk);
        tma_load_4d(dst + C::RAW_T + off, tmv, full, u * C::SUB, srow, c.T.hkv, blk);
      }
      if constexpr (C::SCALES) {
        const int64_t so = (int64_t)blk * p.sc_sb + (int64_t)c.T.hkv * p.sc_sh + (int64_t)srow * 4;
        bulk_load(dst + 2 * C::RAW_T + lane * box * 4, p.k_scale + so, box * 4, full);
        bulk_load(dst + 2 * C::RAW_T + C::RAW_SC + lane * box * 4, p.v_scale + so, box * 4, full);
      }
    }
  }
  if (!ok) {  // let the copies already in flight land before the CTA exits
    for (int k = c.k - 1; k >= 0 && k >= c.k - C::NS; --k)
      (void)mbar_wait_bounded(&bars[C::B_RAW_FULL + k % C::NS], (k / C::NS) & 1);
  }
}

// ---------------------------------------------------------------------------------------
// Warp 1: query rows of a task into Q buffer `qb` (the MMA's B operand) and their logit
// factors (softmax scale * log2 e * query scale * row normalisation [* hi scale]).
template <class C>
__device__ void tc_load_q(const DecodeParams& p, uint8_t* sm, const TcTask& T, int qb, int lane) {
  uint8_t* qs = sm + C::OFF_Q + qb * C::Q_BYTES;
  float* qc = reinterpret_cast<float*>(sm + C::OFF_QC) + qb * C::RPAD;
  const float kst = (C::KIND == KIND_FP8 && C::SKT == SK_TENSOR) ? reinterpret_cast<const float*>(p.k_scale)[0]
                                                                 : 1.f;
  // every row's four elements of this lane (and its scale) first: independent loads
  uint32_t raw[C::RPAD][2];
  float qsc[C::RPAD];
#pragma unroll
  for (int r = 0; r < C::RPAD; ++r) {
    raw[r][0] = raw[r][1] = 0u;
    qsc[r] = 0.f;
    if (r < p.R) {
      const int i = r / p.G, h = T.hkv * p.G + r % p.G;
      const int64_t row = (int64_t)T.s * p.qlen + i;
      const int64_t off = row * p.q_st + (int64_t)h * p.q_sh + 4 * lane;
      if (p.q_fp8) {
        raw[r][0] = *reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint8_t*>(p.q) + off);
        qsc[r] = p.q_scale_per_row ? p.q_scale[row * p.Hq + h] : p.q_scale[0];
      } else {
        const uint2 v = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(p.q) + off);
        raw[r][0] = v.x;
        raw[r][1] = v.y;
        qsc[r] = 1.f;
      }
    }
  }
#pragma unroll
  for (int r = 0; r < C::RPAD; ++r) {
    float x[4];
    if (p.q_fp8) {
      const uint32_t lo = e4m3x2_to_f16x2(raw[r][0] & 0xFFFF), hi = e4m3x2_to_f16x2(raw[r][0] >> 16);
      const __half2 l2 = *reinterpret_cast<const __half2*>(&lo), h2 = *reinterpret_cast<const __half2*>(&hi);
      x[0] = __low2float(l2);
      x[1] = __high2float(l2);
      x[2] = __low2float(h2);
      x[3] = __high2float(h2);
    } else {
      x[0] = __uint_as_float(raw[r][0] << 16);
      x[1] = __uint_as_float(raw[r][0] & 0xFFFF0000u);
      x[2] = __uint_as_float(raw[r][1] << 16);
      x[3] = __uint_as_float(raw[r][1] & 0xFFFF0000u);
    }
    float cr = p.scale_log2 * qsc[r] * kst;  // 0 for padding rows
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if constexpr (C::KIND == KIND_BF16) {
      uint8_t* dst = qs + (lane >> 4) * (C::RPAD * 128) + sw128(r, (lane & 15) * 8);
      *reinterpret_cast<uint2*>(dst) = make_uint2(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]));
    } else if constexpr (!C::QK_F8) {
      // f16 operand: the row's largest magnitude into [256, 512) by a power of two
      int kx = 0;
      if (amax > 0.f) {
        kx = ((__float_as_int(amax) >> 23) & 0xFF) - 127 - 8;
        kx = kx < -100 ? -100 : (kx > 100 ? 100 : kx);
      }
      const float down = exp2i(-kx);
      cr *= exp2i(kx);
      uint8_t* dst = qs + (lane >> 4) * (C::RPAD * 128) + sw128(r, (lane & 15) * 8);
      *reinterpret_cast<uint2*>(dst) =
          make_uint2(pack_f16x2(x[0] * down, x[1] * down), pack_f16x2(x[2] * down, x[3] * down));
    } else {
      // two e4m3 terms: q = s (hi + lo / 16), hi = e4m3(q / s), lo = e4m3(16 (q / s - hi)),
      // s = 2^(floor(log2 amax) - 7), so that q / s keeps q's 8 significant bits and lies
      // in (-256, 256): hi rounds it to 4 significant bits and the residual, a multiple of
      // 2^-7 of q's binade no larger than half hi's spacing, is exact in e4m3 -- the split
      // is exact for every element down to 2^-13 of the row's largest (below that the
      // residual loses bits under 2^-9 s)
      int ex = amax > 0.f ? ((__float_as_int(amax) >> 23) & 0xFF) - 127 - 7 : 0;
      ex = ex < -100 ? -100 : (ex > 100 ? 100 : ex);
      const float s = exp2i(ex);
      const float inv = exp2i(-ex);
      uint32_t hib = 0, lob = 0;
#pragma unroll
      for (int j = 0; j < 4; j += 2) {
        const float a0 = x[j] * inv, a1 = x[j + 1] * inv;
        const __nv_fp8x2_storage_t h2 = __nv_cvt_float2_to_fp8x2(make_float2(a0, a1), __NV_SATFINITE, __NV_E4M3);
        const __half2_raw hb = __nv_cvt_fp8x2_to_halfraw2(h2, __NV_E4M3);
        const __half2 hh = *reinterpret_cast<const __half2*>(&hb);
        const float r0 = (a0 - __low2float(hh)) * 16.f, r1 = (a1 - __high2float(hh)) * 16.f;
        const __nv_fp8x2_storage_t l2 = __nv_cvt_float2_to_fp8x2(make_float2(r0, r1), __NV_SATFINITE, __NV_E4M3);
        hib |= (uint32_t)h2 << (8 * j);
        lob |= (uint32_t)l2 << (8 * j);
      }
      *reinterpret_cast<uint32_t*>(qs + sw128(r, 4 * lane)) = hib;
      *reinterpret_cast<uint32_t*>(qs + sw128(C::RPAD + r, 4 * lane)) = lob;
      cr *= s;
    }
    if (lane == 0) qc[r] = cr;
  }
  fence_proxy_async();  // generic writes, read next by the tensor cores
  __threadfence_block();  // the row factors are read by the consumer warps
  __syncwarp();
}

// Warp 1: MMA issue.  Polls both queues and issues whichever MMA is ready: QK of the next
// tile (at most SBUF tiles ahead of PV, which keeps every S buffer and query buffer it
// writes free) and PV of the oldest tile whose P is written.  Every barrier a role waits
// on can run at most one phase ahead of that wait (one barrier per buffer where needed).
template <class C>
__device__ void tc_mma(const DecodeParams& p, uint8_t* sm, uint64_t* bars, volatile int* abort_flag,
                       uint32_t tmem, int tb, int te, int lane) {
  TileCur cq, cp;
  cur_init(cq, p, tb, te);
  cur_init(cp, p, tb, te);
  const uint32_t ring = smem_u32(sm + C::OFF_RING);
  int qloaded = -1;
  uint64_t idle_since = 0;
  uint32_t idle = 0;
  bool ok = true;
  while (ok && cp.valid) {
    bool prog = false;
    if (cq.valid && cq.k < cp.k + C::SBUF) {
      const int k = cq.k, slot = k % C::NS, sb = k % C::SBUF;
      const int qb = cq.ord % C::NQB;
      if (cq.ord != qloaded) {
        tc_load_q<C>(p, sm, cq.T, qb, lane);
        qloaded = cq.ord;
      }
      const bool rdy = C::KDQ ? mbar_test(&bars[C::B_KF_FULL + (k & 1)], (k >> 1) & 1)
                              : mbar_test(&bars[C::B_RAW_FULL + slot], (k / C::NS) & 1);
      if (__shfl_sync(0xffffffffu, rdy ? 1 : 0, 0)) {
        tc_fence_after();
        if (lane == 0) {
          const uint32_t qa = smem_u32(sm + C::OFF_Q + qb * C::Q_BYTES);
          const uint32_t d = tmem + (uint32_t)(sb * C::NSC);
          if constexpr (C::QK_F8) {
            const uint32_t a = ring + slot * C::SLOT;
#pragma unroll
            for (int s = 0; s < 4; ++s)
              umma_f8(d, umma_desc(a + 32 * s, 16, 1024), umma_desc(qa + 32 * s, 16, 1024), C::IDESC_QK, s > 0);
          } else {
            const uint32_t a = C::KDQ ? smem_u32(sm + C::OFF_BUF + (k & 1) * C::BUF_BYTES + C::P_BYTES + C::VF_BYTES)
                                      : ring + slot * C::SLOT;
#pragma unroll
            for (int s = 0; s < 8; ++s) {
              const uint32_t ao = (s >> 2) * (C::TT * 128) + (s & 3) * 32;
              const uint32_t bo = (s >> 2) * (C::RPAD * 128) + (s & 3) * 32;
              umma_f16(d, umma_desc(a + ao, 16, 1024), umma_desc(qa + bo, 16, 1024), C::IDESC_QK, s > 0);
            }
          }
          umma_commit(&bars[C::B_S_FULL + sb]);
          if constexpr (C::QK_F8) umma_commit(&bars[C::B_RAW_EMPTY + slot]);
        }
        __syncwarp();
        cur_advance(cq, p);
        prog = true;
      }
    }
    {
      const int k = cp.k, slot = k % C::NS;
      const bool rdy = mbar_test(&bars[C::B_PV_READY + (k & 1)], (k >> 1) & 1);
      if (__shfl_sync(0xffffffffu, rdy ? 1 : 0, 0)) {
        tc_fence_after();
        if (lane == 0) {
          const uint8_t* g = sm + C::OFF_BUF + (k & 1) * C::BUF_BYTES;
          const uint32_t a = C::VDQ ? smem_u32(g + C::P_BYTES) : ring + slot * C::SLOT + C::RAW_T;
          const uint32_t b = smem_u32(g);
          const uint32_t d = tmem + (uint32_t)C::COL_O;
          const uint32_t acc = cp.i > 0;  // a task's first tile starts O afresh
#pragma unroll
          for (int s = 0; s < 8; ++s) {
            const uint32_t bo = (s >> 2) * (C::RPAD * 128) + (s & 3) * 32;
            umma_f16(d, umma_desc(a + s * 2048, C::TT * 128, 1024), umma_desc(b + bo, 16, 1024), C::IDESC_PV,
                     s > 0 || acc);
          }
          umma_commit(&bars[C::B_PV_DONE + (k & 1)]);
          if constexpr (C::KIND == KIND_BF16) umma_commit(&bars[C::B_RAW_EMPTY + slot]);
        }
        __syncwarp();
        cur_advance(cp, p);
        prog = true;
      }
    }
    if (prog) {
      idle_since = 0;
      idle = 0;
    } else if ((++idle & 1023) == 0) {  // the wall clock is slow to read: look every 1024 polls
      if (*abort_flag) break;
      const uint64_t now = global_ns();
      if (idle_since == 0) {
        idle_since = now;
      } else if (now - idle_since > 2000000000ull) {
        if (lane == 0) {
          *abort_flag = 1;
          atomicOr(p.status, ST_TIMEOUT);
        }
        ok = false;
      }
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
  }
  // every MMA issued has completed before the tensor memory is freed
  if (lane == 0) umma_commit(&bars[C::B_MMA_DONE]);
  __syncwarp();
  (void)mbar_wait_bounded(&bars[C::B_MMA_DONE], 0);
}

// ---------------------------------------------------------------------------------------
// Consumer group.
// Group-wide barrier with a time limit: lane 0 of each consumer warp arrives.
__device__ __forceinline__ bool grp_sync(uint64_t* bar, uint32_t& phase, volatile int* abort_flag,
                                         int* status, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  const bool ok = tc_wait(bar, phase & 1, abort_flag, status);
  ++phase;
  return ok;
}

// MXFP4 K or V tile (64-byte rows, 64-byte swizzle) to f16 [2 dim atoms][128][128 B]:
// widening thread `ci` (0..255) widens 32-value block (ci & 3) of tokens ci / 4 + 64 j,
// times 2^(e - ref) (K: ref = the token's largest block exponent; V: the running
// reference of block ci & 3).  Rows past the context become zeros.
template <class C, bool ISK>
__device__ __forceinline__ void tc_widen_fp4(const uint8_t* raw, const uint8_t* sc, uint8_t* dst, int ci,
                                             int c0, int L, int vref_b) {
  const int b = ci & 3;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    const int tok = (ci >> 2) + 64 * j;
    const uint4 v = *reinterpret_cast<const uint4*>(raw + tok * 64 + ((b ^ ((tok >> 1) & 3)) << 4));
    const uint32_t sw = *reinterpret_cast<const uint32_t*>(sc + tok * 4);
    const int e = (int)((sw >> (8 * b)) & 0xFF);
    int ref;
    if constexpr (ISK) {
      const int e01 = max((int)(sw & 0xFF), (int)((sw >> 8) & 0xFF));
      const int e23 = max((int)((sw >> 16) & 0xFF), (int)(sw >> 24));
      ref = max(e01, e23);
    } else {
      ref = vref_b;
    }
    const uint32_t fb = (uint32_t)min(max(e - ref + 15, 0), 30) << 10;
    const uint32_t f2 = c0 + tok < L ? (fb | (fb << 16)) : 0u;
    uint32_t h[16];
    e2m1x8_to_f16x2(v.x, *reinterpret_cast<uint32_t(*)[4]>(&h[0]));
    e2m1x8_to_f16x2(v.y, *reinterpret_cast<uint32_t(*)[4]>(&h[4]));
    e2m1x8_to_f16x2(v.z, *reinterpret_cast<uint32_t(*)[4]>(&h[8]));
    e2m1x8_to_f16x2(v.w, *reinterpret_cast<uint32_t(*)[4]>(&h[12]));
#pragma unroll
    for (int i = 0; i < 16; ++i) h[i] = hmul2(h[i], f2);
    uint8_t* row = dst + (b >> 1) * (C::TT * 128) + tok * 128;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int cc = (b & 1) * 4 + u;
      *reinterpret_cast<uint4*>(row + ((cc ^ (tok & 7)) << 4)) =
          make_uint4(h[4 * u], h[4 * u + 1], h[4 * u + 2], h[4 * u + 3]);
    }
  }
}

// fp8 V tile (128-byte rows, 128-byte swizzle) to f16: widening thread `ci` (0..255)
// widens dims 16 (ci & 7) .. +15 of tokens ci / 8 + 32 j.
template <class C>
__device__ __forceinline__ void tc_widen_fp8(const uint8_t* raw, uint8_t* dst, int ci, int c0, int L) {
  const int qd = ci & 7;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int tok = (ci >> 3) + 32 * j;
    const uint4 v = *reinterpret_cast<const uint4*>(raw + tok * 128 + ((qd ^ (tok & 7)) << 4));
    uint32_t h[8];
    e4m3x4_to_f16x2(v.x, h[0], h[1]);
    e4m3x4_to_f16x2(v.y, h[2], h[3]);
    e4m3x4_to_f16x2(v.z, h[4], h[5]);
    e4m3x4_to_f16x2(v.w, h[6], h[7]);
    const uint32_t m = c0 + tok < L ? 0xFFFFFFFFu : 0u;
    uint8_t* row = dst + (qd >> 2) * (C::TT * 128) + tok * 128;
    const int cc = (qd & 3) * 2;
    *reinterpret_cast<uint4*>(row + ((cc ^ (tok & 7)) << 4)) = make_uint4(h[0] & m, h[1] & m, h[2] & m, h[3] & m);
    *reinterpret_cast<uint4*>(row + (((cc + 1) ^ (tok & 7)) << 4)) =
        make_uint4(h[4] & m, h[5] & m, h[6] & m, h[7] & m);
  }
}

// RH consecutive 32-bit TMEM columns of this thread's lane (RH = 8 or 16).
template <class C>
__device__ __forceinline__ void tc_ld_half(uint32_t taddr, float (&v)[C::RH]) {
  uint32_t r[16];
  if constexpr (C::RH == 16) {
    tmem_ld16(taddr, r);
  } else {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                   "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
  }
  tmem_wait_ld();
#pragma unroll
  for (int j = 0; j < C::RH; ++j) v[j] = __uint_as_float(r[j]);
}
template <class C>
__device__ __forceinline__ void tc_st_half(uint32_t taddr, const float (&v)[C::RH]) {
  uint32_t r[16];
#pragma unroll
  for (int j = 0; j < C::RH; ++j) r[j] = __float_as_uint(v[j]);
  if constexpr (C::RH == 16) {
    tmem_st16(taddr, r);
  } else {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
  }
  tmem_wait_st();
}

// Exchange area: a row of RED_W words per consumer warp.  Softmax warps: [0, RH) row
// maxima, [RH, 2 RH) row sums, then raise flags by tile parity [2] and the |v scale|
// maximum.  Widening warps: V reference flags by tile parity [2], then exponent maxima [4].
constexpr int XS_M = 0, XS_VMAX = 2;
constexpr int XW_V = 0, XW_EMAX = 2;

// Softmax group (warps 2-9): scores, lazy max, P, O rescale and the epilogue.
template <class C>
__device__ void tc_softmax(const DecodeParams& p, uint8_t* sm, uint64_t* bars, volatile int* abort_flag,
                           uint32_t tmem, int tb, int te, int wi, int lane) {
  constexpr int R = C::RPAD, RH = C::RH, RW = C::RED_W;
  const int q = (wi + 2) & 3;    // TMEM lane quarter of this warp (warp wi + 2)
  const int h = wi >> 2;         // which half of the query rows
  const int tt = q * 32 + lane;  // token of S, dim of O
  const int r0 = h * RH;         // first query row of this thread
  float* red = reinterpret_cast<float*>(sm + C::OFF_RED);
  int* redi = reinterpret_cast<int*>(red);
  const int* vinfo = reinterpret_cast<const int*>(sm + C::OFF_VINFO);
  const float* qcs = reinterpret_cast<const float*>(sm + C::OFF_QC);
  const uint32_t tl = tmem + ((uint32_t)(q * 32) << 16);
  const uint32_t tO = tl + (uint32_t)(C::COL_O + r0);
  uint64_t* sbar = &bars[C::B_SYNC_S];
  const float vs_tensor = (C::KIND == KIND_FP8 && C::SKT == SK_TENSOR) ? reinterpret_cast<const float*>(p.v_scale)[0]
                                                                       : 1.f;
  auto xr = [&](int w, int j) -> float& { return red[w * RW + j]; };
  auto xl = [&](int w, int j) -> float& { return red[w * RW + RH + j]; };
  auto xi = [&](int w, int slot) -> int& { return redi[w * RW + 2 * RH + slot]; };
  uint32_t sph = 0;
  int ord = -1, k = 0;
  bool ok = true;
  float m[RH], lp[RH], cq[RH];
  float vref = 0.f;
  int vrefq = 127;  // MXFP4: running V reference of this thread's dims' block (q)

  for (int task = tb; task < te && ok; ++task) {
    const TcTask T = tc_task(p, task);
    const int nparts = p.nparts[T.unit];
    if (T.n == 0) {  // empty unit: zeros
#pragma unroll
      for (int j = 0; j < RH; ++j) {
        const int r = r0 + j;
        if (r >= p.R) continue;
        const int i = r / p.G, hh = T.hkv * p.G + r % p.G;
        if (nparts <= 1) {
          p.out[((int64_t)T.s * p.qlen + i) * p.o_st + (int64_t)hh * p.o_sh + tt] = __float2bfloat16_rn(0.f);
        } else {
          const int64_t slot = (int64_t)p.part_base[T.unit] + T.part;
          p.part_o[(slot * p.R + r) * C::D + tt] = 0.f;
          if (tt == 0) reinterpret_cast<float2*>(p.part_ml)[slot * p.R + r] = make_float2(-INFINITY, 0.f);
        }
      }
      continue;
    }
    const int qb = (++ord) % C::NQB;
    for (int i = 0; i < T.n; ++i) {
      const int kk = k + i, slot = kk % C::NS, buf = kk & 1;
      const uint8_t* raw = sm + C::OFF_RING + slot * C::SLOT;
      uint8_t* P = sm + C::OFF_BUF + buf * C::BUF_BYTES;
      const int c0 = T.t0 + i * C::TT;
      const bool own = c0 + tt < T.L;
      const bool first = i == 0;
      if (first) {
#pragma unroll
        for (int j = 0; j < RH; ++j) {
          m[j] = -INFINITY;
          lp[j] = 0.f;
        }
        vref = 0.f;
      }
      if (!tc_wait(&bars[C::B_RAW_FULL + slot], (kk / C::NS) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      float kt = 1.f, vs = 0.f;  // this token's scales, read before the stage is released
      if constexpr (C::TOK) {
        kt = reinterpret_cast<const float*>(raw + 2 * C::RAW_T)[tt];
        vs = own ? reinterpret_cast<const float*>(raw + 2 * C::RAW_T + C::RAW_SC)[tt] : 0.f;
      }
      if constexpr (C::KIND == KIND_FP4) {
        const uint32_t sw = reinterpret_cast<const uint32_t*>(raw + 2 * C::RAW_T)[tt];
        const int e01 = max((int)(sw & 0xFF), (int)((sw >> 8) & 0xFF));
        const int e23 = max((int)((sw >> 16) & 0xFF), (int)(sw >> 24));
        kt = exp2i(max(e01, e23) - 127);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C::B_RAW_EMPTY + slot]);
      // ---- scores of this thread's token and rows ----
      const int sb = kk % C::SBUF;
      if (!tc_wait(&bars[C::B_S_FULL + sb], (kk / C::SBUF) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      if (first) {
#pragma unroll
        for (int j = 0; j < RH; ++j) cq[j] = qcs[qb * R + r0 + j];
      }
      float x[RH];
      {
        const uint32_t tS = tl + (uint32_t)(sb * C::NSC + r0);
        if constexpr (C::QK_F8) {
          float lo[RH];
          tc_ld_half<C>(tS, x);
          tc_ld_half<C>(tS + R, lo);
#pragma unroll
          for (int j = 0; j < RH; ++j) x[j] = fmaf(lo[j], 0.0625f, x[j]) * cq[j] * kt;
        } else {
          tc_ld_half<C>(tS, x);
#pragma unroll
          for (int j = 0; j < RH; ++j) x[j] = x[j] * cq[j] * kt;
        }
#pragma unroll
        for (int j = 0; j < RH; ++j)
          if (!own || r0 + j >= p.R) x[j] = -INFINITY;
      }
      // MXFP4: this tile's V reference moves, decided by the widening group
      int dexpq = 0;
      bool any_dexp = false;
      if constexpr (C::KIND == KIND_FP4) {
        if (!tc_wait(&bars[C::B_VINFO + buf], (kk >> 1) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        const int* vi = vinfo + buf * C::VINFO_W;
        any_dexp = (vi[0] | vi[1] | vi[2] | vi[3]) != 0;
        dexpq = q == 0 ? vi[0] : (q == 1 ? vi[1] : (q == 2 ? vi[2] : vi[3]));
        vrefq = q == 0 ? vi[4] : (q == 1 ? vi[5] : (q == 2 ? vi[6] : vi[7]));
      }
      // ---- lazy raise of the running max (and fp8 per-token V reference), group-wide ----
      bool need_m = false;
#pragma unroll
      for (int j = 0; j < RH; ++j) need_m |= x[j] > m[j] + kLazyLog2;
      const float vsa = fabsf(vs);
      const bool need_v = C::TOK && vsa > vref * kLazyVref;
      const int fl = (__any_sync(0xffffffffu, need_m) ? 1 : 0) | (__any_sync(0xffffffffu, need_v) ? 2 : 0);
      if (lane == 0) xi(wi, XS_M + buf) = fl;
      if (!grp_sync(sbar, sph, abort_flag, p.status, lane)) {
        ok = false;
        break;
      }
      int F = 0;
#pragma unroll
      for (int w = 0; w < C::NSW; ++w) F |= xi(w, XS_M + buf);
      float alpha[RH];
#pragma unroll
      for (int j = 0; j < RH; ++j) alpha[j] = 1.f;
      float beta = 1.f;
      if (F) {
        if (F & 1) {
#pragma unroll
          for (int j = 0; j < RH; ++j) {
            float v = x[j];
#pragma unroll
            for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (lane == 0) xr(wi, j) = v;
          }
        }
        if constexpr (C::TOK) {
          if (F & 2) {
            const uint32_t mv = __reduce_max_sync(0xffffffffu, __float_as_uint(vsa));
            if (lane == 0) xi(wi, XS_VMAX) = (int)mv;
          }
        }
        if (!grp_sync(sbar, sph, abort_flag, p.status, lane)) {
          ok = false;
          break;
        }
        if (F & 1) {
#pragma unroll
          for (int j = 0; j < RH; ++j) {
            const float tm = fmaxf(fmaxf(xr(4 * h, j), xr(4 * h + 1, j)), fmaxf(xr(4 * h + 2, j), xr(4 * h + 3, j)));
            const float mn = fmaxf(m[j], tm);
            if (mn > m[j]) {
              alpha[j] = fast_exp2(m[j] - mn);  // -inf -> 0
              m[j] = mn;
              lp[j] *= alpha[j];
            }
          }
        }
        if constexpr (C::TOK) {
          if (F & 2) {
            int a0 = 0;
#pragma unroll
            for (int w = 0; w < C::NSW; ++w) a0 = max(a0, xi(w, XS_VMAX));
            const float tv = __int_as_float(a0);
            if (tv > vref * kLazyVref) {
              beta = vref > 0.f ? vref / tv : 0.f;
              vref = tv;
            }
          }
        }
      }
      if (!first && (F != 0 || any_dexp)) {  // rescale this thread's part of O (its dim, its rows)
        if (!tc_wait(&bars[C::B_PV_DONE + (buf ^ 1)], ((kk - 1) >> 1) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float bq = C::TOK ? beta : (C::KIND == KIND_FP4 ? exp2i(dexpq) : 1.f);
        float o[RH];
        tc_ld_half<C>(tO, o);
#pragma unroll
        for (int j = 0; j < RH; ++j) o[j] *= alpha[j] * bq;
        tc_st_half<C>(tO, o);
      }
      // ---- P (its buffer is free once the tile two back is through PV) ----
      if (kk >= 2 && !tc_wait(&bars[C::B_PV_DONE + buf], ((kk - 2) >> 1) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      {
        const float vf = C::TOK ? (vref > 0.f ? vs / vref : 0.f) : 1.f;
        uint8_t* pb = P + (tt >> 6) * (R * 128);
        const int bc = (tt & 63) * 2;
#pragma unroll
        for (int j = 0; j < RH; ++j) {
          const float po = own && r0 + j < p.R ? fast_exp2(x[j] - m[j]) : 0.f;
          lp[j] += po;
          const float pv = po * vf;
          uint16_t hv;
          if constexpr (C::KIND == KIND_BF16) {
            const __nv_bfloat16 b16 = __float2bfloat16_rn(pv);
            hv = *reinterpret_cast<const uint16_t*>(&b16);
          } else {
            const __half h16 = __float2half_rn(pv);
            hv = *reinterpret_cast<const uint16_t*>(&h16);
          }
          *reinterpret_cast<uint16_t*>(pb + sw128(r0 + j, bc)) = hv;
        }
      }
      fence_proxy_async();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C::B_PV_READY + buf]);
    }
    if (!ok) break;
    // ---- epilogue: row sums, O, store ----
    const int klast = k + T.n - 1;
#pragma unroll
    for (int j = 0; j < RH; ++j) {
      float v = lp[j];
#pragma unroll
      for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
      if (lane == 0) xl(wi, j) = v;
    }
    if (!grp_sync(sbar, sph, abort_flag, p.status, lane)) break;
    float L[RH];
#pragma unroll
    for (int j = 0; j < RH; ++j) L[j] = ((xl(4 * h, j) + xl(4 * h + 1, j)) + xl(4 * h + 2, j)) + xl(4 * h + 3, j);
    if (!tc_wait(&bars[C::B_PV_DONE + (klast & 1)], (klast >> 1) & 1, abort_flag, p.status)) break;
    tc_fence_after();
    float o[RH];
    tc_ld_half<C>(tO, o);
    tc_fence_before();
    float gam = 1.f;
    if constexpr (C::TOK) gam = vref;
    if constexpr (C::KIND == KIND_FP8 && C::SKT == SK_TENSOR) gam = vs_tensor;
    if constexpr (C::KIND == KIND_FP4) gam = exp2i(vrefq - 127);
    if (nparts <= 1) {
#pragma unroll
      for (int j = 0; j < RH; ++j) {
        const int r = r0 + j;
        if (r >= p.R) continue;
        const int i = r / p.G, hh = T.hkv * p.G + r % p.G;
        const float inv = L[j] > 0.f ? gam / L[j] : 0.f;
        p.out[((int64_t)T.s * p.qlen + i) * p.o_st + (int64_t)hh * p.o_sh + tt] = __float2bfloat16_rn(o[j] * inv);
      }
    } else {
      const int64_t slot = (int64_t)p.part_base[T.unit] + T.part;
#pragma unroll
      for (int j = 0; j < RH; ++j) {
        const int r = r0 + j;
        if (r >= p.R) continue;
        const float inv = L[j] > 0.f ? gam / L[j] : 0.f;
        p.part_o[(slot * p.R + r) * C::D + tt] = o[j] * inv;
        if (tt == 0) reinterpret_cast<float2*>(p.part_ml)[slot * p.R + r] = make_float2(m[j], L[j]);
      }
    }
    k += T.n;
  }
}

// Widening group (warps 10-17): V (and MXFP4 K) of each tile to f16, bf16 unowned rows to
// zero; MXFP4 per-block V references, published for the softmax group.
template <class C>
__device__ void tc_widener(const DecodeParams& p, uint8_t* sm, uint64_t* bars, volatile int* abort_flag, int tb,
                           int te, int wi, int lane) {
  constexpr int RW = C::RED_W;
  const int ci = wi * 32 + lane;  // share of the widening (0 .. 255)
  int* redi = reinterpret_cast<int*>(sm + C::OFF_RED) + C::NSW * RW;  // rows of the widening warps
  int* vinfo = reinterpret_cast<int*>(sm + C::OFF_VINFO);
  uint64_t* wbar = &bars[C::B_SYNC_W];
  auto xw = [&](int w, int slot) -> int& { return redi[w * RW + slot]; };
  uint32_t wph = 0;
  int k = 0;
  bool ok = true;
  int vrefb[4] = {-1000, -1000, -1000, -1000};
  for (int task = tb; task < te && ok; ++task) {
    const TcTask T = tc_task(p, task);
    for (int i = 0; i < T.n; ++i) {
      const int kk = k + i, slot = kk % C::NS, buf = kk & 1;
      const uint8_t* raw = sm + C::OFF_RING + slot * C::SLOT;
      uint8_t* VF = sm + C::OFF_BUF + buf * C::BUF_BYTES + C::P_BYTES;
      uint8_t* KF = VF + C::VF_BYTES;
      const int c0 = T.t0 + i * C::TT;
      const bool first = i == 0;
      if (first) {
#pragma unroll
        for (int b = 0; b < 4; ++b) vrefb[b] = -1000;
      }
      if (!tc_wait(&bars[C::B_RAW_FULL + slot], (kk / C::NS) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      // this parity's buffers are free once the tile two back is through PV (and QK)
      if (kk >= 2 && !tc_wait(&bars[C::B_PV_DONE + buf], ((kk - 2) >> 1) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      if constexpr (C::KDQ) {
        tc_widen_fp4<C, true>(raw, raw + 2 * C::RAW_T, KF, ci, c0, T.L, 0);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[C::B_KF_FULL + buf]);
      }
      if constexpr (C::KIND == KIND_FP4) {
        // V references: raise block b when an owned exponent exceeds it by more than 2^3
        const int b = ci & 3;
        const uint8_t* vsc = raw + 2 * C::RAW_T + C::RAW_SC;
        int emx = 0;
        bool need = false;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int tok = (ci >> 2) + 64 * j;
          const int e = c0 + tok < T.L ? (int)vsc[tok * 4 + b] : 0;
          emx = max(emx, e);
          need |= c0 + tok < T.L && e > vrefb[b] + kLazyExp;
        }
        const int vfl = __any_sync(0xffffffffu, need) ? 1 : 0;
        if (lane == 0) xw(wi, XW_V + buf) = vfl;
        if (!grp_sync(wbar, wph, abort_flag, p.status, lane)) {
          ok = false;
          break;
        }
        int Fv = 0;
#pragma unroll
        for (int w = 0; w < C::NWW; ++w) Fv |= xw(w, XW_V + buf);
        int dexp[4] = {0, 0, 0, 0};
        if (Fv) {
          const int wm = (int)__reduce_max_sync(0x11111111u << (lane & 3), (unsigned)emx);  // lanes of block b
          if (lane < 4) xw(wi, XW_EMAX + lane) = wm;
          if (!grp_sync(wbar, wph, abort_flag, p.status, lane)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            int tv = 0;
#pragma unroll
            for (int w = 0; w < C::NWW; ++w) tv = max(tv, xw(w, XW_EMAX + bb));
            if (tv > vrefb[bb] + kLazyExp) {
              dexp[bb] = first ? 0 : vrefb[bb] - tv;
              vrefb[bb] = tv;
            }
          }
        }
        if (wi == 0 && lane == 0) {
          int* vi = vinfo + buf * C::VINFO_W;
#pragma unroll
          for (int bb = 0; bb < 4; ++bb) {
            vi[bb] = dexp[bb];
            vi[4 + bb] = vrefb[bb];
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[C::B_VINFO + buf]);
      }
      if constexpr (C::KIND == KIND_FP8) {
        tc_widen_fp8<C>(raw + C::RAW_T, VF, ci, c0, T.L);
      } else if constexpr (C::KIND == KIND_FP4) {
        const int bb = ci & 3;
        const int vb = bb == 0 ? vrefb[0] : (bb == 1 ? vrefb[1] : (bb == 2 ? vrefb[2] : vrefb[3]));
        tc_widen_fp4<C, false>(raw + C::RAW_T, raw + 2 * C::RAW_T + C::RAW_SC, VF, ci, c0, T.L, vb);
      } else {
        const int tok = ci >> 1, u = ci & 1;  // bf16 V feeds the MMA as stored: zero unowned rows in place
        if (c0 + tok >= T.L) {
          uint8_t* vr = const_cast<uint8_t*>(raw) + C::RAW_T + u * (C::TT * 128) + tok * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(vr + 16 * c) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async();  // widened / zeroed rows are read next by the tensor cores
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[C::B_PV_READY + buf]);
        mbar_arrive(&bars[C::B_RAW_EMPTY + slot]);  // bf16: the PV commit releases it as well
      }
    }
    k += T.n;
  }
}

// ---------------------------------------------------------------------------------------
template <class C>
__global__ void __launch_bounds__(C::NTHREADS, 1)
    pa_tc_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                 const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_MISC + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBAR; ++i) mbar_init(&bars[i], C::bar_count(i));
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(tslot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  pdl_wait_prior();         // the plan's task list is complete and visible from here on
  pdl_launch_dependents();  // the reduce kernel may launch (after the plan completed); it
                            // waits for this grid's results
  const int tb = p.chunk_first[blockIdx.x], te = p.chunk_first[blockIdx.x + 1];
  if (warp == 0) {
    tc_producer<C>(p, &tmk, &tmv, sm, bars, abort_flag, tb, te, lane);
  } else if (warp == 1) {
    tc_mma<C>(p, sm, bars, abort_flag, tmem, tb, te, lane);
  } else if (warp < 2 + C::NSW) {
    tc_softmax<C>(p, sm, bars, abort_flag, tmem, tb, te, warp - 2, lane);
  } else {
    tc_widener<C>(p, sm, bars, abort_flag, tb, te, warp - 2 - C::NSW, lane);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_free(tmem, C::TMEM_COLS);
}

template <class C>
int launch_tc(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int grid, void* stream) {
  static std::atomic<unsigned long long> attr_done{0};  // per device ordinal
  if (const int rc = set_smem_attr_once(pa_tc_kernel<C>, C::SMEM, attr_done)) return rc;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(C::NTHREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, pa_tc_kernel<C>, p, tk, tv);
  if (e != cudaSuccess) return (int)e;
  return (int)cudaGetLastError();
}

}  // namespace pa
