// pa_tile.cuh -- the sm_103a paged-attention decode tile kernel.
//
// Each CTA walks the tasks of its plan chunk (runs of 256-token tiles of one sequence
// and KV head; a chunk is an equal share of all tiles).  Every warp owns a token slice
// of each CTA stage and runs its own pipeline: it gathers its slice's pages through the
// block table with TMA (K and V land 128- or 64-byte swizzled; per-token or e8m0 scales
// arrive by 1-D bulk copy) into a private ring of mbarrier-guarded slots, NSTAGE slices
// ahead of the one it computes, so no warp ever waits for another inside a task.
// Softmax state and the output accumulators are warp-private; QK^T and PV run on
// mma.sync (m16n8k16, fp32 accumulate) with fp8 / fp4 operands widened to f16 in
// registers.  Only a slice holding tokens at or past the context length (or past a
// query position's causal limit, or before a sliding window's start) runs the masked
// path: scores there become -inf, and V values and per-token scales become 0 by select,
// so unowned rows never reach the output whatever bytes they hold ("[FlyDSL] pa_decode:
// zero V rows past the context before PV", Fix).  At the end of a task the warps merge
// their (max, sum, output) in a fixed order and store either the final bf16 row (units
// with one partition; an attention sink joins the row's sum here) or a partial for the
// reduce kernel ("[FlyDSL] pa_decode: MXFP4 K/V ...", direct output commit).  A
// transposed value cache (fp8) arrives in 16-token pieces, one 16-byte row per head dim,
// and the score columns take tokens in the order its fragments need (kv_token).
#pragma once

#include "pa_params.h"
#include "pa_ptx.cuh"

namespace pa {

enum { KIND_BF16 = 0, KIND_FP8 = 1, KIND_FP4 = 2 };
enum { SK_NONE = 0, SK_TENSOR = 1, SK_TOKEN = 2, SK_E8M0 = 3 };
enum { ST_OK = 0, ST_TIMEOUT = 1, ST_CLAMPED = 2 };

// TileCfg<format, scale kind, head_dim, m-tiles (query rows / 16), token groups, warps per
// token group (head-dim split), tokens per warp slice, slots per warp ring, CTAs per SM,
// a merge buffer of its own (every task merges in one pass, not only a chunk's last),
// transposed value cache [NB, Hkv, D, S] (fp8)>.
template <int KIND_, int SKT_, int D_, int MT_, int NTG_, int NDW_, int TW_, int NSTAGE_,
          int MINB_ = 1, int MRG_ = 0, int TRV_ = 0>
struct TileCfg {
  static constexpr int KIND = KIND_, SKT = SKT_, D = D_, MT = MT_, NTG = NTG_, NDW = NDW_;
  static constexpr int TW = TW_, NSTAGE = NSTAGE_, MINB = MINB_;
  static constexpr bool MRG = MRG_ != 0;
  // Transposed V: each slice's V arrives as 16-token pieces [DW head dims][16 tokens] (one
  // e4m3 byte per token), and the score columns take tokens in the order that makes a
  // lane's 4 consecutive tokens of one head dim its PV B-fragment (see kv_token).
  static constexpr bool TRV = TRV_ != 0;
  static constexpr bool TOK_SCALE = SKT == SK_TOKEN;                 // fp8 per-token scales
  static constexpr bool SCALES = SKT == SK_TOKEN || SKT == SK_E8M0;  // staged per slice
  static constexpr int NCW = NTG * NDW;  // warps (all compute; each loads its own slices)
  static constexpr int NTHREADS = NCW * 32;
  static constexpr int TC = TW * NTG;    // tokens per CTA stage
  static constexpr int NT = TW / 8;      // QK n-tiles per slice
  static constexpr int NKC = TW / 16;    // PV k-chunks per slice
  static constexpr int RPAD = MT * 16;
  static constexpr int ROW_BYTES = KIND == KIND_BF16 ? 2 * D : (KIND == KIND_FP8 ? D : D / 2);
  // swizzle span = sub-tile row: 128 bytes, or 64 where a warp's share of a row is 64 bytes
  static constexpr int SUB = ROW_BYTES / NDW_ >= 128 ? 128 : 64;
  static constexpr int NSUB = ROW_BYTES / SUB;
  static constexpr int NSUBW = NSUB / NDW;  // sub-tiles one warp loads and reads
  static constexpr int WBYTES = ROW_BYTES / NDW;
  static constexpr int NGRP = WBYTES / 64;  // ldmatrix.x4 groups per slice row
  static constexpr int NCP = WBYTES / 32;   // ldmatrix.x4.trans per 16-token chunk
  static constexpr int DW = D / NDW;        // head dims one warp owns
  static constexpr int NKCH = DW / 16;      // QK k-chunks per warp
  static constexpr int NTD = DW / 8;        // PV n-tiles per warp
  static constexpr int NBLK = KIND == KIND_FP4 ? D / 32 : 1;
  static constexpr int SLOT_V = NSUBW * TW * SUB;  // V offset inside a slot
  static constexpr int SLOT_KV = 2 * SLOT_V;       // K + V bytes of one slot
  static constexpr int SLOT_SC = 8 * TW;           // K then V scales (fp32 or 4 e8m0 bytes)
  static constexpr bool Q_IN_REGS = MT * NKCH * 4 <= 32;
  // The last task of a chunk merges its token groups in one pass through the (then idle)
  // load ring when every group's accumulator fits there.
  static constexpr bool PAR_MERGE = NCW * MT * NTD * 32 * 16 <= NCW * NSTAGE * SLOT_KV;
  // Query words are loaded ahead of a task when they take few registers.
  static constexpr bool Q_EARLY = ((RPAD + NCW - 1) / NCW) * (D / 64 + 1) <= 8;
  static constexpr int OFF_RING = 0;
  static constexpr int OFF_SC = OFF_RING + NCW * NSTAGE * SLOT_KV;
  static constexpr int OFF_Q = OFF_SC + NCW * NSTAGE * SLOT_SC;
  static constexpr int OFF_CR = OFF_Q + RPAD * D * 2;
  static constexpr int OFF_X = OFF_CR + RPAD * 4;
  static constexpr int XW = MT * NT * 4 * 32;  // floats per warp per exchange buffer
  // partial-score exchange between the head-dim warps of a token group: double-buffered
  // for two warps, one buffer (and a second barrier) for four
  static constexpr int XBUFS = NDW > 2 ? 1 : 2;
  static constexpr int X_BYTES = NDW > 1 ? NTG * XBUFS * NDW * XW * 4 : 0;
  static constexpr int OFF_OB = OFF_X + X_BYTES;
  // merged rows (RPAD x D floats), reused by the fused partition merge for its weights
  // (RPAD x up to 128 partitions)
  static constexpr int OBW = D > 128 ? D : 128;
  static constexpr int OFF_ML = OFF_OB + RPAD * OBW * 4;
  static constexpr int OFF_FIN = OFF_ML + NTG * RPAD * 8;  // 1 / sum per row
  static constexpr int TAB_BYTES = KIND == KIND_FP4 ? NBLK * TW * 6 : 0;  // K and V e8m0 factor tables
  static constexpr int OFF_TAB = OFF_FIN + RPAD * 8;
  static constexpr int OFF_BAR = (OFF_TAB + NCW * TAB_BYTES + 15) / 16 * 16;
  static constexpr int OFF_FLAG = OFF_BAR + NCW * NSTAGE * 8;
  static constexpr int OFF_NXT = OFF_FLAG + 16;  // the next task's record (16 bytes)
  static constexpr int OFF_ABT = OFF_NXT + 16;  // per warp: where its waits stopped
  static constexpr int OFF_MRG = (OFF_ABT + NCW * 4 + 15) / 16 * 16;
  static constexpr int MRG_BYTES = MRG ? NCW * MT * (D / NDW / 8) * 32 * 16 : 0;
  static constexpr int SMEM = OFF_MRG + MRG_BYTES + 1024;  // + slack to align the base to 1 KiB
  static_assert(TW % 16 == 0, "a warp slice holds whole 16-token k-chunks");
  static_assert(WBYTES % 64 == 0, "a warp row slice is whole ldmatrix.x4 groups");
  static_assert(NSUB % NDW == 0, "head-dim split on sub-tile boundaries");
  static_assert(SLOT_V % 1024 == 0, "swizzled TMA destinations are 1 KiB aligned");
  static_assert(KIND != KIND_FP4 || (D == 128 && NDW == 1 && TW == 32),
                "MXFP4 path: D 128, one warp per row, one lane per slice token");
  static_assert(SMEM * MINB <= 227 * 1024, "shared memory budget");
  static_assert(NTG + 1 < 16, "named barrier ids");
  static_assert(!TRV || KIND == KIND_FP8, "transposed V: e4m3 caches");
  static constexpr int PIECE_V = DW * 16;  // transposed V: bytes of one 16-token piece
  static constexpr int KOFFN = TRV ? 2 * NGRP : NGRP;  // K ldmatrix row offsets per lane
};

// Token (within its 16-token k-chunk) of score column c of a 16-token chunk.  Plain order
// for the token-major caches; with transposed V the columns 2u, 2u + 1, 8 + 2u, 9 + 2u take
// tokens 4u .. 4u + 3, the four consecutive tokens a lane reads from one head-dim row.
template <class C>
__device__ __forceinline__ int kv_token(int c) {
  if constexpr (C::TRV) return 4 * ((c & 7) >> 1) + (c & 1) + 2 * (c >> 3);
  return c;
}

constexpr int BAR_CONSUMERS = 15;  // named barrier id for all warps of the CTA
constexpr uint32_t kNoAbort = 0xFFFFFFFFu;  // a warp's waits have not stopped

template <class C>
__device__ __forceinline__ int swz(int row) {
  return C::SUB == 128 ? (row & 7) : ((row >> 1) & 3);
}

__device__ __forceinline__ int clamped_context(const DecodeParams& p, int s) {
  int L = p.ctx[s];
  const int cap = p.W * p.S;
  L = L < 0 ? 0 : L;
  return L > cap ? cap : L;
}

// Q A-fragment (m16n8k16, row-major A) of k-chunk `kap` of this warp for m-tile `mt`.
// The head-dim order inside a chunk follows the K fragment each format produces.
template <class C>
__device__ __forceinline__ void load_qa(const uint16_t* qs, int mt, int kap, int dw, int g,
                                        int t, uint32_t (&a)[4]) {
  const uint16_t* r0 = qs + (16 * mt + g) * C::D;
  const uint16_t* r8 = r0 + 8 * C::D;
  int d0, d1;
  if constexpr (C::KIND == KIND_BF16) {
    d0 = dw * C::DW + 16 * kap + 2 * t;
    d1 = d0 + 8;
  } else if constexpr (C::KIND == KIND_FP8) {
    d0 = dw * C::DW + 16 * kap + 4 * t;
    d1 = d0 + 2;
  } else {
    d0 = 32 * (kap >> 1) + 8 * t + 4 * (kap & 1);
    d1 = d0 + 2;
  }
  a[0] = *reinterpret_cast<const uint32_t*>(r0 + d0);
  a[1] = *reinterpret_cast<const uint32_t*>(r8 + d0);
  a[2] = *reinterpret_cast<const uint32_t*>(r0 + d1);
  a[3] = *reinterpret_cast<const uint32_t*>(r8 + d1);
}

// Head dim of element j (0..3) of PV n-tile n in this warp's accumulator.
template <class C>
__device__ __forceinline__ int o_dim(int n, int j, int dw, int t) {
  if constexpr (C::KIND == KIND_BF16 || C::TRV) {
    return dw * C::DW + 8 * n + 2 * t + (j & 1);
  } else if constexpr (C::KIND == KIND_FP8) {
    return dw * C::DW + 16 * (n >> 1) + 4 * t + (n & 1) + 2 * (j & 1);
  } else {
    return 32 * (n >> 2) + 8 * t + (n & 3) + 4 * (j & 1);
  }
}

// Inverse of o_dim: the float index, in the fragment-ordered merge buffer, of output
// row `row`, head dim `d` (buffer: per warp of a token group, per (m-tile, n-tile), 32
// lanes x float4).
template <class C>
__device__ __forceinline__ int frag_pos(int row, int d) {
  const int mt = row >> 4, g = row & 7, jh = (row >> 3) & 1;
  const int dw = d / C::DW, dd = d - dw * C::DW;
  int n, t, jl;
  if constexpr (C::KIND == KIND_BF16 || C::TRV) {  // dd = 8n + 2t + jl
    n = dd >> 3;
    t = (dd >> 1) & 3;
    jl = dd & 1;
  } else if constexpr (C::KIND == KIND_FP8) {  // dd = 16 (n >> 1) + 4t + (n & 1) + 2 jl
    const int r = dd & 15;
    n = 2 * (dd >> 4) + (r & 1);
    t = r >> 2;
    jl = (r >> 1) & 1;
  } else {  // dd = 32 (n >> 2) + 8t + (n & 3) + 4 jl
    const int r = dd & 31;
    n = 4 * (dd >> 5) + (r & 3);
    t = r >> 3;
    jl = (r >> 2) & 1;
  }
  return ((dw * (C::MT * C::NTD) + mt * C::NTD + n) * 32 + 4 * g + t) * 4 + 2 * jh + jl;
}

// 2^(e - 127) for an e8m0 byte as fp32 (e = 0 flushes to 0; 255 gives +inf).
__device__ __forceinline__ float e8m0_to_f32(uint32_t e) { return __int_as_float(e << 23); }

// 2^k for an integer k in [-126, 127]; 0 below.
__device__ __forceinline__ float exp2i(int k) {
  return k < -126 ? 0.f : __int_as_float((k + 127) << 23);
}

// MXFP4 K block factors are applied as 2^(e - 127 - 17): a 32-dim partial score of the
// normalised query (|q| < 512, |k| <= 6) stays below 2^17, so the scaled partial stays finite
// for every exponent byte up to 254 (P2 reports logits going to inf at byte 249 when the
// factor is applied unbiased); 2^17 moves into the row's logit factor.
constexpr float kKFactorBias = 1.f / 131072.f;

// The query words a lane reads for its rows of one task: loaded ahead of their use
// (before the ring is first filled, or while the previous task merges) and converted
// when the task starts.
template <class C>
struct QRaw {
  static constexpr int ROWS = (C::RPAD + C::NCW - 1) / C::NCW;  // rows per warp
  static constexpr int EPL = C::D / 32;                          // elements per lane per row
  static constexpr int NW = EPL / 2;  // 32-bit words per row (bf16; e4m3 uses EPL / 4)
  uint32_t w[ROWS][NW];
  float qsc[ROWS];
};

template <class C>
__device__ __forceinline__ void load_q_issue(const DecodeParams& p, int s, int hkv, int cw,
                                             int lane, QRaw<C>& q) {
  constexpr int EPL = QRaw<C>::EPL;
#pragma unroll
  for (int k = 0; k < QRaw<C>::ROWS; ++k) {
    const int r = cw + k * C::NCW;
    q.qsc[k] = 1.f;
    if (r < C::RPAD && r < p.R) {
      const int i = r / p.G, h = hkv * p.G + r % p.G;
      const int64_t row = (int64_t)s * p.qlen + i;
      const int64_t off = row * p.q_st + (int64_t)h * p.q_sh + lane * EPL;
      if (p.q_fp8) {
        const uint8_t* src = reinterpret_cast<const uint8_t*>(p.q) + off;
        if constexpr (EPL >= 4) {
#pragma unroll
          for (int j = 0; j < EPL / 4; ++j) q.w[k][j] = reinterpret_cast<const uint32_t*>(src)[j];
        } else {  // head_dim 64: two e4m3 bytes per lane
          q.w[k][0] = *reinterpret_cast<const uint16_t*>(src);
        }
        q.qsc[k] = p.q_scale_per_row ? p.q_scale[row * p.Hq + h] : p.q_scale[0];
      } else {
        const uint32_t* src =
            reinterpret_cast<const uint32_t*>(reinterpret_cast<const __nv_bfloat16*>(p.q) + off);
#pragma unroll
        for (int j = 0; j < QRaw<C>::NW; ++j) q.w[k][j] = src[j];
      }
    }
  }
}

// Converts a task's query words into shared memory, with the per-row logit factor
// (softmax scale * log2 e * q scale * row normalisation * k scale).
template <class C>
__device__ void load_q_finish(const DecodeParams& p, uint8_t* smem, const QRaw<C>& q, int cw,
                              int lane, float k_scale_tensor) {
  uint16_t* qs = reinterpret_cast<uint16_t*>(smem + C::OFF_Q);
  float* cr = reinterpret_cast<float*>(smem + C::OFF_CR);
  constexpr int EPL = QRaw<C>::EPL;
#pragma unroll
  for (int k = 0; k < QRaw<C>::ROWS; ++k) {
    const int r = cw + k * C::NCW;
    if (r >= C::RPAD) break;
    float x[EPL];
    float crv = 0.f;
    if (r < p.R) {
      if (p.q_fp8) {
#pragma unroll
        for (int j = 0; j < EPL / 4; ++j) {
          uint32_t lo = e4m3x2_to_f16x2(q.w[k][j] & 0xFFFF), hi = e4m3x2_to_f16x2(q.w[k][j] >> 16);
          __half2 l2 = *reinterpret_cast<__half2*>(&lo), h2 = *reinterpret_cast<__half2*>(&hi);
          x[4 * j + 0] = __low2float(l2);
          x[4 * j + 1] = __high2float(l2);
          x[4 * j + 2] = __low2float(h2);
          x[4 * j + 3] = __high2float(h2);
        }
        if constexpr (EPL == 2) {
          uint32_t lo = e4m3x2_to_f16x2(q.w[k][0] & 0xFFFF);
          __half2 l2 = *reinterpret_cast<__half2*>(&lo);
          x[0] = __low2float(l2);
          x[1] = __high2float(l2);
        }
      } else {
#pragma unroll
        for (int j = 0; j < QRaw<C>::NW; ++j) {  // bf16 pair: low half first
          x[2 * j] = __uint_as_float(q.w[k][j] << 16);
          x[2 * j + 1] = __uint_as_float(q.w[k][j] & 0xFFFF0000u);
        }
      }
      float qsck = q.qsc[k];
      if constexpr (C::KIND == KIND_FP4) {
        if (p.q_quant) {  // the row quantised to e4m3, scale amax / 448 (fp32, nearest)
          float amax = 0.f;
#pragma unroll
          for (int j = 0; j < EPL; ++j) amax = fmaxf(amax, fabsf(x[j]));
#pragma unroll
          for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
          const float sq = __fdiv_rn(amax, 448.f);
#pragma unroll
          for (int j = 0; j < EPL; ++j) x[j] = amax > 0.f ? round_e4m3(__fdiv_rn(x[j], sq)) : 0.f;
          qsck = amax > 0.f ? sq : 0.f;
        }
      }
      crv = p.scale_log2 * qsck;
      if constexpr (C::KIND == KIND_FP8) {
        if (p.scale_kind == SK_TENSOR) crv *= k_scale_tensor;
      }
      if constexpr (C::KIND != KIND_BF16) {
        // f16 operands: bring the row's largest magnitude into [256, 512) by a power of 2.
        float amax = 0.f;
#pragma unroll
        for (int j = 0; j < EPL; ++j) amax = fmaxf(amax, fabsf(x[j]));
#pragma unroll
        for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        int kx = 0;
        if (amax > 0.f) {
          kx = ((__float_as_int(amax) >> 23) & 0xFF) - 127 - 8;
          kx = kx < -100 ? -100 : (kx > 100 ? 100 : kx);
        }
        const float down = exp2i(-kx);
#pragma unroll
        for (int j = 0; j < EPL; ++j) x[j] *= down;
        crv *= exp2i(kx);
        if constexpr (C::KIND == KIND_FP4) crv *= 1.f / kKFactorBias;
      }
    } else {
#pragma unroll
      for (int j = 0; j < EPL; ++j) x[j] = 0.f;
    }
    uint16_t* dst = qs + r * C::D + lane * EPL;
#pragma unroll
    for (int j = 0; j < EPL; j += 2) {
      const uint32_t v = C::KIND == KIND_BF16 ? pack_bf16x2(x[j], x[j + 1]) : pack_f16x2(x[j], x[j + 1]);
      *reinterpret_cast<uint32_t*>(dst + j) = v;
    }
    if (lane == 0) cr[r] = crv;
  }
}

// Where a warp's loads stand: the next (task, slice) it will load (tasks of this CTA's
// chunk, in order).  The warp walks the
// same sequence of slices for loading and for computing, the loads NSTAGE ahead.  The
// block-table entries of the next slice are fetched one slice early (blk, one per box,
// held by lanes 0..nbox-1) so that no refill waits on a dependent global load.
struct SliceIt {
  const PlanTask* tasks;  // the plan's task list, or the single-launch mode's one record
  int task, c0, t0, t1, s, hkv, L;
  int lo;  // first token of the lowest query position's sliding window (0: none)
  const int32_t* btrow;
  int blk;
  bool done;
  int bx0, bcur, bnxt;  // blocks of this warp's boxes bx0 + lane and bx0 + 32 + lane in the task
};

__device__ __forceinline__ void it_load_task(SliceIt& it, const DecodeParams& p) {
  const PlanTask tk = it.tasks[it.task];
  it.s = tk.seq;
  it.hkv = tk.hkv_part & 0xFFFF;
  it.L = clamped_context(p, it.s);
  it.lo = p.window > 0 ? it.L - p.qlen - p.window + 1 : 0;
  it.lo = it.lo > 0 ? it.lo : 0;
  it.c0 = tk.tile_begin * kTileTokens;
  it.t0 = it.c0;
  const int t1 = tk.tile_end * kTileTokens;
  it.t1 = t1 < it.L ? t1 : it.L;
  it.btrow = p.bt + (int64_t)it.s * p.bt_stride;
  it.bx0 = -1;
}

// Block of this warp's box ordinal `o` in the task (slice o / bps, box o % bps; 0 past
// the context).
template <class C>
__device__ __forceinline__ int it_bt(const SliceIt& it, int o, int r0, int box_shift, int page_shift) {
  const int bps_shift = (__ffs(C::TW) - 1) - box_shift;  // boxes per slice = 2^bps_shift
  const int n = o >> bps_shift, b = o & ((1 << bps_shift) - 1);
  const int tok = it.t0 + n * C::TC + r0 + (b << box_shift);
  return tok < it.L ? it.btrow[tok >> page_shift] : 0;
}

// Advance to the first slice at or after the current one that holds tokens, and take
// the blocks of its boxes from the warp's block-table window: entries for 32 boxes per
// load, one per lane, the next 32 in flight while these are used.
template <class C>
__device__ __forceinline__ void it_settle(SliceIt& it, const DecodeParams& p, int t_end, int r0,
                                          int lane, int box_shift, int page_shift) {
  while (!it.done && it.c0 + r0 >= it.t1) {
    if (++it.task >= t_end) {
      it.done = true;
      return;
    }
    it_load_task(it, p);
  }
  if (it.done) return;
  if (it.bx0 < 0) {
    it.bx0 = 0;
    it.bcur = it_bt<C>(it, lane, r0, box_shift, page_shift);
    it.bnxt = it_bt<C>(it, 32 + lane, r0, box_shift, page_shift);
  }
  const int bps_shift = (__ffs(C::TW) - 1) - box_shift;
  const int o0 = ((it.c0 - it.t0) / C::TC) << bps_shift;  // first box of this slice
  if (o0 >= it.bx0 + 32) {  // boxes per slice divide 32: a slice never straddles windows
    it.bx0 += 32;
    it.bcur = it.bnxt;
    it.bnxt = it_bt<C>(it, it.bx0 + 32 + lane, r0, box_shift, page_shift);
  }
  const int idx = o0 + lane - it.bx0;
  const int from_cur = __shfl_sync(0xffffffffu, it.bcur, idx & 31);
  const int from_nxt = __shfl_sync(0xffffffffu, it.bnxt, idx & 31);
  it.blk = idx < 32 ? from_cur : from_nxt;
}

// Issue the TMA / bulk copies of one warp slice (tokens [a, min(a + TW, L)) of the
// iterator's sequence and KV head) into ring slot `kv` / `sc`, completing on `bar`.
// Boxes that end at or before the first token of any sliding window are not loaded
// (their slot rows keep stale bytes, which the masked path never lets through).
template <class C>
__device__ __forceinline__ void issue_slice(const DecodeParams& p, const CUtensorMap* tmk,
                                            const CUtensorMap* tmv, uint8_t* kv, uint8_t* sc,
                                            uint64_t* bar, const SliceIt& it, int r0, int dw,
                                            int lane, int box_shift, int page_mask) {
  const int a = it.c0 + r0;
  const int ntok = (it.L - a) < C::TW ? (it.L - a) : C::TW;
  const int box = 1 << box_shift;
  const int nbox = (ntok + box - 1) >> box_shift;
  int fbox = it.lo > a ? (it.lo - a) >> box_shift : 0;  // boxes wholly before the window
  fbox = fbox < nbox ? fbox : nbox;
  if (lane == 0)
    mbar_arrive_expect_tx(bar, (uint32_t)(((nbox - fbox) << box_shift) *
                                          (2 * C::NSUBW * C::SUB + (C::SCALES ? 8 : 0))));
  __syncwarp();
  if (lane >= fbox && lane < nbox) {
    fence_proxy_async();  // the slot was last read through the generic proxy
    const int tok = a + (lane << box_shift);
    int blk = it.blk;
    blk = blk < 0 ? 0 : (blk >= p.NB ? p.NB - 1 : blk);
    const int slot = tok & page_mask;
#pragma unroll
    for (int u = 0; u < C::NSUBW; ++u) {
      const int sub = dw * C::NSUBW + u;
      const int dst = u * (C::TW * C::SUB) + ((lane << box_shift) * C::SUB);
      tma_load_4d(kv + dst, tmk, bar, sub * C::SUB, slot, it.hkv, blk);
      if constexpr (!C::TRV) tma_load_4d(kv + C::SLOT_V + dst, tmv, bar, sub * C::SUB, slot, it.hkv, blk);
    }
    // transposed V: this box is the 16-token piece `lane`, head dims [dw * DW, dw * DW + DW)
    if constexpr (C::TRV) tma_load_4d(kv + C::SLOT_V + lane * C::PIECE_V, tmv, bar, slot, dw * C::DW, it.hkv, blk);
    if constexpr (C::SCALES) {
      const int64_t off = (int64_t)blk * p.sc_sb + (int64_t)it.hkv * p.sc_sh + (int64_t)slot * 4;
      bulk_load(sc + (lane << box_shift) * 4, p.k_scale + off, box * 4, bar);
      bulk_load(sc + 4 * C::TW + (lane << box_shift) * 4, p.v_scale + off, box * 4, bar);
    }
  }
}

// Per-warp softmax and accumulator state of one task.
template <class C>
struct WarpAcc {
  float o[C::MT][C::NTD][4];
  float m[C::MT][2];  // running max (log2 units); probabilities are exp2(s - m) <= 2^kLazyLog2
  float l[C::MT][2];  // thread-partial running sum
  float vref;         // fp8 per-token: V-scale reference (probabilities carry v_scale / vref)
  float vinv;         // 1 / vref (0 while no reference)
  int emax[C::NBLK];  // MXFP4: V e8m0 reference per 32-dim block (-1: none yet)
};

// The running max is only raised when a slice's max exceeds it by more than 2^kLazyLog2
// (probabilities stay <= 256, inside the f16 / bf16 range); the V-scale references move
// only by more than 8x.  Slices that raise nothing skip the accumulator rescale.
constexpr float kLazyLog2 = 8.f;
constexpr float kLazyVref = 8.f;
constexpr int kLazyExp = 3;

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Both halves of a 32-bit word, each two e4m3 values, to two f16x2 words.
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 h0, h1;\n\t"
      "mov.b32 {h0, h1}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, h0;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h1;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// m16n8k16 f16 MMA with a zero accumulator input.
__device__ __forceinline__ void mma_f16_zc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                           uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7},"
      " {%8, %9}, {%10, %10, %10, %10};"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.f));
}

// One slice of one warp: QK^T, online softmax, PV over the slice's tokens.  MASKED is
// the boundary path (tokens >= vw are unowned; with a sliding window, tokens before
// wl - (qm1 - i) are outside query position i's window, and tokens before wl - qm1 are
// outside every window); full slices run no masking instruction.
template <class C, bool MASKED>
__device__ __forceinline__ void stage_compute(
    WarpAcc<C>& A, const uint8_t* kv, const uint8_t* sc, uint8_t* smem, int vw, int lane, int dw,
    int tg, const uint32_t (&qa)[C::Q_IN_REGS ? C::MT : 1][C::Q_IN_REGS ? C::NKCH : 1][4],
    const uint16_t* qs, const float (&crow)[C::MT][2], const uint32_t (&koff)[C::KOFFN],
    const uint32_t (&voff)[C::NCP], int cw, int& xbuf, int cq, int G, int wl, int qm1) {
  constexpr bool tok_scale = C::TOK_SCALE;
  const int g = lane >> 2, t = lane & 3;
  const uint32_t kbase = smem_u32(kv);
  const uint32_t vbase = kbase + C::SLOT_V;
  const int vlo = wl - qm1;  // tokens before vlo: outside every window (stale slot rows)
  const float* ksc = reinterpret_cast<const float*>(sc);
  const float* vsc = reinterpret_cast<const float*>(sc + 4 * C::TW);
  const uint32_t* kex = reinterpret_cast<const uint32_t*>(sc);
  const uint32_t* vex = reinterpret_cast<const uint32_t*>(sc + 4 * C::TW);
  float* ktab = reinterpret_cast<float*>(smem + C::OFF_TAB + cw * C::TAB_BYTES);
  uint16_t* vtab = reinterpret_cast<uint16_t*>(ktab + C::NBLK * C::TW);

  // ---------------- fp8 per-token V-scale reference (lazy) ----------------
  float beta[C::NBLK];
#pragma unroll
  for (int b = 0; b < C::NBLK; ++b) beta[b] = 1.f;
  bool rescale_v = false;
  float vinv = 1.f;
  if constexpr (tok_scale) {
    static_assert(C::TW <= 32, "one lane per slice token");
    // |v_scale| of owned tokens; non-negative floats order like their bit patterns.  The
    // reference moves only when a token passes it by more than kLazyVref: one vote decides,
    // the maximum is reduced only then.
    const float vs =
        (lane < C::TW && (!MASKED || (lane < vw && lane >= vlo))) ? fabsf(vsc[lane]) : 0.f;
    if (__any_sync(0xffffffffu, vs > A.vref * kLazyVref)) {
      const float mx = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(vs)));
      beta[0] = A.vref / mx;
      A.vref = mx;
      A.vinv = 1.f / mx;
      rescale_v = true;
    }
    vinv = A.vinv;
  }
  if constexpr (C::KIND == KIND_FP4) {
    // K: this lane's token's block factors 2^(e-127) x kKFactorBias (the row's logit factor
    // carries the inverse), read back per score pair after the MMAs; an unowned token's
    // scores are overwritten by the boundary mask
    const uint32_t kw = kex[lane];
#pragma unroll
    for (int b = 0; b < C::NBLK; ++b)
      ktab[b * C::TW + lane] = __uint_as_float(((kw >> (8 * b)) & 0xFFu) << 23) * kKFactorBias;
    __syncwarp();
  }
  // ---------------- S = Q K^T over this warp's dims ----------------
  float sacc[C::MT][C::NT][4];
  // fp8 with one m-tile: odd k-chunks accumulate separately (two independent MMA chains
  // per n-tile); the split is summed once before the softmax
  constexpr bool kSplit = C::KIND == KIND_FP8 && C::MT == 1;
  float sacc2[kSplit ? C::MT : 1][kSplit ? C::NT : 1][4];
#pragma unroll
  for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        sacc[mt][nt][j] = 0.f;
        if constexpr (kSplit) sacc2[mt][nt][j] = 0.f;
      }
#pragma unroll
  for (int gi = 0; gi < C::NGRP; ++gi) {
    uint32_t kr[C::NT][4];
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt) {
      if constexpr (C::TRV)  // even / odd n-tiles of a 16-token chunk read their own rows
        ldsm_x4(kbase + koff[(nt & 1) * C::NGRP + gi] + (nt >> 1) * 16 * C::SUB, kr[nt]);
      else
        ldsm_x4(kbase + koff[gi] + nt * 8 * C::SUB, kr[nt]);
    }
    if constexpr (C::KIND == KIND_BF16) {
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
          uint32_t a[4];
          if constexpr (C::Q_IN_REGS) {
#pragma unroll
            for (int z = 0; z < 4; ++z) a[z] = qa[mt][2 * gi + h][z];
          } else {
            load_qa<C>(qs, mt, 2 * gi + h, dw, g, t, a);
          }
#pragma unroll
          for (int nt = 0; nt < C::NT; ++nt) mma_bf16(sacc[mt][nt], a, kr[nt][2 * h], kr[nt][2 * h + 1]);
        }
    } else if constexpr (C::KIND == KIND_FP8) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
          uint32_t a[4];
          if constexpr (C::Q_IN_REGS) {
#pragma unroll
            for (int z = 0; z < 4; ++z) a[z] = qa[mt][4 * gi + q][z];
          } else {
            load_qa<C>(qs, mt, 4 * gi + q, dw, g, t, a);
          }
#pragma unroll
          for (int nt = 0; nt < C::NT; ++nt) {
            uint32_t b0, b1;
            e4m3x4_to_f16x2(kr[nt][q], b0, b1);
            if (kSplit && (q & 1))
              mma_f16(sacc2[kSplit ? mt : 0][kSplit ? nt : 0], a, b0, b1);
            else
              mma_f16(sacc[mt][nt], a, b0, b1);
          }
        }
    } else {
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        float tmp[C::MT][C::NT][4];
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt) {
          uint32_t f[4];
          e2m1x8_to_f16x2(kr[nt][b], f);
#pragma unroll
          for (int mt = 0; mt < C::MT; ++mt) mma_f16_zc(tmp[mt][nt], qa[mt][2 * b], f[0], f[1]);
#pragma unroll
          for (int mt = 0; mt < C::MT; ++mt) mma_f16(tmp[mt][nt], qa[mt][2 * b + 1], f[2], f[3]);
        }
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt) {
          const float2 kf = *reinterpret_cast<const float2*>(ktab + b * C::TW + 8 * nt + 2 * t);
#pragma unroll
          for (int mt = 0; mt < C::MT; ++mt) {
            sacc[mt][nt][0] = fmaf(tmp[mt][nt][0], kf.x, sacc[mt][nt][0]);
            sacc[mt][nt][1] = fmaf(tmp[mt][nt][1], kf.y, sacc[mt][nt][1]);
            sacc[mt][nt][2] = fmaf(tmp[mt][nt][2], kf.x, sacc[mt][nt][2]);
            sacc[mt][nt][3] = fmaf(tmp[mt][nt][3], kf.y, sacc[mt][nt][3]);
          }
        }
      }
    }
  }
  if constexpr (kSplit) {
#pragma unroll
    for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
      for (int j = 0; j < 4; ++j) sacc[0][nt][j] += sacc2[0][nt][j];
  }
  // ---------------- combine the head-dim parts of the token group ----------------
  // Every warp of the group adds the NDW partial scores in the same order (part 0 first),
  // so all of them hold the same scores and run the same softmax.
  if constexpr (C::NDW > 1) {
    float* xb = reinterpret_cast<float*>(smem + C::OFF_X);
    const float* parts = xb + (tg * C::XBUFS + xbuf) * C::NDW * C::XW;
    float* mine = const_cast<float*>(parts) + dw * C::XW;
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) mine[((mt * C::NT + nt) * 4 + j) * 32 + lane] = sacc[mt][nt][j];
    named_bar(1 + tg, C::NDW * 32);
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
      for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int e = ((mt * C::NT + nt) * 4 + j) * 32 + lane;
          float x = dw == 0 ? sacc[mt][nt][j] : parts[e];
#pragma unroll
          for (int i = 1; i < C::NDW; ++i) x = x + (dw == i ? sacc[mt][nt][j] : parts[i * C::XW + e]);
          sacc[mt][nt][j] = x;
        }
    if constexpr (C::XBUFS == 1)
      named_bar(1 + tg, C::NDW * 32);  // one buffer: every part read before the next slice
    else
      xbuf ^= 1;
  }
  // ---------------- MXFP4 V references (lazy) and factor table ----------------
  if constexpr (C::KIND == KIND_FP4) {
    const bool own = !MASKED || (lane < vw && lane >= vlo);  // one lane per slice token
    const uint32_t vwd = vex[lane];
    // A reference moves when none is set yet or a token's exponent passes it by more than
    // kLazyExp: one vote decides; the block maxima are reduced only then.
    bool over = false;
#pragma unroll
    for (int b = 0; b < C::NBLK; ++b)
      over |= A.emax[b] < 0 || (own && (int)((vwd >> (8 * b)) & 0xFF) > A.emax[b] + kLazyExp);
    if (__any_sync(0xffffffffu, over)) {
#pragma unroll
      for (int b = 0; b < C::NBLK; ++b) {
        const uint32_t e = (vwd >> (8 * b)) & 0xFF;
        const int cm = (int)__reduce_max_sync(0xffffffffu, own ? e : 0u);
        const int ne = max(A.emax[b], cm);
        beta[b] = A.emax[b] < 0 ? 0.f : exp2i(A.emax[b] - ne);
        A.emax[b] = ne;
      }
      rescale_v = true;
    }
    // V: 2^(e-emax) as f16 (factors below 2^-14 flush to zero: such a block is at least
    // 2^14 times smaller than the largest one seen for that block); 0 for unowned tokens
    const uint32_t kown = own ? 0xFFFFFFFFu : 0u;
#pragma unroll
    for (int b = 0; b < C::NBLK; ++b) {
      const int ev = (int)((vwd >> (8 * b)) & 0xFF);
      vtab[b * C::TW + lane] = (uint16_t)(((uint32_t)max(ev - A.emax[b] + 15, 0) << 10) & kown);
    }
    __syncwarp();
  }

  // ---------------- logits and boundary mask ----------------
  // Row limits: tokens at or past vw are unowned; with causal masking (cq = qlen - 1 > 0)
  // query position i = row / G sees only the tokens before vw - (cq - i), and with a
  // sliding window only those from wl - (qm1 - i) on.
  int lim[C::MT][2], low[C::MT][2];
#pragma unroll
  for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int i = (16 * mt + g + 8 * hr) / G;
      lim[mt][hr] = MASKED ? vw - (cq > i ? cq - i : 0) : vw;
      low[mt][hr] = MASKED ? wl - (qm1 - i) : 0;
    }
#pragma unroll
  for (int nt = 0; nt < C::NT; ++nt) {
    const int tk0 = 16 * (nt >> 1) + kv_token<C>(8 * (nt & 1) + 2 * t);  // its pair: tk0, tk0 + 1
    float2 ks = make_float2(1.f, 1.f);
    if constexpr (tok_scale) ks = *reinterpret_cast<const float2*>(ksc + tk0);
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float x = sacc[mt][nt][j] * crow[mt][j >> 1];
        if constexpr (tok_scale) x *= (j & 1) ? ks.y : ks.x;
        if (MASKED && (tk0 + (j & 1) >= lim[mt][j >> 1] || tk0 + (j & 1) < low[mt][j >> 1]))
          x = -INFINITY;
        sacc[mt][nt][j] = x;
      }
  }
  // ---------------- online softmax with a lazily raised max ----------------
  float mx[C::MT][2];
  bool need = false;
#pragma unroll
  for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      float vt[C::NT];
#pragma unroll
      for (int nt = 0; nt < C::NT; ++nt) vt[nt] = fmaxf(sacc[mt][nt][2 * hr], sacc[mt][nt][2 * hr + 1]);
#pragma unroll
      for (int w = 1; w < C::NT; w <<= 1)
#pragma unroll
        for (int nt = 0; nt + w < C::NT; nt += 2 * w) vt[nt] = fmaxf(vt[nt], vt[nt + w]);
      float v = vt[0];
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 1));
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 2));
      mx[mt][hr] = v;
      need |= v > A.m[mt][hr] + kLazyLog2;
    }
  need = __any_sync(0xffffffffu, need);
  float alpha[C::MT][2];
#pragma unroll
  for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      alpha[mt][hr] = 1.f;
      if (need) {
        const float mn = fmaxf(A.m[mt][hr], mx[mt][hr]);
        if (mn != A.m[mt][hr]) {
          alpha[mt][hr] = fast_exp2(A.m[mt][hr] - mn);  // -inf -> 0
          A.m[mt][hr] = mn;
          A.l[mt][hr] *= alpha[mt][hr];
        }
      }
      const float base = A.m[mt][hr] == -INFINITY ? 0.f : A.m[mt][hr];
      float rt[C::NT];
#pragma unroll
      for (int nt = 0; nt < C::NT; ++nt) {
        const float p0 = fast_exp2(sacc[mt][nt][2 * hr] - base);
        const float p1 = fast_exp2(sacc[mt][nt][2 * hr + 1] - base);
        sacc[mt][nt][2 * hr] = p0;
        sacc[mt][nt][2 * hr + 1] = p1;
        rt[nt] = p0 + p1;
      }
#pragma unroll
      for (int w = 1; w < C::NT; w <<= 1)
#pragma unroll
        for (int nt = 0; nt + w < C::NT; nt += 2 * w) rt[nt] += rt[nt + w];
      A.l[mt][hr] += rt[0];
    }
  if (need || rescale_v) {
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
      for (int n = 0; n < C::NTD; ++n) {
        const float bb = C::KIND == KIND_FP4 ? beta[n >> 2] : beta[0];
        const float f0 = alpha[mt][0] * bb, f1 = alpha[mt][1] * bb;
        A.o[mt][n][0] *= f0;
        A.o[mt][n][1] *= f0;
        A.o[mt][n][2] *= f1;
        A.o[mt][n][3] *= f1;
      }
  }
  // ---------------- O += P V ----------------
#pragma unroll
  for (int kc = 0; kc < C::NKC; ++kc) {
    if (MASKED && 16 * kc >= vw) break;
    // tokens of this lane's low (k = 2t, 2t + 1) and high (k = 2t + 8, 2t + 9) pairs
    const int tb = 16 * kc + kv_token<C>(2 * t), th = 16 * kc + kv_token<C>(8 + 2 * t);
    uint32_t mlo = 0xFFFFFFFFu, mhi = 0xFFFFFFFFu;
    // a token's V row passes if it is owned and inside some window
    auto in = [&](int x) { return x < vw && x >= vlo; };
    if (MASKED) {
      mlo = (in(tb) ? 0x0000FFFFu : 0u) | (in(tb + 1) ? 0xFFFF0000u : 0u);
      mhi = (in(th) ? 0x0000FFFFu : 0u) | (in(th + 1) ? 0xFFFF0000u : 0u);
    }
    uint32_t pa[C::MT][4];
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt) {
      const float* pl = sacc[mt][2 * kc];
      const float* ph = sacc[mt][2 * kc + 1];
      if constexpr (C::KIND == KIND_BF16) {
        pa[mt][0] = pack_bf16x2(pl[0], pl[1]);
        pa[mt][1] = pack_bf16x2(pl[2], pl[3]);
        pa[mt][2] = pack_bf16x2(ph[0], ph[1]);
        pa[mt][3] = pack_bf16x2(ph[2], ph[3]);
      } else if constexpr (tok_scale) {
        const float2 a = *reinterpret_cast<const float2*>(vsc + tb);
        const float2 c = *reinterpret_cast<const float2*>(vsc + th);
        const float vf0 = (MASKED && !in(tb)) ? 0.f : a.x * vinv;
        const float vf1 = (MASKED && !in(tb + 1)) ? 0.f : a.y * vinv;
        const float vf2 = (MASKED && !in(th)) ? 0.f : c.x * vinv;
        const float vf3 = (MASKED && !in(th + 1)) ? 0.f : c.y * vinv;
        pa[mt][0] = pack_f16x2(pl[0] * vf0, pl[1] * vf1);
        pa[mt][1] = pack_f16x2(pl[2] * vf0, pl[3] * vf1);
        pa[mt][2] = pack_f16x2(ph[0] * vf2, ph[1] * vf3);
        pa[mt][3] = pack_f16x2(ph[2] * vf2, ph[3] * vf3);
      } else {
        pa[mt][0] = pack_f16x2(pl[0], pl[1]);
        pa[mt][1] = pack_f16x2(pl[2], pl[3]);
        pa[mt][2] = pack_f16x2(ph[0], ph[1]);
        pa[mt][3] = pack_f16x2(ph[2], ph[3]);
      }
    }
    if constexpr (C::TRV) {
      // piece kc, head-dim rows of 16 bytes: lane 8q + j points at row 32 cp + 8q + j and
      // gets tokens 4t .. 4t + 3 of head dim 8 (4 cp + q) + g, the B-fragment of n-tile 4 cp + q
#pragma unroll
      for (int cp = 0; cp < C::NTD / 4; ++cp) {
        uint32_t v[4];
        ldsm_x4(vbase + kc * C::PIECE_V + (32 * cp + lane) * 16, v);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t b0, b1;
          e4m3x4_to_f16x2(v[q], b0, b1);
          if (MASKED) {
            b0 &= mlo;
            b1 &= mhi;
          }
#pragma unroll
          for (int mt = 0; mt < C::MT; ++mt) mma_f16(A.o[mt][4 * cp + q], pa[mt], b0, b1);
        }
      }
      continue;
    }
#pragma unroll
    for (int cp = 0; cp < C::NCP; ++cp) {
      uint32_t v[4];
      ldsm_x4_t(vbase + voff[cp] + 16 * kc * C::SUB, v);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int ch = 2 * cp + c;  // 16-byte chunk of the warp's row slice
        if constexpr (C::KIND == KIND_BF16) {
          const uint32_t b0 = MASKED ? v[2 * c] & mlo : v[2 * c];
          const uint32_t b1 = MASKED ? v[2 * c + 1] & mhi : v[2 * c + 1];
#pragma unroll
          for (int mt = 0; mt < C::MT; ++mt) mma_bf16(A.o[mt][ch], pa[mt], b0, b1);
        } else if constexpr (C::KIND == KIND_FP8) {
          uint32_t bA0, bB0, bA1, bB1;
          e4m3x4_to_f16x2(prmt(v[2 * c], v[2 * c], 0x3120), bA0, bB0);
          e4m3x4_to_f16x2(prmt(v[2 * c + 1], v[2 * c + 1], 0x3120), bA1, bB1);
          if (MASKED) {
            bA0 &= mlo;
            bB0 &= mlo;
            bA1 &= mhi;
            bB1 &= mhi;
          }
#pragma unroll
          for (int mt = 0; mt < C::MT; ++mt) {
            mma_f16(A.o[mt][2 * ch], pa[mt], bA0, bA1);
            mma_f16(A.o[mt][2 * ch + 1], pa[mt], bB0, bB1);
          }
        } else {
          // V block `ch`: its e8m0 factors (relative to emax[ch]) go into P, in f16
          const uint32_t vp0 = *reinterpret_cast<const uint32_t*>(vtab + ch * C::TW + tb);
          const uint32_t vp1 = *reinterpret_cast<const uint32_t*>(vtab + ch * C::TW + tb + 8);
          uint32_t pb[C::MT][4];
#pragma unroll
          for (int mt = 0; mt < C::MT; ++mt) {
            pb[mt][0] = hmul2(pa[mt][0], vp0);
            pb[mt][1] = hmul2(pa[mt][1], vp0);
            pb[mt][2] = hmul2(pa[mt][2], vp1);
            pb[mt][3] = hmul2(pa[mt][3], vp1);
          }
          uint32_t fl[4], fh[4];
          e2m1x8_to_f16x2(v[2 * c], fl);
          e2m1x8_to_f16x2(v[2 * c + 1], fh);
          uint32_t b0[4] = {prmt(fl[0], fl[2], 0x5410), prmt(fl[0], fl[2], 0x7632),
                            prmt(fl[1], fl[3], 0x5410), prmt(fl[1], fl[3], 0x7632)};
          uint32_t b1[4] = {prmt(fh[0], fh[2], 0x5410), prmt(fh[0], fh[2], 0x7632),
                            prmt(fh[1], fh[3], 0x5410), prmt(fh[1], fh[3], 0x7632)};
          if (MASKED) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              b0[i] &= mlo;
              b1[i] &= mhi;
            }
          }
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt) mma_f16(A.o[mt][4 * ch + i], pb[mt], b0[i], b1[i]);
        }
      }
    }
  }
}

// Merge partitions [base, base + nparts) of the split unit (s, hkv) in partition order with
// the reduce kernel's formula and store its bf16 rows [r0, r1); every thread of the CTA
// takes part.
template <class C>
__device__ void merge_partials(const DecodeParams& p, float* obuf, int s, int hkv, int64_t base,
                               int nparts, int cw, int lane, int r0, int r1) {
    const float2* pml = reinterpret_cast<const float2*>(p.part_ml);
    float* wts = obuf;  // normalised weights [R][nparts] (nparts <= 128 <= OBW)
    // one warp per row: lanes over partitions, shuffle-tree max and sum
    for (int r = r0 + cw; r < r1; r += C::NCW) {
      float M = -INFINITY;
      for (int q = lane; q < nparts; q += 32) M = fmaxf(M, __ldcg(&pml[(base + q) * p.R + r]).x);
#pragma unroll
      for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      const float mb = M == -INFINITY ? 0.f : M;
      float W = 0.f;
      for (int q = lane; q < nparts; q += 32) {
        const float2 e = __ldcg(&pml[(base + q) * p.R + r]);
        const float w = e.y * fast_exp2(e.x - mb);
        wts[r * nparts + q] = w;
        W += w;
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
      if (p.sinks != nullptr && W > 0.f) W += fast_exp2(p.sinks[hkv * p.G + r % p.G] * kLog2e - mb);
      const float inv = W > 0.f ? 1.f / W : 0.f;
      __syncwarp();
      for (int q = lane; q < nparts; q += 32) wts[r * nparts + q] *= inv;
    }
    named_bar(BAR_CONSUMERS, C::NCW * 32);
    // float4 columns, partitions in order; loads are independent of the sum
    const float4* po4 = reinterpret_cast<const float4*>(p.part_o);
    for (int idx = threadIdx.x + r0 * (C::D / 4); idx < r1 * (C::D / 4); idx += C::NTHREADS) {
      const int r = idx / (C::D / 4), d4 = idx % (C::D / 4);
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      int q = 0;
      for (; q + 4 <= nparts; q += 4) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u] = __ldcg(&po4[((base + q + u) * p.R + r) * (C::D / 4) + d4]);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float w = wts[r * nparts + q + u];
          acc.x += w * v[u].x;
          acc.y += w * v[u].y;
          acc.z += w * v[u].z;
          acc.w += w * v[u].w;
        }
      }
      for (; q < nparts; ++q) {
        const float4 v = __ldcg(&po4[((base + q) * p.R + r) * (C::D / 4) + d4]);
        const float w = wts[r * nparts + q];
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
      }
      const int i = r / p.G, h = hkv * p.G + r % p.G;
      __nv_bfloat16* dst = p.out + ((int64_t)s * p.qlen + i) * p.o_st + (int64_t)h * p.o_sh + 4 * d4;
      dst[0] = __float2bfloat16_rn(acc.x);
      dst[1] = __float2bfloat16_rn(acc.y);
      dst[2] = __float2bfloat16_rn(acc.z);
      dst[3] = __float2bfloat16_rn(acc.w);
    }
}

template <class C>
__device__ void warp_main(const DecodeParams& p, const CUtensorMap* tmk, const CUtensorMap* tmv,
                          uint8_t* smem, uint64_t* full, volatile int* abort_flag,
                          const PlanTask* tasks, int t_begin, int t_end, int pf_nparts,
                          int pf_pbase, int cw, int lane) {
  const int tg = cw / C::NDW, dw = cw % C::NDW;
  const int g = lane >> 2, t = lane & 3;
  const int r0 = tg * C::TW;  // this warp's slice inside a CTA stage
  const uint16_t* qs = reinterpret_cast<const uint16_t*>(smem + C::OFF_Q);
  const float* cr = reinterpret_cast<const float*>(smem + C::OFF_CR);
  float* obuf = reinterpret_cast<float*>(smem + C::OFF_OB);
  float2* ml = reinterpret_cast<float2*>(smem + C::OFF_ML);
  uint8_t* ring = smem + C::OFF_RING + cw * C::NSTAGE * C::SLOT_KV;
  uint8_t* scring = smem + C::OFF_SC + cw * C::NSTAGE * C::SLOT_SC;
  uint64_t* bars = full + cw * C::NSTAGE;
  const float k_scale_tensor = (C::KIND == KIND_FP8 && C::SKT == SK_TENSOR)
                                   ? reinterpret_cast<const float*>(p.k_scale)[0] : 1.f;
  const float v_scale_tensor = (C::KIND == KIND_FP8 && C::SKT == SK_TENSOR)
                                   ? reinterpret_cast<const float*>(p.v_scale)[0] : 1.f;
  const int page_shift = __ffs(p.S) - 1;  // page sizes are powers of two
  // boxes: a page piece of at most one slice; 16 tokens with transposed V (pages >= 16)
  const int box_shift = C::TRV ? 4 : (p.S < C::TW ? page_shift : __ffs(C::TW) - 1);
  const int page_mask = p.S - 1;
  if (lane == 0) {
    tma_prefetch_desc(tmk);
    tma_prefetch_desc(tmv);
  }
  // Per-lane byte offsets of the ldmatrix rows inside a slot (the swizzle phase of a row
  // depends only on its index modulo 8, i.e. on the lane).
  uint32_t koff[C::KOFFN], voff[C::NCP];
  {
    const int j = lane & 7, q = lane >> 3;
#pragma unroll
    for (int par = 0; par < C::KOFFN / C::NGRP; ++par) {
      const int row = kv_token<C>(8 * par + j);  // token row of score column 8 par + j
#pragma unroll
      for (int gi = 0; gi < C::NGRP; ++gi) {
        const int off = gi * 64 + q * 16;
        const int u = off / C::SUB, cin = (off % C::SUB) >> 4;
        koff[par * C::NGRP + gi] = u * (C::TW * C::SUB) + row * C::SUB + ((cin ^ swz<C>(row)) << 4);
      }
    }
#pragma unroll
    for (int cp = 0; cp < C::NCP; ++cp) {
      const int off = (2 * cp + (q >> 1)) * 16;
      const int u = off / C::SUB, cin = (off % C::SUB) >> 4;
      const int row = 8 * (q & 1) + j;
      voff[cp] = u * (C::TW * C::SUB) + row * C::SUB + ((cin ^ swz<C>(row)) << 4);
    }
  }

  QRaw<C> qn;  // query words of the next task to start
  if constexpr (C::Q_EARLY) {
    if (t_begin < t_end) {
      const PlanTask tk0 = tasks[t_begin];
      load_q_issue<C>(p, tk0.seq, tk0.hkv_part & 0xFFFF, cw, lane, qn);
    }
  }
  // prologue: fill the ring
  SliceIt ld;
  ld.tasks = tasks;
  ld.task = t_begin;
  ld.done = ld.task >= t_end;
  ld.blk = 0;
  if (!ld.done) it_load_task(ld, p);
  it_settle<C>(ld, p, t_end, r0, lane, box_shift, page_shift);
  uint32_t issued = 0, consumed = 0;
  // abort_at: consumption index of this warp's first wait that gave up (or that it skipped
  // because another warp of the CTA gave up); from there on it issues no load, and before
  // leaving it waits, with a limit, for every slice it issued but did not wait for.
  volatile uint32_t* abort_at = reinterpret_cast<volatile uint32_t*>(smem + C::OFF_ABT) + cw;
  int lslot = 0;  // ring slot of the next load
  while (!ld.done && issued < (uint32_t)C::NSTAGE) {
    // (test hook: with drop_first_slice, warp 0 of every CTA leaves its first slot empty,
    // so the wait for it gives up after its time limit and the status reports the timeout)
    if (!(p.drop_first_slice && cw == 0 && issued == 0))
      issue_slice<C>(p, tmk, tmv, ring + lslot * C::SLOT_KV, scring + lslot * C::SLOT_SC,
                     &bars[lslot], ld, r0, dw, lane, box_shift, page_mask);
    ++issued;
    lslot = lslot + 1 == C::NSTAGE ? 0 : lslot + 1;
    ld.c0 += C::TC;
    it_settle<C>(ld, p, t_end, r0, lane, box_shift, page_shift);
  }
  int cslot = 0;      // ring slot of the next compute
  uint32_t cpar = 0;  // its phase parity
  int xbuf = 0;
  // tokens a query position may not see past (MXFP4 takes one query position: none)
  const int cq = (C::KIND != KIND_FP4 && p.causal) ? p.qlen - 1 : 0;
  const int qm1 = C::KIND != KIND_FP4 ? p.qlen - 1 : 0;
  // a slice runs the full path only if it starts inside every position's window
  const int wcap = p.window > 0 ? p.window : 0x7FFFFFFF;

  for (int task = t_begin; task < t_end; ++task) {
    const PlanTask tk = tasks[task];
    const int s = tk.seq, hkv = tk.hkv_part & 0xFFFF, part = tk.hkv_part >> 16;
    const int L = clamped_context(p, s);
    const int t0 = tk.tile_begin * kTileTokens;
    int t1 = tk.tile_end * kTileTokens;
    t1 = t1 < L ? t1 : L;
    const int unit = s * p.Hkv + hkv;
    const int nparts = p.pf_split > 0 ? pf_nparts : p.nparts[unit];
    const int64_t slot = nparts > 1 ? (int64_t)(p.pf_split > 0 ? pf_pbase : p.part_base[unit]) + part : 0;

    if constexpr (!C::Q_EARLY) load_q_issue<C>(p, s, hkv, cw, lane, qn);
    load_q_finish<C>(p, smem, qn, cw, lane, k_scale_tensor);
    named_bar(BAR_CONSUMERS, C::NCW * 32);
    // The next task's record, read at this task's merge, copied without waiting for it.
    if (C::Q_EARLY && task + 1 < t_end && cw == 0 && lane == 0) {
      cp_async16(smem + C::OFF_NXT, tasks + task + 1);
      cp_async_commit();
    }
    // Touch this task's output rows now, so that their address translation is not first
    // needed by the stores at the end of the task, with the memory system under load.
    if (cw == 0 && lane == 0) {
      if (nparts > 1) {
        prefetch_l2(p.part_o + slot * p.R * C::D);
        prefetch_l2(p.part_ml + 2 * slot * p.R);
      } else {
        prefetch_l2(p.out + (int64_t)s * p.qlen * p.o_st + (int64_t)hkv * p.G * p.o_sh);
      }
    }

    uint32_t qa[C::Q_IN_REGS ? C::MT : 1][C::Q_IN_REGS ? C::NKCH : 1][4];
    if constexpr (C::Q_IN_REGS) {
#pragma unroll
      for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
        for (int k = 0; k < C::NKCH; ++k) load_qa<C>(qs, mt, k, dw, g, t, qa[mt][k]);
    }
    float crow[C::MT][2];
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt) {
      crow[mt][0] = cr[16 * mt + g];
      crow[mt][1] = cr[16 * mt + g + 8];
    }

    WarpAcc<C> A;
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt) {
#pragma unroll
      for (int n = 0; n < C::NTD; ++n)
#pragma unroll
        for (int j = 0; j < 4; ++j) A.o[mt][n][j] = 0.f;
      A.m[mt][0] = A.m[mt][1] = -INFINITY;
      A.l[mt][0] = A.l[mt][1] = 0.f;
    }
    A.vref = 0.f;
    A.vinv = 0.f;
#pragma unroll
    for (int b = 0; b < C::NBLK; ++b) A.emax[b] = -1;

    for (int c0 = t0; c0 + r0 < t1; c0 += C::TC) {
      bool stop = *abort_flag;  // this warp loads nothing more once set
      if (!stop) {
        if (!mbar_wait_bounded(&bars[cslot], cpar)) {
          *abort_flag = 1;
          if (lane == 0) atomicOr(p.status, ST_TIMEOUT);
          *abort_at = consumed;
          stop = true;
        }
      } else if (*abort_at == kNoAbort) {
        *abort_at = consumed;
      }
      const uint8_t* kv = ring + cslot * C::SLOT_KV;
      const uint8_t* sc = scring + cslot * C::SLOT_SC;
      const int vw = L - (c0 + r0);  // owned tokens in the slice (> 0 here)
      if (vw - cq >= C::TW && vw <= wcap) {
        stage_compute<C, false>(A, kv, sc, smem, vw, lane, dw, tg, qa, qs, crow, koff, voff, cw,
                                xbuf, cq, p.G, 0, qm1);
      } else {
        // the last query position's window starts at slice token vw - window
        const int wl = p.window > 0 ? vw - p.window : -0x40000000;
        stage_compute<C, true>(A, kv, sc, smem, vw, lane, dw, tg, qa, qs, crow, koff, voff, cw,
                               xbuf, cq, p.G, wl, qm1);
      }
      const int done_slot = cslot;
      ++consumed;
      if (++cslot == C::NSTAGE) {
        cslot = 0;
        cpar ^= 1;
      }
      __syncwarp();
      if (!ld.done && !stop) {  // refill the slot just read with the slice NSTAGE ahead
        issue_slice<C>(p, tmk, tmv, ring + done_slot * C::SLOT_KV, scring + done_slot * C::SLOT_SC,
                       &bars[done_slot], ld, r0, dw, lane, box_shift, page_mask);
        ++issued;
        lslot = lslot + 1 == C::NSTAGE ? 0 : lslot + 1;
        ld.c0 += C::TC;
        it_settle<C>(ld, p, t_end, r0, lane, box_shift, page_shift);
      }
    }

    // ---------------- merge the token groups (fixed order) and store ----------------
    if (C::Q_EARLY && task + 1 < t_end && cw == 0 && lane == 0) cp_async_wait_all();
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        float l = A.l[mt][hr];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        A.l[mt][hr] = l;
        if (dw == 0 && t == 0) ml[tg * C::RPAD + 16 * mt + g + 8 * hr] = make_float2(A.m[mt][hr], l);
      }
    named_bar(BAR_CONSUMERS, C::NCW * 32);
    if constexpr (C::Q_EARLY) {  // the next task's query rows load while this one merges
      if (task + 1 < t_end) {
        const PlanTask tn = *reinterpret_cast<const PlanTask*>(smem + C::OFF_NXT);
        load_q_issue<C>(p, tn.seq, tn.hkv_part & 0xFFFF, cw, lane, qn);
      }
    }
    float fac[C::MT][2], Mrow[C::MT][2], Lrow[C::MT][2];
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int row = 16 * mt + g + 8 * hr;
        float M = -INFINITY;
#pragma unroll
        for (int i = 0; i < C::NTG; ++i) M = fmaxf(M, ml[i * C::RPAD + row].x);
        const float base = M == -INFINITY ? 0.f : M;
        fac[mt][hr] = fast_exp2(A.m[mt][hr] - base);
        float Lt = 0.f;
#pragma unroll
        for (int i = 0; i < C::NTG; ++i) {
          const float2 e = ml[i * C::RPAD + row];
          Lt += e.y * fast_exp2(e.x - base);
        }
        Mrow[mt][hr] = M;
        Lrow[mt][hr] = Lt;
      }
    float bfac[C::NBLK];
#pragma unroll
    for (int b = 0; b < C::NBLK; ++b) {
      if constexpr (C::KIND == KIND_FP4) {
        bfac[b] = A.emax[b] < 0 ? 0.f
                                : (A.emax[b] == 0 ? __int_as_float(0x00400000) : __int_as_float(A.emax[b] << 23));
      } else {
        bfac[b] = C::TOK_SCALE ? A.vref : v_scale_tensor;
      }
    }
    // The token groups' scaled accumulators are summed in group order into a buffer kept
    // in fragment order (each lane owns float4 columns: no bank conflicts): all groups write
    // at once -- into the config's own merge buffer, or for the chunk's last task into the
    // idle load ring -- and every thread sums one column over the groups; otherwise the
    // groups add in, one at a time.  Then all threads store the rows, 4 consecutive head
    // dims each, with coalesced writes.
    float4* ob4 = reinterpret_cast<float4*>(obuf) + dw * (C::MT * C::NTD * 32) + lane;
    float* fin = reinterpret_cast<float*>(smem + C::OFF_FIN);
    if (tg == C::NTG - 1 && dw == 0 && t == 0) {
#pragma unroll
      for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const int row = 16 * mt + g + 8 * hr;
          float den = Lrow[mt][hr];
          // a row written here (one partition) takes its query head's sink in the sum
          if (p.sinks != nullptr && nparts <= 1 && den > 0.f && row < p.R)
            den += fast_exp2(p.sinks[hkv * p.G + row % p.G] * kLog2e - Mrow[mt][hr]);
          fin[row] = den > 0.f ? 1.f / den : 0.f;
          if (nparts > 1 && row < p.R)
            reinterpret_cast<float2*>(p.part_ml)[slot * p.R + row] =
                make_float2(Mrow[mt][hr], Lrow[mt][hr]);
        }
    }
    if (C::MRG || (C::PAR_MERGE && task + 1 == t_end && !*abort_flag)) {
      constexpr int NF = C::NDW * C::MT * C::NTD * 32;  // float4 per token group
      float4* all = reinterpret_cast<float4*>(smem + (C::MRG ? C::OFF_MRG : C::OFF_RING));
      float4* mine = all + tg * NF + dw * (C::MT * C::NTD * 32) + lane;
#pragma unroll
      for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
        for (int n = 0; n < C::NTD; ++n) {
          const float bb = C::KIND == KIND_FP4 ? bfac[n >> 2] : bfac[0];
          const float f0 = fac[mt][0] * bb, f1 = fac[mt][1] * bb;
          mine[(mt * C::NTD + n) * 32] = make_float4(A.o[mt][n][0] * f0, A.o[mt][n][1] * f0,
                                                     A.o[mt][n][2] * f1, A.o[mt][n][3] * f1);
        }
      named_bar(BAR_CONSUMERS, C::NCW * 32);
      for (int f = cw * 32 + lane; f < NF; f += C::NTHREADS) {
        float4 a = all[f];
#pragma unroll
        for (int i = 1; i < C::NTG; ++i) {
          const float4 b = all[i * NF + f];
          a = make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
        }
        reinterpret_cast<float4*>(obuf)[f] = a;
      }
      named_bar(BAR_CONSUMERS, C::NCW * 32);
    } else {
#pragma unroll 1
      for (int i = 0; i < C::NTG; ++i) {
        if (tg == i) {
#pragma unroll
          for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
            for (int n = 0; n < C::NTD; ++n) {
              const float bb = C::KIND == KIND_FP4 ? bfac[n >> 2] : bfac[0];
              const float f0 = fac[mt][0] * bb, f1 = fac[mt][1] * bb;
              float4 v = make_float4(A.o[mt][n][0] * f0, A.o[mt][n][1] * f0,
                                     A.o[mt][n][2] * f1, A.o[mt][n][3] * f1);
              float4* dst = ob4 + (mt * C::NTD + n) * 32;
              if (i > 0) {
                const float4 w = *dst;
                v = make_float4(w.x + v.x, w.y + v.y, w.z + v.z, w.w + v.w);
              }
              *dst = v;
            }
        }
        named_bar(BAR_CONSUMERS, C::NCW * 32);
      }
    }
    {
      constexpr int Q4 = C::D / 4;
      for (int c = cw * 32 + lane; c < p.R * Q4; c += C::NTHREADS) {
        const int row = c / Q4, d0 = 4 * (c - row * Q4);
        const float inv = fin[row];
        const float v0 = obuf[frag_pos<C>(row, d0)] * inv, v1 = obuf[frag_pos<C>(row, d0 + 1)] * inv;
        const float v2 = obuf[frag_pos<C>(row, d0 + 2)] * inv, v3 = obuf[frag_pos<C>(row, d0 + 3)] * inv;
        if (nparts <= 1) {
          const int i = row / p.G, h = hkv * p.G + row % p.G;
          const int64_t orow = (int64_t)s * p.qlen + i;
          *reinterpret_cast<uint2*>(p.out + orow * p.o_st + (int64_t)h * p.o_sh + d0) =
              make_uint2(pack_bf16x2(v0, v1), pack_bf16x2(v2, v3));
        } else {
          *reinterpret_cast<float4*>(p.part_o + (slot * p.R + row) * C::D + d0) =
              make_float4(v0, v1, v2, v3);
        }
      }
    }
    // ---------------- fused partition merge (optional) ----------------
    // The task that finishes a split (sequence, KV head) last merges all its partitions,
    // in partition order, with the reduce kernel's formula (counters zeroed by the plan).
    if (p.counters != nullptr && nparts > 1) {
      volatile int* mflag = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG) + 1;
      __threadfence();  // this task's partials are visible before it is counted
      named_bar(BAR_CONSUMERS, C::NCW * 32);
      if (threadIdx.x == 0) *mflag = atomicAdd(p.counters + unit, 1) == nparts - 1;
      named_bar(BAR_CONSUMERS, C::NCW * 32);
      if (*mflag) {
        __threadfence();
        merge_partials<C>(p, obuf, s, hkv, p.part_base[unit], nparts, cw, lane, 0, p.R);
      }
    }
  }
  // Never leave while a copy into this CTA's shared memory may still be in flight (only
  // possible after a wait gave up): slice idx went to slot idx mod NSTAGE, phase idx / NSTAGE.
  for (uint32_t idx = *abort_at; idx < issued; ++idx)
    (void)mbar_wait_bounded(&bars[idx % C::NSTAGE], (idx / C::NSTAGE) & 1, 200000000ull);
}

template <class C>
__global__ void __launch_bounds__(C::NTHREADS, C::MINB)
    pa_tile_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG);
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NCW * C::NSTAGE; ++i) mbar_init(&full[i], 1);
    *abort_flag = 0;
    for (int w = 0; w < C::NCW; ++w) reinterpret_cast<uint32_t*>(smem + C::OFF_ABT)[w] = kNoAbort;
    fence_barrier_init();
  }
  __syncthreads();
  pdl_wait_prior();         // the plan's task list is complete and visible from here on
  pdl_launch_dependents();  // the reduce kernel may launch (after the plan completed); it
                            // waits for this grid's results
  const int cw = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (p.pf_split == 0) {  // planned: this CTA runs its chunk of the plan's task list
    const int t_begin = p.chunk_first[blockIdx.x], t_end = p.chunk_first[blockIdx.x + 1];
    warp_main<C>(p, &tmk, &tmv, smem, full, abort_flag, p.tasks, t_begin, t_end, 0, 0, cw, lane);
    return;
  }
  // Single-launch mode (no plan, no reduce kernel): unit blockIdx / split, one cluster of
  // `split` CTAs per unit, CTA r of it taking the r-th of P = min(split, tiles) equal runs of
  // the unit's tiles (the plan's equal split, restricted to one unit); after a cluster
  // barrier the cluster's CTAs merge a split unit's partials, each a share of its rows.
  const int split = p.pf_split;
  const int rank = split > 1 ? (int)cluster_ctarank() : 0;
  const int unit = blockIdx.x / split;
  const int s = unit / p.Hkv, hkv = unit - s * p.Hkv;
  int first;
  const int n = unit_tiles(clamped_context(p, s), p.qlen, p.window, &first);
  const int P = n < split ? (n > 0 ? n : 1) : split;
  PlanTask* rec = reinterpret_cast<PlanTask*>(smem + C::OFF_NXT);  // no next task here
  if (threadIdx.x == 0) {
    rec->seq = s;
    rec->hkv_part = hkv | (rank << 16);
    rec->tile_begin = first + (int)((int64_t)rank * n / P);
    rec->tile_end = first + (int)((int64_t)(rank + 1) * n / P);
  }
  if (blockIdx.x == 0 && cw == 0) {  // the call's status word (a timeout is ORed in only
    const int cap = p.W * p.S;       // after a wait of 2 s, long after this write)
    bool clamped = false;
    for (int q = lane; q < p.B; q += 32) clamped |= p.ctx[q] > cap;
    clamped = __any_sync(0xffffffffu, clamped);
    if (lane == 0) *p.status = clamped ? ST_CLAMPED : ST_OK;
  }
  if (blockIdx.x == 0) {  // leave no plan behind: empty chunks, one partition per unit
    for (int c = threadIdx.x; c <= p.n_chunks; c += C::NTHREADS) const_cast<int*>(p.chunk_first)[c] = 0;
    for (int u = threadIdx.x; u < p.B * p.Hkv; u += C::NTHREADS) const_cast<int*>(p.nparts)[u] = 1;
  }
  __syncthreads();
  warp_main<C>(p, &tmk, &tmv, smem, full, abort_flag, rec, 0, rank < P ? 1 : 0, P, unit * split,
               cw, lane);
  if (split > 1) {
    __threadfence();   // this CTA's partials, before the cluster barrier releases them
    cluster_sync_all();
    if (P > 1) {  // every CTA of the cluster merges its share of the rows
      const int per = (p.R + split - 1) / split;
      const int r0 = rank * per, r1 = min(p.R, r0 + per);
      if (r0 < r1)
        merge_partials<C>(p, reinterpret_cast<float*>(smem + C::OFF_OB), s, hkv, (int64_t)unit * split,
                          P, cw, lane, r0, r1);
    }
  }
}

// Launch helper: one CTA per plan chunk.
template <class C>
int launch_tile(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                void* stream) {
  static std::atomic<unsigned long long> attr_done{0};  // per device ordinal
  if (const int rc = set_smem_attr_once(pa_tile_kernel<C>, C::SMEM, attr_done)) return rc;
  if (grid < 1) grid = 1;
  // Programmatic serialisation: this grid launches while the plan kernel runs and waits
  // for it (griddepcontrol.wait) before reading the task list.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(C::NTHREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (p.pf_split > 1) {  // single-launch mode: one cluster per (sequence, KV head) unit
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)p.pf_split;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  cudaError_t e = cudaLaunchKernelEx(&cfg, pa_tile_kernel<C>, p, tk, tv);
  if (e != cudaSuccess) return (int)e;
  return (int)cudaGetLastError();
}

}  // namespace pa
