// pa_tile.cuh -- the sm_103a paged-attention decode tile kernel.
//
// One persistent CTA walks planned tasks (runs of 256-token tiles of one sequence
// and KV head).  A producer warp gathers the pages of each pipeline stage through the
// block table with TMA (K and V sub-tiles land 128-/64-byte swizzled; per-token or
// e8m0 scales arrive by 1-D bulk copy) into a ring of mbarrier-guarded stages.
// Consumer warps each own a token slice of every stage, so softmax state and the
// output accumulators are warp-private; they compute QK^T and PV with mma.sync
// (m16n8k16, fp32 accumulate), converting fp8 / fp4 operands to f16 in registers.
// Only a stage holding tokens at or past the context length runs the masked path:
// scores there become -inf, and V values and per-token scales become 0 by select,
// so unowned rows never reach the output whatever bytes they hold
// ("[FlyDSL] pa_decode: zero V rows past the context before PV", Fix).
// At the end of a task the warps merge their (max, sum, output) in a fixed order and
// either store the final bf16 row (single-partition sequences) or a partial for the
// reduce kernel ("[FlyDSL] pa_decode: MXFP4 K/V ...", direct output commit).
#pragma once

#include "pa_params.h"
#include "pa_ptx.cuh"

namespace pa {

enum { KIND_BF16 = 0, KIND_FP8 = 1, KIND_FP4 = 2 };
enum { SK_NONE = 0, SK_TENSOR = 1, SK_TOKEN = 2, SK_E8M0 = 3 };
enum { ST_OK = 0, ST_TIMEOUT = 1, ST_CLAMPED = 2 };

template <int KIND_, int D_, int MT_, int NTG_, int NDW_, int TC_, int NSTAGE_>
struct TileCfg {
  static constexpr int KIND = KIND_, D = D_, MT = MT_, NTG = NTG_, NDW = NDW_, TC = TC_;
  static constexpr int NSTAGE = NSTAGE_;
  static constexpr int NCW = NTG * NDW;            // consumer warps
  static constexpr int NTHREADS = (NCW + 1) * 32;  // plus one producer warp
  static constexpr int TW = TC / NTG;              // tokens per warp slice per stage
  static constexpr int NT = TW / 8;                // QK n-tiles per slice
  static constexpr int NKC = TW / 16;              // PV k-chunks per slice
  static constexpr int RPAD = MT * 16;
  static constexpr int ROW_BYTES = KIND == KIND_BF16 ? 2 * D : (KIND == KIND_FP8 ? D : D / 2);
  static constexpr int SUB = KIND == KIND_FP4 ? 64 : 128;  // swizzle span = sub-tile row
  static constexpr int NSUB = ROW_BYTES / SUB;
  static constexpr int WBYTES = ROW_BYTES / NDW;  // row bytes one warp reads
  static constexpr int NGRP = WBYTES / 64;        // ldmatrix.x4 groups per slice row
  static constexpr int DW = D / NDW;              // head dims one warp owns
  static constexpr int NKCH = DW / 16;            // QK k-chunks per warp
  static constexpr int NTD = DW / 8;              // PV n-tiles per warp
  static constexpr int NBLK = KIND == KIND_FP4 ? D / 32 : 1;
  static constexpr int KV_STAGE = NSUB * TC * SUB;
  static constexpr int SC_STAGE = TC * 4;
  static constexpr int STAGE_BYTES = ((2 * KV_STAGE + 2 * SC_STAGE) + 1023) / 1024 * 1024;
  static constexpr bool Q_IN_REGS = MT * NKCH * 4 <= 32;
  static constexpr int OFF_Q = NSTAGE * STAGE_BYTES;
  static constexpr int OFF_CR = OFF_Q + RPAD * D * 2;
  static constexpr int OFF_X = OFF_CR + RPAD * 4;
  static constexpr int XW = MT * NT * 4 * 32;  // floats per warp per exchange buffer
  static constexpr int X_BYTES = NDW == 2 ? NTG * 2 * 2 * XW * 4 : 0;
  static constexpr int OFF_OB = OFF_X + X_BYTES;
  static constexpr int OFF_ML = OFF_OB + RPAD * D * 4;
  static constexpr int OFF_FIN = OFF_ML + NTG * RPAD * 8;
  static constexpr int OFF_BAR = OFF_FIN + RPAD * 8;
  static constexpr int OFF_FLAG = OFF_BAR + 2 * NSTAGE * 8;
  static constexpr int SMEM = OFF_FLAG + 16 + 1024;  // + slack to align the base to 1 KiB
  static_assert(TW % 16 == 0, "a warp slice holds whole 16-token k-chunks");
  static_assert(WBYTES % 64 == 0, "a warp row slice is whole ldmatrix.x4 groups");
  static_assert(KIND != KIND_FP4 || (D == 128 && NDW == 1), "MXFP4 path: D 128, one warp per row");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static_assert(NTG + 1 < 16, "named barrier ids");
};

constexpr int BAR_CONSUMERS = 15;  // named barrier id for all consumer warps

template <class C>
__device__ __forceinline__ int swz(int row) {
  return C::SUB == 128 ? (row & 7) : ((row >> 1) & 3);
}

// Address of the 16-byte chunk holding byte `off` of token row `row` in a swizzled
// K or V stage buffer.
template <class C>
__device__ __forceinline__ uint32_t chunk_addr(const uint8_t* base, int row, int off) {
  const int sub = off / C::SUB;
  const int cin = (off % C::SUB) >> 4;
  return smem_u32(base + sub * (C::TC * C::SUB) + row * C::SUB + ((cin ^ swz<C>(row)) << 4));
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
  if constexpr (C::KIND == KIND_BF16) {
    return dw * C::DW + 8 * n + 2 * t + (j & 1);
  } else if constexpr (C::KIND == KIND_FP8) {
    return dw * C::DW + 16 * (n >> 1) + 4 * t + (n & 1) + 2 * (j & 1);
  } else {
    return 32 * (n >> 2) + 8 * t + (n & 3) + 4 * (j & 1);
  }
}

// 2^(e - 127) for an e8m0 byte as fp32 (e = 0 flushes to 0; 255 gives +inf).
__device__ __forceinline__ float e8m0_to_f32(uint32_t e) { return __int_as_float(e << 23); }

// 2^k for an integer k in [-126, 127]; 0 below.
__device__ __forceinline__ float exp2i(int k) {
  return k < -126 ? 0.f : __int_as_float((k + 127) << 23);
}

// Load and convert the query rows of (s, hkv) into shared memory, with the per-row
// logit factor (softmax scale * log2 e * q scale * row normalisation * k scale).
template <class C>
__device__ void load_q(const DecodeParams& p, uint8_t* smem, int s, int hkv, int cw, int lane,
                       float k_scale_tensor) {
  uint16_t* qs = reinterpret_cast<uint16_t*>(smem + C::OFF_Q);
  float* cr = reinterpret_cast<float*>(smem + C::OFF_CR);
  constexpr int EPL = C::D / 32;
  for (int r = cw; r < C::RPAD; r += C::NCW) {
    float x[EPL];
    float crv = 0.f;
    if (r < p.R) {
      const int i = r / p.G, h = hkv * p.G + r % p.G;
      const int64_t row = (int64_t)s * p.qlen + i;
      const int64_t off = row * p.q_st + (int64_t)h * p.q_sh + lane * EPL;
      float qsc = 1.f;
      if (p.q_fp8) {
        const uint8_t* src = reinterpret_cast<const uint8_t*>(p.q) + off;
        uint32_t w[EPL / 4];
#pragma unroll
        for (int k = 0; k < EPL / 4; ++k) w[k] = reinterpret_cast<const uint32_t*>(src)[k];
#pragma unroll
        for (int k = 0; k < EPL / 4; ++k) {
          uint32_t lo = e4m3x2_to_f16x2(w[k] & 0xFFFF), hi = e4m3x2_to_f16x2(w[k] >> 16);
          __half2 l2 = *reinterpret_cast<__half2*>(&lo), h2 = *reinterpret_cast<__half2*>(&hi);
          x[4 * k + 0] = __low2float(l2);
          x[4 * k + 1] = __high2float(l2);
          x[4 * k + 2] = __low2float(h2);
          x[4 * k + 3] = __high2float(h2);
        }
        qsc = p.q_scale_per_row ? p.q_scale[row * p.Hq + h] : p.q_scale[0];
      } else {
        const __nv_bfloat16* src = reinterpret_cast<const __nv_bfloat16*>(p.q) + off;
#pragma unroll
        for (int k = 0; k < EPL; ++k) x[k] = __bfloat162float(src[k]);
      }
      crv = p.scale_log2 * qsc;
      if constexpr (C::KIND == KIND_FP8) {
        if (p.scale_kind == SK_TENSOR) crv *= k_scale_tensor;
      }
      if constexpr (C::KIND != KIND_BF16) {
        // f16 operands: bring the row's largest magnitude into [256, 512) by a power of 2.
        float amax = 0.f;
#pragma unroll
        for (int k = 0; k < EPL; ++k) amax = fmaxf(amax, fabsf(x[k]));
#pragma unroll
        for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        int kx = 0;
        if (amax > 0.f) {
          kx = ((__float_as_int(amax) >> 23) & 0xFF) - 127 - 8;
          kx = kx < -100 ? -100 : (kx > 100 ? 100 : kx);
        }
        const float down = exp2i(-kx);
#pragma unroll
        for (int k = 0; k < EPL; ++k) x[k] *= down;
        crv *= exp2i(kx);
      }
    } else {
#pragma unroll
      for (int k = 0; k < EPL; ++k) x[k] = 0.f;
    }
    uint16_t* dst = qs + r * C::D + lane * EPL;
#pragma unroll
    for (int k = 0; k < EPL; k += 2) {
      const uint32_t v = C::KIND == KIND_BF16 ? pack_bf16x2(x[k], x[k + 1]) : pack_f16x2(x[k], x[k + 1]);
      *reinterpret_cast<uint32_t*>(dst + k) = v;
    }
    if (lane == 0) cr[r] = crv;
  }
}

template <class C>
__device__ void producer(const DecodeParams& p, const CUtensorMap* tmk, const CUtensorMap* tmv,
                         uint8_t* smem, uint64_t* full, uint64_t* empty,
                         volatile int* abort_flag, int ntasks, int lane) {
  if (lane == 0) {
    tma_prefetch_desc(tmk);
    tma_prefetch_desc(tmv);
  }
  const bool scales = p.scale_kind == SK_TOKEN || p.scale_kind == SK_E8M0;
  const int box = p.S < C::TC ? p.S : C::TC;
  const uint32_t box_bytes = (uint32_t)box * (2 * C::ROW_BYTES + (scales ? 8 : 0));
  int stage = 0;
  uint32_t phase = 0;
  uint32_t issued = 0;      // stages issued at least once
  uint32_t last_par = 0;    // parity of the last issue per stage
  bool dead = false;
  for (int task = blockIdx.x; task < ntasks && !dead; task += gridDim.x) {
    const PlanTask tk = p.tasks[task];
    const int s = tk.seq, hkv = tk.hkv_part & 0xFFFF;
    const int L = clamped_context(p, s);
    const int t0 = tk.tile_begin * kTileTokens;
    int t1 = tk.tile_end * kTileTokens;
    t1 = t1 < L ? t1 : L;
    const int32_t* btrow = p.bt + (int64_t)s * p.bt_stride;
    for (int c0 = t0; c0 < t1; c0 += C::TC) {
      if (!mbar_wait_bounded(&empty[stage], phase ^ 1)) {
        *abort_flag = 1;
        if (lane == 0) atomicOr(p.status, ST_TIMEOUT);
        dead = true;
        break;
      }
      const int ntok = (L - c0) < C::TC ? (L - c0) : C::TC;
      const int nbox = (ntok + box - 1) / box;
      if (lane == 0) mbar_arrive_expect_tx(&full[stage], nbox * box_bytes);
      __syncwarp();
      uint8_t* st = smem + stage * C::STAGE_BYTES;
      for (int j = lane; j < nbox; j += 32) {
        const int tok = c0 + j * box;
        int blk = btrow[tok / p.S];
        blk = blk < 0 ? 0 : (blk >= p.NB ? p.NB - 1 : blk);
        const int slot = tok % p.S;
#pragma unroll
        for (int sub = 0; sub < C::NSUB; ++sub) {
          const int dst = sub * (C::TC * C::SUB) + j * box * C::SUB;
          tma_load_4d(st + dst, tmk, &full[stage], sub * C::SUB, slot, hkv, blk);
          tma_load_4d(st + C::KV_STAGE + dst, tmv, &full[stage], sub * C::SUB, slot, hkv, blk);
        }
        if (scales) {
          const int64_t off = (int64_t)blk * p.sc_sb + (int64_t)hkv * p.sc_sh + (int64_t)slot * 4;
          bulk_load(st + 2 * C::KV_STAGE + j * box * 4, p.k_scale + off, box * 4, &full[stage]);
          bulk_load(st + 2 * C::KV_STAGE + C::SC_STAGE + j * box * 4, p.v_scale + off, box * 4,
                    &full[stage]);
        }
      }
      issued |= 1u << stage;
      last_par = (last_par & ~(1u << stage)) | (phase << stage);
      if (++stage == C::NSTAGE) {
        stage = 0;
        phase ^= 1;
      }
    }
  }
  // Never leave while a copy into this CTA's shared memory may still be in flight.
  for (int i = 0; i < C::NSTAGE; ++i)
    if (issued & (1u << i)) (void)mbar_wait_bounded(&full[i], (last_par >> i) & 1, 200000000ull);
}

template <class C>
__device__ void consumer(const DecodeParams& p, uint8_t* smem, uint64_t* full, uint64_t* empty,
                        volatile int* abort_flag, int ntasks, int cw, int lane) {
  const int tg = cw / C::NDW, dw = cw % C::NDW;
  const int g = lane >> 2, t = lane & 3;
  const uint16_t* qs = reinterpret_cast<const uint16_t*>(smem + C::OFF_Q);
  const float* cr = reinterpret_cast<const float*>(smem + C::OFF_CR);
  float* obuf = reinterpret_cast<float*>(smem + C::OFF_OB);
  float2* ml = reinterpret_cast<float2*>(smem + C::OFF_ML);
  float2* fin = reinterpret_cast<float2*>(smem + C::OFF_FIN);
  const float k_scale_tensor =
      (C::KIND == KIND_FP8 && p.scale_kind == SK_TENSOR) ? reinterpret_cast<const float*>(p.k_scale)[0] : 1.f;
  const float v_scale_tensor =
      (C::KIND == KIND_FP8 && p.scale_kind == SK_TENSOR) ? reinterpret_cast<const float*>(p.v_scale)[0] : 1.f;
  const bool tok_scale = C::KIND == KIND_FP8 && p.scale_kind == SK_TOKEN;
  int stage = 0;
  uint32_t phase = 0;
  int xbuf = 0;

  for (int task = blockIdx.x; task < ntasks; task += gridDim.x) {
    const PlanTask tk = p.tasks[task];
    const int s = tk.seq, hkv = tk.hkv_part & 0xFFFF, part = tk.hkv_part >> 16;
    const int L = clamped_context(p, s);
    const int t0 = tk.tile_begin * kTileTokens;
    int t1 = tk.tile_end * kTileTokens;
    t1 = t1 < L ? t1 : L;
    const int nparts = p.nparts[s];

    load_q<C>(p, smem, s, hkv, cw, lane, k_scale_tensor);
    named_bar(BAR_CONSUMERS, C::NCW * 32);

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

    float o[C::MT][C::NTD][4];
    float m_run[C::MT][2], l_run[C::MT][2];
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt) {
#pragma unroll
      for (int n = 0; n < C::NTD; ++n)
#pragma unroll
        for (int j = 0; j < 4; ++j) o[mt][n][j] = 0.f;
      m_run[mt][0] = m_run[mt][1] = -INFINITY;
      l_run[mt][0] = l_run[mt][1] = 0.f;
    }
    float vref = 0.f;                 // fp8 per-token: running max |v_scale|
    int emax[C::NBLK];                // MXFP4: running max V e8m0 exponent per block
#pragma unroll
    for (int b = 0; b < C::NBLK; ++b) emax[b] = -1;

    for (int c0 = t0; c0 < t1; c0 += C::TC) {
      if (!*abort_flag) {
        if (!mbar_wait_bounded(&full[stage], phase)) {
          *abort_flag = 1;
          if (lane == 0) atomicOr(p.status, ST_TIMEOUT);
        }
      }
      const uint8_t* st = smem + stage * C::STAGE_BYTES;
      const uint8_t* kst = st;
      const uint8_t* vst = st + C::KV_STAGE;
      const float* ksc = reinterpret_cast<const float*>(st + 2 * C::KV_STAGE);
      const float* vsc = reinterpret_cast<const float*>(st + 2 * C::KV_STAGE + C::SC_STAGE);
      const uint32_t* kex = reinterpret_cast<const uint32_t*>(st + 2 * C::KV_STAGE);
      const uint32_t* vex = reinterpret_cast<const uint32_t*>(st + 2 * C::KV_STAGE + C::SC_STAGE);
      const int r0 = tg * C::TW;
      const int vw = L - (c0 + r0);  // owned tokens in this warp's slice (may be <= 0)
      if (vw > 0) {
        const bool masked = vw < C::TW;
        // ---------------- S = Q K^T over this warp's dims ----------------
        float sacc[C::MT][C::NT][4];
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
          for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
            for (int j = 0; j < 4; ++j) sacc[mt][nt][j] = 0.f;
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt) {
          float kf[C::NBLK][2];
          if constexpr (C::KIND == KIND_FP4) {
            const uint32_t w0 = kex[r0 + 8 * nt + 2 * t], w1 = kex[r0 + 8 * nt + 2 * t + 1];
#pragma unroll
            for (int b = 0; b < C::NBLK; ++b) {
              kf[b][0] = e8m0_to_f32((w0 >> (8 * b)) & 0xFF);
              kf[b][1] = e8m0_to_f32((w1 >> (8 * b)) & 0xFF);
            }
          }
#pragma unroll
          for (int gi = 0; gi < C::NGRP; ++gi) {
            const int rr = r0 + 8 * nt + (lane & 7);
            const int off = dw * C::WBYTES + gi * 64 + (lane >> 3) * 16;
            uint32_t kr[4];
            ldsm_x4(chunk_addr<C>(kst, rr, off), kr);
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
                  mma_bf16(sacc[mt][nt], a, kr[2 * h], kr[2 * h + 1]);
                }
            } else if constexpr (C::KIND == KIND_FP8) {
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const uint32_t b0 = e4m3x2_to_f16x2(kr[q] & 0xFFFF);
                const uint32_t b1 = e4m3x2_to_f16x2(kr[q] >> 16);
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt) {
                  uint32_t a[4];
                  if constexpr (C::Q_IN_REGS) {
#pragma unroll
                    for (int z = 0; z < 4; ++z) a[z] = qa[mt][4 * gi + q][z];
                  } else {
                    load_qa<C>(qs, mt, 4 * gi + q, dw, g, t, a);
                  }
                  mma_f16(sacc[mt][nt], a, b0, b1);
                }
              }
            } else {
#pragma unroll
              for (int b = 0; b < 4; ++b) {
                uint32_t f[4];
                e2m1x8_to_f16x2(kr[b], f);
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt) {
                  float tmp[4] = {0.f, 0.f, 0.f, 0.f};
                  uint32_t a0[4], a1[4];
                  if constexpr (C::Q_IN_REGS) {
#pragma unroll
                    for (int z = 0; z < 4; ++z) {
                      a0[z] = qa[mt][2 * b][z];
                      a1[z] = qa[mt][2 * b + 1][z];
                    }
                  } else {
                    load_qa<C>(qs, mt, 2 * b, dw, g, t, a0);
                    load_qa<C>(qs, mt, 2 * b + 1, dw, g, t, a1);
                  }
                  mma_f16(tmp, a0, f[0], f[1]);
                  mma_f16(tmp, a1, f[2], f[3]);
                  sacc[mt][nt][0] = fmaf(tmp[0], kf[b][0], sacc[mt][nt][0]);
                  sacc[mt][nt][1] = fmaf(tmp[1], kf[b][1], sacc[mt][nt][1]);
                  sacc[mt][nt][2] = fmaf(tmp[2], kf[b][0], sacc[mt][nt][2]);
                  sacc[mt][nt][3] = fmaf(tmp[3], kf[b][1], sacc[mt][nt][3]);
                }
              }
            }
          }
        }
        // ---------------- combine the two head-dim halves ----------------
        if constexpr (C::NDW == 2) {
          float* xb = reinterpret_cast<float*>(smem + C::OFF_X);
          float* mine = xb + ((tg * 2 + xbuf) * 2 + dw) * C::XW;
          const float* other = xb + ((tg * 2 + xbuf) * 2 + (dw ^ 1)) * C::XW;
#pragma unroll
          for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
              for (int j = 0; j < 4; ++j) mine[((mt * C::NT + nt) * 4 + j) * 32 + lane] = sacc[mt][nt][j];
          named_bar(1 + tg, 64);
#pragma unroll
          for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
            for (int nt = 0; nt < C::NT; ++nt)
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float x = other[((mt * C::NT + nt) * 4 + j) * 32 + lane];
                sacc[mt][nt][j] = dw == 0 ? sacc[mt][nt][j] + x : x + sacc[mt][nt][j];
              }
          xbuf ^= 1;
        }
        // ---------------- logits, boundary mask ----------------
#pragma unroll
        for (int nt = 0; nt < C::NT; ++nt) {
          const int tk0 = 8 * nt + 2 * t;
          float ks0 = 1.f, ks1 = 1.f;
          if (tok_scale) {
            const float2 kk = *reinterpret_cast<const float2*>(ksc + r0 + tk0);
            ks0 = kk.x;
            ks1 = kk.y;
          }
#pragma unroll
          for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              float x = sacc[mt][nt][j] * crow[mt][j >> 1];
              if (tok_scale) x *= (j & 1) ? ks1 : ks0;
              if (masked && tk0 + (j & 1) >= vw) x = -INFINITY;
              sacc[mt][nt][j] = x;
            }
        }
        // ---------------- online softmax ----------------
        float alpha[C::MT][2];
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
          for (int hr = 0; hr < 2; ++hr) {
            float mx = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < C::NT; ++nt)
              mx = fmaxf(mx, fmaxf(sacc[mt][nt][2 * hr], sacc[mt][nt][2 * hr + 1]));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float mnew = fmaxf(m_run[mt][hr], mx);
            const float base = mnew == -INFINITY ? 0.f : mnew;
            alpha[mt][hr] = fast_exp2(m_run[mt][hr] - base);
            m_run[mt][hr] = mnew;
            float rs = 0.f;
#pragma unroll
            for (int nt = 0; nt < C::NT; ++nt) {
              const float p0 = fast_exp2(sacc[mt][nt][2 * hr] - base);
              const float p1 = fast_exp2(sacc[mt][nt][2 * hr + 1] - base);
              sacc[mt][nt][2 * hr] = p0;
              sacc[mt][nt][2 * hr + 1] = p1;
              rs += p0 + p1;
            }
            l_run[mt][hr] = l_run[mt][hr] * alpha[mt][hr] + rs;
          }
        // ---------------- V scale references and accumulator rescale ----------------
        float beta[C::NBLK];
        float vinv = 1.f;
#pragma unroll
        for (int b = 0; b < C::NBLK; ++b) beta[b] = 1.f;
        if (tok_scale) {
          float mx = 0.f;
          for (int k = lane; k < vw && k < C::TW; k += 32) mx = fmaxf(mx, fabsf(vsc[r0 + k]));
#pragma unroll
          for (int sh = 16; sh; sh >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, sh));
          const float nref = fmaxf(vref, mx);
          beta[0] = nref > 0.f ? vref / nref : 0.f;
          vinv = nref > 0.f ? 1.f / nref : 0.f;
          vref = nref;
        }
        if constexpr (C::KIND == KIND_FP4) {
          uint32_t mx[C::NBLK];
#pragma unroll
          for (int b = 0; b < C::NBLK; ++b) mx[b] = 0;
          for (int k = lane; k < vw && k < C::TW; k += 32) {
            const uint32_t w = vex[r0 + k];
#pragma unroll
            for (int b = 0; b < C::NBLK; ++b) mx[b] = max(mx[b], (w >> (8 * b)) & 0xFF);
          }
#pragma unroll
          for (int b = 0; b < C::NBLK; ++b) {
            const int cm = (int)__reduce_max_sync(0xffffffffu, mx[b]);
            const int ne = max(emax[b], cm);
            beta[b] = emax[b] < 0 ? 0.f : exp2i(emax[b] - ne);
            emax[b] = ne;
          }
        }
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
          for (int n = 0; n < C::NTD; ++n) {
            const float bb = C::KIND == KIND_FP4 ? beta[n >> 2] : beta[0];
            const float f0 = alpha[mt][0] * bb, f1 = alpha[mt][1] * bb;
            o[mt][n][0] *= f0;
            o[mt][n][1] *= f0;
            o[mt][n][2] *= f1;
            o[mt][n][3] *= f1;
          }
        // ---------------- O += P V ----------------
#pragma unroll
        for (int kc = 0; kc < C::NKC; ++kc) {
          if (masked && 16 * kc >= vw) break;
          const int tb = 16 * kc + 2 * t;  // tokens tb, tb+1 (lo pair) and tb+8, tb+9 (hi pair)
          uint32_t mlo = 0xFFFFFFFFu, mhi = 0xFFFFFFFFu;
          if (masked) {
            mlo = (tb < vw ? 0x0000FFFFu : 0u) | (tb + 1 < vw ? 0xFFFF0000u : 0u);
            mhi = (tb + 8 < vw ? 0x0000FFFFu : 0u) | (tb + 9 < vw ? 0xFFFF0000u : 0u);
          }
          // per-token V factors (0 for unowned tokens, selected, never multiplied)
          float vf[C::NBLK][4];
#pragma unroll
          for (int b = 0; b < C::NBLK; ++b)
#pragma unroll
            for (int z = 0; z < 4; ++z) vf[b][z] = 1.f;
          if (tok_scale) {
            const float2 a = *reinterpret_cast<const float2*>(vsc + r0 + tb);
            const float2 c = *reinterpret_cast<const float2*>(vsc + r0 + tb + 8);
            vf[0][0] = a.x * vinv;
            vf[0][1] = a.y * vinv;
            vf[0][2] = c.x * vinv;
            vf[0][3] = c.y * vinv;
          }
          if constexpr (C::KIND == KIND_FP4) {
            const uint32_t w[4] = {vex[r0 + tb], vex[r0 + tb + 1], vex[r0 + tb + 8], vex[r0 + tb + 9]};
#pragma unroll
            for (int b = 0; b < C::NBLK; ++b)
#pragma unroll
              for (int z = 0; z < 4; ++z) vf[b][z] = exp2i((int)((w[z] >> (8 * b)) & 0xFF) - emax[b]);
          }
          if (masked && (tok_scale || C::KIND == KIND_FP4)) {
#pragma unroll
            for (int b = 0; b < C::NBLK; ++b) {
              if (tb >= vw) vf[b][0] = 0.f;
              if (tb + 1 >= vw) vf[b][1] = 0.f;
              if (tb + 8 >= vw) vf[b][2] = 0.f;
              if (tb + 9 >= vw) vf[b][3] = 0.f;
            }
          }
          // P A-fragments, one set per V block factor
          uint32_t pa[C::NBLK][C::MT][4];
#pragma unroll
          for (int b = 0; b < C::NBLK; ++b)
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt) {
              const float* pl = sacc[mt][2 * kc];
              const float* ph = sacc[mt][2 * kc + 1];
              if constexpr (C::KIND == KIND_BF16) {
                pa[b][mt][0] = pack_bf16x2(pl[0], pl[1]);
                pa[b][mt][1] = pack_bf16x2(pl[2], pl[3]);
                pa[b][mt][2] = pack_bf16x2(ph[0], ph[1]);
                pa[b][mt][3] = pack_bf16x2(ph[2], ph[3]);
              } else {
                pa[b][mt][0] = pack_f16x2(pl[0] * vf[b][0], pl[1] * vf[b][1]);
                pa[b][mt][1] = pack_f16x2(pl[2] * vf[b][0], pl[3] * vf[b][1]);
                pa[b][mt][2] = pack_f16x2(ph[0] * vf[b][2], ph[1] * vf[b][3]);
                pa[b][mt][3] = pack_f16x2(ph[2] * vf[b][2], ph[3] * vf[b][3]);
              }
            }
          // V fragments, two 16-byte chunks per ldmatrix.x4.trans
#pragma unroll
          for (int cp = 0; cp < C::WBYTES / 32; ++cp) {
            const int q = lane >> 3;
            const int rr = r0 + 16 * kc + 8 * (q & 1) + (lane & 7);
            const int off = dw * C::WBYTES + (2 * cp + (q >> 1)) * 16;
            uint32_t v[4];
            ldsm_x4_t(chunk_addr<C>(vst, rr, off), v);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const int ch = 2 * cp + c;  // chunk index within the warp's row slice
              if constexpr (C::KIND == KIND_BF16) {
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt) mma_bf16(o[mt][ch], pa[0][mt], v[2 * c] & mlo, v[2 * c + 1] & mhi);
              } else if constexpr (C::KIND == KIND_FP8) {
                const uint32_t wl = prmt(v[2 * c], v[2 * c], 0x3120);
                const uint32_t wh = prmt(v[2 * c + 1], v[2 * c + 1], 0x3120);
                const uint32_t bA0 = e4m3x2_to_f16x2(wl & 0xFFFF) & mlo;
                const uint32_t bB0 = e4m3x2_to_f16x2(wl >> 16) & mlo;
                const uint32_t bA1 = e4m3x2_to_f16x2(wh & 0xFFFF) & mhi;
                const uint32_t bB1 = e4m3x2_to_f16x2(wh >> 16) & mhi;
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt) {
                  mma_f16(o[mt][2 * ch], pa[0][mt], bA0, bA1);
                  mma_f16(o[mt][2 * ch + 1], pa[0][mt], bB0, bB1);
                }
              } else {
                uint32_t fl[4], fh[4];
                e2m1x8_to_f16x2(v[2 * c], fl);
                e2m1x8_to_f16x2(v[2 * c + 1], fh);
                const uint32_t b0[4] = {prmt(fl[0], fl[2], 0x5410) & mlo, prmt(fl[0], fl[2], 0x7632) & mlo,
                                        prmt(fl[1], fl[3], 0x5410) & mlo, prmt(fl[1], fl[3], 0x7632) & mlo};
                const uint32_t b1[4] = {prmt(fh[0], fh[2], 0x5410) & mhi, prmt(fh[0], fh[2], 0x7632) & mhi,
                                        prmt(fh[1], fh[3], 0x5410) & mhi, prmt(fh[1], fh[3], 0x7632) & mhi};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                  for (int mt = 0; mt < C::MT; ++mt) mma_f16(o[mt][4 * ch + i], pa[ch][mt], b0[i], b1[i]);
              }
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == C::NSTAGE) {
        stage = 0;
        phase ^= 1;
      }
    }

    // ---------------- merge the token groups (fixed order) and store ----------------
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        float l = l_run[mt][hr];
        l += __shfl_xor_sync(0xffffffffu, l, 1);
        l += __shfl_xor_sync(0xffffffffu, l, 2);
        l_run[mt][hr] = l;
        if (dw == 0 && t == 0) ml[tg * C::RPAD + 16 * mt + g + 8 * hr] = make_float2(m_run[mt][hr], l);
      }
    named_bar(BAR_CONSUMERS, C::NCW * 32);
    float fac[C::MT][2];
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int row = 16 * mt + g + 8 * hr;
        float M = -INFINITY;
#pragma unroll
        for (int i = 0; i < C::NTG; ++i) M = fmaxf(M, ml[i * C::RPAD + row].x);
        const float base = M == -INFINITY ? 0.f : M;
        fac[mt][hr] = fast_exp2(m_run[mt][hr] - base);
        if (tg == 0 && dw == 0 && t == 0) {
          float Lt = 0.f;
#pragma unroll
          for (int i = 0; i < C::NTG; ++i) {
            const float2 e = ml[i * C::RPAD + row];
            Lt += e.y * fast_exp2(e.x - base);
          }
          fin[row] = make_float2(M, Lt);
        }
      }
    float bfac[C::NBLK];
#pragma unroll
    for (int b = 0; b < C::NBLK; ++b) {
      if constexpr (C::KIND == KIND_FP4) {
        bfac[b] = emax[b] < 0 ? 0.f : (emax[b] == 0 ? __int_as_float(0x00400000) : __int_as_float(emax[b] << 23));
      } else {
        bfac[b] = tok_scale ? vref : v_scale_tensor;
      }
    }
#pragma unroll 1
    for (int i = 0; i < C::NTG; ++i) {
      if (tg == i) {
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
          for (int n = 0; n < C::NTD; ++n)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const int row = 16 * mt + g + 8 * (j >> 1);
              const int d = o_dim<C>(n, j, dw, t);
              const float bb = C::KIND == KIND_FP4 ? bfac[n >> 2] : bfac[0];
              const float val = o[mt][n][j] * fac[mt][j >> 1] * bb;
              float* dst = obuf + row * C::D + d;
              *dst = (i == 0) ? val : (*dst + val);
            }
      }
      named_bar(BAR_CONSUMERS, C::NCW * 32);
    }
    // final store: coalesced over head_dim
    const int ctid = cw * 32 + lane;
    for (int idx = ctid; idx < p.R * C::D; idx += C::NCW * 32) {
      const int row = idx / C::D, d = idx % C::D;
      const float2 mf = fin[row];
      const float val = mf.y > 0.f ? obuf[idx] / mf.y : 0.f;
      const int i = row / p.G, h = hkv * p.G + row % p.G;
      const int64_t orow = (int64_t)s * p.qlen + i;
      if (nparts <= 1) {
        p.out[orow * p.o_st + (int64_t)h * p.o_sh + d] = __float2bfloat16_rn(val);
      } else {
        const int64_t slot = (int64_t)p.part_base[s] + (int64_t)hkv * nparts + part;
        const int64_t pr = slot * p.R + row;
        p.part_o[pr * C::D + d] = val;
        if (d == 0) reinterpret_cast<float2*>(p.part_ml)[pr] = mf;
      }
    }
  }
}

template <class C>
__global__ void __launch_bounds__(C::NTHREADS, 1)
    pa_tile_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + C::NSTAGE;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NSTAGE; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], C::NCW);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  const int ntasks = *p.ntasks;
  if (warp == C::NCW) {
    producer<C>(p, &tmk, &tmv, smem, full, empty, abort_flag, ntasks, lane);
  } else {
    consumer<C>(p, smem, full, empty, abort_flag, ntasks, warp, lane);
  }
}

// Launch helper: persistent grid of min(capacity, SMs) CTAs, one CTA per SM.
template <class C>
int launch_tile(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int grid_cap,
                int num_sms, void* stream) {
  static bool attr_done = false;  // per process; the attribute is per function
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(pa_tile_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return (int)e;
    attr_done = true;
  }
  int grid = num_sms < grid_cap ? num_sms : grid_cap;
  if (grid < 1) grid = 1;
  pa_tile_kernel<C><<<grid, C::NTHREADS, C::SMEM, reinterpret_cast<cudaStream_t>(stream)>>>(p, tk, tv);
  return (int)cudaGetLastError();
}

}  // namespace pa
