// pa_mx.cuh -- the sm_103a MXFP4 decode kernel: block-scaled tcgen05 QK, mma.sync PV.
//
// The MXFP4 page's QK is one scaled MMA per 32-value block: fp4 K against an 8-bit query
// with K's e8m0 byte as the hardware block scale ("[FlyDSL] pa_decode: MXFP4 K/V in the
// shared PA tile kernel", kernel description).  On sm_103a that is tcgen05.mma
// kind::mxf8f6f4.block_scale: K's e2m1 values are used as stored (two unpack warps only
// spread each 16-value group into the 16-byte slot the operand layout wants), its e8m0 bytes
// sit in tensor memory as the A scales, and the query
// is the B operand in e4m3 (as given, quantised, or a bf16 row split exactly into two e4m3
// terms).  No K value is converted by the CUDA cores.  S^T = K Q^T lands in tensor memory,
// one lane per token, and the softmax warps read it back in mma-fragment order.  PV stays on
// mma.sync: V's e8m0 scales run along the head dim, across the PV reduction, so they fold
// into P per 32-dim block as in the tile kernel, and V is widened to f16 in registers.
//
// Warp roles (one CTA per SM, persistent over the plan chunk, 128-token blocks):
//   warps 0 .. 4*NGRP-1   consumers; warp w reads TMEM lane quarter w % 4 (32 tokens of a
//                         block) and belongs to group w / 4; the groups take turns, block k
//                         going to group k % NGRP; every consumer warp keeps its own
//                         softmax state and a 16 x 128 fp32 output accumulator;
//   warp 4*NGRP           producer: block-table page gather with TMA (K, V, and the two
//                         scale runs) into a ring of NS block slots;
//   warp 4*NGRP+1         MMA: owns tensor memory, builds each task's query operand and row
//                         factors; its lane 0 copies each block's staged K scale bytes into
//                         tensor memory (tcgen05.cp) and issues the block-scaled MMAs (this
//                         loop's issue rate sets the block period).
//   warps 4*NGRP+2, +3    unpack: each spreads half of every block's K into the MMA operand
//                         layout (one of NKU tiles) and stages its scale bytes.
// Each SM sub-partition runs two consumer warps (a warp's TMEM lane quarter fixes its
// sub-partition) and one of the four helper warps.
// (A TMA copy that unpacks 4-bit data on the way in exists, but it delivered about one
// 128-token tile per microsecond per SM, far below what the ring must sustain.)
// A block holding tokens at or past the context length (or before a sliding window's first
// token) runs the masked path: scores become -inf and V values and factors 0 by select, so
// unowned rows never reach the output
// ("[FlyDSL] pa_decode: zero V rows past the context before PV", Fix).  At the end of a
// task the consumer warps merge their (max, sum, output) in a fixed order (groups into group
// 0 per lane quarter, then the quarters) and store the bf16 rows (one partition; a sink joins
// the sum) or a partial for the reduce kernel.  Consumers read a block's V run into
// registers as soon as it lands and release its ring slot before computing, so the whole
// ring is prefetch.
#pragma once

#include "pa_tile.cuh"

namespace pa {

template <int NGRP_, int NS_>
struct MxCfg {
  static constexpr int NGRP = NGRP_, NS = NS_;
  static constexpr int TT = 128, D = 128, RPAD = 16, NTD = 16;
  static constexpr int NCONS = 4 * NGRP;
  static constexpr int WPROD = NCONS, WMMA = NCONS + 1, WUNP = NCONS + 2;  // WUNP, WUNP + 1
  static constexpr int NTHREADS = 32 * (NCONS + 4);
  static_assert(NCONS % 4 == 0, "consumer and helper warps form whole warpgroups");
  static constexpr int MAXREG = (65536 / NTHREADS) / 8 * 8;  // one CTA per SM
  // Registers per thread after the split: the helper warpgroup (producer, MMA, unpack) gives
  // up what its loops do not need and the consumer warpgroups take it; the two shares add
  // up to the launch's MAXREG * NTHREADS.
  static constexpr int REG_HELP = 56;
  static constexpr int REG_CONS = ((MAXREG * NTHREADS - REG_HELP * 128) / (NCONS * 32)) / 8 * 8;
  static_assert(REG_HELP <= MAXREG && REG_CONS >= MAXREG && REG_CONS <= 255, "register split");
  static_assert(REG_HELP * 128 + REG_CONS * NCONS * 32 <= MAXREG * NTHREADS, "register split");
  static constexpr int NSB = 6;  // S buffers in tensor memory (16 columns each)
  static constexpr int NSF = 3;  // K-scale buffers in tensor memory (4 columns each)
  static constexpr int NKU = 3;  // unpacked K tiles (the MMA's A operand)
  static constexpr int NQB = 7;  // query buffers (task ordinal mod NQB); > NSB, see mx_mma
  static constexpr int MAXT = 32;  // task records staged in shared memory (more: global reads)
  // ring slot: K packed [128 tokens][64 B], V [128][64 B] (64-byte swizzle), K and V e8m0
  // words [128][4 B]
  static constexpr int SLOT_K = 0, SLOT_V = 8192, SLOT_KS = 16384, SLOT_VS = 16896;
  static constexpr int SLOT = 17408;
  static constexpr int OFF_RING = 0;
  static constexpr int OFF_KU = OFF_RING + NS * SLOT;     // [NKU][128 tokens][128 B], 128-byte swizzle
  static constexpr int OFF_Q = OFF_KU + NKU * 16384;      // per buffer: hi [16][128], lo [16][128]
  static constexpr int OFF_QRAW = OFF_Q + NQB * 4096;    // next task's rows [16][256 B], scales [16]
  static constexpr int OFF_QC = OFF_QRAW + RPAD * 256 + 64;  // row factors [NQB][16]
  static constexpr int OFF_SFA = OFF_QC + NQB * 64;       // K-scale staging [NSF][32][16 B]
  static constexpr int OFF_SFB = OFF_SFA + NSF * 512;     // query-scale staging [32][16 B]
  static constexpr int OFF_VTAB = OFF_SFB + 512;          // per consumer warp: [4][32] f16 factors
  static constexpr int OFF_TASKS = OFF_VTAB + NCONS * 256;  // MxTask [MAXT]
  static constexpr int OFF_MRG = OFF_TASKS + MAXT * 48;   // per lane quarter: 16 x 128 fp32
  static constexpr int OFF_ML = OFF_MRG + 4 * 8192;       // [NCONS][16] (max, sum)
  static constexpr int OFF_FIN = OFF_ML + NCONS * 16 * 8; // [16] 1/sum, [16] weight base
  static constexpr int OFF_NBLK = OFF_FIN + 128;            // the chunk's block count
  static constexpr int OFF_BAR = OFF_NBLK + 16;
  static constexpr int B_FULL = 0, B_EMPTY = NS, B_SFULL = 2 * NS, B_SFREE = 2 * NS + NSB;
  static constexpr int B_KFULL = 2 * NS + 2 * NSB, B_MDONE = B_KFULL + NKU, B_QRDY = B_MDONE + 1;
  static constexpr int NBAR = B_QRDY + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;     // tmem base, abort flag
  static constexpr int SMEM = OFF_MISC + 16 + 1024;       // + slack to align the base to 1 KiB
  static constexpr int TMEM_COLS = 128;
  // S buffers of 16 columns (query rows 0..15; a split query's two terms accumulate there)
  static constexpr int COL_S = 0, COL_SFA = NSB * 16, COL_SFB = COL_SFA + NSF * 4;
  static_assert(COL_SFB + 4 <= TMEM_COLS, "tensor memory columns");
  static_assert(NQB >= NSB + 1, "a query buffer is rewritten only after its last reader finished");
  static_assert(NSF == NKU && NKU <= NSB, "K tile and scale reuse wait on one S-buffer phase");
  static_assert(SLOT % 1024 == 0 && OFF_KU % 1024 == 0 && OFF_Q % 1024 == 0,
                "swizzled operands on 1 KiB boundaries");
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  // e8m0 bias applied through the query's scale bytes: a 32-value partial of the split
  // query (|q / s| < 256, |k| <= 6) times 2^(e - 127) stays finite for every K byte up to
  // 254 once it carries 2^-17; the row factor carries 2^17 back.  The low query term takes
  // another 2^-4 (it is stored 16 times larger).
  static constexpr uint32_t SFB_HI = 127 - 17, SFB_LO = 127 - 21;
};

// The CTA's block sequence: tasks of the chunk in order, each as ceil((t1 - t0) / 128)
// blocks; every role walks it the same way.
struct MxTask {
  int s, hkv, part, L, t0, t1, nblk, unit;
  int lo;      // first token of the query's sliding window (0: none)
  int nparts;  // partitions of the task's (sequence, KV head) unit
  int pbase;   // its first partial slot (split units)
  int pad;
};
static_assert(sizeof(MxTask) == 48, "task record size");

__device__ __forceinline__ MxTask mx_task_global(const DecodeParams& p, int task) {
  const PlanTask tk = p.tasks[task];
  MxTask r;
  r.s = tk.seq;
  r.hkv = tk.hkv_part & 0xFFFF;
  r.part = tk.hkv_part >> 16;
  r.L = clamped_context(p, r.s);
  r.t0 = tk.tile_begin * kTileTokens;
  const int t1 = tk.tile_end * kTileTokens;
  r.t1 = t1 < r.L ? t1 : r.L;
  r.nblk = r.t1 > r.t0 ? (r.t1 - r.t0 + 127) >> 7 : 0;
  r.unit = r.s * p.Hkv + r.hkv;
  // one query position (MXFP4 takes qlen 1): it sees tokens t > L - 1 - window
  r.lo = p.window > 0 && r.L - p.window > 0 ? r.L - p.window : 0;
  r.nparts = p.nparts[r.unit];
  r.pbase = r.nparts > 1 ? p.part_base[r.unit] : 0;
  r.pad = 0;
  return r;
}

// Task records: the chunk's first MAXT from shared memory (staged at kernel start, before any
// copy loads the memory system), the rest from global memory.
template <class C>
__device__ __forceinline__ MxTask mx_task(const DecodeParams& p, const uint8_t* sm, int tb, int task) {
  if (task - tb < C::MAXT) return reinterpret_cast<const MxTask*>(sm + C::OFF_TASKS)[task - tb];
  return mx_task_global(p, task);
}

// Next task at or after `task` that holds a block (te when none).
template <class C>
__device__ __forceinline__ int mx_next_task(const DecodeParams& p, const uint8_t* sm, int tb, int task, int te) {
  while (task < te && mx_task<C>(p, sm, tb, task).nblk == 0) ++task;
  return task;
}

// Bounded wait that stops every later wait of the CTA once any role has given up.
__device__ __forceinline__ bool mx_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                        int* status) {
  if (*abort_flag) return false;
  if (mbar_wait_bounded(bar, parity)) return true;
  *abort_flag = 1;
  atomicOr(status, ST_TIMEOUT);
  return false;
}

// Byte offset of (row, byte column) in a region of 128-byte rows swizzled in 1 KiB atoms.
__device__ __forceinline__ uint32_t mx_sw128(int row, int bcol) {
  return (uint32_t)(row * 128 + ((((bcol >> 4) ^ (row & 7)) << 4) | (bcol & 15)));
}

// ---------------------------------------------------------------------------------------
// Producer warp: block-table entries for 32 boxes per load, one per lane, the next 32 in
// flight, so no TMA issue waits on a dependent global load.
template <class C>
__device__ void mx_producer(const DecodeParams& p, const CUtensorMap* tmk, const CUtensorMap* tmv,
                            uint8_t* sm, uint64_t* bars, volatile int* abort_flag, int tb, int te,
                            int lane) {
  const int page_shift = __ffs(p.S) - 1, page_mask = p.S - 1;
  const int box = p.S < C::TT ? p.S : C::TT;
  const int box_shift = __ffs(box) - 1;
  const int bpb = C::TT >> box_shift;  // boxes per block (<= 8)
  if (lane == 0) {
    tma_prefetch_desc(tmk);
    tma_prefetch_desc(tmv);
  }
  // block of box b of task T (0 past the context)
  auto bt_load = [&](const MxTask& T, int b) -> int {
    const int tok = T.t0 + b * box;
    return tok < T.L ? p.bt[(int64_t)T.s * p.bt_stride + (tok >> page_shift)] : 0;
  };
  int task = mx_next_task<C>(p, sm, tb, tb, te);
  bool ok_start = true;
  int ncur = 0, nnxt = 0;  // the first two windows of the task to come
  if (task < te) {
    const MxTask T0 = mx_task<C>(p, sm, tb, task);
    ncur = bt_load(T0, lane);
    nnxt = bt_load(T0, 32 + lane);
  }
  // the MMA warp holds the first copies back until it has the first task's query rows
  if (!mx_wait(&bars[C::B_QRDY], 0, abort_flag, p.status)) ok_start = false;
  int k = 0;
  bool ok = ok_start;
  while (task < te && ok) {
    const MxTask T = mx_task<C>(p, sm, tb, task);
    int bbase = 0;
    int bcur = ncur, bnxt = nnxt;
    // the next task's first windows load while this task streams
    const int next = mx_next_task<C>(p, sm, tb, task + 1, te);
    if (next < te) {
      const MxTask Tn = mx_task<C>(p, sm, tb, next);
      ncur = bt_load(Tn, lane);
      nnxt = bt_load(Tn, 32 + lane);
    }
    for (int i = 0; i < T.nblk; ++i, ++k) {
      const int b0 = i * bpb;  // first box of this block
      if (b0 >= bbase + 32) {  // bpb divides 32: a block never straddles windows
        bbase += 32;
        bcur = bnxt;
        bnxt = bt_load(T, bbase + 32 + lane);
      }
      const int slot = k % C::NS, f = k / C::NS;
      if (f > 0 && !mx_wait(&bars[C::B_EMPTY + slot], (f - 1) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      const int c0 = T.t0 + i * C::TT;
      const int ntok = min(C::TT, T.L - c0);
      const int nbox = (ntok + box - 1) >> box_shift;
      // boxes that end at or before the window's first token are not loaded (their slot rows
      // keep stale bytes, which the masked path never lets through)
      int fbox = T.lo > c0 ? (T.lo - c0) >> box_shift : 0;
      fbox = fbox < nbox ? fbox : nbox;
      uint8_t* dst = sm + C::OFF_RING + slot * C::SLOT;
      uint64_t* full = &bars[C::B_FULL + slot];
      const int idx = b0 + lane - bbase;
      const int from_cur = __shfl_sync(0xffffffffu, bcur, idx & 31);
      const int from_nxt = __shfl_sync(0xffffffffu, bnxt, idx & 31);
      int blk = idx < 32 ? from_cur : from_nxt;
      blk = blk < 0 ? 0 : (blk >= p.NB ? p.NB - 1 : blk);
      // K and V arrive as 64 bytes per token, and 4 + 4 e8m0 bytes
      if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)((nbox - fbox) * box * (64 + 64 + 8)));
      __syncwarp();
      // (test hook: with drop_first_slice the chunk's first block is announced but never
      // loaded, so every wait on it runs out and the status word reports the timeout)
      if (lane >= fbox && lane < nbox && !(p.drop_first_slice && k == 0)) {
        fence_proxy_async();  // the slot was last read through the generic proxy
        const int tok = c0 + lane * box;
        const int srow = tok & page_mask;
        tma_load_4d(dst + C::SLOT_K + lane * box * 64, tmk, full, 0, srow, T.hkv, blk);
        tma_load_4d(dst + C::SLOT_V + lane * box * 64, tmv, full, 0, srow, T.hkv, blk);
        const int64_t so = (int64_t)blk * p.sc_sb + (int64_t)T.hkv * p.sc_sh + (int64_t)srow * 4;
        bulk_load(dst + C::SLOT_KS + lane * box * 4, p.k_scale + so, box * 4, full);
        bulk_load(dst + C::SLOT_VS + lane * box * 4, p.v_scale + so, box * 4, full);
      }
    }
    task = next;
  }
  if (!ok) {  // let the copies already in flight land before the CTA exits
    for (int j = k - 1; j >= 0 && j >= k - C::NS; --j)
      (void)mbar_wait_bounded(&bars[C::B_FULL + j % C::NS], (j / C::NS) & 1, 200000000ull);
  }
}

// ---------------------------------------------------------------------------------------
// MMA warp: a task's query rows (and per-row e4m3 scales) copied ahead of their use into a
// staging area of 16 rows x 256 bytes with cp.async, so that no register holds them while
// the task before streams.
template <class C>
__device__ __forceinline__ void mx_q_issue(const DecodeParams& p, uint8_t* sm, const MxTask& T, int lane) {
  uint8_t* st = sm + C::OFF_QRAW;
  const int rb = p.q_fp8 ? C::D : 2 * C::D;  // bytes of one query row
  const int per_row = rb >> 4;                // 16-byte pieces per row
  for (int i = lane; i < p.R * per_row; i += 32) {
    const int r = i / per_row, c = i - r * per_row;
    const int h = T.hkv * p.G + r;  // qlen 1: row r is query head hkv * G + r
    const uint8_t* src = reinterpret_cast<const uint8_t*>(p.q) +
                         ((int64_t)T.s * p.q_st + (int64_t)h * p.q_sh) * (p.q_fp8 ? 1 : 2) + 16 * c;
    cp_async16(st + r * 256 + 16 * c, src);
  }
  if (p.q_fp8 && lane < p.R) {
    const int h = T.hkv * p.G + lane;
    cp_async4(st + C::RPAD * 256 + 4 * lane, p.q_scale_per_row ? p.q_scale + (int64_t)T.s * p.Hq + h : p.q_scale);
  }
  cp_async_commit();
}

template <class C>
__device__ void mx_load_q(const DecodeParams& p, uint8_t* sm, int qb, int lane) {
  cp_async_wait_all();  // this lane's pieces of the staged rows
  __syncwarp();         // and every other lane's
  const uint8_t* st = sm + C::OFF_QRAW;
  uint8_t* qh = sm + C::OFF_Q + qb * 4096;
  uint8_t* ql = qh + 2048;
  float* qc = reinterpret_cast<float*>(sm + C::OFF_QC) + qb * C::RPAD;
  // rows one at a time (a rolled loop: this code runs once per task, cold, and its
  // instruction fetches cost more than its arithmetic)
#pragma unroll 1
  for (int r = 0; r < C::RPAD; ++r) {
    uint32_t hib = 0, lob = 0;
    const bool real = r < p.R;  // padding rows: zero words and a zero factor
    const float qsc = !real ? 0.f : (p.q_fp8 ? reinterpret_cast<const float*>(st + C::RPAD * 256)[r] : 1.f);
    float cr = p.scale_log2 * qsc * (1.f / kKFactorBias);
    if (p.q_fp8) {
      hib = real ? *reinterpret_cast<const uint32_t*>(st + r * 256 + 4 * lane) : 0u;  // e4m3 as stored
    } else {
      const uint2 w = real ? *reinterpret_cast<const uint2*>(st + r * 256 + 8 * lane) : make_uint2(0u, 0u);
      float x[4];
      x[0] = __uint_as_float(w.x << 16);
      x[1] = __uint_as_float(w.x & 0xFFFF0000u);
      x[2] = __uint_as_float(w.y << 16);
      x[3] = __uint_as_float(w.y & 0xFFFF0000u);
      float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
      for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      if (p.q_quant) {
        // the row quantised to e4m3 with scale amax / 448 (fp32, nearest), as the MXFP4 page
        // does; the codes are decided as in the oracle (same precision, same rounding)
        const float sq = __fdiv_rn(amax, 448.f);
#pragma unroll
        for (int j = 0; j < 4; j += 2) {
          const float a0 = amax > 0.f ? __fdiv_rn(x[j], sq) : 0.f;
          const float a1 = amax > 0.f ? __fdiv_rn(x[j + 1], sq) : 0.f;
          uint16_t b;
          asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(b) : "f"(a1), "f"(a0));
          hib |= (uint32_t)b << (8 * j);
        }
        cr *= amax > 0.f ? sq : 0.f;
      } else {
        // two e4m3 terms: q = s (hi + lo / 16), s = 2^(floor(log2 amax) - 7): q / s keeps q's
        // 8 significant bits inside (-256, 256), hi rounds it to 4 and the residual is exact in
        // e4m3 for every element down to 2^-13 of the row's largest
        int ex = amax > 0.f ? ((__float_as_int(amax) >> 23) & 0xFF) - 127 - 7 : 0;
        ex = ex < -100 ? -100 : (ex > 100 ? 100 : ex);
        const float inv = exp2i(-ex);
#pragma unroll
        for (int j = 0; j < 4; j += 2) {
          const float a0 = x[j] * inv, a1 = x[j + 1] * inv;
          uint16_t h2;
          asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(h2) : "f"(a1), "f"(a0));
          const uint32_t hf = e4m3x2_to_f16x2(h2);
          const __half2 hh = *reinterpret_cast<const __half2*>(&hf);
          const float r0 = (a0 - __low2float(hh)) * 16.f, r1 = (a1 - __high2float(hh)) * 16.f;
          uint16_t l2;
          asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(l2) : "f"(r1), "f"(r0));
          hib |= (uint32_t)h2 << (8 * j);
          lob |= (uint32_t)l2 << (8 * j);
        }
        cr *= exp2i(ex);
      }
    }
    *reinterpret_cast<uint32_t*>(qh + mx_sw128(r, 4 * lane)) = hib;
    *reinterpret_cast<uint32_t*>(ql + mx_sw128(r, 4 * lane)) = lob;
    if (lane == 0) qc[r] = cr;
  }
  fence_proxy_async();    // generic writes, read next by the tensor cores
  __threadfence_block();  // the row factors are read by the consumer warps
  __syncwarp();
}

template <class C>
__device__ void mx_mma(const DecodeParams& p, uint8_t* sm, uint64_t* bars, volatile int* abort_flag,
                       uint32_t tmem, int tb, int te, int lane) {
  const bool two_terms = !p.q_fp8 && !p.q_quant;  // a bf16 query split into hi + lo
  // The first task's query rows are in shared memory before the producer starts its copies
  // (the QRDY barrier): once the ring fills, the memory system is busy and a late load waits
  // long.  They are converted while the first blocks land.
  int task = mx_next_task<C>(p, sm, tb, tb, te);
  if (task < te) {
    mx_q_issue<C>(p, sm, mx_task<C>(p, sm, tb, task), lane);
    cp_async_wait_all();
  }
  __syncwarp();
  if (lane == 0) mbar_arrive(&bars[C::B_QRDY]);  // the rows are in; they convert while K lands
  if (task < te) mx_load_q<C>(p, sm, 0, lane);
  // the query scale bytes, once, in every lane of every quarter: byte 0 the hi term's factor,
  // byte 1 the lo term's (the MMA's scale-byte selector picks one per term)
  {
    uint8_t* st = sm + C::OFF_SFB;
    const uint32_t w = C::SFB_HI | (C::SFB_LO << 8) | (C::SFB_HI << 16) | (C::SFB_LO << 24);
    *reinterpret_cast<uint4*>(st + 16 * lane) = make_uint4(w, w, w, w);
    fence_proxy_async();
    __syncwarp();
    if (lane == 0) tmem_cp_32x128b_x4(tmem + C::COL_SFB, umma_desc_noswz(smem_u32(st), 128));
    __syncwarp();
  }
  int k = 0, ord = 0;
  bool ok = true;
  for (; task < te && ok;) {
    const MxTask T = mx_task<C>(p, sm, tb, task);
    const int qb = ord % C::NQB;
    (void)T;
    // Query buffer qb last served task ord - NQB, whose blocks all lie at or before block
    // k - NQB <= k - 1 - NSB (every task in between holds a block); the S buffers of those
    // blocks were released (waited below, in block order) before this point, and a consumer
    // reads a task's row factors before it releases the S buffer of its first block.
    if (ord > 0) mx_load_q<C>(p, sm, qb, lane);  // the first was converted at the start
    const int next = mx_next_task<C>(p, sm, tb, task + 1, te);  // its query rows load now
    if (next < te) mx_q_issue<C>(p, sm, mx_task<C>(p, sm, tb, next), lane);
    const uint32_t qh = smem_u32(sm + C::OFF_Q + qb * 4096);
    // The block loop runs on lane 0 alone: this warp's issue rate sets the block period, so
    // the loop holds no warp-wide step.  Both barriers of a block are probed back to back
    // (their latencies overlap), and the bounded wait with its abort check runs only when a
    // probe finds the phase open.
    if (lane == 0) {
      const uint64_t db = umma_desc(qh, 16, 1024);
      // one MMA of N = 16 query rows per 32-value block (K-step s: descriptor start + 32 s
      // bytes, scale byte s); a split query's lo term (rows 16..31 of the buffer, 2048 bytes
      // on, its own scale byte) accumulates into the same columns
      constexpr uint32_t H0 = umma_idesc_mx(5u, 0u, 16u, 128u, 0u, 0u), H1 = umma_idesc_mx(5u, 0u, 16u, 128u, 1u, 0u);
      constexpr uint32_t H2 = umma_idesc_mx(5u, 0u, 16u, 128u, 2u, 0u), H3 = umma_idesc_mx(5u, 0u, 16u, 128u, 3u, 0u);
      constexpr uint32_t L0 = umma_idesc_mx(5u, 0u, 16u, 128u, 0u, 1u), L1 = umma_idesc_mx(5u, 0u, 16u, 128u, 1u, 1u);
      constexpr uint32_t L2 = umma_idesc_mx(5u, 0u, 16u, 128u, 2u, 1u), L3 = umma_idesc_mx(5u, 0u, 16u, 128u, 3u, 1u);
      for (int i = 0; i < T.nblk; ++i, ++k) {
        const int sb = k % C::NSB, sf = k % C::NSF, ku = k % C::NKU;
        const uint32_t kpar = (k / C::NKU) & 1, spar = ((k - C::NSB) / C::NSB) & 1;
        const bool kready = mbar_try_wait(&bars[C::B_KFULL + ku], kpar);
        const bool sready = k < C::NSB || mbar_try_wait(&bars[C::B_SFREE + sb], spar);
        if (!kready && !mx_wait(&bars[C::B_KFULL + ku], kpar, abort_flag, p.status)) {
          ok = false;
          break;
        }
        if (!sready && !mx_wait(&bars[C::B_SFREE + sb], spar, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint64_t da = umma_desc(smem_u32(sm + C::OFF_KU + ku * 16384), 16, 1024);
        const uint32_t d = tmem + (uint32_t)(C::COL_S + sb * 16);
        const uint32_t sfa = tmem + (uint32_t)(C::COL_SFA + sf * 4), sfb = tmem + (uint32_t)C::COL_SFB;
        // lane quarter q of the tokens reads its scales from column sfa + q
        tmem_cp_32x128b_x4(sfa, umma_desc_noswz(smem_u32(sm + C::OFF_SFA + sf * 512), 128));
        // (a descriptor's start address is its low 14 bits, in 16-byte units: + 2 per 32
        // bytes; shared addresses stay below 227 KiB + 2 KiB, so the field never carries)
        umma_mxf8f6f4(d, da, db, H0, sfa, sfb, 0u);
        umma_mxf8f6f4(d, da + 2, db + 2, H1, sfa, sfb, 1u);
        umma_mxf8f6f4(d, da + 4, db + 4, H2, sfa, sfb, 1u);
        umma_mxf8f6f4(d, da + 6, db + 6, H3, sfa, sfb, 1u);
        if (two_terms) {
          umma_mxf8f6f4(d, da, db + 128, L0, sfa, sfb, 1u);
          umma_mxf8f6f4(d, da + 2, db + 130, L1, sfa, sfb, 1u);
          umma_mxf8f6f4(d, da + 4, db + 132, L2, sfa, sfb, 1u);
          umma_mxf8f6f4(d, da + 6, db + 134, L3, sfa, sfb, 1u);
        }
        umma_commit(&bars[C::B_SFULL + sb]);
      }
    }
    __syncwarp();
    ok = __shfl_sync(0xffffffffu, ok, 0) != 0;
    k = __shfl_sync(0xffffffffu, k, 0);
    ++ord;
    task = next;
  }
  // every MMA issued has completed before tensor memory is freed
  if (lane == 0) umma_commit(&bars[C::B_MDONE]);
  __syncwarp();
  (void)mbar_wait_bounded(&bars[C::B_MDONE], 0);
}

// Unpack warps (two): each block's K into the MMA operand layout (each 16 values, 8 packed
// bytes, into the lower half of a 16-byte slot of a 128-byte row, 128-byte swizzle; the upper
// halves are zero for good) in one of NKU tiles, and its scale words into the tcgen05.cp
// staging layout (row r holds the words of tokens r, r + 32, r + 64, r + 96); warp h takes
// tokens 64 h .. 64 h + 63.  Then K's part of the ring slot is released.
template <class C>
__device__ void mx_unpack(const DecodeParams& p, uint8_t* sm, uint64_t* bars, volatile int* abort_flag, int tb,
                          int te, int h, int lane) {
  if (h == 0) {  // the upper 8 bytes of every 16-byte slot: zero, set once
    for (int i = lane; i < C::NKU * 16384 / 16; i += 32)
      *reinterpret_cast<uint4*>(sm + C::OFF_KU + 16 * i) = make_uint4(0u, 0u, 0u, 0u);
  }
  named_bar(3, 64);  // both unpack warps: the tiles are zeroed
  // lane l moves 16-byte unit 32 j + l of the half (token 64 h + 8 j + l / 4, values
  // 32 (l % 4) ..); the swizzled slots depend on l only (token mod 8 = (l / 4) mod 8)
  const int rl = lane >> 2, c = 2 * (lane & 3);
  const uint32_t d0 = (uint32_t)(rl * 128 + ((c ^ (rl & 7)) << 4));
  const uint32_t d1 = (uint32_t)(rl * 128 + (((c + 1) ^ (rl & 7)) << 4));
  int k = 0;
  bool ok = true;
  for (int task = tb; task < te && ok; ++task) {
    const MxTask T = mx_task<C>(p, sm, tb, task);
    for (int i = 0; i < T.nblk; ++i, ++k) {
      const int slot = k % C::NS;
      if (!mx_wait(&bars[C::B_FULL + slot], (k / C::NS) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      // the tile and staging of block k - NKU are free once its MMAs are done, which its
      // S-full commit (issued after them) reports
      if (k >= C::NKU &&
          !mx_wait(&bars[C::B_SFULL + (k - C::NKU) % C::NSB], ((k - C::NKU) / C::NSB) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      const uint8_t* sl = sm + C::OFF_RING + slot * C::SLOT + C::SLOT_K + 4096 * h;
      uint8_t* ku = sm + C::OFF_KU + (k % C::NKU) * 16384 + 8192 * h;
      uint4 w[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) w[j] = *reinterpret_cast<const uint4*>(sl + 16 * (32 * j + lane));
      const uint32_t* ks = reinterpret_cast<const uint32_t*>(sm + C::OFF_RING + slot * C::SLOT + C::SLOT_KS);
      const uint2 sw = make_uint2(ks[64 * h + lane], ks[64 * h + 32 + lane]);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        *reinterpret_cast<uint2*>(ku + 1024 * j + d0) = make_uint2(w[j].x, w[j].y);
        *reinterpret_cast<uint2*>(ku + 1024 * j + d1) = make_uint2(w[j].z, w[j].w);
      }
      // staging row r = lane: columns 2 h, 2 h + 1 hold tokens 64 h + r, 64 h + 32 + r
      *reinterpret_cast<uint2*>(sm + C::OFF_SFA + (k % C::NSF) * 512 + 16 * lane + 8 * h) = sw;
      fence_proxy_async();  // generic writes, read next by the tensor cores
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bars[C::B_EMPTY + slot]);  // this half of K and its scales read
        mbar_arrive(&bars[C::B_KFULL + k % C::NKU]);
      }
    }
  }
}

// ---------------------------------------------------------------------------------------
// Consumer warps.
template <class C>
struct MxAcc {
  float o[C::NTD][4];  // rows g, g + 8 (mma accumulator order), head dims per o_dim
  float m[4];          // rows 2t, 2t + 1, 8 + 2t, 9 + 2t: running max (log2 units)
  float l[4];          // thread-partial sums of those rows
  int emax[4];         // V e8m0 reference per 32-dim block (-1: none yet)
};

// One consumer warp on one block: its 32 tokens (TMEM lane quarter q), S in registers.
// MASKED: tokens at or past vw (quarter-local) are unowned, and tokens before vlo lie before
// the sliding window.
template <class C, bool MASKED>
__device__ __forceinline__ void mx_block(MxAcc<C>& A, const uint32_t (&sraw)[16], const float (&crow)[4],
                                         const uint32_t (&vf)[2][2][4], uint32_t vwd, uint16_t* vtab,
                                         int vw, int vlo, int lane) {
  const int g = lane >> 2, t = lane & 3;
  // sraw[4 * c + e]: c = 0: tokens g, g + 8, rows 2t, 2t + 1; c = 1: rows 8 + 2t, 9 + 2t;
  // c = 2, 3: the same for tokens g + 16, g + 24.  e: (tok lo, row a), (tok lo, row b),
  // (tok hi, row a), (tok hi, row b).
  // ---------------- V references (lazy) and factor table ----------------
  float beta[4] = {1.f, 1.f, 1.f, 1.f};
  bool rescale_v = false;
  {
    const bool own = !MASKED || (lane < vw && lane >= vlo);  // one lane per token of the quarter
    bool over = false;
#pragma unroll
    for (int b = 0; b < 4; ++b) over |= A.emax[b] < 0 || (own && (int)((vwd >> (8 * b)) & 0xFF) > A.emax[b] + kLazyExp);
    if (__any_sync(0xffffffffu, over)) {
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const uint32_t e = (vwd >> (8 * b)) & 0xFF;
        const int cm = (int)__reduce_max_sync(0xffffffffu, own ? e : 0u);
        const int ne = max(A.emax[b], cm);
        beta[b] = A.emax[b] < 0 ? 0.f : exp2i(A.emax[b] - ne);
        A.emax[b] = ne;
      }
      rescale_v = true;
    }
    // 2^(e - emax) as f16 (below 2^-14 flushes to zero: such a block is at least 2^14 times
    // smaller than the largest one seen for it); 0 for unowned tokens
    const uint32_t kown = own ? 0xFFFFFFFFu : 0u;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int ev = (int)((vwd >> (8 * b)) & 0xFF);
      vtab[b * 32 + lane] = (uint16_t)(((uint32_t)max(ev - A.emax[b] + 15, 0) << 10) & kown);
    }
    __syncwarp();
  }
  // ---------------- logits, boundary mask, lazy max ----------------
  float x[16];
  bool need = false;
  float mx[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) mx[r] = -INFINITY;
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = 2 * (c & 1) + (e & 1);                 // row slot
      const int tok = g + 8 * (e >> 1) + 16 * (c >> 1);    // quarter-local token
      float v = __uint_as_float(sraw[4 * c + e]) * crow[r];
      if (MASKED && (tok >= vw || tok < vlo)) v = -INFINITY;
      x[4 * c + e] = v;
      mx[r] = fmaxf(mx[r], v);
    }
#pragma unroll
  for (int r = 0; r < 4; ++r) need |= mx[r] > A.m[r] + kLazyLog2;
  need = __any_sync(0xffffffffu, need);
  float alpha[4] = {1.f, 1.f, 1.f, 1.f};
  if (need) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float v = mx[r];  // row max over the warp's tokens: lanes with this t
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 4));
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 8));
      v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, 16));
      const float mn = fmaxf(A.m[r], v);
      if (mn != A.m[r]) {
        alpha[r] = fast_exp2(A.m[r] - mn);  // -inf -> 0
        A.m[r] = mn;
        A.l[r] *= alpha[r];
      }
    }
  }
  float base[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) base[r] = A.m[r] == -INFINITY ? 0.f : A.m[r];
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = 2 * (c & 1) + (e & 1);
      const float pv = fast_exp2(x[4 * c + e] - base[r]);
      x[4 * c + e] = pv;
      A.l[r] += pv;
    }
  if (need || rescale_v) {
    // the output accumulator holds rows g and g + 8: their factors come from lane g / 2,
    // whose row slots 0 / 1 (rows 2t, 2t + 1) and 2 / 3 (rows 8 + 2t, 9 + 2t) hold them
    const float a0 = __shfl_sync(0xffffffffu, alpha[0], g >> 1);
    const float a1 = __shfl_sync(0xffffffffu, alpha[1], g >> 1);
    const float a2 = __shfl_sync(0xffffffffu, alpha[2], g >> 1);
    const float a3 = __shfl_sync(0xffffffffu, alpha[3], g >> 1);
    const float fg = (g & 1) ? a1 : a0, fg8 = (g & 1) ? a3 : a2;
#pragma unroll
    for (int n = 0; n < C::NTD; ++n) {
      const float bb = beta[n >> 2];
      A.o[n][0] *= fg * bb;
      A.o[n][1] *= fg * bb;
      A.o[n][2] *= fg8 * bb;
      A.o[n][3] *= fg8 * bb;
    }
  }
  // ---------------- P into A fragments (rows on M, tokens on K) ----------------
  // an f16 pair (token j, rows 2t, 2t + 1) is the (row j, column pair t) element of an 8x8
  // matrix in fragment order; its transpose gives (row g, tokens 2t, 2t + 1)
  uint32_t pa[2][4];
#pragma unroll
  for (int kc = 0; kc < 2; ++kc) {
    const float* xa = x + 8 * kc;  // c = 2 kc (rows 2t, 2t + 1), 2 kc + 1 (rows 8 + 2t, 9 + 2t)
    pa[kc][0] = movmatrix_t(pack_f16x2(xa[0], xa[1]));  // tokens g: rows g; tokens 2t, 2t + 1
    pa[kc][2] = movmatrix_t(pack_f16x2(xa[2], xa[3]));  // tokens g + 8: row g, tokens 8 + 2t ..
    pa[kc][1] = movmatrix_t(pack_f16x2(xa[4], xa[5]));  // rows 8 + g
    pa[kc][3] = movmatrix_t(pack_f16x2(xa[6], xa[7]));
  }
  // ---------------- O += P V ----------------
#pragma unroll
  for (int kc = 0; kc < 2; ++kc) {
    if (MASKED && (16 * kc >= vw || 16 * kc + 16 <= vlo)) continue;
    const int tb = 16 * kc + 2 * t, th = tb + 8;  // this lane's token pairs
    uint32_t mlo = 0xFFFFFFFFu, mhi = 0xFFFFFFFFu;
    if (MASKED) {
      auto in = [&](int x) { return x < vw && x >= vlo; };
      mlo = (in(tb) ? 0x0000FFFFu : 0u) | (in(tb + 1) ? 0xFFFF0000u : 0u);
      mhi = (in(th) ? 0x0000FFFFu : 0u) | (in(th + 1) ? 0xFFFF0000u : 0u);
    }
#pragma unroll
    for (int cp = 0; cp < 2; ++cp) {
      const uint32_t(&v)[4] = vf[kc][cp];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int ch = 2 * cp + cc;  // 32-dim block
        const uint32_t vp0 = *reinterpret_cast<const uint32_t*>(vtab + ch * 32 + tb);
        const uint32_t vp1 = *reinterpret_cast<const uint32_t*>(vtab + ch * 32 + th);
        uint32_t pb[4] = {hmul2(pa[kc][0], vp0), hmul2(pa[kc][1], vp0), hmul2(pa[kc][2], vp1),
                          hmul2(pa[kc][3], vp1)};
        uint32_t fl[4], fh[4];
        e2m1x8_to_f16x2(v[2 * cc], fl);
        e2m1x8_to_f16x2(v[2 * cc + 1], fh);
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
        for (int i = 0; i < 4; ++i) mma_f16(A.o[4 * ch + i], pb, b0[i], b1[i]);
      }
    }
  }
}

template <class C>
__device__ void mx_consumer(const DecodeParams& p, uint8_t* sm, uint64_t* bars, volatile int* abort_flag,
                            uint32_t tmem, int tb, int te, int cw, int lane) {
  const int q = cw & 3, grp = cw >> 2;
  const int g = lane >> 2, t = lane & 3;
  uint16_t* vtab = reinterpret_cast<uint16_t*>(sm + C::OFF_VTAB + cw * 256);
  float2* ml = reinterpret_cast<float2*>(sm + C::OFF_ML);
  float* fin = reinterpret_cast<float*>(sm + C::OFF_FIN);
  // ldmatrix.trans row offsets inside a 32-token, 64-byte-swizzled V run (see the tile kernel)
  uint32_t voff[2];
  {
    const int j = lane & 7, qq = lane >> 3;
#pragma unroll
    for (int cp = 0; cp < 2; ++cp) {
      const int off = (2 * cp + (qq >> 1)) * 16;
      const int row = 8 * (qq & 1) + j;
      voff[cp] = row * 64 + (((off >> 4) ^ ((row >> 1) & 3)) << 4);
    }
  }
  const uint32_t lane_base = (uint32_t)(32 * q) << 16;
  bool ok = true;
  int k = 0, ord = 0;
  for (int task = tb; task < te; ++task) {
    const MxTask T = mx_task<C>(p, sm, tb, task);
    const int nparts = T.nparts;
    const int64_t pslot = nparts > 1 ? (int64_t)T.pbase + T.part : 0;
    MxAcc<C> A;
#pragma unroll
    for (int n = 0; n < C::NTD; ++n)
#pragma unroll
      for (int j = 0; j < 4; ++j) A.o[n][j] = 0.f;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      A.m[r] = -INFINITY;
      A.l[r] = 0.f;
      A.emax[r] = -1;
    }
    if (T.nblk > 0) {
      const float* qc = reinterpret_cast<const float*>(sm + C::OFF_QC) + (ord % C::NQB) * C::RPAD;
      float crow[4];
      bool crow_read = false;
      for (int i = 0; i < T.nblk; ++i, ++k) {
        if (k % C::NGRP != grp || !ok) continue;
        const int slot = k % C::NS, sb = k % C::NSB;
        if (!mx_wait(&bars[C::B_SFULL + sb], (k / C::NSB) & 1, abort_flag, p.status)) {
          ok = false;
          continue;
        }
        // this warp's V run and scale words (landed: the MMA warp saw the slot full); the
        // slot is released right after (the unpack warps read K before the MMA ran)
        if (!mx_wait(&bars[C::B_FULL + slot], (k / C::NS) & 1, abort_flag, p.status)) {
          ok = false;
          continue;
        }
        const uint8_t* sl = sm + C::OFF_RING + slot * C::SLOT;
        uint32_t vf[2][2][4];
        {
          const uint32_t vbase = smem_u32(sl + C::SLOT_V + 32 * q * 64);
#pragma unroll
          for (int kc = 0; kc < 2; ++kc)
#pragma unroll
            for (int cp = 0; cp < 2; ++cp) ldsm_x4_t(vbase + voff[cp] + 16 * kc * 64, vf[kc][cp]);
        }
        const uint32_t vwd = reinterpret_cast<const uint32_t*>(sl + C::SLOT_VS + 32 * q * 4)[lane];
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[C::B_EMPTY + slot]);
        tc_fence_after();
        uint32_t sraw[16];
        const uint32_t col = tmem + (uint32_t)(C::COL_S + sb * 16);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r4[4];
          tmem_ld_16x256b(col + lane_base + ((uint32_t)(16 * (c >> 1)) << 16) + 8 * (c & 1), r4);
#pragma unroll
          for (int e = 0; e < 4; ++e) sraw[4 * c + e] = r4[e];
        }
        tmem_wait_ld();
        if (!crow_read) {  // written by the MMA warp before its first commit of the task
          crow[0] = qc[2 * t];
          crow[1] = qc[2 * t + 1];
          crow[2] = qc[8 + 2 * t];
          crow[3] = qc[9 + 2 * t];
          crow_read = true;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[C::B_SFREE + sb]);
        const int c0 = T.t0 + i * C::TT + 32 * q;  // first token of this warp's quarter
        const int vw = T.L - c0, vlo = T.lo - c0;
        if (vw >= 32 && vlo <= 0)
          mx_block<C, false>(A, sraw, crow, vf, vwd, vtab, vw, vlo, lane);
        else
          mx_block<C, true>(A, sraw, crow, vf, vwd, vtab, vw, vlo, lane);
        __syncwarp();
      }
      ++ord;
    }
    // ---------------- merge the consumer warps (warp order) and store ----------------
    // row sums over the lanes holding a row (same t), then (max, sum) per row into shared
    // memory by the lanes of g = 0 (rows 2t, 2t + 1, 8 + 2t, 9 + 2t)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      float l = A.l[r];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      A.l[r] = l;
    }
    if (g == 0) {
      ml[cw * 16 + 2 * t] = make_float2(A.m[0], A.l[0]);
      ml[cw * 16 + 2 * t + 1] = make_float2(A.m[1], A.l[1]);
      ml[cw * 16 + 8 + 2 * t] = make_float2(A.m[2], A.l[2]);
      ml[cw * 16 + 9 + 2 * t] = make_float2(A.m[3], A.l[3]);
    }
    named_bar(1, C::NCONS * 32);
    // this warp's factor for rows g and g + 8: exp2(m_w - M) times the V block factors
    float fac[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
      const int row = g + 8 * hr;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < C::NCONS; ++w) M = fmaxf(M, ml[w * 16 + row].x);
      const float base = M == -INFINITY ? 0.f : M;
      fac[hr] = fast_exp2(ml[cw * 16 + row].x - base);
    }
    if (cw == 0 && t == 0) {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int row = g + 8 * hr;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < C::NCONS; ++w) M = fmaxf(M, ml[w * 16 + row].x);
        const float base = M == -INFINITY ? 0.f : M;
        float den = 0.f;
#pragma unroll
        for (int w = 0; w < C::NCONS; ++w) {
          const float2 e = ml[w * 16 + row];
          den += e.y * fast_exp2(e.x - base);
        }
        const float Lrow = den;
        if (p.sinks != nullptr && nparts <= 1 && den > 0.f && row < p.R)
          den += fast_exp2(p.sinks[T.hkv * p.G + row] * kLog2e - M);
        fin[row] = den > 0.f ? 1.f / den : 0.f;
        if (nparts > 1 && row < p.R)
          reinterpret_cast<float2*>(p.part_ml)[pslot * p.R + row] = make_float2(M, Lrow);
      }
    }
    {
      // each warp's scaled accumulator; group g > 0 hands its part to the group-0 warp of the
      // same lane quarter through that quarter's buffer (groups in order), then the group-0
      // warps hold the sums and write them
#pragma unroll
      for (int n = 0; n < C::NTD; ++n) {
        const float bb = A.emax[n >> 2] < 0 ? 0.f
                         : (A.emax[n >> 2] == 0 ? __int_as_float(0x00400000) : __int_as_float(A.emax[n >> 2] << 23));
        const float f0 = fac[0] * bb, f1 = fac[1] * bb;
        A.o[n][0] *= f0;
        A.o[n][1] *= f0;
        A.o[n][2] *= f1;
        A.o[n][3] *= f1;
      }
      float4* mine = reinterpret_cast<float4*>(sm + C::OFF_MRG) + q * (C::NTD * 32) + lane;
#pragma unroll 1
      for (int gi = 1; gi < C::NGRP; ++gi) {
        if (grp == gi) {
#pragma unroll
          for (int n = 0; n < C::NTD; ++n) mine[n * 32] = make_float4(A.o[n][0], A.o[n][1], A.o[n][2], A.o[n][3]);
        }
        named_bar(1, C::NCONS * 32);
        if (grp == 0) {
#pragma unroll
          for (int n = 0; n < C::NTD; ++n) {
            const float4 w = mine[n * 32];
            A.o[n][0] += w.x;
            A.o[n][1] += w.y;
            A.o[n][2] += w.z;
            A.o[n][3] += w.w;
          }
        }
        named_bar(1, C::NCONS * 32);
      }
      if (grp == 0) {
#pragma unroll
        for (int n = 0; n < C::NTD; ++n) mine[n * 32] = make_float4(A.o[n][0], A.o[n][1], A.o[n][2], A.o[n][3]);
      }
    }
    named_bar(1, C::NCONS * 32);
    {
      // rows, 4 consecutive head dims per thread: the lane quarters' parts summed in order,
      // then one coalesced store
      const float* all = reinterpret_cast<const float*>(sm + C::OFF_MRG);
      using Cfg = TileCfg<KIND_FP4, SK_E8M0, 128, 1, 8, 1, 32, 3, 1, 1>;  // its o_dim / frag_pos
      for (int c = cw * 32 + lane; c < p.R * 32; c += C::NCONS * 32) {
        const int row = c >> 5, d0 = 4 * (c & 31);
        const int f0 = frag_pos<Cfg>(row, d0), f1 = frag_pos<Cfg>(row, d0 + 1);
        const int f2 = frag_pos<Cfg>(row, d0 + 2), f3 = frag_pos<Cfg>(row, d0 + 3);
        float v0 = 0.f, v1 = 0.f, v2 = 0.f, v3 = 0.f;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float* a = all + w * 2048;
          v0 += a[f0];
          v1 += a[f1];
          v2 += a[f2];
          v3 += a[f3];
        }
        const float inv = fin[row];
        v0 *= inv;
        v1 *= inv;
        v2 *= inv;
        v3 *= inv;
        if (nparts <= 1) {
          const int h = T.hkv * p.G + row;
          *reinterpret_cast<uint2*>(p.out + (int64_t)T.s * p.o_st + (int64_t)h * p.o_sh + d0) =
              make_uint2(pack_bf16x2(v0, v1), pack_bf16x2(v2, v3));
        } else {
          *reinterpret_cast<float4*>(p.part_o + (pslot * p.R + row) * C::D + d0) = make_float4(v0, v1, v2, v3);
        }
      }
    }
    named_bar(1, C::NCONS * 32);  // the merge buffer and row factors are reused by the next task
  }
}

template <class C>
__global__ void __launch_bounds__(C::NTHREADS, 1) __maxnreg__(C::MAXREG)
    pa_mx_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                 const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + C::OFF_MISC + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(&bars[C::B_FULL + i], 1);
      mbar_init(&bars[C::B_EMPTY + i], 2 + 4);  // the 2 unpack warps + the 4 consumer warps
    }
    for (int i = 0; i < C::NSB; ++i) {
      mbar_init(&bars[C::B_SFULL + i], 1);
      mbar_init(&bars[C::B_SFREE + i], 4);
    }
    for (int i = 0; i < C::NKU; ++i) mbar_init(&bars[C::B_KFULL + i], 2);
    mbar_init(&bars[C::B_MDONE], 1);
    mbar_init(&bars[C::B_QRDY], 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == C::WMMA) tmem_alloc(tslot, C::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  pdl_wait_prior();         // the plan's task list is complete and visible from here on
  pdl_launch_dependents();  // the reduce kernel may launch; it waits for this grid's results
  const int tb = p.chunk_first[blockIdx.x], te = p.chunk_first[blockIdx.x + 1];
  // the chunk's task records (with context lengths and partition slots) into shared memory
  if ((int)threadIdx.x < min(te - tb, C::MAXT))
    reinterpret_cast<MxTask*>(sm + C::OFF_TASKS)[threadIdx.x] = mx_task_global(p, tb + threadIdx.x);
  __syncthreads();
  if (threadIdx.x == 0) {  // blocks of the whole chunk
    int n = 0;
    for (int t = tb; t < te; ++t) n += mx_task<C>(p, sm, tb, t).nblk;
    *reinterpret_cast<int*>(sm + C::OFF_NBLK) = n;
  }
  __syncthreads();
  if (warp < C::NCONS) {
    setmaxnreg_inc<C::REG_CONS>();
    mx_consumer<C>(p, sm, bars, abort_flag, tmem, tb, te, warp, lane);
  } else {
    setmaxnreg_dec<C::REG_HELP>();
    if (warp == C::WPROD)
      mx_producer<C>(p, &tmk, &tmv, sm, bars, abort_flag, tb, te, lane);
    else if (warp >= C::WUNP)
      mx_unpack<C>(p, sm, bars, abort_flag, tb, te, warp - C::WUNP, lane);
    else
      mx_mma<C>(p, sm, bars, abort_flag, tmem, tb, te, lane);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == C::WMMA) tmem_free(tmem, C::TMEM_COLS);
}

template <class C>
int launch_mx(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int grid, void* stream) {
  static std::atomic<unsigned long long> attr_done{0};  // per device ordinal
  if (const int rc = set_smem_attr_once(pa_mx_kernel<C>, C::SMEM, attr_done)) return rc;
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
  cudaError_t e = cudaLaunchKernelEx(&cfg, pa_mx_kernel<C>, p, tk, tv);
  if (e != cudaSuccess) return (int)e;
  return (int)cudaGetLastError();
}

}  // namespace pa
