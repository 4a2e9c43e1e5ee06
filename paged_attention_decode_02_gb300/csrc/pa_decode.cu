// pa_decode.cu -- plan and reduce kernels, and the host side of the C ABI
// (validation, workspace layout, TMA descriptors, launches).  See include/pa_decode.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "pa_configs.cuh"
#include "pa_tc.cuh"
#include "../../include/pa_decode.h"

namespace pa {

// ------------------------------------------------------------------------------------
// Plan: ceil(L/256) tiles per (sequence, KV head) unit ("[FlyDSL] pa_decode: zero V rows
// past the context before PV", Root cause).  The units are laid end to end, each as a
// gap of kUnitCostTiles (the fixed cost of starting and finishing a task: query load,
// first-slice latency, masked tail, merge) followed by its tiles, and the line is cut
// into `budget` chunks of equal length, one per tile-kernel CTA; a unit crossing a chunk
// boundary becomes several partitions whose partials are merged afterwards ("[FlyDSL]
// pa_decode: MXFP4 K/V ...", commit messages: planned tasks, direct output with one
// partition, tasks from a CU budget; max_partitions caps the split).  Equal chunks keep
// every CTA busy for the same time whatever the mix of context lengths.
// Splitting is dropped where it buys nothing: when no unit is longer than a chunk plus its
// gap, the units are also laid out whole (each in the chunk its tiles start in), and that
// layout is taken if no chunk then carries more than two unit gaps beyond the chunk
// length (checked for up to one round of sequences, 1024). A split unit costs a second task (its end-of-task merge), the partial writes and
// a reduce pass, which batches of many short, even sequences do not win back.
// ------------------------------------------------------------------------------------
constexpr int kWholeUnitChunks = 2048;  // chunks the whole-unit check covers (more: split)
__device__ __forceinline__ int clamp_len(int L, int cap, int* clamped) {
  if (L < 0) return 0;
  if (L > cap) {
    *clamped = 1;
    return cap;
  }
  return L;
}


template <typename T>
__device__ T block_exclusive_scan(T v, T* total, T* sh) {  // sh: >= 32 elements
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  T x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    T y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[wid] = x;
  __syncthreads();
  if (wid == 0) {
    T w = lane < nw ? sh[lane] : T(0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      T y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    sh[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const T before = (wid == 0 ? T(0) : sh[wid - 1]) + (x - v);
  *total = sh[nw - 1];
  __syncthreads();
  return before;
}

// How a unit of n tiles whose first tile sits at position U of the line splits: one
// partition per chunk it touches (one in all when it is empty or splitting is off).
// Positions are 32-bit: the plan serves lines shorter than 2^31 tiles in one call.
struct ChunkGrid {
  uint32_t C;        // line positions (tiles and unit gaps) per chunk
  uint32_t nchunks;  // chunks that hold tiles (>= 1)
  int maxp;
};

__device__ __forceinline__ int unit_parts(const ChunkGrid& cg, uint32_t U, int n) {
  if (n == 0 || cg.maxp < 2) return 1;
  return (int)((U + (uint32_t)n - 1) / cg.C - U / cg.C + 1);
}

// Tiles [begin, end) of partition q of the unit, and its chunk.
__device__ __forceinline__ void unit_part(const ChunkGrid& cg, uint32_t U, int n, int q, int* begin,
                                          int* end, int* chunk) {
  const uint32_t c0 = U / cg.C;
  if (n == 0 || cg.maxp < 2) {
    *begin = 0;
    *end = n;
    *chunk = (int)(c0 < cg.nchunks - 1 ? c0 : cg.nchunks - 1);
    return;
  }
  const uint32_t c = c0 + (uint32_t)q;
  const uint32_t g0 = c * cg.C > U ? c * cg.C : U;
  const uint32_t g1 = (c + 1) * cg.C < U + (uint32_t)n ? (c + 1) * cg.C : U + (uint32_t)n;
  *begin = (int)(g0 - U);
  *end = (int)(g1 - U);
  *chunk = (int)c;
}

// Chunk of the last task of a unit (its last partition).
__device__ __forceinline__ int unit_last_chunk(const ChunkGrid& cg, uint32_t U, int n) {
  int b, e, c;
  unit_part(cg, U, n, unit_parts(cg, U, n) - 1, &b, &e, &c);
  return c;
}

__global__ void __launch_bounds__(1024) pa_plan_kernel(const PlanParams pp) {
  __shared__ long long sh64[32];
  __shared__ int sh32[32];
  __shared__ int sh32b[32];
  __shared__ int shmax, shclamp;
  __shared__ int sh_last[1024];  // chunk of each thread's last task in the current round
  __shared__ int sh_load[kWholeUnitChunks];  // line positions per chunk, units laid out whole
  __shared__ int sh_load_max;
  const int tid = threadIdx.x;
  const int cap = pp.W * pp.S;
  // Until the first write this kernel only reads the context lengths, which no kernel of
  // this library writes: it runs that part while the previous kernel in the stream
  // finishes (that kernel may still read this workspace), and waits before writing.
  pdl_launch_dependents();  // the tile kernel may launch now; it waits for this grid
  if (tid == 0) {
    shmax = 0;
    shclamp = 0;
  }
  __syncthreads();
  int clamped = 0, lmax = 0, n_own = 0;  // n_own: tiles of sequence tid (one round of sequences)
  int f_own = 0;                          // and the first of them
  long long local = 0;
  for (int s = tid; s < pp.B; s += blockDim.x) {
    int f;
    const int n = unit_tiles(clamp_len(pp.ctx[s], cap, &clamped), pp.qlen, pp.window, &f);
    if (s == tid) {
      n_own = n;
      f_own = f;
    }
    local += n;
    lmax = n > lmax ? n : lmax;
  }
  if (lmax > 0) atomicMax(&shmax, lmax);
  if (clamped) atomicOr(&shclamp, 1);
  long long seq_tiles;
  (void)block_exclusive_scan<long long>(local, &seq_tiles, sh64);  // also orders shmax
  const int w = kUnitCostTiles;
  long long T64 = (seq_tiles + (long long)w * pp.B) * pp.Hkv;  // length of the line
  const bool overflow = T64 > 0x7FFFFFFFll;  // beyond the plan's range: flagged, results undefined
  if (overflow) T64 = 0x7FFFFFFFll;
  const uint32_t T = (uint32_t)T64;
  ChunkGrid cg;
  cg.maxp = pp.max_partitions;
  cg.C = (T + (uint32_t)pp.budget - 1) / (uint32_t)pp.budget;
  if (cg.C < 1) cg.C = 1;
  if (cg.maxp >= 2 && shmax > 0) {  // no unit may touch more than max_partitions chunks
    const uint32_t cmin = (uint32_t)(shmax - 1) / (uint32_t)(cg.maxp - 1) + 1;
    if (cg.C < cmin) cg.C = cmin;
  }
  cg.nchunks = T > 0 ? (T + cg.C - 1) / cg.C : 1;
  // (the condition is the same in every thread: shmax is read after the scan's barriers;
  // one round of sequences, so the check costs one scan)
  if (cg.maxp >= 2 && shmax > 0 && (uint32_t)shmax <= cg.C + (uint32_t)w && pp.B <= (int)blockDim.x &&
      cg.nchunks <= (uint32_t)kWholeUnitChunks) {
    for (int c = tid; c < (int)cg.nchunks; c += blockDim.x) sh_load[c] = 0;
    if (tid == 0) sh_load_max = 0;
    __syncthreads();
    const int n = tid < pp.B ? n_own : 0;
    long long all_tiles;
    const long long before = block_exclusive_scan<long long>((long long)n, &all_tiles, sh64);
    if (tid < pp.B) {
      const uint32_t U0 = (uint32_t)(before * pp.Hkv + (long long)w * ((long long)tid * pp.Hkv + 1));
      for (int h = 0; h < pp.Hkv; ++h) {
        const uint32_t c = (U0 + (uint32_t)(h * (n + w))) / cg.C;
        atomicAdd(&sh_load[c < cg.nchunks - 1 ? c : cg.nchunks - 1], n + w);
      }
    }
    __syncthreads();
    int mx = 0;
    for (int c = tid; c < (int)cg.nchunks; c += blockDim.x) mx = sh_load[c] > mx ? sh_load[c] : mx;
    atomicMax(&sh_load_max, mx);
    __syncthreads();
    if ((uint32_t)sh_load_max <= cg.C + 2u * (uint32_t)w) cg.maxp = 1;  // whole units
  }

  long long carry_tiles = 0;
  int carry_tasks = 0, carry_slots = 0, carry_chunk = -1;  // chunk of the last task so far
  for (int base = 0; base < pp.B; base += blockDim.x) {
    const int s = base + tid;
    int n = 0, first = 0;
    if (s < pp.B) {
      int dummy = 0;
      if (base == 0) {
        n = n_own;
        first = f_own;
      } else {
        n = unit_tiles(clamp_len(pp.ctx[s], cap, &dummy), pp.qlen, pp.window, &first);
      }
    }
    long long round_tiles;
    const long long before = block_exclusive_scan<long long>((long long)n, &round_tiles, sh64);
    // position of the first tile of unit (s, 0); unit (s, h) starts h * (n + w) later
    const uint32_t U0 =
        (uint32_t)((carry_tiles + before) * pp.Hkv + (long long)w * ((long long)s * pp.Hkv + 1));
    int ntask = 0, nslot = 0;
    if (s < pp.B) {
      for (int h = 0; h < pp.Hkv; ++h) {
        const int P = unit_parts(cg, U0 + (uint32_t)(h * (n + w)), n);
        ntask += P;
        nslot += P >= 2 ? P : 0;
      }
      sh_last[tid] = unit_last_chunk(cg, U0 + (uint32_t)((pp.Hkv - 1) * (n + w)), n);
    }
    int tot_t, tot_s;
    const int off_t = block_exclusive_scan<int>(ntask, &tot_t, sh32);  // its syncs order sh_last
    const int off_s = block_exclusive_scan<int>(nslot, &tot_s, sh32b);
    if (base == 0) {  // first write: the previous kernel is done with the workspace
      pdl_wait_prior();
      if (tid == 0) *pp.status = (shclamp || overflow) ? ST_CLAMPED : ST_OK;
    }
    if (s < pp.B) {
      int t = carry_tasks + off_t, slot = carry_slots + off_s;
      // tasks are in unit order, hence in non-decreasing chunk order: chunk c runs tasks
      // [chunk_first[c], chunk_first[c + 1]); every chunk that begins at a task is set here
      int prev = tid > 0 ? sh_last[tid - 1] : carry_chunk;
      for (int h = 0; h < pp.Hkv; ++h) {
        const uint32_t U = U0 + (uint32_t)(h * (n + w));
        const int P = unit_parts(cg, U, n);
        const int u = s * pp.Hkv + h;
        pp.nparts[u] = P;
        pp.part_base[u] = P >= 2 ? slot : 0;
        pp.counters[u] = 0;
        if (P >= 2) slot += P;
        for (int q = 0; q < P; ++q, ++t) {
          PlanTask tk;
          int chunk;
          tk.seq = s;
          tk.hkv_part = h | (q << 16);
          unit_part(cg, U, n, q, &tk.tile_begin, &tk.tile_end, &chunk);
          tk.tile_begin += first;
          tk.tile_end += first;
          pp.tasks[t] = tk;
          pp.task_chunk[t] = chunk;
          for (int k = prev + 1; k <= chunk; ++k) pp.chunk_first[k] = t;
          prev = chunk;
        }
      }
    }
    const int last_s = min(pp.B, base + (int)blockDim.x) - 1 - base;
    carry_chunk = sh_last[last_s];
    carry_tiles += round_tiles;
    carry_tasks += tot_t;
    carry_slots += tot_s;
    __syncthreads();  // sh_last is rewritten by the next round
  }
  if (tid == 0) *pp.ntasks = carry_tasks;
  // chunks past the last task hold none
  for (int c = carry_chunk + 1 + tid; c <= pp.budget; c += blockDim.x) pp.chunk_first[c] = carry_tasks;
}

// ------------------------------------------------------------------------------------
// Reduce: merge the partitions of each split (sequence, KV head) unit in a fixed order
// ("[FlyDSL] pa_decode: MXFP4 K/V ...", Self-Review: the partition reducer).
// One warp per output row.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) pa_reduce_kernel(const ReduceParams rp) {
  __shared__ float wsh[8][128];  // normalised partition weights of each warp's row
  pdl_launch_dependents();  // a following plan may launch; it waits before writing
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const long long row = (long long)blockIdx.x * 8 + wid;
  const long long rows = (long long)rp.B * rp.qlen * rp.Hq;
  // The partition counts and bases come from the plan, which completed before the tile
  // kernel (the grid this one follows) let it launch: they are read before the wait.
  int P = 0;
  long long base = 0;
  int s = 0, i = 0, h = 0;
  if (row < rows) {
    s = (int)(row / ((long long)rp.qlen * rp.Hq));
    const int rem = (int)(row % ((long long)rp.qlen * rp.Hq));
    i = rem / rp.Hq;
    h = rem % rp.Hq;
    const int u = s * rp.Hkv + h / rp.G;
    P = __ldcg(rp.nparts + u);  // through L2: no line cached in L1 by an earlier grid
    base = __ldcg(rp.part_base + u);
  }
  pdl_wait_prior();  // the tile kernel's partials are complete and visible from here on
  if (P < 2) return;
  const int r = i * rp.G + h % rp.G;
  const float2* ml = reinterpret_cast<const float2*>(rp.part_ml);
  float* w = wsh[wid];
  // The first partials' outputs load together with the (max, sum) pairs.
  constexpr int PRE = 8;
  float4 pre[PRE];
  if (rp.D == 128) {
#pragma unroll
    for (int q = 0; q < PRE; ++q)
      if (q < P) pre[q] = *reinterpret_cast<const float4*>(rp.part_o + ((base + q) * rp.R + r) * 128 + 4 * lane);
  }
  // M and the weights: lanes over partitions, then a fixed shuffle tree
  float M = -INFINITY;
  for (int q = lane; q < P; q += 32) M = fmaxf(M, ml[(base + q) * rp.R + r].x);
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float mb = M == -INFINITY ? 0.f : M;
  float W = 0.f;
  for (int q = lane; q < P; q += 32) {
    const float2 e = ml[(base + q) * rp.R + r];
    w[q] = e.y * fast_exp2(e.x - mb);
    W += w[q];
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) W += __shfl_xor_sync(0xffffffffu, W, o);
  if (rp.sinks != nullptr && W > 0.f) W += fast_exp2(rp.sinks[h] * kLog2e - mb);  // the sink's term
  const float inv = W > 0.f ? 1.f / W : 0.f;
  __syncwarp();
  for (int q = lane; q < P; q += 32) w[q] *= inv;
  __syncwarp();
  __nv_bfloat16* dst = rp.out + (long long)(s * rp.qlen + i) * rp.o_st + (long long)h * rp.o_sh;
  // each lane owns 4 consecutive dims per 128; partitions are added in a fixed order
  for (int d0 = 4 * lane; d0 < rp.D; d0 += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int q = 0;
    if (rp.D == 128) {
#pragma unroll
      for (int k = 0; k < PRE; ++k)
        if (k < P) {
          acc.x += w[k] * pre[k].x;
          acc.y += w[k] * pre[k].y;
          acc.z += w[k] * pre[k].z;
          acc.w += w[k] * pre[k].w;
        }
      q = P < PRE ? P : PRE;
    }
    for (; q + 4 <= P; q += 4) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        v[u] = *reinterpret_cast<const float4*>(rp.part_o + ((base + q + u) * rp.R + r) * rp.D + d0);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        acc.x += w[q + u] * v[u].x;
        acc.y += w[q + u] * v[u].y;
        acc.z += w[q + u] * v[u].z;
        acc.w += w[q + u] * v[u].w;
      }
    }
    for (; q < P; ++q) {
      const float4 v = *reinterpret_cast<const float4*>(rp.part_o + ((base + q) * rp.R + r) * rp.D + d0);
      acc.x += w[q] * v.x;
      acc.y += w[q] * v.y;
      acc.z += w[q] * v.z;
      acc.w += w[q] * v.w;
    }
    *reinterpret_cast<uint2*>(dst + d0) = make_uint2(pack_bf16x2(acc.x, acc.y), pack_bf16x2(acc.z, acc.w));
  }
}

// Tokens per warp slice (the TMA box is min(S, this) rows high), swizzle span and head dims
// per warp of the tile kernel that serves a format / head_dim / query-row count.
template <class C>
static void geometry_of(int* tw, int* sub, int* dw) {
  *tw = C::TW;
  *sub = C::SUB;
  *dw = C::DW;
}

void tile_geometry(int kind, int head_dim, int rows, int* tw, int* sub, int* dw) {
  const int m = rows <= 16 ? 1 : (rows <= 32 ? 2 : 4);
  if (kind == KIND_BF16) {
    if (head_dim == 64)
      m == 1 ? geometry_of<CfgBf16D64M1>(tw, sub, dw)
             : (m == 2 ? geometry_of<CfgBf16D64M2>(tw, sub, dw) : geometry_of<CfgBf16D64M4>(tw, sub, dw));
    else if (head_dim == 128)
      m == 1 ? geometry_of<CfgBf16D128M1>(tw, sub, dw)
             : (m == 2 ? geometry_of<CfgBf16D128M2>(tw, sub, dw) : geometry_of<CfgBf16D128M4>(tw, sub, dw));
    else
      m == 1 ? geometry_of<CfgBf16D256M1>(tw, sub, dw)
             : (m == 2 ? geometry_of<CfgBf16D256M2>(tw, sub, dw) : geometry_of<CfgBf16D256M4>(tw, sub, dw));
  } else if (kind == KIND_FP8) {
    if (head_dim == 64)
      m == 1 ? geometry_of<CfgFp8D64M1<SK_TOKEN>>(tw, sub, dw)
             : (m == 2 ? geometry_of<CfgFp8D64M2<SK_TOKEN>>(tw, sub, dw)
                       : geometry_of<CfgFp8D64M4<SK_TOKEN>>(tw, sub, dw));
    else if (head_dim == 128)
      m == 1 ? geometry_of<CfgFp8D128M1<SK_TOKEN>>(tw, sub, dw)
             : (m == 2 ? geometry_of<CfgFp8D128M2<SK_TOKEN>>(tw, sub, dw)
                       : geometry_of<CfgFp8D128M4<SK_TOKEN>>(tw, sub, dw));
    else
      m == 1 ? geometry_of<CfgFp8D256M1<SK_TOKEN>>(tw, sub, dw)
             : (m == 2 ? geometry_of<CfgFp8D256M2<SK_TOKEN>>(tw, sub, dw)
                       : geometry_of<CfgFp8D256M4<SK_TOKEN>>(tw, sub, dw));
  } else {
    geometry_of<CfgFp4D128M1>(tw, sub, dw);
  }
}

}  // namespace pa

// ======================================================================================
// Host side
// ======================================================================================
namespace {

using pa::WsLayout;

constexpr int kMaxRows = 64;         // G * qlen served by the tile kernels
constexpr int kDefaultMaxParts = 128;
constexpr int kMaxParts = 128;  // the in-decode merge keeps [rows, partitions] weights in smem

int device_sms(int* out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  static std::mutex mu;
  static int cache[64] = {0};
  std::lock_guard<std::mutex> lk(mu);
  if (dev < 64 && cache[dev] > 0) {
    *out = cache[dev];
    return 0;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
  if (dev < 64) cache[dev] = n;
  *out = n;
  return 0;
}

int64_t row_bytes(const pa_decode_args* a) {
  if (a->kv_dtype == PA_KV_BF16) return 2LL * a->head_dim;
  if (a->kv_dtype == PA_KV_FP8_E4M3) return a->head_dim;
  return a->head_dim / 2;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

pa_status validate(const pa_decode_args* a) {
  if (!a) return PA_ERR_INVALID_ARG;
  if (a->batch < 0 || a->qlen < 1 || a->num_kv_heads < 1 || a->num_q_heads < 1) return PA_ERR_INVALID_ARG;
  if (a->num_q_heads % a->num_kv_heads) return PA_ERR_INVALID_ARG;
  if (a->num_q_heads > 65535 * a->num_kv_heads || a->num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
  if (a->head_dim < 1 || a->page_size < 1 || a->num_blocks < 1 || a->max_blocks_per_seq < 1)
    return PA_ERR_INVALID_ARG;
  if ((int64_t)a->max_blocks_per_seq * a->page_size > (int64_t)1 << 30) return PA_ERR_UNSUPPORTED;
  if ((int64_t)a->batch * a->num_kv_heads > ((int64_t)1 << 30)) return PA_ERR_UNSUPPORTED;
  if (a->head_dim != 64 && a->head_dim != 128 && a->head_dim != 256) return PA_ERR_UNSUPPORTED;
  switch (a->page_size) {
    case 16: case 32: case 64: case 128: case 256: break;
    default: return PA_ERR_UNSUPPORTED;
  }
  const bool combo = (a->kv_dtype == PA_KV_BF16 && a->kv_scale == PA_SCALE_NONE) ||
                     (a->kv_dtype == PA_KV_FP8_E4M3 &&
                      (a->kv_scale == PA_SCALE_PER_TENSOR || a->kv_scale == PA_SCALE_PER_TOKEN)) ||
                     (a->kv_dtype == PA_KV_MXFP4 && a->kv_scale == PA_SCALE_E8M0_32);
  if (a->kv_dtype < 0 || a->kv_dtype > 2 || a->kv_scale < 0 || a->kv_scale > 3) return PA_ERR_INVALID_ARG;
  if (!combo) return PA_ERR_UNSUPPORTED;
  if (a->q_dtype != PA_Q_BF16 && a->q_dtype != PA_Q_FP8_E4M3 && a->q_dtype != PA_Q_BF16_TO_E4M3)
    return PA_ERR_INVALID_ARG;
  if (a->q_dtype == PA_Q_BF16_TO_E4M3 && a->kv_dtype != PA_KV_MXFP4) return PA_ERR_UNSUPPORTED;
  if (a->merge_in_decode != 0 && a->merge_in_decode != 1) return PA_ERR_INVALID_ARG;
  if (a->causal != 0 && a->causal != 1) return PA_ERR_INVALID_ARG;
  if (a->sliding_window < 0) return PA_ERR_INVALID_ARG;
  if (a->trans_v != 0 && a->trans_v != 1) return PA_ERR_INVALID_ARG;
  if (a->kernel < PA_KERNEL_DEFAULT || a->kernel > PA_KERNEL_TCGEN05) return PA_ERR_INVALID_ARG;
  if (a->trans_v && !(a->kv_dtype == PA_KV_FP8_E4M3 && a->kv_scale == PA_SCALE_PER_TENSOR))
    return PA_ERR_UNSUPPORTED;
  const int G = a->num_q_heads / a->num_kv_heads;
  const int R = G * a->qlen;
  if (R > kMaxRows) return PA_ERR_UNSUPPORTED;
  if (a->kv_dtype == PA_KV_MXFP4 && (a->head_dim != 128 || a->qlen != 1 || G > 16)) return PA_ERR_UNSUPPORTED;
  if (a->batch == 0) return PA_OK;
  if (!a->query || !a->key_cache || !a->value_cache || !a->block_tables || !a->context_lens || !a->out)
    return PA_ERR_INVALID_ARG;
  if (a->q_dtype == PA_Q_FP8_E4M3 && !a->q_scale) return PA_ERR_INVALID_ARG;
  if (a->kv_scale != PA_SCALE_NONE && (!a->key_scale || !a->value_scale)) return PA_ERR_INVALID_ARG;
  // query / output: head_dim contiguous; vector loads need 16-byte aligned rows
  const int qel = a->q_dtype == PA_Q_FP8_E4M3 ? 1 : 2;
  if (a->q_stride_head < a->head_dim || a->q_stride_token < 0) return PA_ERR_INVALID_ARG;
  if (!aligned16(a->query) || (a->q_stride_head * qel) % 16 || (a->q_stride_token * qel) % 16)
    return PA_ERR_UNSUPPORTED;
  if (a->out_stride_head < a->head_dim || a->out_stride_token < 0) return PA_ERR_INVALID_ARG;
  if (a->bt_stride < a->max_blocks_per_seq) return PA_ERR_INVALID_ARG;
  // caches: dense token rows, non-overlapping heads and blocks, 16-byte granularity (TMA)
  const int64_t rb = row_bytes(a);
  if (a->kv_stride_token != rb) return PA_ERR_UNSUPPORTED;
  if (a->kv_stride_head < rb * a->page_size ||
      a->kv_stride_block < a->kv_stride_head * a->num_kv_heads)
    return PA_ERR_INVALID_ARG;
  if (a->kv_stride_head % 16 || a->kv_stride_block % 16 || !aligned16(a->key_cache) ||
      !aligned16(a->value_cache))
    return PA_ERR_UNSUPPORTED;
  if (a->kv_stride_block >= ((int64_t)1 << 40)) return PA_ERR_UNSUPPORTED;
  if (a->kv_scale == PA_SCALE_PER_TOKEN || a->kv_scale == PA_SCALE_E8M0_32) {
    const int64_t tb = 4;  // fp32 per token, or 4 e8m0 bytes per token at head_dim 128
    if (a->scale_stride_head < tb * a->page_size ||
        a->scale_stride_block < a->scale_stride_head * a->num_kv_heads)
      return PA_ERR_INVALID_ARG;
    if (a->scale_stride_head % 16 || a->scale_stride_block % 16 || !aligned16(a->key_scale) ||
        !aligned16(a->value_scale))
      return PA_ERR_UNSUPPORTED;
  }
  return PA_OK;
}

// Work-split parameters that every call derives identically from the arguments.
pa_status split_params(const pa_decode_args* a, int* budget, int* maxp) {
  int b = a->task_budget;
  if (b <= 0) {
    int sms = 0;
    if (device_sms(&sms)) return PA_ERR_CUDA;
    b = sms;
  }
  *budget = b;
  *maxp = a->max_partitions > 0 ? a->max_partitions : kDefaultMaxParts;
  if (*maxp > kMaxParts) *maxp = kMaxParts;
  return PA_OK;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The tensor-core (tcgen05) kernel covers head_dim 128, up to 32 query rows per KV head
// and pages of at least 8 tokens, with the separate reduce, not causal, without a sliding
// window or sinks, and with token-major V.  It runs when the caller asks for it
// (kernel = PA_KERNEL_TCGEN05) and covers the shape; otherwise the mma.sync tile kernel
// runs, the faster of the two on the long-context workloads.
bool tc_kernel_applies(const pa_decode_args* a, int rows) {
  return a->kernel == PA_KERNEL_TCGEN05 && a->head_dim == 128 && rows <= 32 && a->page_size >= 8 &&
         !a->merge_in_decode && !(a->causal && a->qlen > 1) && a->sliding_window == 0 &&
         !a->trans_v && !a->sinks && a->q_dtype != PA_Q_BF16_TO_E4M3;
}

// The MXFP4 kernel with block-scaled tcgen05 QK serves MXFP4 caches by default: any page
// size and sliding window, without the in-decode merge (that runs on the tile kernel).
bool mx_kernel_applies(const pa_decode_args* a) {
  return a->kv_dtype == PA_KV_MXFP4 && a->kernel == PA_KERNEL_DEFAULT && !a->merge_in_decode;
}

// Test hook, read once per process: when the environment holds PA_DECODE_TEST_DROP_SLICE=1
// at the library's first decode call, that one call (and no later one) has the first warp
// of every CTA leave its first ring slot unloaded, so that wait runs out and the status
// word reports it; the next call shows that the context is still usable.
bool drop_first_slice_hook() {
  static std::once_flag once;
  static std::atomic<bool> armed{false};
  std::call_once(once, [] {
    const char* d = getenv("PA_DECODE_TEST_DROP_SLICE");
    armed.store(d != nullptr && strcmp(d, "1") == 0);
  });
  return armed.load(std::memory_order_relaxed) && armed.exchange(false);
}

pa_status make_layout(const pa_decode_args* a, WsLayout* L) {
  int budget = 0, maxp = 0;
  pa_status st = split_params(a, &budget, &maxp);
  if (st != PA_OK) return st;
  const int G = a->num_q_heads / a->num_kv_heads;
  const int R = G * a->qlen;
  const int B = a->batch;
  L->budget = budget;
  L->max_partitions = maxp;
  // tasks <= units + chunks - 1; a split unit holds >= 1 of the chunks - 1 interior chunk
  // boundaries and has one partition more than it holds, so split partitions <= 2 * budget
  L->capacity = B * a->num_kv_heads + budget;
  L->slots = maxp >= 2 ? 2 * budget : 0;
  size_t off = 0;
  L->status = off;
  L->ntasks = off + 4;
  off = 256;
  const size_t units = (size_t)B * a->num_kv_heads;
  L->nparts = off;
  off = align_up(off + 4 * units, 256);
  L->part_base = off;
  off = align_up(off + 4 * units, 256);
  L->counters = off;
  off = align_up(off + 4 * units, 256);
  L->tasks = off;
  off = align_up(off + sizeof(pa::PlanTask) * (size_t)L->capacity, 256);
  L->task_chunk = off;
  off = align_up(off + 4 * (size_t)L->capacity, 256);
  L->chunk_first = off;
  off = align_up(off + 4 * ((size_t)budget + 1), 256);
  L->part_ml = off;
  off = align_up(off + 8 * (size_t)L->slots * R, 256);
  L->part_o = off;
  off = align_up(off + 4 * (size_t)L->slots * R * a->head_dim, 256);
  L->total = off;
  return PA_OK;
}

pa_status check_ws(const pa_decode_args* a, const void* ws, size_t bytes, WsLayout* L) {
  pa_status st = make_layout(a, L);
  if (st != PA_OK) return st;
  if (!ws || bytes < L->total || (reinterpret_cast<uintptr_t>(ws) & 255)) return PA_ERR_WORKSPACE;
  return PA_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// K or V cache as a 4-D byte tensor {row bytes, page slots, KV heads, blocks}; the box is
// one swizzle span wide and min(S, stage tokens) slots high.
pa_status cache_map(const pa_decode_args* a, const void* base, int sub, int box_rows, CUtensorMap* m) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  cuuint64_t dims[4] = {(cuuint64_t)row_bytes(a), (cuuint64_t)a->page_size,
                        (cuuint64_t)a->num_kv_heads, (cuuint64_t)a->num_blocks};
  cuuint64_t strides[3] = {(cuuint64_t)a->kv_stride_token, (cuuint64_t)a->kv_stride_head,
                           (cuuint64_t)a->kv_stride_block};
  cuuint32_t box[4] = {(cuuint32_t)sub, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  sub == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_UNSUPPORTED;
}

// A cache as a 4-D byte tensor {row bytes, page slots, KV heads, blocks} with unswizzled
// boxes of whole rows by `box_rows` slots (rows land back to back in shared memory).
pa_status cache_map_rows(const pa_decode_args* a, const void* base, int box_rows, CUtensorMap* m) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  cuuint64_t dims[4] = {(cuuint64_t)row_bytes(a), (cuuint64_t)a->page_size, (cuuint64_t)a->num_kv_heads,
                        (cuuint64_t)a->num_blocks};
  cuuint64_t strides[3] = {(cuuint64_t)a->kv_stride_token, (cuuint64_t)a->kv_stride_head,
                           (cuuint64_t)a->kv_stride_block};
  cuuint32_t box[4] = {(cuuint32_t)row_bytes(a), (cuuint32_t)box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_UNSUPPORTED;
}

// Tensor map of a transposed e4m3 value cache [NB, Hkv, D, S]: boxes of 16 tokens (16
// bytes) by `dims` head dims, unswizzled (rows of 16 bytes are read conflict-free).
pa_status cache_map_vt(const pa_decode_args* a, int dims, CUtensorMap* m) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return PA_ERR_CUDA;
  cuuint64_t gdim[4] = {(cuuint64_t)a->page_size, (cuuint64_t)a->head_dim,
                        (cuuint64_t)a->num_kv_heads, (cuuint64_t)a->num_blocks};
  cuuint64_t strides[3] = {(cuuint64_t)a->page_size, (cuuint64_t)a->kv_stride_head,
                           (cuuint64_t)a->kv_stride_block};
  cuuint32_t box[4] = {16, (cuuint32_t)dims, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(a->value_cache), gdim,
                  strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_UNSUPPORTED;
}

// Single-launch mode of pa_decode_run for small problems: no plan and no reduce kernel;
// the tile kernel takes one cluster of `split` CTAs per (sequence, KV head) unit and each
// CTA a run of the unit's tiles, the cluster's CTAs then merging the partials (rows split
// among them).  It runs
// when every unit fits the CTA budget, a unit's tiles (bounded by the block-table width,
// or by the sliding window) give each CTA at most kSingleLaunchTiles of them, and the
// caller did not ask for the tcgen05 tile kernel.  Returns the split, or 0 (planned path).
// The mode leaves the workspace's plan empty (no chunk holds a task, every unit one
// partition), so a pa_decode or pa_decode_reduce that follows without a new plan finds
// nothing to do.
constexpr int kSingleLaunchTiles = 3;
constexpr int kMaxClusterCtas = 8;  // portable cluster size
int single_launch_split(const pa_decode_args* a, const WsLayout& L) {
  if (a->kernel == PA_KERNEL_TCGEN05) return 0;
  const int64_t units = (int64_t)a->batch * a->num_kv_heads;
  if (units < 1 || units > L.budget) return 0;
  const int64_t TT = pa::kTileTokens;
  int64_t tiles = ((int64_t)a->max_blocks_per_seq * a->page_size + TT - 1) / TT;
  if (a->sliding_window > 0) {
    const int64_t wt = ((int64_t)a->sliding_window + a->qlen - 1 + TT - 1) / TT + 1;
    tiles = wt < tiles ? wt : tiles;
  }
  if (tiles < 1) tiles = 1;
  int64_t split = L.budget / units;  // one wave: units * split <= budget CTAs
  if (split > kMaxClusterCtas) split = kMaxClusterCtas;
  if (split > tiles) split = tiles;
  if (split > L.max_partitions) split = L.max_partitions;
  if (split < 1) split = 1;
  if (split > 1 && units * split > L.slots) return 0;  // partial slots (units <= budget: never)
  if ((tiles + split - 1) / split > kSingleLaunchTiles) return 0;
  return (int)split;
}

pa_status decode_launch(const pa_decode_args* a, void* ws, size_t bytes, void* stream, int pf_split) {
  pa_status st = validate(a);
  if (st != PA_OK) return st;
  WsLayout L;
  if ((st = check_ws(a, ws, bytes, &L)) != PA_OK) return st;
  if (a->batch == 0) return PA_OK;
  const int G = a->num_q_heads / a->num_kv_heads;
  const int R = G * a->qlen;
  const int kind = a->kv_dtype == PA_KV_BF16 ? pa::KIND_BF16 : (a->kv_dtype == PA_KV_FP8_E4M3 ? pa::KIND_FP8 : pa::KIND_FP4);
  // the single-launch mode runs the mma.sync tile kernel
  const bool use_tc = pf_split == 0 && tc_kernel_applies(a, R);
  const bool use_mx = pf_split == 0 && !use_tc && mx_kernel_applies(a);
  int tc = 0, sub = 0, dims = a->head_dim;
  if (use_mx) {
    tc = 128;
    sub = 64;
  } else if (use_tc) {
    tc = 128;
    sub = kind == pa::KIND_FP4 ? 64 : 128;
  } else {
    pa::tile_geometry(kind, a->head_dim, R, &tc, &sub, &dims);
  }
  // transposed V is loaded in 16-token pieces, and K in boxes of the same height
  const int box = a->trans_v ? 16 : (a->page_size < tc ? a->page_size : tc);
  CUtensorMap tk, tv;
  if (use_mx)
    st = cache_map_rows(a, a->key_cache, box, &tk);
  else
    st = cache_map(a, a->key_cache, sub, box, &tk);
  if (st != PA_OK) return st;
  if (a->trans_v)
    st = cache_map_vt(a, dims, &tv);
  else
    st = cache_map(a, a->value_cache, sub, box, &tv);
  if (st != PA_OK) return st;

  uint8_t* w = static_cast<uint8_t*>(ws);
  pa::DecodeParams p;
  p.B = a->batch;
  p.qlen = a->qlen;
  p.causal = a->causal && a->qlen > 1;
  p.window = a->sliding_window;
  p.trans_v = a->trans_v;
  p.sinks = a->sinks;
  p.Hq = a->num_q_heads;
  p.Hkv = a->num_kv_heads;
  p.G = G;
  p.R = R;
  p.D = a->head_dim;
  p.S = a->page_size;
  p.W = a->max_blocks_per_seq;
  p.NB = a->num_blocks;
  p.bt_stride = a->bt_stride;
  const float sc = a->softmax_scale > 0.f ? a->softmax_scale : 1.0f / sqrtf((float)a->head_dim);
  p.scale_log2 = sc * 1.4426950408889634f;
  p.q_fp8 = a->q_dtype == PA_Q_FP8_E4M3;
  p.q_quant = a->q_dtype == PA_Q_BF16_TO_E4M3;
  p.drop_first_slice = drop_first_slice_hook();
  p.q_scale_per_row = a->q_scale_per_row != 0;
  p.scale_kind = a->kv_scale;
  p.q = a->query;
  p.q_st = a->q_stride_token;
  p.q_sh = a->q_stride_head;
  p.q_scale = a->q_scale;
  p.k_scale = static_cast<const uint8_t*>(a->key_scale);
  p.v_scale = static_cast<const uint8_t*>(a->value_scale);
  p.sc_sb = a->scale_stride_block;
  p.sc_sh = a->scale_stride_head;
  p.bt = a->block_tables;
  p.ctx = a->context_lens;
  p.out = static_cast<__nv_bfloat16*>(a->out);
  p.o_st = a->out_stride_token;
  p.o_sh = a->out_stride_head;
  p.status = reinterpret_cast<int*>(w + L.status);
  p.ntasks = reinterpret_cast<const int*>(w + L.ntasks);
  p.nparts = reinterpret_cast<const int*>(w + L.nparts);
  p.part_base = reinterpret_cast<const int*>(w + L.part_base);
  p.tasks = reinterpret_cast<const pa::PlanTask*>(w + L.tasks);
  p.chunk_first = reinterpret_cast<const int*>(w + L.chunk_first);
  p.part_ml = reinterpret_cast<float*>(w + L.part_ml);
  p.part_o = reinterpret_cast<float*>(w + L.part_o);
  p.counters = a->merge_in_decode && pf_split == 0 ? reinterpret_cast<int*>(w + L.counters) : nullptr;
  p.pf_split = pf_split;
  p.n_chunks = L.budget;
  const int grid = pf_split > 0 ? a->batch * a->num_kv_heads * pf_split : L.budget;
  int rc;
  if (use_mx) {
    rc = pa::launch_mx_mxfp4(p, tk, tv, grid, stream);
  } else if (use_tc) {
    if (kind == pa::KIND_BF16)
      rc = pa::launch_tc_bf16(p, tk, tv, L.budget, stream);
    else if (kind == pa::KIND_FP8)
      rc = pa::launch_tc_fp8(p, tk, tv, L.budget, stream);
    else
      rc = pa::launch_tc_mxfp4(p, tk, tv, L.budget, stream);
  } else if (kind == pa::KIND_BF16)
    rc = pa::launch_tile_bf16(p, tk, tv, grid, stream);
  else if (kind == pa::KIND_FP8)
    rc = pa::launch_tile_fp8(p, tk, tv, grid, stream);
  else
    rc = pa::launch_tile_mxfp4(p, tk, tv, grid, stream);
  return rc == 0 ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

extern "C" {

int32_t pa_decode_abi_version(void) { return PA_DECODE_ABI_VERSION; }

const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported combination";
    case PA_ERR_WORKSPACE: return "workspace missing, too small or not 256-byte aligned";
    case PA_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

pa_status pa_decode_validate(const pa_decode_args* a) { return validate(a); }

size_t pa_decode_workspace_size(const pa_decode_args* a) {
  if (validate(a) != PA_OK) return 0;
  WsLayout L;
  if (make_layout(a, &L) != PA_OK) return 0;
  return L.total;
}

pa_status pa_decode_plan(const pa_decode_args* a, void* ws, size_t bytes, void* stream) {
  pa_status st = validate(a);
  if (st != PA_OK) return st;
  WsLayout L;
  if ((st = check_ws(a, ws, bytes, &L)) != PA_OK) return st;
  uint8_t* w = static_cast<uint8_t*>(ws);
  pa::PlanParams pp;
  pp.B = a->batch;
  pp.Hkv = a->num_kv_heads;
  pp.W = a->max_blocks_per_seq;
  pp.S = a->page_size;
  pp.qlen = a->qlen;
  pp.window = a->sliding_window;
  pp.max_partitions = L.max_partitions;
  pp.budget = L.budget;
  pp.ctx = a->context_lens;
  pp.status = reinterpret_cast<int*>(w + L.status);
  pp.ntasks = reinterpret_cast<int*>(w + L.ntasks);
  pp.nparts = reinterpret_cast<int*>(w + L.nparts);
  pp.part_base = reinterpret_cast<int*>(w + L.part_base);
  pp.counters = reinterpret_cast<int*>(w + L.counters);
  pp.tasks = reinterpret_cast<pa::PlanTask*>(w + L.tasks);
  pp.task_chunk = reinterpret_cast<int*>(w + L.task_chunk);
  pp.chunk_first = reinterpret_cast<int*>(w + L.chunk_first);
  int threads = (a->batch + 31) / 32 * 32;  // one thread per sequence, up to 1024
  threads = threads < 32 ? 32 : (threads > 1024 ? 1024 : threads);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1);
  cfg.blockDim = dim3(threads);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, pa::pa_plan_kernel, pp) != cudaSuccess) return PA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_decode(const pa_decode_args* a, void* ws, size_t bytes, void* stream) {
  return decode_launch(a, ws, bytes, stream, 0);
}

pa_status pa_decode_reduce(const pa_decode_args* a, void* ws, size_t bytes, void* stream) {
  pa_status st = validate(a);
  if (st != PA_OK) return st;
  WsLayout L;
  if ((st = check_ws(a, ws, bytes, &L)) != PA_OK) return st;
  if (a->batch == 0 || L.max_partitions < 2 || a->merge_in_decode) return PA_OK;
  uint8_t* w = static_cast<uint8_t*>(ws);
  pa::ReduceParams rp;
  rp.B = a->batch;
  rp.sinks = a->sinks;
  rp.qlen = a->qlen;
  rp.Hq = a->num_q_heads;
  rp.Hkv = a->num_kv_heads;
  rp.G = a->num_q_heads / a->num_kv_heads;
  rp.R = rp.G * a->qlen;
  rp.D = a->head_dim;
  rp.nparts = reinterpret_cast<const int*>(w + L.nparts);
  rp.part_base = reinterpret_cast<const int*>(w + L.part_base);
  rp.part_ml = reinterpret_cast<const float*>(w + L.part_ml);
  rp.part_o = reinterpret_cast<const float*>(w + L.part_o);
  rp.out = static_cast<__nv_bfloat16*>(a->out);
  rp.o_st = a->out_stride_token;
  rp.o_sh = a->out_stride_head;
  const long long rows = (long long)a->batch * a->qlen * a->num_q_heads;
  const unsigned grid = (unsigned)((rows + 7) / 8);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, pa::pa_reduce_kernel, rp) != cudaSuccess) return PA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

pa_status pa_decode_run(const pa_decode_args* a, void* ws, size_t bytes, void* stream) {
  pa_status st = validate(a);
  if (st != PA_OK) return st;
  WsLayout L;
  if ((st = check_ws(a, ws, bytes, &L)) != PA_OK) return st;
  const int split = single_launch_split(a, L);
  if (split > 0) return decode_launch(a, ws, bytes, stream, split);
  st = pa_decode_plan(a, ws, bytes, stream);
  if (st != PA_OK) return st;
  if ((st = pa_decode(a, ws, bytes, stream)) != PA_OK) return st;
  return pa_decode_reduce(a, ws, bytes, stream);
}

pa_status pa_decode_read_status(const void* ws, int32_t* host_status, void* stream) {
  if (!ws || !host_status) return PA_ERR_INVALID_ARG;
  cudaError_t e = cudaMemcpyAsync(host_status, ws, sizeof(int32_t), cudaMemcpyDeviceToHost,
                                  reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // extern "C"
