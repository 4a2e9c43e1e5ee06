// pa_decode.cu -- plan and reduce kernels, and the host side of the C ABI
// (validation, workspace layout, TMA descriptors, launches).  See include/pa_decode.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "pa_configs.cuh"
#include "../../include/pa_decode.h"

namespace pa {

// ------------------------------------------------------------------------------------
// Plan: ceil(L/256) tiles per sequence ("[FlyDSL] pa_decode: zero V rows past the context
// before PV", Root cause), split into partitions proportional to the sequence's share of
// all tiles so that the task count stays within the budget ("[FlyDSL] pa_decode: MXFP4
// K/V ...", plan-free commit: tasks from a 2 x CU budget; max_partitions caps the split).
// ------------------------------------------------------------------------------------
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

__global__ void __launch_bounds__(1024) pa_plan_kernel(const PlanParams pp) {
  __shared__ long long sh64[32];
  __shared__ int sh32[32];
  __shared__ int sh32b[32];
  const int tid = threadIdx.x;
  const int cap = pp.W * pp.S;
  pdl_wait_prior();          // the previous kernel may still read this workspace
  pdl_launch_dependents();  // the tile kernel may launch now; it waits for this grid
  if (tid == 0) *pp.status = 0;
  __syncthreads();
  int clamped = 0;
  long long local = 0;
  for (int s = tid; s < pp.B; s += blockDim.x)
    local += (clamp_len(pp.ctx[s], cap, &clamped) + kTileTokens - 1) / kTileTokens;
  long long total_tiles;
  (void)block_exclusive_scan<long long>(local, &total_tiles, sh64);
  total_tiles *= pp.Hkv;
  if (clamped) atomicOr(pp.status, ST_CLAMPED);

  int carry_tasks = 0, carry_slots = 0;
  for (int base = 0; base < pp.B; base += blockDim.x) {
    const int s = base + tid;
    int P = 0, tiles = 0;
    if (s < pp.B) {
      int dummy = 0;
      tiles = (clamp_len(pp.ctx[s], cap, &dummy) + kTileTokens - 1) / kTileTokens;
      if (tiles == 0) {
        P = 1;
      } else {
        long long share = total_tiles > 0 ? (long long)tiles * pp.budget / total_tiles : 1;
        if (share < 1) share = 1;
        if (share > pp.max_partitions) share = pp.max_partitions;
        if (share > tiles) share = tiles;
        P = (int)share;
      }
    }
    const int ntask = s < pp.B ? P * pp.Hkv : 0;
    const int nslot = (s < pp.B && P >= 2) ? P * pp.Hkv : 0;
    int tot_t, tot_s;
    const int off_t = block_exclusive_scan<int>(ntask, &tot_t, sh32);
    const int off_s = block_exclusive_scan<int>(nslot, &tot_s, sh32b);
    if (s < pp.B) {
      pp.nparts[s] = P;
      pp.part_base[s] = carry_slots + off_s;
      for (int h = 0; h < pp.Hkv; ++h) pp.counters[s * pp.Hkv + h] = 0;
      for (int h = 0; h < pp.Hkv; ++h)
        for (int q = 0; q < P; ++q) {
          PlanTask tk;
          tk.seq = s;
          tk.hkv_part = h | (q << 16);
          tk.tile_begin = (int)((long long)q * tiles / P);
          tk.tile_end = (int)((long long)(q + 1) * tiles / P);
          pp.tasks[carry_tasks + off_t + h * P + q] = tk;
        }
    }
    carry_tasks += tot_t;
    carry_slots += tot_s;
  }
  if (tid == 0) *pp.ntasks = carry_tasks;
}

// ------------------------------------------------------------------------------------
// Reduce: merge the partitions of each split sequence in a fixed order
// ("[FlyDSL] pa_decode: MXFP4 K/V ...", Self-Review: the partition reducer).
// One warp per output row.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) pa_reduce_kernel(const ReduceParams rp) {
  __shared__ float wsh[8][128];  // normalised partition weights of each warp's row
  pdl_wait_prior();  // the tile kernel's partials are complete and visible from here on
  pdl_launch_dependents();  // a following plan may launch; it waits before writing
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const long long row = (long long)blockIdx.x * 8 + wid;
  const long long rows = (long long)rp.B * rp.qlen * rp.Hq;
  if (row >= rows) return;
  const int s = (int)(row / ((long long)rp.qlen * rp.Hq));
  const int P = rp.nparts[s];
  if (P < 2) return;
  const int rem = (int)(row % ((long long)rp.qlen * rp.Hq));
  const int i = rem / rp.Hq, h = rem % rp.Hq, hkv = h / rp.G;
  const int r = i * rp.G + h % rp.G;
  const long long base = (long long)rp.part_base[s] + (long long)hkv * P;
  const float2* ml = reinterpret_cast<const float2*>(rp.part_ml);
  float* w = wsh[wid];
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
  const float inv = W > 0.f ? 1.f / W : 0.f;
  __syncwarp();
  for (int q = lane; q < P; q += 32) w[q] *= inv;
  __syncwarp();
  __nv_bfloat16* dst = rp.out + (long long)(s * rp.qlen + i) * rp.o_st + (long long)h * rp.o_sh;
  // each lane owns 4 consecutive dims per 128; partitions are added in a fixed order
  for (int d0 = 4 * lane; d0 < rp.D; d0 += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int q = 0;
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
    dst[d0] = __float2bfloat16_rn(acc.x);
    dst[d0 + 1] = __float2bfloat16_rn(acc.y);
    dst[d0 + 2] = __float2bfloat16_rn(acc.z);
    dst[d0 + 3] = __float2bfloat16_rn(acc.w);
  }
}

// Tokens per warp slice (the TMA box is min(S, this) rows high) and swizzle span of the
// tile kernel that serves a format / head_dim / query-row count.
void tile_geometry(int kind, int head_dim, int rows, int* tw, int* sub) {
  if (kind == KIND_BF16) {
    if (head_dim == 128) {
      *tw = rows <= 16 ? CfgBf16D128M1::TW : CfgBf16D128M2::TW;
    } else {
      *tw = rows <= 16 ? CfgBf16D256M1::TW : CfgBf16D256M2::TW;
    }
    *sub = 128;
  } else if (kind == KIND_FP8) {
    if (head_dim == 128) {
      *tw = rows <= 16 ? CfgFp8D128M1<SK_TOKEN>::TW : CfgFp8D128M2<SK_TOKEN>::TW;
    } else {
      *tw = rows <= 16 ? CfgFp8D256M1<SK_TOKEN>::TW : CfgFp8D256M2<SK_TOKEN>::TW;
    }
    *sub = 128;
  } else {
    *tw = CfgFp4D128M1::TW;
    *sub = CfgFp4D128M1::SUB;
  }
}

}  // namespace pa

// ======================================================================================
// Host side
// ======================================================================================
namespace {

using pa::WsLayout;

constexpr int kMaxRows = 32;         // G * qlen served by the tile kernels
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
  if (a->head_dim != 128 && a->head_dim != 256) return PA_ERR_UNSUPPORTED;
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
  if (a->q_dtype != PA_Q_BF16 && a->q_dtype != PA_Q_FP8_E4M3) return PA_ERR_INVALID_ARG;
  if (a->merge_in_decode != 0 && a->merge_in_decode != 1) return PA_ERR_INVALID_ARG;
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
  const int qel = a->q_dtype == PA_Q_BF16 ? 2 : 1;
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

pa_status make_layout(const pa_decode_args* a, WsLayout* L) {
  int budget = 0, maxp = 0;
  pa_status st = split_params(a, &budget, &maxp);
  if (st != PA_OK) return st;
  const int G = a->num_q_heads / a->num_kv_heads;
  const int R = G * a->qlen;
  const int B = a->batch;
  L->budget = budget;
  L->max_partitions = maxp;
  L->capacity = B * a->num_kv_heads + budget;
  L->slots = maxp >= 2 ? budget : 0;
  size_t off = 0;
  L->status = off;
  L->ntasks = off + 4;
  off = 256;
  L->nparts = off;
  off = align_up(off + 4 * (size_t)B, 256);
  L->part_base = off;
  off = align_up(off + 4 * (size_t)B, 256);
  L->counters = off;
  off = align_up(off + 4 * (size_t)B * a->num_kv_heads, 256);
  L->tasks = off;
  off = align_up(off + sizeof(pa::PlanTask) * (size_t)L->capacity, 256);
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
  pp.max_partitions = L.max_partitions;
  pp.budget = L.budget;
  pp.ctx = a->context_lens;
  pp.status = reinterpret_cast<int*>(w + L.status);
  pp.ntasks = reinterpret_cast<int*>(w + L.ntasks);
  pp.nparts = reinterpret_cast<int*>(w + L.nparts);
  pp.part_base = reinterpret_cast<int*>(w + L.part_base);
  pp.counters = reinterpret_cast<int*>(w + L.counters);
  pp.tasks = reinterpret_cast<pa::PlanTask*>(w + L.tasks);
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
  pa_status st = validate(a);
  if (st != PA_OK) return st;
  WsLayout L;
  if ((st = check_ws(a, ws, bytes, &L)) != PA_OK) return st;
  if (a->batch == 0) return PA_OK;
  int sms = 0;
  if (device_sms(&sms)) return PA_ERR_CUDA;
  const int G = a->num_q_heads / a->num_kv_heads;
  const int R = G * a->qlen;
  const int kind = a->kv_dtype == PA_KV_BF16 ? pa::KIND_BF16 : (a->kv_dtype == PA_KV_FP8_E4M3 ? pa::KIND_FP8 : pa::KIND_FP4);
  int tc = 0, sub = 0;
  pa::tile_geometry(kind, a->head_dim, R, &tc, &sub);
  const int box = a->page_size < tc ? a->page_size : tc;
  CUtensorMap tk, tv;
  if ((st = cache_map(a, a->key_cache, sub, box, &tk)) != PA_OK) return st;
  if ((st = cache_map(a, a->value_cache, sub, box, &tv)) != PA_OK) return st;

  uint8_t* w = static_cast<uint8_t*>(ws);
  pa::DecodeParams p;
  p.B = a->batch;
  p.qlen = a->qlen;
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
  p.part_ml = reinterpret_cast<float*>(w + L.part_ml);
  p.part_o = reinterpret_cast<float*>(w + L.part_o);
  p.counters = a->merge_in_decode ? reinterpret_cast<int*>(w + L.counters) : nullptr;
  int rc;
  if (kind == pa::KIND_BF16)
    rc = pa::launch_tile_bf16(p, tk, tv, L.capacity, sms, stream);
  else if (kind == pa::KIND_FP8)
    rc = pa::launch_tile_fp8(p, tk, tv, L.capacity, sms, stream);
  else
    rc = pa::launch_tile_mxfp4(p, tk, tv, L.capacity, sms, stream);
  return rc == 0 ? PA_OK : PA_ERR_CUDA;
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
  rp.qlen = a->qlen;
  rp.Hq = a->num_q_heads;
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
  pa_status st = pa_decode_plan(a, ws, bytes, stream);
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
