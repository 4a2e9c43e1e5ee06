// pa_params.h -- parameter blocks shared by the host API and the sm_103a kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

namespace pa {

constexpr int kTileTokens = 256;  // the plan's work unit: ceil(L / 256) tiles per sequence
// What the plan charges each (sequence, KV head) unit on top of its tiles: a task's fixed
// cost (query load, first-slice latency, masked tail, merge and store) measured at about
// two tiles' worth of streaming on the long-context workloads.
constexpr int kUnitCostTiles = 2;
constexpr float kLog2e = 1.4426950408889634f;  // sinks are natural-log logits; scores are log2

// One task = a run of consecutive 256-token tiles of one (sequence, KV head) unit.
struct PlanTask {
  int32_t seq;
  int32_t hkv_part;  // hkv | (partition << 16)
  int32_t tile_begin;
  int32_t tile_end;
};

// Byte offsets of the workspace regions.
struct WsLayout {
  size_t status;   // int32 device status word (PA_DEVICE_*), then ntasks
  size_t ntasks;
  size_t nparts;       // int32 [B*Hkv]: partitions of each (sequence, KV head) unit
  size_t part_base;    // int32 [B*Hkv]: first partial slot of each split unit
  size_t counters;     // int32 [B*Hkv]: finished tasks per split unit
  size_t tasks;        // PlanTask [capacity], in unit order (and so in chunk order)
  size_t task_chunk;   // int32 [capacity]: the chunk (CTA) each task belongs to
  size_t chunk_first;  // int32 [budget + 1]: first task of each chunk; [budget] = ntasks
  size_t part_ml;    // float2 [slots, R]: (max in log2 units, sum)
  size_t part_o;     // float [slots, R, D]: normalised partial outputs
  size_t total;
  int32_t capacity;  // task capacity = B*Hkv + budget
  int32_t slots;     // partial slots = 2 * budget (split units only)
  int32_t budget;    // chunks = tile-kernel CTAs
  int32_t max_partitions;
};

// Tiles of a (sequence, KV head) unit: [*first, ceil(L / 256)), where *first is the tile
// holding the first token that any query position's sliding window reaches (0 without a
// window).  Returns the count.  The plan and the single-launch path both split units by it.
__device__ __forceinline__ int unit_tiles(int L, int qlen, int window, int* first) {
  int lo = window > 0 ? L - qlen - window + 1 : 0;
  lo = lo > 0 ? lo : 0;
  *first = lo / kTileTokens;
  return (L + kTileTokens - 1) / kTileTokens - *first;
}

struct DecodeParams {
  // single-launch mode (no plan, no reduce kernel): CTAs per (sequence, KV head) unit,
  // one thread-block cluster per unit, partials merged inside the cluster; 0: planned
  int pf_split;
  int n_chunks;  // the workspace's chunk count (its task list has n_chunks + 1 boundaries)
  int B, qlen, Hq, Hkv, G, R, D, S, W, NB;
  int64_t bt_stride;
  float scale_log2;  // softmax_scale * log2(e)
  int q_fp8, q_scale_per_row, scale_kind;
  int causal;  // qlen > 1: query position i sees tokens < L - qlen + 1 + i
  int window;  // > 0: query position i sees tokens > L - qlen + i - window
  int trans_v;  // value cache [NB, Hkv, D, S] (fp8 per-tensor)
  const float* sinks;  // [Hq] logits joining every row's softmax with a zero value, or null
  int q_quant;  // bf16 query quantised per head row to e4m3 (scale amax / 448)
  int drop_first_slice;  // test hook: warp 0 of each CTA never loads its first slice
  const void* q;
  int64_t q_st, q_sh;
  const float* q_scale;
  const uint8_t* k_scale;
  const uint8_t* v_scale;
  int64_t sc_sb, sc_sh;
  const int32_t* bt;
  const int32_t* ctx;
  __nv_bfloat16* out;
  int64_t o_st, o_sh;
  // workspace views
  int* status;
  const int* ntasks;
  const int* nparts;       // per unit
  const int* part_base;    // per unit
  const PlanTask* tasks;
  const int* chunk_first;  // CTA b runs tasks [chunk_first[b], chunk_first[b + 1])
  float* part_ml;
  float* part_o;
  int* counters;  // non-null: merge split sequences at the end of the tile kernel
};

struct PlanParams {
  int B, Hkv, W, S;
  int qlen, window;  // a unit's tiles start at the first tile any position's window holds
  int max_partitions;
  int budget;
  const int32_t* ctx;
  int* status;
  int* ntasks;
  int* nparts;
  int* part_base;
  int* counters;
  PlanTask* tasks;
  int* task_chunk;
  int* chunk_first;
};

struct ReduceParams {
  int B, qlen, Hq, Hkv, G, R, D;
  const float* sinks;  // [Hq] or null
  const int* nparts;
  const int* part_base;
  const float* part_ml;
  const float* part_o;
  __nv_bfloat16* out;
  int64_t o_st, o_sh;
};

// Kernel launchers, one per KV format (defined in the per-format translation units):
// `grid` CTAs, one per plan chunk.  Each returns a cudaError_t value (0 = success).
int launch_tile_bf16(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                     int grid, void* stream);
int launch_tile_fp8(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                    int grid, void* stream);
int launch_tile_mxfp4(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                      int grid, void* stream);

// Tensor-core (tcgen05) kernel launchers, head_dim 128, up to 32 query rows per KV
// head; the K / V tensor maps have boxes of min(page size, 128) rows.
int launch_tc_bf16(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                   int grid, void* stream);
int launch_tc_fp8(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                  int grid, void* stream);
int launch_tc_mxfp4(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                    int grid, void* stream);

// MXFP4 kernel with block-scaled tcgen05 QK and mma.sync PV (head_dim 128, up to 16 query
// rows); `tk` maps the key cache as unswizzled 64-byte rows, `tv` the value cache as
// 64-byte-swizzled rows, both in boxes of min(page size, 128) tokens.
int launch_mx_mxfp4(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                    int grid, void* stream);

// Tokens per warp slice, swizzle span (bytes) and head dims per warp of the tile kernel
// chosen for a format / head_dim / query-row count; the TMA box is min(S, slice tokens)
// rows high (16 with a transposed value cache, whose boxes are `dims_per_warp` high).
void tile_geometry(int kind, int head_dim, int rows, int* slice_tokens, int* swizzle_bytes,
                   int* dims_per_warp);

}  // namespace pa
