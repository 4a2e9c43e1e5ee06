// pa_params.h -- parameter blocks shared by the host API and the sm_103a kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

namespace pa {

constexpr int kTileTokens = 256;  // the plan's work unit: ceil(L / 256) tiles per sequence

// One task = a run of consecutive 256-token tiles of one (sequence, KV head).
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
  size_t nparts;     // int32 [B]: partitions of each sequence
  size_t part_base;  // int32 [B]: first partial slot of each split sequence
  size_t counters;   // int32 [B*Hkv]: finished tasks per split (sequence, KV head)
  size_t tasks;      // PlanTask [capacity]
  size_t part_ml;    // float2 [slots, R]: (max in log2 units, sum)
  size_t part_o;     // float [slots, R, D]: normalised partial outputs
  size_t total;
  int32_t capacity;  // task capacity = B*Hkv + budget
  int32_t slots;     // partial slots = budget (split sequences only)
  int32_t budget;
  int32_t max_partitions;
};

struct DecodeParams {
  int B, qlen, Hq, Hkv, G, R, D, S, W, NB;
  int64_t bt_stride;
  float scale_log2;  // softmax_scale * log2(e)
  int q_fp8, q_scale_per_row, scale_kind;
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
  const int* nparts;
  const int* part_base;
  const PlanTask* tasks;
  float* part_ml;
  float* part_o;
  int* counters;  // non-null: merge split sequences at the end of the tile kernel
};

struct PlanParams {
  int B, Hkv, W, S;
  int max_partitions;
  int budget;
  const int32_t* ctx;
  int* status;
  int* ntasks;
  int* nparts;
  int* part_base;
  int* counters;
  PlanTask* tasks;
};

struct ReduceParams {
  int B, qlen, Hq, G, R, D;
  const int* nparts;
  const int* part_base;
  const float* part_ml;
  const float* part_o;
  __nv_bfloat16* out;
  int64_t o_st, o_sh;
};

// Kernel launchers, one per KV format (defined in the per-format translation units).
// Each returns a cudaError_t value (0 = success).
int launch_tile_bf16(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                     int grid_cap, int num_sms, void* stream);
int launch_tile_fp8(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                    int grid_cap, int num_sms, void* stream);
int launch_tile_mxfp4(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                      int grid_cap, int num_sms, void* stream);

// Tokens per warp slice and swizzle span (bytes) of the tile kernel chosen for a
// format / head_dim / query-row count; the TMA box is min(S, slice tokens) rows high.
void tile_geometry(int kind, int head_dim, int rows, int* slice_tokens, int* swizzle_bytes);

}  // namespace pa
