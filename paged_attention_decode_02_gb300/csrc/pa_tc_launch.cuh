// Tensor-core (tcgen05) decode kernel specialisations: one per KV format, scale kind and
// padded query-row count (16 or 32).  Each pa_tc_<format>.cu defines one PA_TC_PART_*.
#pragma once

#include "pa_tc.cuh"

namespace pa {

#if defined(PA_TC_PART_BF16)
int launch_tc_bf16(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int grid, void* stream) {
  return p.R <= 16 ? launch_tc<TcCfg<KIND_BF16, SK_NONE, 16, 3>>(p, tk, tv, grid, stream)
                   : launch_tc<TcCfg<KIND_BF16, SK_NONE, 32, 2>>(p, tk, tv, grid, stream);
}
#elif defined(PA_TC_PART_FP8)
int launch_tc_fp8(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int grid, void* stream) {
  if (p.scale_kind == SK_TOKEN)
    return p.R <= 16 ? launch_tc<TcCfg<KIND_FP8, SK_TOKEN, 16, 4>>(p, tk, tv, grid, stream)
                     : launch_tc<TcCfg<KIND_FP8, SK_TOKEN, 32, 3>>(p, tk, tv, grid, stream);
  return p.R <= 16 ? launch_tc<TcCfg<KIND_FP8, SK_TENSOR, 16, 4>>(p, tk, tv, grid, stream)
                   : launch_tc<TcCfg<KIND_FP8, SK_TENSOR, 32, 3>>(p, tk, tv, grid, stream);
}
#elif defined(PA_TC_PART_FP4)
int launch_tc_mxfp4(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int grid, void* stream) {
  return p.R <= 16 ? launch_tc<TcCfg<KIND_FP4, SK_E8M0, 16, 4>>(p, tk, tv, grid, stream)
                   : launch_tc<TcCfg<KIND_FP4, SK_E8M0, 32, 3>>(p, tk, tv, grid, stream);
}
#endif

}  // namespace pa
