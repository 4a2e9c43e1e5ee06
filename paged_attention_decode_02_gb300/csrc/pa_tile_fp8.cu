// fp8 e4m3 KV (per-tensor or per-token scales) specialisations of the tile kernel.
#include "pa_configs.cuh"

namespace pa {

template <int SKT, int TRV>
static int launch_fp8(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                      int grid, void* stream) {
  if (p.D == 64)
    return p.R <= 16   ? launch_tile<CfgFp8D64M1<SKT, TRV>>(p, tk, tv, grid, stream)
           : p.R <= 32 ? launch_tile<CfgFp8D64M2<SKT, TRV>>(p, tk, tv, grid, stream)
                       : launch_tile<CfgFp8D64M4<SKT, TRV>>(p, tk, tv, grid, stream);
  if (p.D == 128)
    return p.R <= 16   ? launch_tile<CfgFp8D128M1<SKT, TRV>>(p, tk, tv, grid, stream)
           : p.R <= 32 ? launch_tile<CfgFp8D128M2<SKT, TRV>>(p, tk, tv, grid, stream)
                       : launch_tile<CfgFp8D128M4<SKT, TRV>>(p, tk, tv, grid, stream);
  return p.R <= 16   ? launch_tile<CfgFp8D256M1<SKT, TRV>>(p, tk, tv, grid, stream)
         : p.R <= 32 ? launch_tile<CfgFp8D256M2<SKT, TRV>>(p, tk, tv, grid, stream)
                     : launch_tile<CfgFp8D256M4<SKT, TRV>>(p, tk, tv, grid, stream);
}

int launch_tile_fp8(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                    int grid, void* stream) {
  if (p.trans_v) return launch_fp8<SK_TENSOR, 1>(p, tk, tv, grid, stream);  // per tensor only
  return p.scale_kind == SK_TOKEN ? launch_fp8<SK_TOKEN, 0>(p, tk, tv, grid, stream)
                                  : launch_fp8<SK_TENSOR, 0>(p, tk, tv, grid, stream);
}

}  // namespace pa
