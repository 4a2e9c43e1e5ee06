// bf16 KV specialisations of the tile kernel.
#include "pa_configs.cuh"

namespace pa {

int launch_tile_bf16(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                     int grid, void* stream) {
  if (p.D == 64)
    return p.R <= 16   ? launch_tile<CfgBf16D64M1>(p, tk, tv, grid, stream)
           : p.R <= 32 ? launch_tile<CfgBf16D64M2>(p, tk, tv, grid, stream)
                       : launch_tile<CfgBf16D64M4>(p, tk, tv, grid, stream);
  if (p.D == 128)
    return p.R <= 16   ? launch_tile<CfgBf16D128M1>(p, tk, tv, grid, stream)
           : p.R <= 32 ? launch_tile<CfgBf16D128M2>(p, tk, tv, grid, stream)
                       : launch_tile<CfgBf16D128M4>(p, tk, tv, grid, stream);
  return p.R <= 16   ? launch_tile<CfgBf16D256M1>(p, tk, tv, grid, stream)
         : p.R <= 32 ? launch_tile<CfgBf16D256M2>(p, tk, tv, grid, stream)
                     : launch_tile<CfgBf16D256M4>(p, tk, tv, grid, stream);
}

}  // namespace pa
