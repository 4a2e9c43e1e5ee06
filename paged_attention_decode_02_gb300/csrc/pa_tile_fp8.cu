// fp8 e4m3 KV (per-tensor or per-token scales) specialisations of the tile kernel.
#include "pa_configs.cuh"

namespace pa {

int launch_tile_fp8(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                    int grid_cap, int num_sms, void* stream) {
  if (p.D == 128)
    return p.R <= 16 ? launch_tile<CfgFp8D128M1>(p, tk, tv, grid_cap, num_sms, stream)
                     : launch_tile<CfgFp8D128M2>(p, tk, tv, grid_cap, num_sms, stream);
  return p.R <= 16 ? launch_tile<CfgFp8D256M1>(p, tk, tv, grid_cap, num_sms, stream)
                   : launch_tile<CfgFp8D256M2>(p, tk, tv, grid_cap, num_sms, stream);
}

}  // namespace pa
