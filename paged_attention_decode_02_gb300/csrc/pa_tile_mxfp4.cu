// MXFP4 KV (e2m1 + e8m0 per 32 values) specialisation of the tile kernel.
#include "pa_configs.cuh"

namespace pa {

int launch_tile_mxfp4(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                      int grid, void* stream) {
  return launch_tile<CfgFp4D128M1>(p, tk, tv, grid, stream);
}

}  // namespace pa
