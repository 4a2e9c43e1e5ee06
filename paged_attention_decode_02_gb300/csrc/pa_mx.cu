// MXFP4 decode kernel with block-scaled tcgen05 QK (see pa_mx.cuh).
#include "pa_mx.cuh"

namespace pa {

int launch_mx_mxfp4(const DecodeParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int grid,
                    void* stream) {
  return launch_mx<MxCfg<3, 5>>(p, tk, tv, grid, stream);
}

}  // namespace pa
