// pa_configs.cuh -- the tile-kernel specialisations this library builds.
//
// TileCfg<format, head_dim, m-tiles (query rows / 16), token groups, warps per
// row (head-dim split), tokens per pipeline stage, stages>.  A stage holds about
// 32 KiB of K+V; one persistent CTA per SM.
#pragma once

#include "pa_tile.cuh"

namespace pa {

using CfgBf16D128M1 = TileCfg<KIND_BF16, 128, 1, 4, 1, 64, 4>;
using CfgBf16D128M2 = TileCfg<KIND_BF16, 128, 2, 4, 1, 64, 4>;
using CfgBf16D256M1 = TileCfg<KIND_BF16, 256, 1, 2, 2, 32, 4>;
using CfgBf16D256M2 = TileCfg<KIND_BF16, 256, 2, 2, 2, 32, 4>;
using CfgFp8D128M1 = TileCfg<KIND_FP8, 128, 1, 4, 1, 128, 4>;
using CfgFp8D128M2 = TileCfg<KIND_FP8, 128, 2, 4, 1, 128, 4>;
using CfgFp8D256M1 = TileCfg<KIND_FP8, 256, 1, 2, 2, 64, 4>;
using CfgFp8D256M2 = TileCfg<KIND_FP8, 256, 2, 2, 2, 64, 4>;
using CfgFp4D128M1 = TileCfg<KIND_FP4, 128, 1, 4, 1, 256, 4>;

}  // namespace pa
