// pa_configs.cuh -- the tile-kernel specialisations this library builds.
//
// TileCfg<format, scale kind, head_dim, m-tiles (query rows / 16), token groups, warps per
// token group (head-dim split), tokens per warp slice, slots per warp ring, CTAs per SM,
// own merge buffer>.  The head_dim-128 fp8 and MXFP4 shapes keep 2 and 3 slices in flight
// per warp (enough to cover HBM latency at their per-warp rate) and spend the freed shared
// memory on a merge buffer, so every task merges in one pass; head_dim 64 (64- or 128-byte
// rows) streams 32-token slices, 2-4 in flight, with a merge buffer too.  64 query rows
// (four m-tiles) keep a 64 x head_dim fp32 accumulator: at head_dim 256 four warps and at
// head_dim 128 two warps split the head dim (64 dims each), at head_dim 64 one warp holds
// it.  One
// persistent CTA per SM; every warp streams its own slices.  The long-context shapes
// (fp8 / MXFP4, head_dim 128, up to 16 query rows) run eight warps, two per scheduler.
#pragma once

#include "pa_tile.cuh"

namespace pa {

using CfgBf16D64M1 = TileCfg<KIND_BF16, SK_NONE, 64, 1, 8, 1, 32, 2, 1, 1>;
using CfgBf16D64M2 = TileCfg<KIND_BF16, SK_NONE, 64, 2, 8, 1, 32, 2, 1, 1>;
using CfgBf16D64M4 = TileCfg<KIND_BF16, SK_NONE, 64, 4, 8, 1, 16, 3>;
using CfgBf16D128M1 = TileCfg<KIND_BF16, SK_NONE, 128, 1, 8, 1, 16, 2, 1, 1>;
using CfgBf16D128M2 = TileCfg<KIND_BF16, SK_NONE, 128, 2, 8, 1, 16, 3>;
using CfgBf16D128M4 = TileCfg<KIND_BF16, SK_NONE, 128, 4, 4, 2, 16, 3>;
using CfgBf16D256M1 = TileCfg<KIND_BF16, SK_NONE, 256, 1, 4, 2, 16, 2>;
using CfgBf16D256M2 = TileCfg<KIND_BF16, SK_NONE, 256, 2, 4, 2, 16, 2>;
using CfgBf16D256M4 = TileCfg<KIND_BF16, SK_NONE, 256, 4, 2, 4, 16, 2>;
// (TRV = 1: transposed value cache, per-tensor scales)
template <int SKT, int TRV = 0> using CfgFp8D64M1 = TileCfg<KIND_FP8, SKT, 64, 1, 8, 1, 32, 4, 1, 1, TRV>;
template <int SKT, int TRV = 0> using CfgFp8D64M2 = TileCfg<KIND_FP8, SKT, 64, 2, 8, 1, 32, 4, 1, 1, TRV>;
template <int SKT, int TRV = 0> using CfgFp8D64M4 = TileCfg<KIND_FP8, SKT, 64, 4, 8, 1, 16, 4, 1, 0, TRV>;
template <int SKT, int TRV = 0> using CfgFp8D128M1 = TileCfg<KIND_FP8, SKT, 128, 1, 8, 1, 32, 2, 1, 1, TRV>;
template <int SKT, int TRV = 0> using CfgFp8D128M2 = TileCfg<KIND_FP8, SKT, 128, 2, 8, 1, 16, 4, 1, 0, TRV>;
template <int SKT, int TRV = 0> using CfgFp8D128M4 = TileCfg<KIND_FP8, SKT, 128, 4, 4, 2, 16, 4, 1, 0, TRV>;
template <int SKT, int TRV = 0> using CfgFp8D256M1 = TileCfg<KIND_FP8, SKT, 256, 1, 4, 2, 32, 2, 1, 0, TRV>;
template <int SKT, int TRV = 0> using CfgFp8D256M2 = TileCfg<KIND_FP8, SKT, 256, 2, 4, 2, 16, 3, 1, 0, TRV>;
template <int SKT, int TRV = 0> using CfgFp8D256M4 = TileCfg<KIND_FP8, SKT, 256, 4, 2, 4, 16, 4, 1, 0, TRV>;
using CfgFp4D128M1 = TileCfg<KIND_FP4, SK_E8M0, 128, 1, 8, 1, 32, 3, 1, 1>;

}  // namespace pa
