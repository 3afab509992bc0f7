// plans_t64x128k32.cu -- the twin of plans_t128x64k32.cu with 64 x 128 tiles
// (warps 2 x 2, each 32 x 64): 32-k stages, 3 stages of 24 KB, A transposed
// ([BK][BM] in shared memory), packed two-lane FP32 FMAs, in its own
// translation unit.  The table takes it instead of the 128 x 64 kernel when
// 64-row tiles cover less padded area (M = 64 or 192: a 128-row tile would
// pad a quarter or half of its rows); at 4096^3 both run at the same rate.
// The four plans: A stored K x M (tmaT_), row-major A transposed into a
// workspace first (pre_), both operands packed aligned into a workspace first
// (pack_), B stored N x K transposed (and A unless stored K x M) into a
// workspace first (pret_).  Fields as in plans_tma.cu.
#include "plan_registry.h"
#include "sgemm_ffma.cuh"

namespace b2g {

const Plan kPlansT64x128k32[] = {
    B2G_FFMA_PLAN("tmaT_64x128x32_s3_o5", 64, 128, 32, 2, 2, 8, 3, kAKMajor, kFeedTMA, 1, 5),
    B2G_FFMA_PLAN_PRE("pre_64x128x32_s3_o5", 64, 128, 32, 2, 2, 8, 3, 1, 5, 1),
    B2G_FFMA_PLAN_PRE("pack_64x128x32_s3_o5", 64, 128, 32, 2, 2, 8, 3, 1, 5, 2),
    B2G_FFMA_PLAN_PRE("pret_64x128x32_s3_o5", 64, 128, 32, 2, 2, 8, 3, 1, 5, 3),
};
const int kNumPlansT64x128k32 = sizeof(kPlansT64x128k32) / sizeof(kPlansT64x128k32[0]);

}  // namespace b2g
