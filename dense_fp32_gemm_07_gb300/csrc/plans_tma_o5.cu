// plans_tma_o5.cu -- the split-tail kernel for products below about 1e9
// multiply-adds that the one-launch wk_ plans leave to it (64 x 128 tiles,
// 16-k stages, 6 stages, A k-chunked by a 3-D bulk-tensor view: no transpose
// before it) with packed two-lane FP32 FMAs instead of scalar ones, in its
// own translation unit.  Fields as in plans_tma.cu.
#include "plan_registry.h"
#include "sgemm_ffma.cuh"

namespace b2g {

const Plan kPlansTmaO5[] = {
    B2G_FFMA_PLAN("tma_64x128x16_s6_o5", 64, 128, 16, 2, 2, 8, 6, kAKChunk, kFeedTMA, 1, 5),
};
const int kNumPlansTmaO5 = sizeof(kPlansTmaO5) / sizeof(kPlansTmaO5[0]);

}  // namespace b2g
