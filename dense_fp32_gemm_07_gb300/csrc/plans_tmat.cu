// plans_tmat.cu -- alternative FFMA issue orders of the transposed-A kernels
// (A stored K x M), kept for comparison sweeps; the plans the tune table uses
// live one kernel per file in plans_t*.cu.  Fields as in plans_tma.cu.
#include "plan_registry.h"
#include "sgemm_ffma.cuh"

namespace b2g {

const Plan kPlansT[] = {
    B2G_FFMA_PLAN("tmaT_64x128x16_s6", 64, 128, 16, 2, 2, 8, 6, kAKMajor, kFeedTMA, 1, 0),
    B2G_FFMA_PLAN("tmaT_64x128x16_s6_o4", 64, 128, 16, 2, 2, 8, 6, kAKMajor, kFeedTMA, 1, 4),
    B2G_FFMA_PLAN("tmaT_128x128x16_s6_o1", 128, 128, 16, 4, 2, 8, 6, kAKMajor, kFeedTMA, 1, 1),
};
const int kNumPlansT = sizeof(kPlansT) / sizeof(kPlansT[0]);

}  // namespace b2g
