// plans_tma.cu -- bulk-tensor fed FFMA plans that read row-major A directly.
// Each line instantiates one kernel of sgemm_ffma.cuh: name, BM, BN, BK, warps
// along M, warps along N, per-thread columns TN, stages, A layout, feed,
// producer warps, FFMA issue order.
#include "plan_registry.h"
#include "sgemm_ffma.cuh"

namespace b2g {

const Plan kPlansTMA[] = {
    // A k-chunked by a 3-D bulk-tensor view ([BK/4][BM][4] in shared memory)
    B2G_FFMA_PLAN("tma_128x128x16_s6", 128, 128, 16, 4, 2, 8, 6, kAKChunk, kFeedTMA, 1, 0),
    B2G_FFMA_PLAN("tma_64x128x16_s6_o1", 64, 128, 16, 2, 2, 8, 6, kAKChunk, kFeedTMA, 1, 1),
    B2G_FFMA_PLAN("tma_64x128x16_s6_o2", 64, 128, 16, 2, 2, 8, 6, kAKChunk, kFeedTMA, 1, 2),
    // A staged k-chunked, rewritten transposed by each consumer warp for its rows
    B2G_FFMA_PLAN("tmaX_128x128x16_s6_o2", 128, 128, 16, 4, 2, 8, 6, kAKMajor, kFeedTMATrans, 1, 2),
    B2G_FFMA_PLAN("tmaX_64x128x16_s6_o1", 64, 128, 16, 2, 2, 8, 6, kAKMajor, kFeedTMATrans, 1, 1),
};
const int kNumPlansTMA = sizeof(kPlansTMA) / sizeof(kPlansTMA[0]);

}  // namespace b2g
