// plans_cs.cu -- the cluster-split form of the FFMA kernel for small problems:
// one CTA per (output tile, k slice), the k slices of a tile in one
// thread-block cluster, their sums added through distributed shared memory
// in slice order (one launch, no workspace, no reduction kernel).  The
// kernel is the 64 x 128 tile, 16-k stage, k-chunked-A kernel of the
// tma_64x128x16_s6_o2 plan in that form, compiled in its own
// translation unit; the plans differ only in the most k slices per tile
// (2, 4, 8 -- the portable cluster size -- or 16).  Fields as in plans_tma.cu, then the
// largest cluster.
#include "plan_registry.h"
#include "sgemm_ffma.cuh"

namespace b2g {

const Plan kPlansCs[] = {
    B2G_FFMA_PLAN_CS("cs2_64x128x16_s6_o2", 64, 128, 16, 2, 2, 8, 6, kAKChunk, 1, 2, 2),
    B2G_FFMA_PLAN_CS("cs4_64x128x16_s6_o2", 64, 128, 16, 2, 2, 8, 6, kAKChunk, 1, 2, 4),
    B2G_FFMA_PLAN_CS("cs8_64x128x16_s6_o2", 64, 128, 16, 2, 2, 8, 6, kAKChunk, 1, 2, 8),
    B2G_FFMA_PLAN_CS("cs16_64x128x16_s6_o2", 64, 128, 16, 2, 2, 8, 6, kAKChunk, 1, 2, 16),
};
const int kNumPlansCs = sizeof(kPlansCs) / sizeof(kPlansCs[0]);

}  // namespace b2g
