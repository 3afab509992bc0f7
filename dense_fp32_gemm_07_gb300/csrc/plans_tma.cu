// plans_tma.cu -- the bulk-tensor (TMA) fed FFMA plans.  Each line instantiates
// one kernel of sgemm_ffma.cuh: name, BM, BN, BK, warps along M, warps along N,
// per-thread columns TN, stages, A layout, feed, producer warps, FFMA order.
#include "sgemm_ffma.cuh"

namespace b2g {

const Plan kPlansTMA[] = {
    B2G_FFMA_PLAN("tma_128x128x16_s6", 128, 128, 16, 4, 2, 8, 6, kAKChunk, kFeedTMA, 1, 0),
    B2G_FFMA_PLAN("tma_128x128x16_s6_o1", 128, 128, 16, 4, 2, 8, 6, kAKChunk, kFeedTMA, 1, 1),
    B2G_FFMA_PLAN("tma_128x128x16_s6_o2", 128, 128, 16, 4, 2, 8, 6, kAKChunk, kFeedTMA, 1, 2),
    B2G_FFMA_PLAN("tma_128x128x32_s4", 128, 128, 32, 4, 2, 8, 4, kAKChunk, kFeedTMA, 1, 0),
    B2G_FFMA_PLAN("tma_64x128x16_s6", 64, 128, 16, 2, 2, 8, 6, kAKChunk, kFeedTMA, 1, 0),
    B2G_FFMA_PLAN("tma_64x128x16_s6_o1", 64, 128, 16, 2, 2, 8, 6, kAKChunk, kFeedTMA, 1, 1),
    B2G_FFMA_PLAN("tma_64x128x16_s6_o2", 64, 128, 16, 2, 2, 8, 6, kAKChunk, kFeedTMA, 1, 2),
    B2G_FFMA_PLAN("tma_128x64x16_s6", 128, 64, 16, 4, 1, 8, 6, kAKChunk, kFeedTMA, 1, 0),
    B2G_FFMA_PLAN("tma_32x64x32_s6", 32, 64, 32, 1, 1, 8, 6, kAKChunk, kFeedTMA, 1, 0),
    // A lands k-chunked in a staging slot; the producer warp writes it [BK][BM]
    B2G_FFMA_PLAN("tmaX_128x128x16_s6", 128, 128, 16, 4, 2, 8, 6, kAKMajor, kFeedTMATrans, 1, 0),
    B2G_FFMA_PLAN("tmaX_128x128x16_s6_o1", 128, 128, 16, 4, 2, 8, 6, kAKMajor, kFeedTMATrans, 1, 1),
    B2G_FFMA_PLAN("tmaX_128x128x16_s6_o2", 128, 128, 16, 4, 2, 8, 6, kAKMajor, kFeedTMATrans, 1, 2),
    B2G_FFMA_PLAN("tmaX_64x128x16_s6_o1", 64, 128, 16, 2, 2, 8, 6, kAKMajor, kFeedTMATrans, 1, 1),
    B2G_FFMA_PLAN("tmaX_128x128x32_s4_o1", 128, 128, 32, 4, 2, 8, 4, kAKMajor, kFeedTMATrans, 1, 1),
    B2G_FFMA_PLAN("tmaX_128x128x16_s8_o1", 128, 128, 16, 4, 2, 8, 8, kAKMajor, kFeedTMATrans, 1, 1),
    B2G_FFMA_PLAN("tmaX_128x128x16_s9_o1", 128, 128, 16, 4, 2, 8, 9, kAKMajor, kFeedTMATrans, 1, 1),
    // A stored K x M (op(A) = A^T): the copy lands transposed, [BK][BM]
    B2G_FFMA_PLAN("tmaT_128x128x16_s6", 128, 128, 16, 4, 2, 8, 6, kAKMajor, kFeedTMA, 1, 0),
    B2G_FFMA_PLAN("tmaT_128x128x16_s6_o1", 128, 128, 16, 4, 2, 8, 6, kAKMajor, kFeedTMA, 1, 1),
    B2G_FFMA_PLAN("tmaT_64x128x16_s6", 64, 128, 16, 2, 2, 8, 6, kAKMajor, kFeedTMA, 1, 0),
    // row-major A: transposed into a workspace first, then the kernels above
    B2G_FFMA_PLAN_PRE("pre_128x128x16_s6_o1", 128, 128, 16, 4, 2, 8, 6, 1, 1, 1),
    B2G_FFMA_PLAN_PRE("pre_64x128x16_s6", 64, 128, 16, 2, 2, 8, 6, 1, 0, 1),
    // any operands: A^T and B packed aligned into a workspace first
    B2G_FFMA_PLAN_PRE("pack_128x128x16_s6_o1", 128, 128, 16, 4, 2, 8, 6, 1, 1, 2),
    B2G_FFMA_PLAN_PRE("pack_64x128x16_s6", 64, 128, 16, 2, 2, 8, 6, 1, 0, 2),
};
const int kNumPlansTMA = sizeof(kPlansTMA) / sizeof(kPlansTMA[0]);

}  // namespace b2g
