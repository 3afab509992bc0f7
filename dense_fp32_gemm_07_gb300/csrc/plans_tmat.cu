// plans_tmat.cu -- bulk-tensor fed FFMA plans whose A arrives transposed
// ([BK][BM] in shared memory): A stored K x M (op(A) = A^T), row-major A
// transposed into a workspace first (pre_), or both operands packed aligned
// into a workspace first (pack_).  Same fields as plans_tma.cu.
#include "sgemm_ffma.cuh"

namespace b2g {

const Plan kPlansT[] = {
    B2G_FFMA_PLAN("tmaT_64x128x16_s6", 64, 128, 16, 2, 2, 8, 6, kAKMajor, kFeedTMA, 1, 0),
    B2G_FFMA_PLAN("tmaT_64x128x16_s6_o2", 64, 128, 16, 2, 2, 8, 6, kAKMajor, kFeedTMA, 1, 2),
    B2G_FFMA_PLAN("tmaT_64x128x16_s6_o4", 64, 128, 16, 2, 2, 8, 6, kAKMajor, kFeedTMA, 1, 4),
    B2G_FFMA_PLAN("tmaT_128x64x16_s6_o2", 128, 64, 16, 4, 1, 8, 6, kAKMajor, kFeedTMA, 1, 2),
    B2G_FFMA_PLAN("tmaT_128x128x16_s6_o1", 128, 128, 16, 4, 2, 8, 6, kAKMajor, kFeedTMA, 1, 1),
    B2G_FFMA_PLAN("tmaT_128x128x16_s6_o2", 128, 128, 16, 4, 2, 8, 6, kAKMajor, kFeedTMA, 1, 2),
    // row-major A: transposed into a workspace first, then the kernels above
    B2G_FFMA_PLAN_PRE("pre_64x128x16_s6_o2", 64, 128, 16, 2, 2, 8, 6, 1, 2, 1),
    B2G_FFMA_PLAN_PRE("pre_128x64x16_s6_o2", 128, 64, 16, 4, 1, 8, 6, 1, 2, 1),
    B2G_FFMA_PLAN_PRE("pre_128x128x16_s6_o2", 128, 128, 16, 4, 2, 8, 6, 1, 2, 1),
    // any operands: A^T and B packed aligned into a workspace first
    B2G_FFMA_PLAN_PRE("pack_64x128x16_s6_o2", 64, 128, 16, 2, 2, 8, 6, 1, 2, 2),
    B2G_FFMA_PLAN_PRE("pack_128x64x16_s6_o2", 128, 64, 16, 4, 1, 8, 6, 1, 2, 2),
    B2G_FFMA_PLAN_PRE("pack_128x128x16_s6_o2", 128, 128, 16, 4, 2, 8, 6, 1, 2, 2),
};
const int kNumPlansT = sizeof(kPlansT) / sizeof(kPlansT[0]);

}  // namespace b2g
