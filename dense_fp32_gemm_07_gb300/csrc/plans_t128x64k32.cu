// plans_t128x64k32.cu -- one FFMA kernel, 128 x 64 tiles of 32 k, 3 stages
// (the same 72 KB ring as 6 stages of 16 k, so still three CTAs per SM, but
// half the full/empty barrier round trips per k), A transposed ([BK][BM] in
// shared memory), packed two-lane FP32 FMAs, in its own translation unit so
// that its machine code does not depend on what else is compiled, and the
// four plans that run it: A stored K x M (tmaT_), row-major A transposed into
// a workspace first (pre_), both operands packed aligned into a workspace
// first (pack_), B stored N x K transposed (and A unless stored K x M) into a
// workspace first (pret_).
// Fields as in plans_tma.cu.
#include "plan_registry.h"
#include "sgemm_ffma.cuh"

namespace b2g {

const Plan kPlansT128x64k32[] = {
    B2G_FFMA_PLAN("tmaT_128x64x32_s3_o5", 128, 64, 32, 4, 1, 8, 3, kAKMajor, kFeedTMA, 1, 5),
    B2G_FFMA_PLAN_PRE("pre_128x64x32_s3_o5", 128, 64, 32, 4, 1, 8, 3, 1, 5, 1),
    B2G_FFMA_PLAN_PRE("pack_128x64x32_s3_o5", 128, 64, 32, 4, 1, 8, 3, 1, 5, 2),
    B2G_FFMA_PLAN_PRE("pret_128x64x32_s3_o5", 128, 64, 32, 4, 1, 8, 3, 1, 5, 3),
};
const int kNumPlansT128x64k32 = sizeof(kPlansT128x64k32) / sizeof(kPlansT128x64k32[0]);

}  // namespace b2g
