// plans_t128x128.cu -- one FFMA kernel, 128 x 128 tiles of 16 k, 6 stages, A
// transposed ([BK][BM] in shared memory), zigzag FFMA order, in its own
// translation unit so that its machine code does not depend on what else is
// compiled, and the three plans that run it: A stored K x M (tmaT_), row-major
// A transposed into a workspace first (pre_), both operands packed aligned
// into a workspace first (pack_).  Fields as in plans_tma.cu.
#include "plan_registry.h"
#include "sgemm_ffma.cuh"

namespace b2g {

const Plan kPlansT128x128[] = {
    B2G_FFMA_PLAN("tmaT_128x128x16_s6_o2", 128, 128, 16, 4, 2, 8, 6, kAKMajor, kFeedTMA, 1, 2),
    B2G_FFMA_PLAN_PRE("pre_128x128x16_s6_o2", 128, 128, 16, 4, 2, 8, 6, 1, 2, 1),
    B2G_FFMA_PLAN_PRE("pack_128x128x16_s6_o2", 128, 128, 16, 4, 2, 8, 6, 1, 2, 2),
};
const int kNumPlansT128x128 = sizeof(kPlansT128x128) / sizeof(kPlansT128x128[0]);

}  // namespace b2g
