// plans_general.cu -- the 4-byte cp.async fed FFMA plans: any alignment, any
// leading dimension, both op() flags.  Same fields as plans_tma.cu.
#include "plan_registry.h"
#include "sgemm_ffma.cuh"

namespace b2g {

const Plan kPlansGeneral[] = {
    B2G_FFMA_PLAN("gen_128x128x16_s4", 128, 128, 16, 4, 2, 8, 4, kAKMajor, kFeedCpAsync, 4, 0),
    B2G_FFMA_PLAN("gen_64x64x16_s4", 64, 64, 16, 2, 1, 8, 4, kAKMajor, kFeedCpAsync, 2, 0),
};
const int kNumPlansGeneral = sizeof(kPlansGeneral) / sizeof(kPlansGeneral[0]);

}  // namespace b2g
