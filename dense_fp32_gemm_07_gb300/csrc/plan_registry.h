// plan_registry.h -- the plan tables each kernel translation unit compiles,
// and the launchers of the reduction kernels, for the C-ABI layer (host.cu).
// A translation unit that defines a table includes this header so the table
// has external linkage.
#pragma once
#include <cstddef>

#include "sgemm_params.h"

namespace b2g {

// Skinny-M plans (M <= BM), compiled in skinny.cu and skinny_tma.cu.
extern const Plan kPlansSkinny[];
extern const int kNumPlansSkinny;
extern const Plan kPlansSkinnyTma[];
extern const int kNumPlansSkinnyTma;
// C = alpha * sum_s P[s] + beta * C over the M x N window (split-K reduction).
// dependent: launched as a programmatic dependent of the kernel just before it
// on `stream` (it may start early and waits for that kernel's results).
cudaError_t launch_splitk_reduce(const SgemmParams& p, cudaStream_t stream, int num_sms,
                                 bool dependent);

// FFMA plans' split tail: C = alpha * (slice 0 + slice 1 + ...) + beta * C for
// every split tile (p.tail_splits > 1), BM x BN the plan's tile.
cudaError_t launch_tail_reduce(const SgemmParams& p, int BM, int BN, cudaStream_t stream);

// Workspace bytes that the tune table's plan cannot do without for these
// row-major arguments (A^T for the transposing plans; 0 when none).  It is at
// most what b2g_sgemm_workspace_size reports, which adds room for the split
// tail's partial sums; with less than that the plan runs without the split.
// Returns 0 or a B2G_ERR_* code.
int sgemm_min_workspace_bytes(int M, int N, int K, float alpha, const float* A, int lda,
                              const float* B, int ldb, const float* C, int ldc, size_t* bytes);

// Plans compiled in each kernel translation unit.
extern const Plan kPlansTMA[];
extern const int kNumPlansTMA;
extern const Plan kPlansT[];
extern const int kNumPlansT;
extern const Plan kPlansT64x128[];
extern const int kNumPlansT64x128;
extern const Plan kPlansT128x64[];
extern const int kNumPlansT128x64;
extern const Plan kPlansT128x64k32[];
extern const int kNumPlansT128x64k32;
extern const Plan kPlansT64x128k32[];
extern const int kNumPlansT64x128k32;
extern const Plan kPlansT128x128[];
extern const int kNumPlansT128x128;
extern const Plan kPlansGeneral[];
extern const int kNumPlansGeneral;
extern const Plan kPlansCs[];
extern const int kNumPlansCs;
extern const Plan kPlansTmaO5[];
extern const int kNumPlansTmaO5;
extern const Plan kPlansWarpk[];
extern const int kNumPlansWarpk;

}  // namespace b2g
