// tf32x3.h -- launchers of the 3xTF32 tensor-core SGEMM (tf32x3.cu).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

namespace b2g {

struct Tf32x3Params {
  int M, N, K;
  float alpha, beta;
  float* C;
  long long ldc;
  int c_vec4;  // C 16-byte aligned and ldc % 4 == 0
  int tiles_m, tiles_n, group_m, k_tiles;
  unsigned long long wait_limit_ns;
  int debug_stop_ktile;  // < 0 normally; >= 0 stops the copy issuer (timeout test)
  unsigned int* status;
  // Split tail (CTA-pair kernels): output tiles tail_first .. tiles-1 are each
  // cut into tail_splits k slices (1: none); a slice writes its raw sums, a
  // 256 x pn block, to work + (slice unit index) * 256 * pn, and
  // launch_tf32x3_tail_reduce adds each tile's slices in order.
  float* work;
  int tail_first, tail_splits;
};

// Tile shape of the tensor-core kernel.
constexpr int kTcBM = 128, kTcBN = 128, kTcBK = 32, kTcStages = 3;

// A -> Ahi, Alo (M x K, ld K) and B -> Bhi^T, Blo^T (N x K, ld K), in one
// launch.  A 16-byte aligned, lda % 4 == 0, K % 4 == 0; B read element by
// element.
cudaError_t launch_split_ab(const float* A, int M, int K, long long lda, float* Ahi, float* Alo,
                            const float* B, int N, long long ldb, float* Bhi, float* Blo,
                            int num_sms, cudaStream_t stream);

// The GEMM on the split operands.  maps: Ahi, Alo, Bhi^T, Blo^T as 2-D tensors
// {K, rows} with 128-byte swizzle and boxes {32, 128}.  tiles_m counts
// 128-row tiles.
cudaError_t launch_tf32x3(const Tf32x3Params& p, const CUtensorMap* maps, int num_sms,
                          cudaStream_t stream);

// The same GEMM with a CTA pair per 256 x pn output tile, pn = 128 or 256 (a
// cluster of two CTAs, one tcgen05.mma.cta_group::2 per step).  maps: boxes
// {32, 128} for A_hi and A_lo, {32, pn / 2} for B_hi^T and B_lo^T.  tiles_m
// counts 256-row tiles, tiles_n pn-column tiles.
cudaError_t launch_tf32x3_pair(const Tf32x3Params& p, const CUtensorMap* maps, int pn,
                               int num_sms, cudaStream_t stream);

// CTA pairs of the pn kernel resident at once on the current device (0 on
// failure): the persistent grid's size, which the host's split tail needs.
int tf32x3_pair_capacity(int pn, int num_sms);

// C = alpha * (slice 0 + ... ) + beta * C for every split tile of the pn kernel.
cudaError_t launch_tf32x3_tail_reduce(const Tf32x3Params& p, int pn, cudaStream_t stream);

}  // namespace b2g
