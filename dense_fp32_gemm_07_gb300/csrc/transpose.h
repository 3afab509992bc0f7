// transpose.h -- launcher of the A -> A^T workspace kernel (transpose.cu).
#pragma once
#include <cuda_runtime.h>

namespace b2g {

// At[k][m] = A[m][k] for m < M, k < K; columns M .. ldat-1 of At get zeros.
// A: 16-byte aligned, lda % 4 == 0, K % 4 == 0.  At: 16-byte aligned,
// ldat % 4 == 0, ldat >= M, K x ldat floats.
// `batch` problems, A and At advancing by strideA and strideAt elements.
cudaError_t launch_transpose_a(const float* A, int M, int K, long long lda, float* At,
                               long long ldat, cudaStream_t stream, int batch = 1,
                               long long strideA = 0, long long strideAt = 0);

// One packing job: out (R x Cc, leading dimension ldo) = trans ? in^T : in,
// in read element by element (any alignment and leading dimension ld), in 32 x
// 32 tiles; `batch` problems advance by stride_in and stride_out elements.
struct PackJob {
  const float* in;
  long long ld;
  int trans, R, Cc;
  float* out;
  long long ldo, stride_in, stride_out;
  int tiles_x, tiles_y;  // 32 x 32 tiles along Cc and R
};
PackJob pack_job(const float* in, long long ld, int trans, int R, int Cc, float* out,
                 long long ldo, long long stride_in = 0, long long stride_out = 0);

// Both jobs in one launch (the packed plans' A^T and B); at most 2^31 - 1
// tiles in all.
cudaError_t launch_pack2(const PackJob& a, const PackJob& b, cudaStream_t stream, int batch = 1);

}  // namespace b2g
