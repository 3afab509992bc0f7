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

// out (R x Cc, leading dimension ldo) = trans ? in^T : in, in read element by
// element: any alignment and leading dimension ld.  Grid-limited to R and Cc
// below 2^31 / 32 tiles.
cudaError_t launch_pack(const float* in, long long ld, int trans, int R, int Cc, float* out,
                        long long ldo, cudaStream_t stream, int batch = 1,
                        long long stride_in = 0, long long stride_out = 0);

}  // namespace b2g
