// transpose.cu -- At = A^T for the pre-transposed GEMM plans.
//
// The FFMA kernels run fastest when A reaches shared memory as [k][m] rows
// (a thread's eight m values in two 16-byte vectors).  Row-major A has k
// contiguous instead, so the pre-transposed plans first write At (K x ldat,
// row-major, ldat = M rounded up to 4) into a workspace with this HBM-bound
// kernel: 64 x 64 tiles, 16-byte loads of A rows, a [64 k][64 m] shared tile
// written by 32 consecutive m per warp store (no bank conflicts), and 16-byte
// stores of At rows.  Requires A 16-byte aligned with lda % 4 == 0 and
// K % 4 == 0 (the callers check); M is arbitrary.  Columns M .. ldat-1 of At
// are padding and receive zeros.
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "transpose.h"

namespace b2g {

constexpr int kTT = 64;  // tile edge (m and k)

__global__ void __launch_bounds__(256) transpose_a_kernel(const float* __restrict__ A, int M,
                                                          int K, long long lda,
                                                          float* __restrict__ At,
                                                          long long ldat, long long strideA,
                                                          long long strideAt) {
  __shared__ __align__(16) float tile[kTT][kTT];  // [k][m]
  pdl_launch_dependents();
  pdl_wait();
  A += (long long)blockIdx.z * strideA;  // problem blockIdx.z of a batch
  At += (long long)blockIdx.z * strideAt;
  const int m0 = blockIdx.x * kTT, k0 = blockIdx.y * kTT;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // load: warp w takes 4-k chunks c = w, w+8; lanes take 32 consecutive rows
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int m = m0 + h * 32 + lane;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      const int c = warp + 8 * cc;  // 0..15
      const int k = k0 + 4 * c;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (m < M && k < K) v = *reinterpret_cast<const float4*>(A + (long long)m * lda + k);
      tile[4 * c + 0][h * 32 + lane] = v.x;
      tile[4 * c + 1][h * 32 + lane] = v.y;
      tile[4 * c + 2][h * 32 + lane] = v.z;
      tile[4 * c + 3][h * 32 + lane] = v.w;
    }
  }
  __syncthreads();
  // store: 16 threads cover one At row segment of 64 m as 16-byte vectors
  const int t = threadIdx.x & 15, r = threadIdx.x >> 4;  // r = 0..15
#pragma unroll
  for (int rr = 0; rr < kTT / 16; ++rr) {
    const int kl = r + 16 * rr;
    const int k = k0 + kl, m = m0 + 4 * t;
    if (k < K && m < ldat) {
      const float4 v = *reinterpret_cast<const float4*>(&tile[kl][4 * t]);
      *reinterpret_cast<float4*>(At + (long long)k * ldat + m) = v;
    }
  }
}

cudaError_t launch_transpose_a(const float* A, int M, int K, long long lda, float* At,
                               long long ldat, cudaStream_t stream, int batch,
                               long long strideA, long long strideAt) {
  for (int b0 = 0; b0 < batch; b0 += 65535) {  // grid z is at most 65535
    const int nb = batch - b0 < 65535 ? batch - b0 : 65535;
    const float* Ab = A + (long long)b0 * strideA;
    float* Atb = At + (long long)b0 * strideAt;
    const dim3 grid((unsigned)((M + kTT - 1) / kTT), (unsigned)((K + kTT - 1) / kTT),
                    (unsigned)nb);
    void* args[] = {(void*)&Ab, (void*)&M, (void*)&K, (void*)&lda, (void*)&Atb, (void*)&ldat,
                    (void*)&strideA, (void*)&strideAt};
    const cudaError_t e = launch_pdl(reinterpret_cast<const void*>(&transpose_a_kernel), grid,
                                     dim3(256), args, 0, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace b2g

namespace b2g {

// out (R x Cc, row-major, leading dimension ldo) = trans ? in^T : in, where in
// is read element by element (any alignment, any leading dimension):
//   trans == 0: out[r][c] = in[r * ld + c]
//   trans != 0: out[r][c] = in[c * ld + r]
// 32 x 32 tiles through shared memory (rows padded to 33: no bank conflicts),
// coalesced on both sides in either direction.
__global__ void __launch_bounds__(256) pack_kernel(const float* __restrict__ in, long long ld,
                                                   int trans, int R, int Cc,
                                                   float* __restrict__ out, long long ldo,
                                                   long long stride_in, long long stride_out) {
  __shared__ float tile[32][33];
  pdl_launch_dependents();
  pdl_wait();
  in += (long long)blockIdx.z * stride_in;  // problem blockIdx.z of a batch
  out += (long long)blockIdx.z * stride_out;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  if (trans) {
    // read in rows (c0 + i), columns r0 + tx: coalesced along r
#pragma unroll
    for (int i = ty; i < 32; i += 8) {
      const int c = c0 + i, r = r0 + tx;
      tile[i][tx] = (c < Cc && r < R) ? in[(long long)c * ld + r] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int i = ty; i < 32; i += 8) {
      const int r = r0 + i, c = c0 + tx;
      if (r < R && c < Cc) out[(long long)r * ldo + c] = tile[tx][i];
    }
  } else {
#pragma unroll
    for (int i = ty; i < 32; i += 8) {
      const int r = r0 + i, c = c0 + tx;
      if (r < R && c < Cc) out[(long long)r * ldo + c] = in[(long long)r * ld + c];
    }
  }
}

cudaError_t launch_pack(const float* in, long long ld, int trans, int R, int Cc, float* out,
                        long long ldo, cudaStream_t stream, int batch, long long stride_in,
                        long long stride_out) {
  for (int b0 = 0; b0 < batch; b0 += 65535) {
    const int nb = batch - b0 < 65535 ? batch - b0 : 65535;
    const float* ib = in + (long long)b0 * stride_in;
    float* ob = out + (long long)b0 * stride_out;
    const dim3 grid((unsigned)((Cc + 31) / 32), (unsigned)((R + 31) / 32), (unsigned)nb);
    void* args[] = {(void*)&ib, (void*)&ld, (void*)&trans, (void*)&R, (void*)&Cc, (void*)&ob,
                    (void*)&ldo, (void*)&stride_in, (void*)&stride_out};
    const cudaError_t e =
        launch_pdl(reinterpret_cast<const void*>(&pack_kernel), grid, dim3(256), args, 0, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace b2g
