// transpose.cu -- At = A^T for the pre-transposed GEMM plans.
//
// The FFMA kernels run fastest when A reaches shared memory as [k][m] rows
// (a thread's eight m values in two 16-byte vectors).  Row-major A has k
// contiguous instead, so the pre-transposed plans first write At (K x ldat,
// row-major, ldat = M rounded up to 4) into a workspace with this HBM-bound
// kernel: 64 x 64 tiles, each row of A's tile read by 16 consecutive threads
// as 16-byte vectors (a warp's load covers two whole 256-byte row segments:
// one request per line rather than one per thread), a [64 k][65] shared tile,
// and At rows written the same way.  Requires A 16-byte aligned with lda % 4 == 0 and
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
  // [k][m] with rows of 65 floats: the scalar writes of a warp (16 k chunks x
  // 2 rows of A) and the scalar reads (2 k rows x 16 m chunks) both meet
  // bank conflicts of at most two ways.
  __shared__ float tile[kTT][kTT + 1];
  pdl_wait();
  A += (long long)blockIdx.z * strideA;  // problem blockIdx.z of a batch
  At += (long long)blockIdx.z * strideAt;
  const int m0 = blockIdx.x * kTT, k0 = blockIdx.y * kTT;
  const int q = threadIdx.x & 15, r = threadIdx.x >> 4;  // 16-byte chunk, row (0..15)
  // load: 16 consecutive threads read one row of A's tile as 16-byte vectors
  // (a warp takes two whole 256-byte row segments)
  float4 v[kTT / 16];
#pragma unroll
  for (int i = 0; i < kTT / 16; ++i) {
    const int m = m0 + r + 16 * i, k = k0 + 4 * q;
    v[i] = (m < M && k < K) ? *reinterpret_cast<const float4*>(A + (long long)m * lda + k)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int i = 0; i < kTT / 16; ++i) {
    const int ml = r + 16 * i;
    tile[4 * q + 0][ml] = v[i].x;
    tile[4 * q + 1][ml] = v[i].y;
    tile[4 * q + 2][ml] = v[i].z;
    tile[4 * q + 3][ml] = v[i].w;
  }
  __syncthreads();
  // store: 16 consecutive threads write one At row segment of 64 m as 16-byte
  // vectors; columns M .. ldat-1 receive the zeros loaded for rows past M
#pragma unroll
  for (int i = 0; i < kTT / 16; ++i) {
    const int kl = r + 16 * i;
    const int k = k0 + kl, m = m0 + 4 * q;
    if (k < K && m < ldat) {
      const float4 o = make_float4(tile[kl][4 * q], tile[kl][4 * q + 1], tile[kl][4 * q + 2],
                                   tile[kl][4 * q + 3]);
      *reinterpret_cast<float4*>(At + (long long)k * ldat + m) = o;
    }
  }
  // The GEMM that reads At may launch once every CTA is here: launched while
  // this grid still held the SMs, its persistent CTAs were placed unevenly
  // (up to three on some SMs, none on others: 1536^3 ran at 42 instead of
  // 60 TFLOP/s).
  pdl_launch_dependents();
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
__device__ __forceinline__ void pack_tile(const PackJob& j, int bx, int by, int bz,
                                          float (&tile)[32][33]) {
  const float* __restrict__ in = j.in + (long long)bz * j.stride_in;  // problem bz of a batch
  float* __restrict__ out = j.out + (long long)bz * j.stride_out;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  const int r0 = by * 32, c0 = bx * 32;
  if (j.trans) {
    // read in rows (c0 + i), columns r0 + tx: coalesced along r
#pragma unroll
    for (int i = ty; i < 32; i += 8) {
      const int c = c0 + i, r = r0 + tx;
      tile[i][tx] = (c < j.Cc && r < j.R) ? in[(long long)c * j.ld + r] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int i = ty; i < 32; i += 8) {
      const int r = r0 + i, c = c0 + tx;
      if (r < j.R && c < j.Cc) out[(long long)r * j.ldo + c] = tile[tx][i];
    }
  } else {
#pragma unroll
    for (int i = ty; i < 32; i += 8) {
      const int r = r0 + i, c = c0 + tx;
      if (r < j.R && c < j.Cc) out[(long long)r * j.ldo + c] = in[(long long)r * j.ld + c];
    }
  }
}

// Both operands in one launch: blocks 0 .. tiles(a)-1 pack job a, the rest
// job b (a block's job is uniform across its threads, so the barrier in the
// transposing branch is reached by all of them).
__global__ void __launch_bounds__(256) pack2_kernel(const __grid_constant__ PackJob a,
                                                    const __grid_constant__ PackJob b) {
  __shared__ float tile[32][33];
  pdl_wait();
  const int ta = a.tiles_x * a.tiles_y;
  const int t = (int)blockIdx.x;
  if (t < ta)
    pack_tile(a, t % a.tiles_x, t / a.tiles_x, (int)blockIdx.z, tile);
  else
    pack_tile(b, (t - ta) % b.tiles_x, (t - ta) / b.tiles_x, (int)blockIdx.z, tile);
  pdl_launch_dependents();  // after the work: the GEMM's CTAs then find the SMs free
}

PackJob pack_job(const float* in, long long ld, int trans, int R, int Cc, float* out,
                 long long ldo, long long stride_in, long long stride_out) {
  PackJob j{in, ld, trans, R, Cc, out, ldo, stride_in, stride_out, (Cc + 31) / 32,
            (R + 31) / 32};
  return j;
}

cudaError_t launch_pack2(const PackJob& a, const PackJob& b, cudaStream_t stream, int batch) {
  const long long tiles = (long long)a.tiles_x * a.tiles_y + (long long)b.tiles_x * b.tiles_y;
  if (tiles <= 0) return cudaSuccess;
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
  for (int b0 = 0; b0 < batch; b0 += 65535) {  // grid z is at most 65535
    const int nb = batch - b0 < 65535 ? batch - b0 : 65535;
    PackJob ja = a, jb = b;
    ja.in += (long long)b0 * a.stride_in, ja.out += (long long)b0 * a.stride_out;
    jb.in += (long long)b0 * b.stride_in, jb.out += (long long)b0 * b.stride_out;
    void* args[] = {&ja, &jb};
    const cudaError_t e = launch_pdl(reinterpret_cast<const void*>(&pack2_kernel),
                                     dim3((unsigned)tiles, 1, (unsigned)nb), dim3(256), args, 0,
                                     stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace b2g
