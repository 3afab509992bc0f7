// tail.cu -- the second half of the FFMA plans' split tail.
//
// A persistent grid of G CTAs that runs T output tiles finishes when its
// busiest SM does: with T = q*G + r (0 < r < G) the last round keeps only r
// CTAs busy.  The host therefore cuts the tiles from tail_first on into S k
// slices of at least 64 k: by default the last r tiles with S = G / r, so
// every CTA gets q whole tiles plus at most one slice, or, where a per-SM
// balance model expects it to be faster, the tiles of the last rounds into
// more slices.  The GEMM kernel writes each slice's raw BM x BN sums to the
// workspace; this kernel adds a tile's S slices in slice order (a fixed
// order: results are reproducible run to run) and applies the same epilogue
// as the GEMM kernel, C = alpha * sum + beta * C, reading C only when
// beta != 0.
#include <cuda_runtime.h>

#include "sgemm_ffma.cuh"

namespace b2g {

// blockIdx.x: split tile (tail_first + blockIdx.x); blockIdx.y and the
// threads stride over the tile's BM x BN / 4 float4 positions.
__global__ void __launch_bounds__(256) tail_reduce_kernel(const __grid_constant__ SgemmParams p,
                                                          int BM, int BN) {
  // No early signal to the next grid: this short grid leaves most slots free,
  // and a persistent GEMM launched into them would land unevenly (its CTAs
  // launch as these exit instead: 1024^3 41.4 -> 45.4 TFLOP/s).
  pdl_wait();  // the partial sums are the previous grid's output
  int b, tm, tn;
  tile_coords(p, p.tail_first + (int)blockIdx.x, b, tm, tn);
  const int S = p.tail_splits;
  const size_t tile_elems = (size_t)BM * BN;
  const float* __restrict__ P = p.work + (size_t)blockIdx.x * S * tile_elems;
  float* __restrict__ Cb = p.C + (long long)b * p.strideC;
  const int n4 = BN / 4;
  const int m0 = tm * BM, n0 = tn * BN;
  const float alpha = p.alpha, beta = p.beta;
  for (int q = blockIdx.y * blockDim.x + threadIdx.x; q < BM * n4;
       q += gridDim.y * blockDim.x) {
    const int r = q / n4, c = (q - r * n4) * 4;
    const int gr = m0 + r, gc = n0 + c;
    if (gr >= p.M || gc >= p.N) continue;
    float* crow = Cb + (long long)gr * p.ldc;
    const bool vec = p.c_vec4 && gc + 3 < p.N;
    // C's values first, so that their trip from memory overlaps the slices'
    // (element by element where C's rows are not 16-byte aligned)
    float4 cv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (beta != 0.f) {
      if (vec) {
        cv = *reinterpret_cast<const float4*>(crow + gc);
      } else {
        cv.x = crow[gc];
        if (gc + 1 < p.N) cv.y = crow[gc + 1];
        if (gc + 2 < p.N) cv.z = crow[gc + 2];
        if (gc + 3 < p.N) cv.w = crow[gc + 3];
      }
    }
    float4 acc = *reinterpret_cast<const float4*>(P + (size_t)q * 4);
    for (int s = 1; s < S; ++s) {
      const float4 v = *reinterpret_cast<const float4*>(P + s * tile_elems + (size_t)q * 4);
      acc.x += v.x, acc.y += v.y, acc.z += v.z, acc.w += v.w;
    }
    const float av[4] = {acc.x, acc.y, acc.z, acc.w};
    if (vec) {
      float4 o;
      if (beta != 0.f) {
        o.x = fmaf(alpha, av[0], beta * cv.x);
        o.y = fmaf(alpha, av[1], beta * cv.y);
        o.z = fmaf(alpha, av[2], beta * cv.z);
        o.w = fmaf(alpha, av[3], beta * cv.w);
      } else {
        o.x = alpha * av[0], o.y = alpha * av[1], o.z = alpha * av[2], o.w = alpha * av[3];
      }
      *reinterpret_cast<float4*>(crow + gc) = o;
    } else {
      const float cs[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (gc + e < p.N)
          crow[gc + e] = (beta != 0.f) ? fmaf(alpha, av[e], beta * cs[e]) : alpha * av[e];
      }
    }
  }
}

cudaError_t launch_tail_reduce(const SgemmParams& p, int BM, int BN, cudaStream_t stream) {
  const long long tiles = (long long)p.tiles_m * p.tiles_n * p.batch;
  const long long n = tiles - p.tail_first;
  if (p.tail_splits <= 1 || n <= 0) return cudaSuccess;
  // one float4 position per thread: every load of a thread in flight at once
  const unsigned gy = (unsigned)((BM * BN / 4 + 255) / 256);
  SgemmParams pc = p;
  void* args[] = {&pc, &BM, &BN};
  return launch_pdl(reinterpret_cast<const void*>(&tail_reduce_kernel), dim3((unsigned)n, gy),
                    dim3(256), args, 0, stream);
}

}  // namespace b2g
