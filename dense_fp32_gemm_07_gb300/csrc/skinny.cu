// skinny.cu -- SGEMM for skinny M (M <= 32): split-K FFMA kernel and its
// deterministic reduction.
//
// With M this small the GEMM is a stream over B (the 16 x 4096 x 4096 case
// moves 64 MiB of B for 0.5 GFLOP): it is bound by HBM, not by the FFMA pipe,
// and the tiled kernels leave most SMs idle (one row of output tiles).  The
// handbook names split-K as the remedy for small M ("GEMM 优化之路", section
// 接下来的优化方向, 参数自动调优).  Here:
//  * a CTA owns 128 columns of C and one k slab; each thread keeps all MR rows
//    x 4 columns of accumulators, so every element of B is read once, with
//    16-byte loads straight from global memory (a warp reads 512 contiguous
//    bytes of a B row);
//  * the CTA stages A's rows for the slab transposed in shared memory, [k][m],
//    and every thread reads them as broadcast 16-byte vectors;
//  * the 4 warps split the slab and add their accumulators in warp order;
//  * with a workspace, the k slabs of different CTAs land as partial sums
//    P[s][m][n] and a second kernel adds them in s order and applies
//    alpha/beta; without one, one CTA per column slab runs the whole K and
//    writes C directly.
// Every output element is summed in a fixed order, so results are bitwise
// reproducible for a given split.
#include <cuda_runtime.h>

#include <atomic>

#include "plan_registry.h"
#include "ptx.cuh"
#include "sgemm_params.h"

namespace b2g {

constexpr int kSkCols = 128;    // columns of C per CTA
constexpr int kSkThreads = 128;
constexpr int kSkChunk = 256;   // k extent of A staged at a time

template <int MR, int UNR = 4>
struct SkinnyCfg {
  static constexpr int kSmemBytes = (kSkChunk * MR + 3 * MR * kSkCols) * 4;
};

template <int MR, int UNR>
__global__ void __launch_bounds__(kSkThreads) skinny_kernel(const __grid_constant__ SgemmParams p) {
  extern __shared__ __align__(16) float sm[];
  pdl_wait();  // after the previous grid on the stream (see launch_pdl)
  float* As = sm;                    // [kSkChunk][MR]
  float* red = sm + kSkChunk * MR;   // [3][MR][kSkCols]: warps 1..3 hand their sums to warp 0
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.y;
  const int kb = s * p.kc, ke = min(p.K, kb + p.kc);
  const int bz = blockIdx.z;  // problem of a batch
  const float* Ab = p.A + (long long)bz * p.strideA;
  const float* Bb = p.B + (long long)bz * p.strideB;
  float* Cb = p.C + (long long)bz * p.strideC;
  float* Wb = p.splits > 1 ? p.work + (long long)bz * p.splits * p.M * p.N : nullptr;
  const int col = blockIdx.x * kSkCols + 4 * lane;
  const bool col_ok = col < p.N;  // N % 4 == 0, so col + 3 < N as well
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);

  float acc[MR][4];
#pragma unroll
  for (int i = 0; i < MR; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;

  static_assert(MR % 4 == 0, "rows come in 16-byte vectors");
  for (int c0 = kb; c0 < ke; c0 += kSkChunk) {
    const int cl = min(kSkChunk, ke - c0);  // a multiple of 4 (K % 4 == 0, kc % 16 == 0)
    // A[0..MR)[c0 .. c0+cl) -> As[k][m]; rows at or past M are zero
    for (int idx = threadIdx.x; idx < MR * (cl / 4); idx += kSkThreads) {
      const int m = idx % MR, k4 = idx / MR;
      const float4 v = (m < p.M)
                           ? *reinterpret_cast<const float4*>(Ab + (long long)m * p.lda + c0 + 4 * k4)
                           : zero;
      As[(4 * k4 + 0) * MR + m] = v.x;
      As[(4 * k4 + 1) * MR + m] = v.y;
      As[(4 * k4 + 2) * MR + m] = v.z;
      As[(4 * k4 + 3) * MR + m] = v.w;
    }
    __syncthreads();
    const int kw = cl / 4;  // this warp's share of the chunk
    const float* bp = Bb + (long long)(c0 + warp * kw) * p.ldb + col;
    const float* ap = As + warp * kw * MR;
#pragma unroll UNR
    for (int k = 0; k < kw; ++k) {
      const float4 b =
          col_ok ? __ldg(reinterpret_cast<const float4*>(bp + (long long)k * p.ldb)) : zero;
#pragma unroll
      for (int i4 = 0; i4 < MR / 4; ++i4) {
        const float4 a = *reinterpret_cast<const float4*>(ap + k * MR + 4 * i4);
        const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          float* c = acc[4 * i4 + r];
          c[0] = fmaf(av[r], b.x, c[0]);
          c[1] = fmaf(av[r], b.y, c[1]);
          c[2] = fmaf(av[r], b.z, c[2]);
          c[3] = fmaf(av[r], b.w, c[3]);
        }
      }
    }
    __syncthreads();  // As is restaged by the next chunk
  }
  // the reduction kernel may launch now; it waits for this grid's results
  pdl_launch_dependents();

  // warps 1..3 -> shared memory; warp 0 adds them in warp order
  if (warp > 0) {
#pragma unroll
    for (int i = 0; i < MR; ++i)
      *reinterpret_cast<float4*>(red + ((warp - 1) * MR + i) * kSkCols + 4 * lane) =
          make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  }
  __syncthreads();
  if (warp != 0 || !col_ok) return;
#pragma unroll
  for (int w = 0; w < 3; ++w)
#pragma unroll
    for (int i = 0; i < MR; ++i) {
      const float4 v = *reinterpret_cast<const float4*>(red + (w * MR + i) * kSkCols + 4 * lane);
      acc[i][0] += v.x, acc[i][1] += v.y, acc[i][2] += v.z, acc[i][3] += v.w;
    }
  const float alpha = p.alpha, beta = p.beta;
#pragma unroll
  for (int i = 0; i < MR; ++i) {
    if (i >= p.M) break;
    if (p.splits > 1) {
      *reinterpret_cast<float4*>(Wb + ((long long)s * p.M + i) * p.N + col) =
          make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
    } else {
      float* crow = Cb + (long long)i * p.ldc + col;
      if (p.c_vec4) {
        float4 o;
        if (beta != 0.f) {
          const float4 cv = *reinterpret_cast<const float4*>(crow);
          o = make_float4(fmaf(alpha, acc[i][0], beta * cv.x), fmaf(alpha, acc[i][1], beta * cv.y),
                          fmaf(alpha, acc[i][2], beta * cv.z), fmaf(alpha, acc[i][3], beta * cv.w));
        } else {
          o = make_float4(alpha * acc[i][0], alpha * acc[i][1], alpha * acc[i][2],
                          alpha * acc[i][3]);
        }
        *reinterpret_cast<float4*>(crow) = o;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e)
          crow[e] = (beta != 0.f) ? fmaf(alpha, acc[i][e], beta * crow[e]) : alpha * acc[i][e];
      }
    }
  }
}

// C = alpha * (P[0] + P[1] + ... + P[S-1]) + beta * C, partials added in s order
// (eight loads in flight per thread, the additions still in s order).  When
// launched as a programmatic dependent of the split-K kernel it starts early
// and waits here until that kernel has finished and its writes are visible.
__global__ void __launch_bounds__(256) splitk_reduce_kernel(const __grid_constant__ SgemmParams p) {
  pdl_wait();  // the partial sums are the previous grid's output
  const long long nv = p.N / 4;
  const long long per = (long long)p.M * nv;
  const long long total = per * p.batch;
  const long long plane = (long long)p.M * p.N;
  const float alpha = p.alpha, beta = p.beta;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long bz = idx / per, r = idx - bz * per;
    const long long m = r / nv, c = (r - m * nv) * 4;
    const float* w = p.work + bz * p.splits * plane + m * p.N + c;
    float4 sum = *reinterpret_cast<const float4*>(w);
    int s = 1;
    for (; s + 8 <= p.splits; s += 8) {
      float4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = *reinterpret_cast<const float4*>(w + (s + j) * plane);
#pragma unroll
      for (int j = 0; j < 8; ++j) sum.x += v[j].x, sum.y += v[j].y, sum.z += v[j].z, sum.w += v[j].w;
    }
    for (; s < p.splits; ++s) {
      const float4 v = *reinterpret_cast<const float4*>(w + s * plane);
      sum.x += v.x, sum.y += v.y, sum.z += v.z, sum.w += v.w;
    }
    const float sv[4] = {sum.x, sum.y, sum.z, sum.w};
    float* crow = p.C + bz * p.strideC + m * p.ldc + c;
    if (p.c_vec4) {
      float4 o;
      if (beta != 0.f) {
        const float4 cv = *reinterpret_cast<const float4*>(crow);
        o = make_float4(fmaf(alpha, sv[0], beta * cv.x), fmaf(alpha, sv[1], beta * cv.y),
                        fmaf(alpha, sv[2], beta * cv.z), fmaf(alpha, sv[3], beta * cv.w));
      } else {
        o = make_float4(alpha * sv[0], alpha * sv[1], alpha * sv[2], alpha * sv[3]);
      }
      *reinterpret_cast<float4*>(crow) = o;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        crow[e] = (beta != 0.f) ? fmaf(alpha, sv[e], beta * crow[e]) : alpha * sv[e];
    }
  }
}

cudaError_t launch_splitk_reduce(const SgemmParams& p, cudaStream_t stream, int num_sms,
                                 bool dependent) {
  const long long total = (long long)p.M * (p.N / 4) * p.batch;
  long long blocks = (total + 255) / 256;
  const long long cap = (long long)num_sms * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  SgemmParams pc = p;
  void* args[] = {&pc};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = dependent ? 1 : 0;
  return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(&splitk_reduce_kernel), args);
}

// CTAs of skinny_kernel<MR, UNR> resident per SM on the current device (the
// host sizes the split so the whole grid is one resident wave); 0 on failure.
template <int MR, int UNR>
int skinny_occupancy() {
  static std::atomic<int> cached[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int occ = cached[dev].load(std::memory_order_acquire);
  if (occ) return occ;
  auto kern = skinny_kernel<MR, UNR>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SkinnyCfg<MR>::kSmemBytes) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kSkThreads,
                                                    SkinnyCfg<MR>::kSmemBytes) != cudaSuccess)
    return 0;
  cached[dev].store(occ, std::memory_order_release);
  return occ;
}

template <int MR, int UNR>
cudaError_t launch_skinny(const SgemmParams& p, const CUtensorMap*, const CUtensorMap*,
                          int num_sms, cudaStream_t stream) {
  auto kern = skinny_kernel<MR, UNR>;
  static std::atomic<int> configured[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SkinnyCfg<MR>::kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev].store(1, std::memory_order_release);
  }
  const dim3 grid((unsigned)((p.N + kSkCols - 1) / kSkCols), (unsigned)p.splits,
                  (unsigned)p.batch);
  SgemmParams pc = p;
  void* args[] = {&pc};
  e = launch_pdl(reinterpret_cast<const void*>(kern), grid, dim3(kSkThreads), args,
                 SkinnyCfg<MR>::kSmemBytes, stream);
  if (e == cudaSuccess && p.splits > 1) e = launch_splitk_reduce(p, stream, num_sms, true);
  return e;
}

#define B2G_SKINNY_PLAN(NAME, MR, UNR)                                                           \
  Plan {                                                                                         \
    NAME, MR, kSkCols, kSkChunk, 1, 4, kAKMajor, kFeedSkinny, kSkThreads,                        \
        SkinnyCfg<MR>::kSmemBytes, &launch_skinny<MR, UNR>, 0, &skinny_occupancy<MR, UNR>        \
  }

const Plan kPlansSkinny[] = {
    B2G_SKINNY_PLAN("skinny_m8", 8, 16),
    B2G_SKINNY_PLAN("skinny_m16", 16, 8),
    B2G_SKINNY_PLAN("skinny_m32", 32, 8),
};
const int kNumPlansSkinny = sizeof(kPlansSkinny) / sizeof(kPlansSkinny[0]);

}  // namespace b2g
