// skinny_tma.cu -- SGEMM for skinny M (M <= 32) with bulk-tensor fed operands
// and the split-K sums added inside a thread-block cluster.
//
// With M this small the product is a stream over B (16 x 4096 x 4096 moves
// 64 MiB of B for 0.5 GFLOP), so the work is cut along K ("GEMM 优化之路",
// section 接下来的优化方向: split-K for small M): a CTA owns 128 columns of C
// and one k slab.  B and A reach shared memory through bulk-tensor copies
// issued by a producer warp into a ring of 32-k stages, so each CTA keeps tens
// of KB of B in flight.  Per stage: B rows k..k+31, columns n0..n0+127
// ([32][128], 16 KB) and A rows 0..MR-1, columns k..k+31 ([MR][32]); rows of A
// at or past M and k at or past K arrive as zeros.
//
// Consumers: (MR / 8) row groups x 4 k groups of warps.  The warp of row group
// g and k group q takes rows 8q..8q+7 of every stage, in two steps of 4 k: one
// 16-byte load of B per k row (a warp reads 512 contiguous bytes), and per row
// m of its 8 rows of A one 16-byte load giving A[m][k..k+3] (the same address
// for every lane: a broadcast).  Each thread keeps 8 rows x 4 columns of
// accumulators, updated by packed two-lane FP32 FMAs (sm_100's fma.rn.f32x2,
// each lane rounded as fmaf: the same results in half the FMA instructions,
// which matters here because with 16 rows the multiply-adds, not the stream of
// B, set the pace on the SMs that run two CTAs); the 4 k groups of a row group
// then add their sums in k-group order through shared memory (the drained
// ring).
//
// The S k slabs of one column slab run as one cluster of S CTAs (S <= 8).
// Each CTA leaves its MR x 128 sums in its own shared memory; after a cluster
// barrier the CTA of rank r takes 1/S of the tile's elements, reads their S
// partial sums through distributed shared memory (all S loads in flight), adds
// them in rank (= slab) order, applies C = alpha * sum + beta * C and writes
// C; a second cluster barrier keeps every CTA until all have read.
// So there is no partial-sum workspace and no second kernel, and every output
// is summed in a fixed order (bitwise reproducible).  With S = 1 the CTA
// writes C itself.  Every wait is bounded, and every thread of every CTA
// reaches both cluster barriers, timeouts included.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "ptx.cuh"
#include "plan_registry.h"
#include "sgemm_params.h"
#include "tcgen05.cuh"

namespace b2g {

constexpr int kStBK = 32;   // k rows per stage
constexpr int kStBN = 128;  // columns of C per CTA
constexpr int kStStages = 4;
constexpr int kStMaxCluster = 8;  // portable cluster size: at most 8 k slabs per column slab
constexpr int kStPrefetch = 2;    // stages of B and A fetched into L2 before the dependency wait
// Where a CTA lets the next grid on the stream launch (cold-L2 timings at
// 4096 x 4096, back to back): 8 rows best without an early signal (CTAs launch
// as these exit: 14.1 us against 16.1 signalling at the start), 16 and 32 rows
// best after the main loop (18.4 / 29.1 us against 18.7 / 29.4 at the start,
// 19.2 / 29.8 at exit).
template <int MR>
constexpr bool kStSignalAfterLoop = MR > 8;

// Fetch the 128-byte line holding `p` into L2 (no register or shared-memory
// result; like tma_prefetch_3d it cannot read a stale value).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p) : "memory");
}

template <int MR>
struct SkinnyTmaCfg {
  static constexpr int kGroups = MR / 8;                       // row groups of 8
  static constexpr int kConsumerWarps = 4 * kGroups;           // x 4 k groups
  static constexpr int kConsumers = kConsumerWarps * 32;
  static constexpr int kThreads = kConsumers + 32;             // + the producer warp
  static constexpr int kBStage = kStBK * kStBN;                // floats
  static constexpr int kAStage = MR * kStBK;                   // floats
  static constexpr int kStageBytes = (kBStage + kAStage) * 4;
  static constexpr int kRing = kStStages * (kBStage + kAStage);  // floats
  static constexpr int kRed = 3 * MR * kStBN;                     // floats (in the drained ring)
  static constexpr int kPart = MR * kStBN;                        // floats, after kRed
  static_assert(MR % 8 == 0, "rows come in groups of 8");
  static_assert(kRed + kPart <= kRing, "the sums reuse the drained ring");
  static constexpr int kSmemBytes = kRing * 4 + 2 * kStStages * 8 + 16;  // + failure flag
};

template <int MR>
__global__ void __launch_bounds__(SkinnyTmaCfg<MR>::kThreads)
    skinny_tma_kernel(const __grid_constant__ SgemmParams p,
                      const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB) {
  using Cfg = SkinnyTmaCfg<MR>;
  extern __shared__ __align__(128) float sm[];
  float* Bs = sm;                               // [stages][32][128]
  float* As = sm + kStStages * Cfg::kBStage;    // [stages][MR][32]
  float* red = sm;                              // [3][MR][128], after the last stage
  float* part = sm + Cfg::kRed;                 // [MR][128]: this CTA's sums (cluster mode)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Cfg::kRing);
  const uint32_t full0 = smem_addr(bars), empty0 = smem_addr(bars + kStStages);
  volatile int* failed = reinterpret_cast<volatile int*>(bars + 2 * kStStages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int s = blockIdx.y, bz = blockIdx.z;
  const int kb = s * p.kc, ke = min(p.K, kb + p.kc);
  const int nst = ke > kb ? (ke - kb + kStBK - 1) / kStBK : 0;  // kc is a multiple of 32
  const int n0 = blockIdx.x * kStBN;
  const bool clustered = p.splits > 1;  // the grid's y extent is one cluster
  const float alpha = p.alpha, beta = p.beta;
  float* Cb = p.C + (long long)bz * p.strideC;

  // Launched as a programmatic dependent: this grid touches global memory only
  // after the previous grid on the stream has completed and its writes are
  // visible; the next grid may launch once every CTA here has passed its main
  // loop (kStSignalAfterLoop) or exited.
  if (threadIdx.x == 0) {
    for (int i = 0; i < kStStages; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, Cfg::kConsumerWarps);
    }
    fence_mbar_init();
    fence_proxy_async_smem();
    *failed = 0;
  }
  if (warp == Cfg::kConsumerWarps && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    // the first stages into L2 while the previous grid finishes (its writes,
    // should it write these operands, still land in L2 before they are read)
    for (int c = 0; c < nst && c < kStPrefetch; ++c) {
      tma_prefetch_3d(&tmB, n0, kb + c * kStBK, bz);
      tma_prefetch_3d(&tmA, kb + c * kStBK, 0, bz);
    }
  }
  if (warp == Cfg::kConsumerWarps && beta != 0.f) {
    // and the lines of C this CTA will read at the end (its share of the
    // tile in a cluster, the whole tile alone), in bounds only: one line of
    // 8 float4 per lane and step
    constexpr int E = MR * (kStBN / 4);
    const int S = clustered ? p.splits : 1, r = clustered ? s : 0;
    for (int e = r * E / S + 8 * lane; e < (r + 1) * E / S; e += 8 * 32) {
      const int i = e / (kStBN / 4), col = n0 + 4 * (e % (kStBN / 4));
      if (i < p.M && col < p.N) prefetch_l2(Cb + (long long)i * p.ldc + col);
    }
  }
  __syncthreads();
  pdl_wait();

  if (warp == Cfg::kConsumerWarps) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      int st = 0, issued = 0;
      uint32_t ph = 0;
      for (int c = 0; c < nst; ++c) {
        if (p.debug_stop_ktile >= 0 && issued >= p.debug_stop_ktile) break;
        if (!mbar_wait(empty0 + 8 * st, ph ^ 1u, p.wait_limit_ns, p.status, kStatusTimeoutEmpty))
          break;
        const uint32_t fb = full0 + 8 * st;
        const int k = kb + c * kStBK;
        mbar_arrive_expect_tx(fb, Cfg::kStageBytes);
        tma_load_3d(smem_addr(Bs + st * Cfg::kBStage), &tmB, n0, k, bz, fb);  // {N, K, batch}
        tma_load_3d(smem_addr(As + st * Cfg::kAStage), &tmA, k, 0, bz, fb);   // {K, M, batch}
        ++issued;
        if (++st == kStStages) st = 0, ph ^= 1u;
      }
      // leave only after every copy started here has landed
      for (int d = 0, pending = min(issued, kStStages); d < pending; ++d) {
        if (--st < 0) st = kStStages - 1, ph ^= 1u;
        if (!mbar_wait(full0 + 8 * st, ph, p.wait_limit_ns, p.status, kStatusTimeoutDrain)) break;
      }
    }
    __syncwarp();
    if (kStSignalAfterLoop<MR>) pdl_launch_dependents();
  } else {
    // ---------------------------------------------------------- consumers
    const int rg = warp >> 2, kg = warp & 3;  // row group, k group
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
    int st = 0;
    uint32_t ph = 0;
    for (int c = 0; c < nst; ++c) {
      const bool landed =
          mbar_wait(full0 + 8 * st, ph, p.wait_limit_ns, p.status, kStatusTimeoutFull);
      if (!__all_sync(0xffffffffu, landed)) {  // the whole warp gives up together
        if (lane == 0) *failed = 1;
        break;
      }
      const float* bsm = Bs + st * Cfg::kBStage + 4 * lane;
      const float* asm_ = As + st * Cfg::kAStage + rg * 8 * kStBK;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int k = kg * 8 + 4 * h;  // rows k..k+3 of the stage
        float4 b[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          b[kk] = *reinterpret_cast<const float4*>(bsm + (k + kk) * kStBN);
        float4 a4[8];
#pragma unroll
        for (int m = 0; m < 8; ++m) a4[m] = *reinterpret_cast<const float4*>(asm_ + m * kStBK + k);
        // k outer, rows inner: consecutive packed FMAs share the B pair
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const float2 b01 = make_float2(b[kk].x, b[kk].y), b23 = make_float2(b[kk].z, b[kk].w);
#pragma unroll
          for (int m = 0; m < 8; ++m) {
            const float av = kk == 0 ? a4[m].x : kk == 1 ? a4[m].y : kk == 2 ? a4[m].z : a4[m].w;
            const float2 aa = make_float2(av, av);
            const float2 r0 = __ffma2_rn(aa, b01, make_float2(acc[m][0], acc[m][1]));
            const float2 r1 = __ffma2_rn(aa, b23, make_float2(acc[m][2], acc[m][3]));
            acc[m][0] = r0.x, acc[m][1] = r0.y, acc[m][2] = r1.x, acc[m][3] = r1.y;
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * st);
      if (++st == kStStages) st = 0, ph ^= 1u;
    }
    if (kStSignalAfterLoop<MR>) pdl_launch_dependents();

    // k groups 1..3 -> shared memory (the drained ring); k group 0 adds them in
    // k-group order and keeps (cluster) or writes (alone) the CTA's sums
    asm volatile("bar.sync 1, %0;" ::"n"(Cfg::kConsumers) : "memory");  // all past the ring
    if (!*failed) {
      if (kg > 0) {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          *reinterpret_cast<float4*>(red + ((kg - 1) * MR + rg * 8 + i) * kStBN + 4 * lane) =
              make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
      }
      asm volatile("bar.sync 1, %0;" ::"n"(Cfg::kConsumers) : "memory");
      if (kg == 0) {
#pragma unroll
        for (int w = 0; w < 3; ++w)
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float4 v =
                *reinterpret_cast<const float4*>(red + (w * MR + rg * 8 + i) * kStBN + 4 * lane);
            acc[i][0] += v.x, acc[i][1] += v.y, acc[i][2] += v.z, acc[i][3] += v.w;
          }
        const int col = n0 + 4 * lane;
#pragma unroll
        for (int ii = 0; ii < 8; ++ii) {
          const int i = rg * 8 + ii;  // row of the tile
          if (clustered) {
            *reinterpret_cast<float4*>(part + i * kStBN + 4 * lane) =
                make_float4(acc[ii][0], acc[ii][1], acc[ii][2], acc[ii][3]);
          } else if (i < p.M && col < p.N) {  // N % 4 == 0: col + 3 < N as well
            float* crow = Cb + (long long)i * p.ldc + col;
            if (p.c_vec4) {
              float4 o;
              if (beta != 0.f) {
                const float4 cv = *reinterpret_cast<const float4*>(crow);
                o = make_float4(fmaf(alpha, acc[ii][0], beta * cv.x),
                                fmaf(alpha, acc[ii][1], beta * cv.y),
                                fmaf(alpha, acc[ii][2], beta * cv.z),
                                fmaf(alpha, acc[ii][3], beta * cv.w));
              } else {
                o = make_float4(alpha * acc[ii][0], alpha * acc[ii][1], alpha * acc[ii][2],
                                alpha * acc[ii][3]);
              }
              *reinterpret_cast<float4*>(crow) = o;
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e)
                crow[e] = (beta != 0.f) ? fmaf(alpha, acc[ii][e], beta * crow[e])
                                        : alpha * acc[ii][e];
            }
          }
        }
      }
    }
  }

  if (!clustered) return;
  // ------------------------------------------------------------ cluster sum
  __syncwarp();
  cluster_sync();  // every CTA's sums (or its failure flag) are in its shared memory
  if (threadIdx.x < Cfg::kConsumers) {
    const int S = p.splits;
    const int rank = (int)cluster_ctarank();
    bool any_failed = false;
    for (int r = 0; r < S; ++r)
      any_failed |= ld_shared_cluster_u32(mapa_shared(smem_addr((const void*)failed), r)) != 0;
    if (!any_failed) {  // otherwise the status word says why and C is left alone
      constexpr int E = MR * (kStBN / 4);  // float4 elements of the tile
      const int e0 = rank * E / S, e1 = (rank + 1) * E / S;
      const uint32_t part0 = smem_addr(part);
      for (int e = e0 + threadIdx.x; e < e1; e += Cfg::kConsumers) {
        const int i = e / (kStBN / 4), col = n0 + 4 * (e % (kStBN / 4));
        if (i >= p.M || col >= p.N) continue;
        float4 v[kStMaxCluster];
#pragma unroll
        for (int r = 0; r < kStMaxCluster; ++r)
          if (r < S) v[r] = ld_shared_cluster_f4(mapa_shared(part0 + 16u * e, r));
        float4 sum = v[0];
#pragma unroll
        for (int r = 1; r < kStMaxCluster; ++r)
          if (r < S) sum.x += v[r].x, sum.y += v[r].y, sum.z += v[r].z, sum.w += v[r].w;
        const float sv[4] = {sum.x, sum.y, sum.z, sum.w};
        float* crow = Cb + (long long)i * p.ldc + col;
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
          for (int q = 0; q < 4; ++q)
            crow[q] = (beta != 0.f) ? fmaf(alpha, sv[q], beta * crow[q]) : alpha * sv[q];
        }
      }
    }
  }
  // The others keep their shared memory until every CTA has read it.  The
  // arrive is relaxed: the distributed-shared-memory loads it must follow have
  // already been consumed, and the global stores of C need no order with the
  // barrier, so no CTA waits for its stores to drain (1-2% faster).
  __syncwarp();
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::
                   : "memory");
}

template <int MR>
int skinny_tma_occupancy() {
  static std::atomic<int> cached[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int occ = cached[dev].load(std::memory_order_acquire);
  if (occ) return occ;
  auto kern = skinny_tma_kernel<MR>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           SkinnyTmaCfg<MR>::kSmemBytes) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, SkinnyTmaCfg<MR>::kThreads,
                                                    SkinnyTmaCfg<MR>::kSmemBytes) != cudaSuccess)
    return 0;
  cached[dev].store(occ, std::memory_order_release);
  return occ;
}

template <int MR>
cudaError_t launch_skinny_tma(const SgemmParams& p, const CUtensorMap* tmA, const CUtensorMap* tmB,
                              int, cudaStream_t stream) {
  if (!tmA || !tmB) return cudaErrorInvalidValue;
  if (p.splits < 1 || p.splits > kStMaxCluster) return cudaErrorInvalidConfiguration;
  if (skinny_tma_occupancy<MR>() < 1) return cudaErrorInvalidConfiguration;
  SgemmParams pc = p;
  CUtensorMap a = *tmA, b = *tmB;
  void* args[] = {&pc, &a, &b};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = (unsigned)p.splits;  // the k slabs of a column slab
  attr[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((p.N + kStBN - 1) / kStBN), (unsigned)p.splits, (unsigned)p.batch);
  cfg.blockDim = dim3(SkinnyTmaCfg<MR>::kThreads);
  cfg.dynamicSmemBytes = SkinnyTmaCfg<MR>::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = p.splits > 1 ? 2 : 1;
  return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(&skinny_tma_kernel<MR>), args);
}

#define B2G_SKINNY_TMA_PLAN(NAME, MR)                                                            \
  Plan {                                                                                         \
    NAME, MR, kStBN, kStBK, kStStages, 4, kAKMajor, kFeedSkinnyTMA, SkinnyTmaCfg<MR>::kThreads,  \
        SkinnyTmaCfg<MR>::kSmemBytes, &launch_skinny_tma<MR>, 0, &skinny_tma_occupancy<MR>      \
  }

const Plan kPlansSkinnyTma[] = {
    B2G_SKINNY_TMA_PLAN("skinnyT_m8", 8),
    B2G_SKINNY_TMA_PLAN("skinnyT_m16", 16),
    B2G_SKINNY_TMA_PLAN("skinnyT_m32", 32),
};
const int kNumPlansSkinnyTma = sizeof(kPlansSkinnyTma) / sizeof(kPlansSkinnyTma[0]);

}  // namespace b2g
