// sgemm_ffma.cuh -- persistent, warp-specialised FP32 SGEMM on the CUDA cores.
//
//   C = alpha * op(A) * op(B) + beta * C      (row-major, FP32 FFMA throughout)
//
// The problem statement is the GEMM handbook's ("GEMM 优化之路", section
// 问题定义与性能上限).  The design keeps what the pages' optimisation chain
// establishes -- block tiling in shared memory (section v2), an 8x8 per-thread
// register outer product (section v4), 128-bit fragment loads (section v5),
// overlapped loading with several stages (section 接下来的优化方向: double
// buffering / cp.async pipelining) and masked edges (练习 2) -- and re-builds it
// around sm_103a's asynchronous machinery:
//
//  * one CTA per SM, persistent over output tiles (grouped along M for L2 reuse);
//  * an S-stage shared-memory ring with `full`/`empty` mbarriers;
//  * producer warp(s) fill the ring: either one elected thread issuing
//    bulk-tensor (TMA) copies, or warps issuing 4-byte cp.async with zero fill
//    for arbitrary alignment, leading dimensions and transposes;
//  * consumer warps each own a 32 x (8*TN) warp tile, as 4 x 8 threads with an
//    8 x TN register tile; per k they run 8*TN FFMAs from registers;
//  * B is staged [BK][BN] and a quarter-warp's 16-byte loads cover 128
//    contiguous bytes, so B fragment loads are free of bank conflicts;
//  * A is staged either k-chunked ([BK/4][BM][4], written directly by a 3-D
//    TMA view, one 16-byte load gives a row's next 4 k) or transposed
//    ([BK][BM], one 16-byte load gives 4 rows at one k); both give 128-bit
//    fragment loads without bank conflicts;
//  * every mbarrier wait is bounded: on timeout a flag goes to the status word
//    and the kernel leaves instead of hanging.
//
// Every output element is a k-ordered chain of FP32 FFMAs, so a given plan is
// bitwise reproducible run to run.
#pragma once
#include <algorithm>
#include <atomic>
#include <cstring>

#include "ptx.cuh"
#include "sgemm_params.h"
#include "tcgen05.cuh"

namespace b2g {

template <int BM, int BN, int BK, int WM, int WN, int TN, int STAGES, int ALAY, int FEED,
          int PWARPS, int ORD = 0, int CS = 0>
struct FfmaCfg {
  static constexpr int TM = 8;
  static constexpr int kConsumerWarps = WM * WN;
  static constexpr int kConsumers = kConsumerWarps * 32;
  static constexpr int kProducers = PWARPS * 32;
  static constexpr int kThreads = kConsumers + kProducers;
  // Staged feed: A lands k-chunked in a staging slot and each consumer warp
  // rewrites the 32 rows it owns, transposed, into a private double buffer.
  static constexpr bool kStaged = FEED == kFeedTMATrans;
  static constexpr int kAStage = kStaged ? 0 : BM * BK;  // floats per stage, shared A
  static constexpr int kBStage = BK * BN;
  static constexpr int kStaging = kStaged ? BM * BK : 0;                 // k-chunked A copy
  static constexpr int kPrivate = kStaged ? kConsumerWarps * 2 * BK * 32 : 0;  // per-warp A
  static constexpr int kARow = kStaged ? 32 : BM;  // row stride of the transposed A a warp reads
  static constexpr int kStageBytes = (BM * BK + kBStage) * 4;  // bytes one stage's copies land
  // Cluster split (CS = 1): one work unit per CTA, the k slices of a tile
  // summed in a cluster through distributed shared memory; each slice's sums
  // wait in the drained ring, and a flag word follows the barriers.
  static constexpr int kCsFlagBytes = CS ? 16 : 0;
  static constexpr int kSmemBytes =
      (STAGES * (kAStage + kBStage + kStaging) + kPrivate) * 4 + 2 * STAGES * 8 + kCsFlagBytes;
  static_assert(!CS || BM * BN <= STAGES * (kAStage + kBStage), "a slice's sums fit in the ring");
  static_assert(!CS || (FEED == kFeedTMA && !kStaged), "cluster split: bulk-tensor feed");
  static_assert(BM == WM * 32, "a warp tile is 32 rows");
  static_assert(BN == WN * 8 * TN, "a warp tile is 8*TN columns");
  static_assert(TN % 4 == 0 && BK % 4 == 0, "16-byte fragments");
  static_assert(BM <= 256 && BN <= 256, "bulk-tensor box dimensions are at most 256");
  static_assert(FEED == kFeedCpAsync ? PWARPS >= 1 : PWARPS == 1, "producer warps");
  static_assert(FEED == kFeedTMA || ALAY == kAKMajor, "4-byte feed writes the transposed layout");
  // The packed order (5) pairs accumulators in 64-bit registers and needs a
  // 128-register cap to keep three 160-thread CTAs per SM; its 32-k stage runs
  // fully unrolled.  The scalar orders unroll at most 16 k (unrolled 32 times
  // the scalar loop was measured 13% slower).
  // With A k-chunked the packed order keeps eight float4 fragments and would
  // spill under that cap, so those kernels ask for two CTAs per SM instead.
  static constexpr int kMinBlocks = ORD == 5 ? (ALAY == kAKChunk ? 2 : 3) : 1;
  static constexpr int kUnroll = ORD == 5 ? 32 : 16;
};

// One k step of the register outer product, acc[i][j] += a[i] * b[j].
// ORD picks the issue order of the scalar FP32 FMAs (0: row by row, 1: column
// by column, 2: rows with alternating column direction, 3: 2 x 2 blocks walked
// as a snake, 4: columns with alternating row direction), or 5: packed FMAs
// (sm_100's two-lane FP32 FMA, each lane rounded as fmaf), one per pair of
// columns j, j+1 and row i, walked pair of columns by pair of columns so that
// consecutive instructions share the B pair.  A packed FMA still occupies the
// FP32 pipe for both lanes but takes one issue slot instead of two, which
// leaves the slots for the fragment loads and the loop.  Every order performs
// the same fused multiply-adds on the same accumulators in the same k order,
// so results are identical.
template <int ORD, int TN>
__device__ __forceinline__ void outer_product(float (&acc)[8][TN], const float (&a)[8],
                                              const float (&b)[TN]) {
  if constexpr (ORD == 5) {
#pragma unroll
    for (int j2 = 0; j2 < TN / 2; ++j2) {
      const float2 bj = make_float2(b[2 * j2], b[2 * j2 + 1]);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float2 r = __ffma2_rn(make_float2(a[i], a[i]), bj,
                                    make_float2(acc[i][2 * j2], acc[i][2 * j2 + 1]));
        acc[i][2 * j2] = r.x, acc[i][2 * j2 + 1] = r.y;
      }
    }
  } else if constexpr (ORD == 1) {
#pragma unroll
    for (int j = 0; j < TN; ++j)
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
  } else if constexpr (ORD == 3) {
#pragma unroll
    for (int i2 = 0; i2 < 4; ++i2)
#pragma unroll
      for (int jj = 0; jj < TN / 2; ++jj) {
        const int j2 = (i2 & 1) ? TN / 2 - 1 - jj : jj;
        const int i = 2 * i2, j = 2 * j2;
        acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        acc[i][j + 1] = fmaf(a[i], b[j + 1], acc[i][j + 1]);
        acc[i + 1][j + 1] = fmaf(a[i + 1], b[j + 1], acc[i + 1][j + 1]);
        acc[i + 1][j] = fmaf(a[i + 1], b[j], acc[i + 1][j]);
      }
  } else if constexpr (ORD == 4) {
#pragma unroll
    for (int j = 0; j < TN; ++j)
#pragma unroll
      for (int ii = 0; ii < 8; ++ii) {
        const int i = (j & 1) ? 7 - ii : ii;
        acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      }
  } else if constexpr (ORD == 2) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int jj = 0; jj < TN; ++jj) {
        const int j = (i & 1) ? TN - 1 - jj : jj;
        acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
      }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
  }
}

// Output tile of linear index `tile`: problem b = tile / (tiles_m * tiles_n) of
// a batch; inside a problem, tiles run down a group of `group_m` tile rows
// before moving one tile column right, so CTAs that run together share A row
// panels and B column panels in L2.
__device__ __forceinline__ void tile_coords(const SgemmParams& p, int tile, int& b, int& tm,
                                            int& tn) {
  const int per_batch = p.tiles_m * p.tiles_n;
  b = tile / per_batch;
  tile -= b * per_batch;
  const int per_group = p.group_m * p.tiles_n;
  const int g = tile / per_group;
  const int first_m = g * p.group_m;
  const int gsize = min(p.tiles_m - first_m, p.group_m);
  const int r = tile - g * per_group;
  tm = first_m + r % gsize;
  tn = r / gsize;
}

// Work unit u of the persistent loop: the first tail_first units are whole
// output tiles (k tiles 0 .. k_tiles-1); with a split tail (tail_splits > 1)
// every later tile is tail_splits units, slice s covering k tiles
// [s*k_tiles/S, (s+1)*k_tiles/S).  part is the slice's index among all slices
// (where its partial sums go), -1 for a whole tile.
__device__ __forceinline__ void unit_range(const SgemmParams& p, int u, int& tile, int& kt0,
                                           int& kt1, int& part) {
  if (p.tail_splits <= 1 || u < p.tail_first) {
    tile = u, kt0 = 0, kt1 = p.k_tiles, part = -1;
    return;
  }
  const int v = u - p.tail_first;
  const int S = p.tail_splits;
  const int s = v % S;
  tile = p.tail_first + v / S;
  kt0 = (int)((long long)s * p.k_tiles / S);
  kt1 = (int)((long long)(s + 1) * p.k_tiles / S);
  part = v;
}

__device__ __forceinline__ int total_units(const SgemmParams& p) {
  const int tiles = p.tiles_m * p.tiles_n * p.batch;
  return p.tail_splits > 1 ? p.tail_first + (tiles - p.tail_first) * p.tail_splits : tiles;
}

// Cluster split: the S = p.tail_splits CTAs of a cluster are the k slices
// of one output tile (blockIdx.x = tile * S + slice, the slice being the
// CTA's rank in the cluster), and each has left its raw BM x BN sums in its
// own shared memory at `part` (rows of BN floats).  After a cluster barrier
// the CTA of rank r takes 1/S of the tile's float4 positions, adds their S
// partial sums in rank (= slice) order through distributed shared memory,
// applies C = alpha * sum + beta * C (C read only when beta != 0) and writes
// C.  A second barrier keeps every CTA until all have read.  When any CTA of
// the cluster gave up on a wait (its flag word), C is left alone; the status
// word says why.  Every thread of the CTA calls this, on every path.
template <int BM, int BN, int NT>
__device__ __forceinline__ void cs_finish(const SgemmParams& p, const float* part,
                                          const volatile int* failed) {
  const int S = p.tail_splits;
  if (S <= 1) return;  // no cluster: the CTA wrote C itself
  // Not the .aligned barrier forms: the producer warp's lanes arrive from two
  // places (lane 0 after its copies, the others at once).
  // Every CTA's sums (or its failure flag) are in its shared memory after this.
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
  const uint32_t rank = cluster_ctarank();
  bool any_failed = false;
  for (int r = 0; r < S; ++r)
    any_failed |=
        ld_shared_cluster_u32(mapa_shared(smem_addr((const void*)failed), (uint32_t)r)) != 0;
  if (!any_failed) {
    int bt, tm, tn;
    tile_coords(p, (int)blockIdx.x / S, bt, tm, tn);
    float* Cb = p.C + (long long)bt * p.strideC;
    constexpr int E = BM * BN / 4;  // float4 positions of the tile
    const int e0 = (int)rank * E / S, e1 = ((int)rank + 1) * E / S;
    const uint32_t part0 = smem_addr(part);
    const float alpha = p.alpha, beta = p.beta;
    for (int e = e0 + (int)threadIdx.x; e < e1; e += NT) {
      const int gr = tm * BM + e / (BN / 4), gc = tn * BN + 4 * (e % (BN / 4));
      if (gr >= p.M || gc >= p.N) continue;
      float4 v[16];
#pragma unroll
      for (int r = 0; r < 16; ++r)
        if (r < S) v[r] = ld_shared_cluster_f4(mapa_shared(part0 + 16u * e, (uint32_t)r));
      float4 sum = v[0];
#pragma unroll
      for (int r = 1; r < 16; ++r)
        if (r < S) sum.x += v[r].x, sum.y += v[r].y, sum.z += v[r].z, sum.w += v[r].w;
      const float sv[4] = {sum.x, sum.y, sum.z, sum.w};
      float* crow = Cb + (long long)gr * p.ldc;
      if (p.c_vec4 && gc + 3 < p.N) {
        float4 o;
        if (beta != 0.f) {
          const float4 cv = *reinterpret_cast<const float4*>(crow + gc);
          o = make_float4(fmaf(alpha, sv[0], beta * cv.x), fmaf(alpha, sv[1], beta * cv.y),
                          fmaf(alpha, sv[2], beta * cv.z), fmaf(alpha, sv[3], beta * cv.w));
        } else {
          o = make_float4(alpha * sv[0], alpha * sv[1], alpha * sv[2], alpha * sv[3]);
        }
        *reinterpret_cast<float4*>(crow + gc) = o;
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (gc + q < p.N) {
            float* o = crow + gc + q;
            *o = (beta != 0.f) ? fmaf(alpha, sv[q], beta * *o) : alpha * sv[q];
          }
      }
    }
  }
  // the others keep their shared memory until every CTA has read it; the
  // arrive is relaxed (the loads it follows have been consumed, and the
  // stores of C need no order with it)
  asm volatile("barrier.cluster.arrive.relaxed;\n\tbarrier.cluster.wait;" ::: "memory");
}

template <int BM, int BN, int BK, int WM, int WN, int TN, int STAGES, int ALAY, int FEED,
          int PWARPS, int ORD, int CS>
__global__ void __launch_bounds__((WM * WN + PWARPS) * 32,
                                  (FfmaCfg<BM, BN, BK, WM, WN, TN, STAGES, ALAY, FEED, PWARPS,
                                           ORD>::kMinBlocks))
    sgemm_ffma_kernel(const __grid_constant__ SgemmParams p,
                      const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB) {
  using Cfg = FfmaCfg<BM, BN, BK, WM, WN, TN, STAGES, ALAY, FEED, PWARPS, ORD, CS>;
  extern __shared__ __align__(1024) unsigned char smem[];
  float* sA = reinterpret_cast<float*>(smem);
  float* sB = sA + STAGES * Cfg::kAStage;
  float* sAst = sB + STAGES * Cfg::kBStage;     // staging (staged feed only)
  float* sAp = sAst + STAGES * Cfg::kStaging;   // per-warp A buffers (staged feed only)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sAp + Cfg::kPrivate);
  const uint32_t full0 = smem_addr(bars);
  const uint32_t empty0 = smem_addr(bars + STAGES);
  volatile int* cs_failed = reinterpret_cast<volatile int*>(bars + 2 * STAGES);  // CS only
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // the next grid may set up while this one runs, unless this grid leaves
  // slots free for it to land in unevenly (then it launches as CTAs exit)
  if (!p.pdl_late) pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, FEED == kFeedCpAsync ? Cfg::kProducers : 1);
      mbar_init(empty0 + 8 * s, Cfg::kConsumerWarps);
    }
    fence_mbar_init();
    fence_proxy_async_smem();
    if constexpr (CS) *cs_failed = 0;
  }
  __syncthreads();
  pdl_wait();  // global memory only once the previous grid has completed

  const int units = total_units(p);

  // ------------------------------------------------------------------ producer
  // Producer warps come first (warps 0 .. PWARPS-1), consumers after them.
  if (warp < PWARPS) {
    int stage = 0;
    uint32_t phase = 0;
    int issued = 0;
    if constexpr (FEED == kFeedTMA || FEED == kFeedTMATrans) {
      if (lane != 0) {
        if constexpr (CS) cs_finish<BM, BN, Cfg::kThreads>(p, sA, cs_failed);
        return;
      }
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      for (int u = blockIdx.x; u < units; u += gridDim.x) {
        int tile, kt0, kt1, part;
        unit_range(p, u, tile, kt0, kt1, part);
        int bt, tm, tn;
        tile_coords(p, tile, bt, tm, tn);
        const int m0 = tm * BM, n0 = tn * BN;
        for (int kt = kt0; kt < kt1; ++kt) {
          if (p.debug_stop_ktile >= 0 && issued >= p.debug_stop_ktile) goto drain_tma;
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, p.wait_limit_ns, p.status,
                         kStatusTimeoutEmpty))
            goto drain_tma;
          // the staged feed lands A in the staging slot
          const uint32_t fb = full0 + 8 * stage;
          mbar_arrive_expect_tx(fb, Cfg::kStageBytes);
          const uint32_t dA = smem_addr(FEED == kFeedTMATrans ? sAst + stage * Cfg::kStaging
                                                              : sA + stage * Cfg::kAStage);
          const uint32_t dB = smem_addr(sB + stage * Cfg::kBStage);
          // the batch index is each view's outermost coordinate
          if constexpr (ALAY == kAKChunk || FEED == kFeedTMATrans)
            tma_load_4d(dA, &tmA, 0, m0, kt * (BK / 4), bt, fb);  // view {4, M, K/4, batch}
          else
            tma_load_3d(dA, &tmA, m0, kt * BK, bt, fb);  // A stored K x M: {M, K, batch}
          tma_load_3d(dB, &tmB, n0, kt * BK, bt, fb);    // {N, K, batch}
          ++issued;
          if (++stage == STAGES) stage = 0, phase ^= 1u;
        }
      }
    drain_tma:
      // Leave only after every copy this thread started has landed.
      for (int d = 0, pending = min(issued, STAGES); d < pending; ++d) {
        if (--stage < 0) stage = STAGES - 1, phase ^= 1u;
        if (!mbar_wait(full0 + 8 * stage, phase, p.wait_limit_ns, p.status, kStatusTimeoutDrain))
          break;
      }
    } else {
      const int pt = threadIdx.x;
      for (int u = blockIdx.x; u < units; u += gridDim.x) {
        int tile, kt0, kt1, part;
        unit_range(p, u, tile, kt0, kt1, part);
        int bt, tm, tn;
        tile_coords(p, tile, bt, tm, tn);
        const int m0 = tm * BM, n0 = tn * BN;
        const float* Ab = p.A + (long long)bt * p.strideA;
        const float* Bb = p.B + (long long)bt * p.strideB;
        for (int kt = kt0; kt < kt1; ++kt) {
          if (p.debug_stop_ktile >= 0 && issued >= p.debug_stop_ktile) goto drain_cp;
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, p.wait_limit_ns, p.status,
                         kStatusTimeoutEmpty))
            goto drain_cp;
          const int k0 = kt * BK;
          const uint32_t dA = smem_addr(sA + stage * Cfg::kAStage);
          const uint32_t dB = smem_addr(sB + stage * Cfg::kBStage);
          // A tile -> As[k][m]; consecutive threads take consecutive m, so the
          // shared-memory writes hit consecutive banks.
#pragma unroll 4
          for (int it = 0; it < (BM * BK) / Cfg::kProducers; ++it) {
            const int idx = it * Cfg::kProducers + pt;
            const int r = idx % BM, k = idx / BM;
            const int gr = m0 + r, gk = k0 + k;
            const bool ok = gr < p.M && gk < p.K;
            const long long off = ok ? (p.transA ? (long long)gk * p.lda + gr
                                                 : (long long)gr * p.lda + gk)
                                     : 0;
            cp_async_4(dA + 4u * (k * BM + r), Ab + off, ok ? 4u : 0u);
          }
          // B tile -> Bs[k][n]
#pragma unroll 4
          for (int it = 0; it < (BK * BN) / Cfg::kProducers; ++it) {
            const int idx = it * Cfg::kProducers + pt;
            const int n = idx % BN, k = idx / BN;
            const int gn = n0 + n, gk = k0 + k;
            const bool ok = gn < p.N && gk < p.K;
            const long long off = ok ? (p.transB ? (long long)gn * p.ldb + gk
                                                 : (long long)gk * p.ldb + gn)
                                     : 0;
            cp_async_4(dB + 4u * (k * BN + n), Bb + off, ok ? 4u : 0u);
          }
          cp_async_arrive_noinc(full0 + 8 * stage);
          ++issued;
          if (++stage == STAGES) stage = 0, phase ^= 1u;
        }
      }
    drain_cp:
      cp_async_wait_all();
    }
    if constexpr (CS) cs_finish<BM, BN, Cfg::kThreads>(p, sA, cs_failed);
    return;
  }

  // ------------------------------------------------------------------ consumers
  const int cw = warp - PWARPS;  // consumer warp index
  const int wm = cw % WM, wn = cw / WM;
  const int tr = lane >> 3, tc = lane & 7;
  // Thread rows: k-chunked A gives rows wm*32 + tr + 4i (the 4 thread rows of a
  // warp read 4 consecutive 16-byte vectors); transposed A gives rows
  // wm*32 + 4tr + (i & 3) + 16(i >> 2).  Thread columns:
  // wn*8*TN + 4tc + 32(j >> 2) + (j & 3).
  const int a_off = (ALAY == kAKChunk) ? (wm * 32 + tr) * 4 : wm * 32 + 4 * tr;
  const int b_off = wn * (8 * TN) + 4 * tc;
  int stage = 0;
  uint32_t phase = 0;

  // Staged feed: before computing stage t each warp reads its 32 rows of stage
  // t+1 from the k-chunked staging copy (one 16-byte load per 4 k, 32
  // consecutive rows per warp load), and after computing stage t writes them
  // transposed, [BK][32], into its other private buffer (32 consecutive rows per
  // warp store).  Neither side has bank conflicts, the latency hides under the
  // FFMAs, and no warp waits for another.
  long long t_all = 0, total_stages = 0;
  float4 xv[Cfg::kStaged ? BK / 4 : 1];
  float* priv = sAp + cw * 2 * BK * 32;
  auto x_load = [&](int slot) {
    const float* st = sAst + slot * Cfg::kStaging + (wm * 32 + lane) * 4;
#pragma unroll
    for (int q = 0; q < BK / 4; ++q) xv[q] = *reinterpret_cast<const float4*>(st + q * BM * 4);
  };
  auto x_store = [&](int buf) {
    float* d = priv + buf * BK * 32 + lane;
#pragma unroll
    for (int q = 0; q < BK / 4; ++q) {
      d[(4 * q + 0) * 32] = xv[q].x;
      d[(4 * q + 1) * 32] = xv[q].y;
      d[(4 * q + 2) * 32] = xv[q].z;
      d[(4 * q + 3) * 32] = xv[q].w;
    }
  };
  if constexpr (Cfg::kStaged) {
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      int tile, kt0, kt1, part;
      unit_range(p, u, tile, kt0, kt1, part);
      total_stages += kt1 - kt0;
    }
    if (total_stages > 0) {
      if (!mbar_wait(full0, 0, p.wait_limit_ns, p.status, kStatusTimeoutFull)) return;
      x_load(0);
      x_store(0);
      __syncwarp();
    }
  }

  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    int tile, kt0, kt1, part;
    unit_range(p, u, tile, kt0, kt1, part);
    int bt, tm, tn;
    tile_coords(p, tile, bt, tm, tn);
    float acc[8][TN];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

    for (int kt = kt0; kt < kt1; ++kt) {
      const float* As;
      bool next = false;
      if constexpr (Cfg::kStaged) {
        next = t_all + 1 < total_stages;
        if (next) {
          const int ns = stage + 1 == STAGES ? 0 : stage + 1;
          const uint32_t np = stage + 1 == STAGES ? phase ^ 1u : phase;
          if (!mbar_wait(full0 + 8 * ns, np, p.wait_limit_ns, p.status, kStatusTimeoutFull))
            return;
          x_load(ns);
        }
        As = priv + (int)(t_all & 1) * BK * 32 + 4 * tr;
      } else {
        if constexpr (CS) {
          // the whole warp gives up together, and still reaches the barriers below
          const bool landed =
              mbar_wait(full0 + 8 * stage, phase, p.wait_limit_ns, p.status, kStatusTimeoutFull);
          if (!__all_sync(0xffffffffu, landed)) {
            if (lane == 0) *cs_failed = 1;
            break;
          }
        } else {
          if (!mbar_wait(full0 + 8 * stage, phase, p.wait_limit_ns, p.status, kStatusTimeoutFull))
            return;  // the status word says why; the producer drains and leaves too
        }
        As = sA + stage * Cfg::kAStage + a_off;
      }
      const float* Bs = sB + stage * Cfg::kBStage + b_off;
      if constexpr (ALAY == kAKChunk) {
#pragma unroll
        for (int q = 0; q < BK / 4; ++q) {
          float4 a4[8];
#pragma unroll
          for (int i = 0; i < 8; ++i)
            a4[i] = *reinterpret_cast<const float4*>(As + q * BM * 4 + 16 * i);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            float b[TN];
#pragma unroll
            for (int j4 = 0; j4 < TN / 4; ++j4) {
              const float4 v =
                  *reinterpret_cast<const float4*>(Bs + (4 * q + kk) * BN + 32 * j4);
              b[4 * j4 + 0] = v.x, b[4 * j4 + 1] = v.y, b[4 * j4 + 2] = v.z, b[4 * j4 + 3] = v.w;
            }
            float a[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
              a[i] = kk == 0 ? a4[i].x : kk == 1 ? a4[i].y : kk == 2 ? a4[i].z : a4[i].w;
            outer_product<ORD, TN>(acc, a, b);
          }
        }
      } else {
        // a 32-k stage (half the barrier round trips per k of a 16-k stage)
        // runs its scalar loop body twice, its packed loop body once
#pragma unroll Cfg::kUnroll
        for (int k = 0; k < BK; ++k) {
          const float4 a0 = *reinterpret_cast<const float4*>(As + k * Cfg::kARow);
          const float4 a1 = *reinterpret_cast<const float4*>(As + k * Cfg::kARow + 16);
          const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
          float b[TN];
#pragma unroll
          for (int j4 = 0; j4 < TN / 4; ++j4) {
            const float4 v = *reinterpret_cast<const float4*>(Bs + k * BN + 32 * j4);
            b[4 * j4 + 0] = v.x, b[4 * j4 + 1] = v.y, b[4 * j4 + 2] = v.z, b[4 * j4 + 3] = v.w;
          }
          outer_product<ORD, TN>(acc, a, b);
        }
      }
      if constexpr (Cfg::kStaged) {
        if (next) x_store((int)((t_all + 1) & 1));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty0 + 8 * stage);
      if (++stage == STAGES) stage = 0, phase ^= 1u;
      ++t_all;
    }

    // Epilogue: C = alpha*acc + beta*C, C read only when beta != 0, float4
    // where the 4 columns are in range and C is 16-byte aligned.  A slice of a
    // split tile instead stores its raw sums (alpha 1, beta 0: exact) as a
    // whole BM x BN block with leading dimension BN for the tail reduction.
    const bool slice = part >= 0;
    if constexpr (CS) {
      // every consumer warp has left the ring before a slice's sums overwrite it
      asm volatile("bar.sync 1, %0;" ::"n"(Cfg::kConsumers) : "memory");
      if (*cs_failed) break;
    }
    float* const cb = slice ? (CS ? sA : p.work + (size_t)part * (BM * BN))
                            : p.C + (long long)bt * p.strideC;
    const long long ldc = slice ? BN : p.ldc;
    const int m0 = slice ? 0 : tm * BM, n0 = slice ? 0 : tn * BN;
    const int mlim = slice ? BM : p.M, nlim = slice ? BN : p.N;
    const bool vec4 = slice || p.c_vec4;
    const float alpha = slice ? 1.f : p.alpha, beta = slice ? 0.f : p.beta;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = m0 + ((ALAY == kAKChunk) ? wm * 32 + tr + 4 * i
                                            : wm * 32 + 4 * tr + (i & 3) + 16 * (i >> 2));
      if (r >= mlim) continue;
      float* crow = cb + (long long)r * ldc;
#pragma unroll
      for (int j4 = 0; j4 < TN / 4; ++j4) {
        const int c = n0 + b_off + 32 * j4;
        const float* av = &acc[i][4 * j4];
        if (vec4 && c + 3 < nlim) {
          float4 o;
          if (beta != 0.f) {
            const float4 cv = *reinterpret_cast<const float4*>(crow + c);
            o.x = fmaf(alpha, av[0], beta * cv.x);
            o.y = fmaf(alpha, av[1], beta * cv.y);
            o.z = fmaf(alpha, av[2], beta * cv.z);
            o.w = fmaf(alpha, av[3], beta * cv.w);
          } else {
            o.x = alpha * av[0], o.y = alpha * av[1], o.z = alpha * av[2], o.w = alpha * av[3];
          }
          *reinterpret_cast<float4*>(crow + c) = o;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            if (c + e < nlim) {
              float* q = crow + c + e;
              *q = (beta != 0.f) ? fmaf(alpha, av[e], beta * *q) : alpha * av[e];
            }
          }
        }
      }
    }
  }
  if constexpr (CS) cs_finish<BM, BN, Cfg::kThreads>(p, sA, cs_failed);
}

// CTAs of one plan resident per SM on the current device, queried once per
// device (after opting in to the plan's dynamic shared memory); 0 on failure.
template <int BM, int BN, int BK, int WM, int WN, int TN, int STAGES, int ALAY, int FEED,
          int PWARPS, int ORD, int CS = 0>
int ffma_occupancy() {
  using Cfg = FfmaCfg<BM, BN, BK, WM, WN, TN, STAGES, ALAY, FEED, PWARPS, ORD, CS>;
  auto kern = sgemm_ffma_kernel<BM, BN, BK, WM, WN, TN, STAGES, ALAY, FEED, PWARPS, ORD, CS>;
  static std::atomic<int> resident[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  int occ = resident[dev].load(std::memory_order_acquire);
  if (occ == 0) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Cfg::kSmemBytes) != cudaSuccess)
      return 0;
    // clusters of up to 16 k slices (more than the portable 8)
    if (CS && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
                  cudaSuccess)
      return 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, Cfg::kThreads,
                                                      Cfg::kSmemBytes) != cudaSuccess ||
        occ < 1)
      return 0;
    resident[dev].store(occ, std::memory_order_release);
  }
  return occ;
}

template <int BM, int BN, int BK, int WM, int WN, int TN, int STAGES, int ALAY, int FEED,
          int PWARPS, int ORD, int CS = 0>
cudaError_t launch_ffma(const SgemmParams& p, const CUtensorMap* tmA, const CUtensorMap* tmB,
                        int num_sms, cudaStream_t stream) {
  using Cfg = FfmaCfg<BM, BN, BK, WM, WN, TN, STAGES, ALAY, FEED, PWARPS, ORD, CS>;
  auto kern = sgemm_ffma_kernel<BM, BN, BK, WM, WN, TN, STAGES, ALAY, FEED, PWARPS, ORD, CS>;
  // The persistent grid is SMs x resident CTAs, or one CTA per work unit;
  // a cluster-split grid is always one CTA per work unit.
  const int occ = ffma_occupancy<BM, BN, BK, WM, WN, TN, STAGES, ALAY, FEED, PWARPS, ORD, CS>();
  if (occ < 1) return cudaErrorInvalidConfiguration;
  const long long tiles = (long long)p.tiles_m * p.tiles_n * p.batch;
  const long long units =
      p.tail_splits > 1 ? p.tail_first + (tiles - p.tail_first) * p.tail_splits : tiles;
  if (CS && (p.tail_first != 0 || p.tail_splits > 16 || units > 0x7fffffffLL))
    return cudaErrorInvalidConfiguration;
  const int grid = CS ? (int)units : (int)std::min<long long>(units, (long long)num_sms * occ);
  CUtensorMap none;
  memset(&none, 0, sizeof(none));
  SgemmParams pc = p;
  pc.pdl_late = grid < (long long)num_sms * occ ? 1 : 0;
  CUtensorMap a = tmA ? *tmA : none, b = tmB ? *tmB : none;
  void* args[] = {&pc, &a, &b};
  if (CS && p.tail_splits > 1) {  // the k slices of a tile form one cluster
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = (unsigned)p.tail_splits;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(Cfg::kThreads);
    cfg.dynamicSmemBytes = Cfg::kSmemBytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelExC(&cfg, reinterpret_cast<const void*>(kern), args);
  }
  return launch_pdl(reinterpret_cast<const void*>(kern), dim3(grid), dim3(Cfg::kThreads), args,
                    Cfg::kSmemBytes, stream);
}

#define B2G_FFMA_PLAN(NAME, BM, BN, BK, WM, WN, TN, ST, ALAY, FEED, PW, ORD)                      \
  Plan {                                                                                         \
    NAME, BM, BN, BK, ST, TN, ALAY, FEED,                                                        \
        FfmaCfg<BM, BN, BK, WM, WN, TN, ST, ALAY, FEED, PW, ORD>::kThreads,                      \
        FfmaCfg<BM, BN, BK, WM, WN, TN, ST, ALAY, FEED, PW, ORD>::kSmemBytes,                    \
        &launch_ffma<BM, BN, BK, WM, WN, TN, ST, ALAY, FEED, PW, ORD>, 0,                        \
        &ffma_occupancy<BM, BN, BK, WM, WN, TN, ST, ALAY, FEED, PW, ORD>                         \
  }

// The kernel in its cluster-split form: one CTA per (tile, k slice), the k
// slices of a tile (at most SMAX, one cluster) summed through distributed
// shared memory; one launch, no workspace.
#define B2G_FFMA_PLAN_CS(NAME, BM, BN, BK, WM, WN, TN, ST, ALAY, PW, ORD, SMAX)                   \
  Plan {                                                                                         \
    NAME, BM, BN, BK, ST, TN, ALAY, kFeedTMA,                                                    \
        FfmaCfg<BM, BN, BK, WM, WN, TN, ST, ALAY, kFeedTMA, PW, ORD, 1>::kThreads,               \
        FfmaCfg<BM, BN, BK, WM, WN, TN, ST, ALAY, kFeedTMA, PW, ORD, 1>::kSmemBytes,             \
        &launch_ffma<BM, BN, BK, WM, WN, TN, ST, ALAY, kFeedTMA, PW, ORD, 1>, 0,                 \
        &ffma_occupancy<BM, BN, BK, WM, WN, TN, ST, ALAY, kFeedTMA, PW, ORD, 1>, SMAX            \
  }

// The same kernel behind a transpose of row-major A (PRE = 1) or a packing of
// both operands (PRE = 2) into a workspace.
#define B2G_FFMA_PLAN_PRE(NAME, BM, BN, BK, WM, WN, TN, ST, PW, ORD, PRE)                         \
  Plan {                                                                                         \
    NAME, BM, BN, BK, ST, TN, kAKMajor, kFeedTMA,                                                \
        FfmaCfg<BM, BN, BK, WM, WN, TN, ST, kAKMajor, kFeedTMA, PW, ORD>::kThreads,              \
        FfmaCfg<BM, BN, BK, WM, WN, TN, ST, kAKMajor, kFeedTMA, PW, ORD>::kSmemBytes,            \
        &launch_ffma<BM, BN, BK, WM, WN, TN, ST, kAKMajor, kFeedTMA, PW, ORD>, PRE,              \
        &ffma_occupancy<BM, BN, BK, WM, WN, TN, ST, kAKMajor, kFeedTMA, PW, ORD>                 \
  }

}  // namespace b2g
