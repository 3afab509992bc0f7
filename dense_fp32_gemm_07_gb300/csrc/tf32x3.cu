// tf32x3.cu -- row-major SGEMM on the 5th-generation tensor cores with the
// 3xTF32 split, reported apart from the FP32 FFMA path.
//
// The handbook ("GEMM 优化之路", section 接下来的优化方向, 使用 Tensor Core)
// points out that tensor cores run the same tiled GEMM with the innermost step
// replaced by matrix instructions, and that TF32 keeps FP32 inputs but only a
// 10-bit mantissa.  Three TF32 products recover FP32 accuracy: every operand x
// is split into hi = x rounded to TF32 and lo = x - hi (exact in FP32, at most
// 2^-11 |x|), and
//     A*B ~= A_lo*B_hi + A_hi*B_lo + A_hi*B_hi
// (the dropped A_lo*B_lo term and the TF32 rounding of lo are below 2^-21 of
// |a||b| per product), accumulated in FP32 in tensor memory.
//
// Stages:
//  1. one split kernel (HBM bound): A -> A_hi, A_lo (M x K, row-major =
//     K-major) and B -> B_hi^T, B_lo^T (N x K, transposed so that B is
//     K-major too);
//  2. a persistent tcgen05 kernel: one lane issues bulk-tensor copies of the
//     four 128 x 32 tiles per stage (128-byte swizzle), one lane issues the
//     three tcgen05.mma kind::tf32 per K step into a double-buffered 128 x 128
//     FP32 accumulator in tensor memory, four warps read finished accumulators
//     back (tcgen05.ld) and apply C = alpha*acc + beta*C.
// Every wait is bounded; on a timeout the kernel flags the status word, waits
// (bounded) for the work it started, frees its tensor memory and returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstring>

#include "ptx.cuh"
#include "tcgen05.cuh"
#include "sgemm_params.h"
#include "tf32x3.h"

namespace b2g {

// ----------------------------------------------------------------- the split

// hi = x rounded to the nearest TF32 value (ties away from zero); lo = x - hi,
// exact.  Non-finite x passes through in hi with lo = 0; a finite x whose
// rounding would overflow is truncated instead.
__device__ __forceinline__ void tf32_split(float x, float& hi, float& lo) {
  if (!isfinite(x)) {
    hi = x;
    lo = 0.f;
    return;
  }
  const uint32_t u = __float_as_uint(x);
  float h = __uint_as_float((u + 0x1000u) & 0xFFFFE000u);
  if (!isfinite(h)) h = __uint_as_float(u & 0xFFFFE000u);
  hi = h;
  lo = x - h;
}

// A (M x K, lda) -> Ahi, Alo (M x K, leading dimension K).  16-byte vectors:
// A 16-byte aligned, lda and K multiples of 4.  Block `blk` of `nblk` takes
// every nblk-th group of 256 vectors.
__device__ __forceinline__ void split_a_part(const float* __restrict__ A, int M, int K,
                                             long long lda, float* __restrict__ Ahi,
                                             float* __restrict__ Alo, int blk, int nblk) {
  const long long kv = K / 4;
  const long long total = (long long)M * kv;
  for (long long i = (long long)blk * blockDim.x + threadIdx.x; i < total;
       i += (long long)nblk * blockDim.x) {
    const long long r = i / kv, c = (i - r * kv) * 4;
    const float4 v = *reinterpret_cast<const float4*>(A + r * lda + c);
    float4 h, l;
    tf32_split(v.x, h.x, l.x);
    tf32_split(v.y, h.y, l.y);
    tf32_split(v.z, h.z, l.z);
    tf32_split(v.w, h.w, l.w);
    *reinterpret_cast<float4*>(Ahi + r * K + c) = h;
    *reinterpret_cast<float4*>(Alo + r * K + c) = l;
  }
}

// B (K x N, ldb) -> Bhi^T, Blo^T (N x K, leading dimension K) in 64 x 64
// tiles: coalesced reads of B rows, 16-byte writes of the transposed rows.  The
// scalar shared-memory writes of the [n][k] tile (rows padded to 68 floats so
// the 16-byte reads stay aligned) are 4-way bank conflicted, which the
// HBM-bound kernel does not notice.  K % 4 == 0; N arbitrary.  This block
// takes the tile of columns 64 bx and rows 64 by.
__device__ __forceinline__ void split_bt_part(const float* __restrict__ B, int K, int N,
                                              long long ldb, float* __restrict__ Bhi,
                                              float* __restrict__ Blo, int bx, int by,
                                              float (&tile)[64][68]) {
  const int k0 = by * 64, n0 = bx * 64;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // load: warp w takes rows k = k0 + w + 8j; lanes take 32 consecutive n (twice)
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int kl = warp + 8 * j, k = k0 + kl;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int nl = h * 32 + lane, n = n0 + nl;
      tile[nl][kl] = (k < K && n < N) ? B[(long long)k * ldb + n] : 0.f;
    }
  }
  __syncthreads();
  // store: 16 threads per transposed row (64 k as 16 vectors), 16 rows per pass
  const int t = threadIdx.x & 15, r = threadIdx.x >> 4;
#pragma unroll
  for (int rr = 0; rr < 4; ++rr) {
    const int nl = r + 16 * rr, n = n0 + nl, k = k0 + 4 * t;
    if (n < N && k < K) {
      const float4 v = *reinterpret_cast<const float4*>(&tile[nl][4 * t]);
      float4 h, l;
      tf32_split(v.x, h.x, l.x);
      tf32_split(v.y, h.y, l.y);
      tf32_split(v.z, h.z, l.z);
      tf32_split(v.w, h.w, l.w);
      *reinterpret_cast<float4*>(Bhi + (long long)n * K + k) = h;
      *reinterpret_cast<float4*>(Blo + (long long)n * K + k) = l;
    }
  }
}

// Both splits in one launch: blocks 0 .. na-1 split A, the rest take B's 64 x
// 64 tiles (a block's part is uniform across its threads, so the barrier in
// B's part is reached by all of them).
__global__ void __launch_bounds__(256) split_ab_kernel(const float* __restrict__ A, int M, int K,
                                                       long long lda, float* __restrict__ Ahi,
                                                       float* __restrict__ Alo, int na,
                                                       const float* __restrict__ B, int N,
                                                       long long ldb, float* __restrict__ Bhi,
                                                       float* __restrict__ Blo, int tiles_x) {
  __shared__ __align__(16) float tile[64][68];  // [n][k], rows padded to keep 16-byte reads aligned
  pdl_wait();
  const int b = (int)blockIdx.x;
  if (b < na)
    split_a_part(A, M, K, lda, Ahi, Alo, b, na);
  else
    split_bt_part(B, K, N, ldb, Bhi, Blo, (b - na) % tiles_x, (b - na) / tiles_x, tile);
  pdl_launch_dependents();  // after the work, as in the transpose kernel
}

// ------------------------------------------------------------- the tensor-core GEMM

constexpr int kTcThreads = 192;  // warp 0 copies, warp 1 MMA, warps 2-5 epilogue
constexpr uint32_t kTcTileBytes = kTcBM * kTcBK * 4;    // one 128 x 32 FP32 tile: 16 KB
constexpr uint32_t kTcStageBytes = 4 * kTcTileBytes;    // A_hi, A_lo, B_hi^T, B_lo^T
constexpr uint32_t kTcTmemCols = 2 * kTcBN;             // two FP32 accumulators
constexpr int kTcNumBars = 2 * kTcStages + 5;
constexpr int kTcSmemBytes = kTcStages * kTcStageBytes + 1024 + kTcNumBars * 8 + 16;

__device__ __forceinline__ void tc_tile_coords(const Tf32x3Params& p, int tile, int& tm, int& tn) {
  const int per_group = p.group_m * p.tiles_n;
  const int g = tile / per_group;
  const int first_m = g * p.group_m;
  const int gsize = min(p.tiles_m - first_m, p.group_m);
  const int r = tile - g * per_group;
  tm = first_m + r % gsize;
  tn = r / gsize;
}

__global__ void __launch_bounds__(kTcThreads, 1)
    sgemm_tf32x3_kernel(const __grid_constant__ Tf32x3Params p,
                        const __grid_constant__ CUtensorMap mAhi,
                        const __grid_constant__ CUtensorMap mAlo,
                        const __grid_constant__ CUtensorMap mBhi,
                        const __grid_constant__ CUtensorMap mBlo) {
  extern __shared__ unsigned char smem_raw[];
  // the 128-byte swizzle atoms need 1024-byte aligned tiles
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + kTcStages * kTcStageBytes;
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (kTcStages + s); };
  auto tfull = [&](int a) { return bars + 8u * (2 * kTcStages + a); };
  auto tempty = [&](int a) { return bars + 8u * (2 * kTcStages + 2 + a); };
  const uint32_t drain = bars + 8u * (2 * kTcStages + 4);
  uint32_t* tmem_slot =
      reinterpret_cast<uint32_t*>(gbase + kTcStages * kTcStageBytes + kTcNumBars * 8);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTcStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull(a), 1);
      mbar_init(tempty(a), 4);  // one arrival per epilogue warp
    }
    mbar_init(drain, 1);
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), kTcTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  pdl_wait();  // operands and C only once the previous grid has completed
  const uint32_t tmem = *tmem_slot;
  const int total_tiles = p.tiles_m * p.tiles_n;

  if (warp == 0) {
    // ---------------------------------------------------------- copy issuer
    if (lane == 0) {
      prefetch_tmap(&mAhi);
      prefetch_tmap(&mAlo);
      prefetch_tmap(&mBhi);
      prefetch_tmap(&mBlo);
      int s = 0, issued = 0;
      uint32_t ph = 0;
      for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
        int tm, tn;
        tc_tile_coords(p, tile, tm, tn);
        const int m0 = tm * kTcBM, n0 = tn * kTcBN;
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          if (p.debug_stop_ktile >= 0 && issued >= p.debug_stop_ktile) goto copies_done;
          if (!mbar_wait(empty(s), ph ^ 1u, p.wait_limit_ns, p.status, kStatusTimeoutEmpty))
            goto copies_done;
          const uint32_t st = base + s * kTcStageBytes;
          mbar_arrive_expect_tx(full(s), kTcStageBytes);
          tma_load_2d(st, &mAhi, kt * kTcBK, m0, full(s));
          tma_load_2d(st + kTcTileBytes, &mAlo, kt * kTcBK, m0, full(s));
          tma_load_2d(st + 2 * kTcTileBytes, &mBhi, kt * kTcBK, n0, full(s));
          tma_load_2d(st + 3 * kTcTileBytes, &mBlo, kt * kTcBK, n0, full(s));
          ++issued;
          if (++s == kTcStages) s = 0, ph ^= 1u;
        }
      }
    copies_done:
      // leave only after every copy started here has landed
      for (int d = 0, pending = min(issued, kTcStages); d < pending; ++d) {
        if (--s < 0) s = kTcStages - 1, ph ^= 1u;
        if (!mbar_wait(full(s), ph, p.wait_limit_ns, p.status, kStatusTimeoutDrain)) break;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_tf32(kTcBM, kTcBN);
      int s = 0, a = 0;
      uint32_t ph = 0, aph = 0;
      for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
        if (!mbar_wait(tempty(a), aph ^ 1u, p.wait_limit_ns, p.status, kStatusTimeoutTmem))
          goto mma_done;
        tc_fence_after_sync();
        const uint32_t d = tmem + (uint32_t)(a * kTcBN);
        for (int kt = 0; kt < p.k_tiles; ++kt) {
          if (!mbar_wait(full(s), ph, p.wait_limit_ns, p.status, kStatusTimeoutFull)) goto mma_done;
          tc_fence_after_sync();
          const uint32_t st = base + s * kTcStageBytes;
#pragma unroll
          for (int kk = 0; kk < kTcBK / 8; ++kk) {  // 8 TF32 = 32 bytes per K step
            const uint32_t off = kk * 32u;
            const uint64_t ahi = smem_desc_sw128_kmajor(st + off);
            const uint64_t alo = smem_desc_sw128_kmajor(st + kTcTileBytes + off);
            const uint64_t bhi = smem_desc_sw128_kmajor(st + 2 * kTcTileBytes + off);
            const uint64_t blo = smem_desc_sw128_kmajor(st + 3 * kTcTileBytes + off);
            mma_tf32(d, alo, bhi, idesc, (kt > 0 || kk > 0) ? 1u : 0u);
            mma_tf32(d, ahi, blo, idesc, 1u);
            mma_tf32(d, ahi, bhi, idesc, 1u);
          }
          mma_commit(empty(s));  // the stage is free once these MMAs have read it
          if (++s == kTcStages) s = 0, ph ^= 1u;
        }
        mma_commit(tfull(a));  // the accumulator is final once every MMA is done
        if (++a == 2) a = 0, aph ^= 1u;
      }
    mma_done:
      // leave only after every MMA issued here has completed
      mma_commit(drain);
      mbar_wait(drain, 0, p.wait_limit_ns, p.status, kStatusTimeoutTmem);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;  // tensor-memory lanes 32q .. 32q+31 belong to this warp
    int a = 0;
    uint32_t aph = 0;
    const float alpha = p.alpha, beta = p.beta;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
      int tm, tn;
      tc_tile_coords(p, tile, tm, tn);
      if (!mbar_wait(tfull(a), aph, p.wait_limit_ns, p.status, kStatusTimeoutTmem)) break;
      tc_fence_after_sync();
      const int r = tm * kTcBM + 32 * q + lane;
      float* crow = p.C + (long long)r * p.ldc;
#pragma unroll 1
      for (int c = 0; c < kTcBN / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(a * kTcBN + 32 * c), v);
        tmem_ld_wait();
        if (r < p.M) {
          const int n = tn * kTcBN + 32 * c;
          if (p.c_vec4 && n + 31 < p.N) {
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              float4 o;
              const float a0 = __uint_as_float(v[j]), a1 = __uint_as_float(v[j + 1]);
              const float a2 = __uint_as_float(v[j + 2]), a3 = __uint_as_float(v[j + 3]);
              if (beta != 0.f) {
                const float4 cv = *reinterpret_cast<const float4*>(crow + n + j);
                o = make_float4(fmaf(alpha, a0, beta * cv.x), fmaf(alpha, a1, beta * cv.y),
                                fmaf(alpha, a2, beta * cv.z), fmaf(alpha, a3, beta * cv.w));
              } else {
                o = make_float4(alpha * a0, alpha * a1, alpha * a2, alpha * a3);
              }
              *reinterpret_cast<float4*>(crow + n + j) = o;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (n + j < p.N) {
                float* qp = crow + n + j;
                const float acc = __uint_as_float(v[j]);
                *qp = (beta != 0.f) ? fmaf(alpha, acc, beta * *qp) : alpha * acc;
              }
            }
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty(a));
      if (++a == 2) a = 0, aph ^= 1u;
    }
  }

  // teardown: every role is done with tensor memory; warp 1 frees it
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTcTmemCols);
  }
}

// ------------------------------------------------- the CTA-pair tensor-core GEMM
//
// Two CTAs of a cluster share each 256 x 128 output tile: CTA r stages rows
// 128r .. 128r+127 of A (hi and lo) and rows 64r .. 64r+63 of B^T (columns of
// B), and holds rows 128r .. 128r+127 of the accumulator in its own tensor
// memory.  One lane of the even CTA issues tcgen05.mma.cta_group::2 (M 256,
// N 128), which reads both CTAs' shared memory.  Per SM this stages 48 KB per
// 32-k step instead of 64 KB (4 stages fit where 3 did) and reads B once for
// two SMs.
//
// Signalling: both CTAs' copies of a stage complete on the even CTA's `full`
// barrier (the pair form of the bulk-tensor copy); the MMA issuer commits
// "stage read" and "accumulator final" to its own barriers and to the odd
// CTA's (a second commit aimed at the peer's address); the odd CTA's epilogue
// warps arrive remotely on the even CTA's "accumulator drained" barrier.
// Every wait is bounded; every thread of both CTAs reaches the final cluster
// barrier before tensor memory is freed.

constexpr int kTpThreads = 192;  // warp 0 copies, 1 MMA, 2-5 epilogue
constexpr uint32_t kTpATile = 128 * kTcBK * 4;  // this CTA's 128 rows of A_hi or A_lo: 16 KB

// PN: the pair's N per MMA (128 or 256); each CTA stages PN/2 rows of B^T.
template <int PN>
struct PairCfg {
  static constexpr int kStages = PN == 128 ? 4 : 3;
  static constexpr uint32_t kBTile = (PN / 2) * kTcBK * 4;  // 8 or 16 KB
  static constexpr uint32_t kStageBytes = 2 * kTpATile + 2 * kBTile;  // 48 or 64 KB
  static constexpr uint32_t kTmemCols = 2 * PN;                      // two accumulators
  static constexpr int kNumBars = 2 * kStages + 5;
  // 8 KB of slack after the barriers: an operand read one B tile longer than
  // intended would still stay inside this CTA's shared memory.
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024 + kNumBars * 8 + 16 + 8192;
  static_assert(PN == 128 || PN == 256, "pair tiles are 256 x 128 or 256 x 256");
};

// Work unit u of the pair kernels: the first tail_first units are whole tiles,
// then (with a split tail) every later tile is tail_splits units, slice s
// covering k tiles [s*k_tiles/S, (s+1)*k_tiles/S); part is the slice's index
// among all slices (where its raw sums go), -1 for a whole tile.
__device__ __forceinline__ void tc_unit(const Tf32x3Params& p, int u, int& tile, int& kt0,
                                        int& kt1, int& part) {
  if (p.tail_splits <= 1 || u < p.tail_first) {
    tile = u, kt0 = 0, kt1 = p.k_tiles, part = -1;
    return;
  }
  const int v = u - p.tail_first, S = p.tail_splits, sl = v % S;
  tile = p.tail_first + v / S;
  kt0 = (int)((long long)sl * p.k_tiles / S);
  kt1 = (int)((long long)(sl + 1) * p.k_tiles / S);
  part = v;
}

__device__ __forceinline__ int tc_units(const Tf32x3Params& p) {
  const int tiles = p.tiles_m * p.tiles_n;
  return p.tail_splits > 1 ? p.tail_first + (tiles - p.tail_first) * p.tail_splits : tiles;
}

template <int PN>
__global__ void __launch_bounds__(kTpThreads, 1)
    sgemm_tf32x3_pair_kernel(const __grid_constant__ Tf32x3Params p,
                             const __grid_constant__ CUtensorMap mAhi,
                             const __grid_constant__ CUtensorMap mAlo,
                             const __grid_constant__ CUtensorMap mBhi,
                             const __grid_constant__ CUtensorMap mBlo) {
  using Cfg = PairCfg<PN>;
  constexpr int kTpStages = Cfg::kStages;
  constexpr uint32_t kTpBTile = Cfg::kBTile, kTpStageBytes = Cfg::kStageBytes;
  constexpr uint32_t kTpTmemCols = Cfg::kTmemCols;
  constexpr int kTpNumBars = Cfg::kNumBars;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;  // 128-byte swizzle atoms: 1024-byte aligned
  unsigned char* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + kTpStages * kTpStageBytes;
  auto full = [&](int s) { return bars + 8u * s; };  // even CTA: both CTAs' copies landed
  auto empty = [&](int s) { return bars + 8u * (kTpStages + s); };  // stage read by the MMAs
  auto tfull = [&](int a) { return bars + 8u * (2 * kTpStages + a); };
  auto tempty = [&](int a) { return bars + 8u * (2 * kTpStages + 2 + a); };
  const uint32_t drain = bars + 8u * (2 * kTpStages + 4);
  uint32_t* tmem_slot =
      reinterpret_cast<uint32_t*>(gbase + kTpStages * kTpStageBytes + kTpNumBars * 8);

  const uint32_t rank = cluster_ctarank() & 1u;
  const bool even = rank == 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTpStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull(a), 1);
      mbar_init(tempty(a), 8);  // four epilogue warps in each CTA
    }
    mbar_init(drain, 1);
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_addr(tmem_slot), kTpTmemCols);
    tmem_relinquish_pair();
  }
  __syncwarp();
  tc_fence_before_sync();
  cluster_sync();  // barriers initialised and tensor memory allocated in both CTAs
  tc_fence_after_sync();
  pdl_wait();  // operands and C only once the previous grid has completed
  // The even CTA's base address names the pair's accumulator columns in both.
  const uint32_t tmem =
      even ? *tmem_slot : ld_shared_cluster_u32(mapa_shared(smem_addr(tmem_slot), 0));
  const int units = tc_units(p);
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

  if (warp == 0) {
    // ---------------------------------------------------------- copy issuer
    if (lane == 0) {
      prefetch_tmap(&mAhi);
      prefetch_tmap(&mAlo);
      prefetch_tmap(&mBhi);
      prefetch_tmap(&mBlo);
      int s = 0, issued = 0;
      uint32_t ph = 0;
      for (int u = pair; u < units; u += npairs) {
        int tile, kt0, kt1, part;
        tc_unit(p, u, tile, kt0, kt1, part);
        int tm, tn;
        tc_tile_coords(p, tile, tm, tn);
        const int ma = tm * 2 * kTcBM + (int)rank * kTcBM;    // this CTA's rows of A
        const int nb = tn * PN + (int)rank * (PN / 2);  // this CTA's rows of B^T
        for (int kt = kt0; kt < kt1; ++kt) {
          if (p.debug_stop_ktile >= 0 && issued >= p.debug_stop_ktile) goto copies_done;
          if (!mbar_wait(empty(s), ph ^ 1u, p.wait_limit_ns, p.status, kStatusTimeoutEmpty))
            goto copies_done;
          const uint32_t st = base + s * kTpStageBytes;
          // both CTAs' bytes complete on the even CTA's barrier
          if (even) mbar_arrive_expect_tx(full(s), 2 * kTpStageBytes);
          const uint32_t fb = even ? full(s) : mapa_shared(full(s), 0);
          tma_load_2d_pair(st, &mAhi, kt * kTcBK, ma, fb);
          tma_load_2d_pair(st + kTpATile, &mAlo, kt * kTcBK, ma, fb);
          tma_load_2d_pair(st + 2 * kTpATile, &mBhi, kt * kTcBK, nb, fb);
          tma_load_2d_pair(st + 2 * kTpATile + kTpBTile, &mBlo, kt * kTcBK, nb, fb);
          ++issued;
          if (++s == kTpStages) s = 0, ph ^= 1u;
        }
      }
    copies_done:
      // Leave only after the copies started here have landed: the even CTA
      // sees its `full` barriers complete (they count both CTAs' bytes), the
      // odd CTA sees the MMAs release the stages (they read what landed).
      for (int d = 0, pending = min(issued, kTpStages); d < pending; ++d) {
        if (--s < 0) s = kTpStages - 1, ph ^= 1u;
        if (!mbar_wait(even ? full(s) : empty(s), ph, p.wait_limit_ns, p.status,
                       kStatusTimeoutDrain))
          break;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer (even CTA)
    if (even && lane == 0) {
      constexpr uint32_t idesc = idesc_tf32(2 * kTcBM, PN);
      int s = 0, a = 0;
      uint32_t ph = 0, aph = 0;
      for (int u = pair; u < units; u += npairs) {
        int tile, kt0, kt1, part;
        tc_unit(p, u, tile, kt0, kt1, part);
        if (!mbar_wait(tempty(a), aph ^ 1u, p.wait_limit_ns, p.status, kStatusTimeoutTmem))
          goto mma_done;
        tc_fence_after_sync();
        const uint32_t d = tmem + (uint32_t)(a * PN);
        for (int kt = kt0; kt < kt1; ++kt) {
          if (!mbar_wait(full(s), ph, p.wait_limit_ns, p.status, kStatusTimeoutFull)) goto mma_done;
          tc_fence_after_sync();
          const uint32_t st = base + s * kTpStageBytes;
#pragma unroll
          for (int kk = 0; kk < kTcBK / 8; ++kk) {  // 8 TF32 = 32 bytes per K step
            const uint32_t off = kk * 32u;
            const uint64_t ahi = smem_desc_sw128_kmajor(st + off);
            const uint64_t alo = smem_desc_sw128_kmajor(st + kTpATile + off);
            const uint64_t bhi = smem_desc_sw128_kmajor(st + 2 * kTpATile + off);
            const uint64_t blo = smem_desc_sw128_kmajor(st + 2 * kTpATile + kTpBTile + off);
            mma_tf32_pair(d, alo, bhi, idesc, (kt > kt0 || kk > 0) ? 1u : 0u);
            mma_tf32_pair(d, ahi, blo, idesc, 1u);
            mma_tf32_pair(d, ahi, bhi, idesc, 1u);
          }
          mma_commit_pair(empty(s));                  // this CTA may refill the stage
          mma_commit_pair(mapa_shared(empty(s), 1));  // and so may the odd one
          if (++s == kTpStages) s = 0, ph ^= 1u;
        }
        mma_commit_pair(tfull(a));  // the accumulator is final in both CTAs
        mma_commit_pair(mapa_shared(tfull(a), 1));
        if (++a == 2) a = 0, aph ^= 1u;
      }
    mma_done:
      mma_commit_pair(drain);
      mbar_wait(drain, 0, p.wait_limit_ns, p.status, kStatusTimeoutTmem);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;  // tensor-memory lanes 32q .. 32q+31 belong to this warp
    int a = 0;
    uint32_t aph = 0;
    const float alpha = p.alpha, beta = p.beta;
    for (int u = pair; u < units; u += npairs) {
      int tile, kt0, kt1, part;
      tc_unit(p, u, tile, kt0, kt1, part);
      int tm, tn;
      tc_tile_coords(p, tile, tm, tn);
      if (!mbar_wait(tfull(a), aph, p.wait_limit_ns, p.status, kStatusTimeoutTmem)) break;
      tc_fence_after_sync();
      const int r = tm * 2 * kTcBM + (int)rank * kTcBM + 32 * q + lane;
      float* crow = p.C + (long long)r * p.ldc;
      // a slice of a split tile: its raw sums, this CTA's 128 rows of the
      // 256 x PN block, for the tail reduction
      float* wrow = part >= 0 ? p.work + (size_t)part * (2 * kTcBM * PN) +
                                    (size_t)((int)rank * kTcBM + 32 * q + lane) * PN
                              : nullptr;
#pragma unroll 1
      for (int c = 0; c < PN / 32; ++c) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(a * PN + 32 * c), v);
        tmem_ld_wait();
        if (wrow) {
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(wrow + 32 * c + j) =
                make_float4(__uint_as_float(v[j]), __uint_as_float(v[j + 1]),
                            __uint_as_float(v[j + 2]), __uint_as_float(v[j + 3]));
        } else if (r < p.M) {
          const int n = tn * PN + 32 * c;
          if (p.c_vec4 && n + 31 < p.N) {
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
              float4 o;
              const float a0 = __uint_as_float(v[j]), a1 = __uint_as_float(v[j + 1]);
              const float a2 = __uint_as_float(v[j + 2]), a3 = __uint_as_float(v[j + 3]);
              if (beta != 0.f) {
                const float4 cv = *reinterpret_cast<const float4*>(crow + n + j);
                o = make_float4(fmaf(alpha, a0, beta * cv.x), fmaf(alpha, a1, beta * cv.y),
                                fmaf(alpha, a2, beta * cv.z), fmaf(alpha, a3, beta * cv.w));
              } else {
                o = make_float4(alpha * a0, alpha * a1, alpha * a2, alpha * a3);
              }
              *reinterpret_cast<float4*>(crow + n + j) = o;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              if (n + j < p.N) {
                float* qp = crow + n + j;
                const float acc = __uint_as_float(v[j]);
                *qp = (beta != 0.f) ? fmaf(alpha, acc, beta * *qp) : alpha * acc;
              }
            }
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if (even)
          mbar_arrive(tempty(a));
        else
          mbar_arrive_remote(mapa_shared(tempty(a), 0));
      }
      if (++a == 2) a = 0, aph ^= 1u;
    }
  }

  // teardown: no copy, MMA, remote arrival or tensor-memory read of either
  // CTA is still outstanding once both have passed this barrier
  __syncwarp();
  tc_fence_before_sync();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(*tmem_slot, kTpTmemCols);
  }
}

// ------------------------------------------------------------------- launchers

cudaError_t launch_split_ab(const float* A, int M, int K, long long lda, float* Ahi, float* Alo,
                            const float* B, int N, long long ldb, float* Bhi, float* Blo,
                            int num_sms, cudaStream_t stream) {
  const long long total = (long long)M * (K / 4);
  long long na = (total + 255) / 256;
  const long long cap = (long long)num_sms * 8;
  if (na > cap) na = cap;
  if (na < 1) na = 1;
  const long long tx = (N + 63) / 64, ty = (K + 63) / 64;
  const long long blocks = na + tx * ty;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  int na_i = (int)na, tx_i = (int)tx;
  void* args[] = {(void*)&A,   (void*)&M,   (void*)&K,   (void*)&lda, (void*)&Ahi, (void*)&Alo,
                  (void*)&na_i, (void*)&B,  (void*)&N,   (void*)&ldb, (void*)&Bhi, (void*)&Blo,
                  (void*)&tx_i};
  return launch_pdl(reinterpret_cast<const void*>(&split_ab_kernel), dim3((unsigned)blocks),
                    dim3(256), args, 0, stream);
}

cudaError_t launch_tf32x3(const Tf32x3Params& p, const CUtensorMap* maps, int num_sms,
                          cudaStream_t stream) {
  static std::atomic<int> configured[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(sgemm_tf32x3_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kTcSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev].store(1, std::memory_order_release);
  }
  const long long tiles = (long long)p.tiles_m * p.tiles_n;
  const int grid = (int)(tiles < num_sms ? tiles : num_sms);
  Tf32x3Params pc = p;
  CUtensorMap m0 = maps[0], m1 = maps[1], m2 = maps[2], m3 = maps[3];
  void* args[] = {&pc, &m0, &m1, &m2, &m3};
  return launch_pdl(reinterpret_cast<const void*>(&sgemm_tf32x3_kernel), dim3(grid),
                    dim3(kTcThreads), args, kTcSmemBytes, stream);
}

template <int PN>
cudaError_t launch_pair(const Tf32x3Params& p, const CUtensorMap* maps, int num_sms,
                        cudaStream_t stream) {
  using Cfg = PairCfg<PN>;
  // Per device, once: opt in to the shared memory and ask how many CTA pairs
  // can be resident at once (the persistent grid is that many pairs).
  static std::atomic<int> resident_pairs[kMaxDevices];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kTpThreads);
  cfg.dynamicSmemBytes = Cfg::kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const void* kern = reinterpret_cast<const void*>(&sgemm_tf32x3_pair_kernel<PN>);
  int pairs = resident_pairs[dev].load(std::memory_order_acquire);
  if (pairs == 0) {
    e = cudaFuncSetAttribute(sgemm_tf32x3_pair_kernel<PN>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3((unsigned)(num_sms & ~1));
    e = cudaOccupancyMaxActiveClusters(&pairs, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (pairs < 1) return cudaErrorInvalidConfiguration;
    resident_pairs[dev].store(pairs, std::memory_order_release);
  }
  const long long tiles = (long long)p.tiles_m * p.tiles_n;
  cfg.gridDim = dim3((unsigned)(2 * (tiles < pairs ? tiles : pairs)));
  cfg.numAttrs = 2;  // the occupancy query above used the cluster shape alone
  Tf32x3Params pc = p;
  CUtensorMap m0 = maps[0], m1 = maps[1], m2 = maps[2], m3 = maps[3];
  void* args[] = {&pc, &m0, &m1, &m2, &m3};
  return cudaLaunchKernelExC(&cfg, kern, args);
}

cudaError_t launch_tf32x3_pair(const Tf32x3Params& p, const CUtensorMap* maps, int pn,
                               int num_sms, cudaStream_t stream) {
  return pn == 256 ? launch_pair<256>(p, maps, num_sms, stream)
                   : launch_pair<128>(p, maps, num_sms, stream);
}

int tf32x3_pair_capacity(int pn, int num_sms) {
  static std::atomic<int> cached[2][kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  const int w = pn == 256 ? 1 : 0;
  int pairs = cached[w][dev].load(std::memory_order_acquire);
  if (pairs) return pairs;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kTpThreads);
  cfg.gridDim = dim3((unsigned)(num_sms & ~1));
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const void* kern = pn == 256 ? reinterpret_cast<const void*>(&sgemm_tf32x3_pair_kernel<256>)
                               : reinterpret_cast<const void*>(&sgemm_tf32x3_pair_kernel<128>);
  cfg.dynamicSmemBytes = pn == 256 ? PairCfg<256>::kSmemBytes : PairCfg<128>::kSmemBytes;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)cfg.dynamicSmemBytes) != cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&pairs, kern, &cfg) != cudaSuccess || pairs < 1)
    return 0;
  cached[w][dev].store(pairs, std::memory_order_release);
  return pairs;
}

// blockIdx.x: split tile (tail_first + blockIdx.x); blockIdx.y and the threads
// stride over the tile's 256 x pn / 4 float4 positions; slices added in order.
__global__ void __launch_bounds__(256) tc_tail_reduce_kernel(const __grid_constant__ Tf32x3Params p,
                                                             int pn) {
  pdl_launch_dependents();
  pdl_wait();  // the partial sums are the previous grid's output
  int tm, tn;
  tc_tile_coords(p, p.tail_first + (int)blockIdx.x, tm, tn);
  const int S = p.tail_splits;
  const size_t tile_elems = (size_t)2 * kTcBM * pn;
  const float* __restrict__ P = p.work + (size_t)blockIdx.x * S * tile_elems;
  const int n4 = pn / 4;
  const int m0 = tm * 2 * kTcBM, n0 = tn * pn;
  const float alpha = p.alpha, beta = p.beta;
  for (int q = blockIdx.y * blockDim.x + threadIdx.x; q < 2 * kTcBM * n4;
       q += gridDim.y * blockDim.x) {
    const int r = q / n4, c = (q - r * n4) * 4;
    const int gr = m0 + r, gc = n0 + c;
    if (gr >= p.M || gc >= p.N) continue;
    float* crow = p.C + (long long)gr * p.ldc;
    const bool vec = p.c_vec4 && gc + 3 < p.N;
    // C's values first, so that their trip from memory overlaps the slices'
    float4 cv = make_float4(0.f, 0.f, 0.f, 0.f);
    if (vec && beta != 0.f) cv = *reinterpret_cast<const float4*>(crow + gc);
    float4 acc = *reinterpret_cast<const float4*>(P + (size_t)q * 4);
    for (int s = 1; s < S; ++s) {
      const float4 v = *reinterpret_cast<const float4*>(P + s * tile_elems + (size_t)q * 4);
      acc.x += v.x, acc.y += v.y, acc.z += v.z, acc.w += v.w;
    }
    const float av[4] = {acc.x, acc.y, acc.z, acc.w};
    if (vec) {
      float4 o;
      if (beta != 0.f) {
        o = make_float4(fmaf(alpha, av[0], beta * cv.x), fmaf(alpha, av[1], beta * cv.y),
                        fmaf(alpha, av[2], beta * cv.z), fmaf(alpha, av[3], beta * cv.w));
      } else {
        o = make_float4(alpha * av[0], alpha * av[1], alpha * av[2], alpha * av[3]);
      }
      *reinterpret_cast<float4*>(crow + gc) = o;
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (gc + e < p.N) {
          float* o = crow + gc + e;
          *o = (beta != 0.f) ? fmaf(alpha, av[e], beta * *o) : alpha * av[e];
        }
    }
  }
}

cudaError_t launch_tf32x3_tail_reduce(const Tf32x3Params& p, int pn, cudaStream_t stream) {
  const long long n = (long long)p.tiles_m * p.tiles_n - p.tail_first;
  if (p.tail_splits <= 1 || n <= 0) return cudaSuccess;
  const unsigned gy = (unsigned)((2 * kTcBM * pn / 4 + 255) / 256);  // 1 float4 per thread
  Tf32x3Params pc = p;
  void* args[] = {&pc, &pn};
  return launch_pdl(reinterpret_cast<const void*>(&tc_tail_reduce_kernel), dim3((unsigned)n, gy),
                    dim3(256), args, 0, stream);
}

}  // namespace b2g
