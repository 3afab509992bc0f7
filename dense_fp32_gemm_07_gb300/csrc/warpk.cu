// warpk.cu -- small problems in one launch: the k range of each output tile
// is split between the warps of its CTA.
//
// For a small product the FFMA plans cannot fill the GPU with whole tiles
// (512^3 is 32 tiles of 64 x 128 for 456 CTA slots), so they cut the k range
// into slices that write partial sums to a workspace and add them in a
// second kernel: two launches, the partial sums' round trip through L2 and a
// dependency between them, about 8 us a call even at 128^3.  Here one CTA
// takes one small output tile (BM x BN = 32 WM x 64 WN), and KG groups of
// WM x WN consumer warps take its k tiles in turn (k tile t goes to group
// t % KG).  Each warp keeps the 8 x 8 register outer product of the FFMA
// plans (packed two-lane FMAs; B row-major; A either row-major, k-chunked by
// a 3-D bulk-tensor view, or stored K x M, landing transposed).  When the
// groups are done, their partial tiles meet in the drained shared-memory ring
// and are added in group order, then C = alpha * sum + beta * C is written:
// one launch, no workspace.  Every output element is a fixed-order sum (k
// order inside a group, group order across them), so the results are bitwise
// reproducible run to run.
//
// One elected producer thread fills an S-stage ring of 32-k stages with
// bulk-tensor copies (full/empty mbarriers; S a multiple of KG, so that a
// slot always serves the same group).  With one slot a group (the 8-group
// tile) a group waits for its slot's refill after every stage: two slots
// took 64 x 4096 x 4096 from 50.5 to 47.4 us but 512^3 from 8.42 to 8.58, and
// the table sends long k ranges to the split-tail plans anyway.  16-k stages measured 4-11% slower from
// 384^3 to 1024^3 (twice the barrier round trips).  Every wait is bounded and
// a timeout leaves C untouched, with the reason in the status word.
#include "plan_registry.h"
#include "sgemm_ffma.cuh"

namespace b2g {

template <int WM, int WN, int KG, int BK, int STAGES, int ALAY>
struct WarpkCfg {
  static constexpr int BM = 32 * WM, BN = 64 * WN, TN = 8;
  static constexpr int kGroupWarps = WM * WN;  // the warps of one k group
  static constexpr int kConsumerWarps = kGroupWarps * KG;
  static constexpr int kConsumers = kConsumerWarps * 32;
  static constexpr int kThreads = kConsumers + 32;
  static constexpr int kAStage = BM * BK, kBStage = BK * BN;  // floats
  static constexpr int kStageBytes = (kAStage + kBStage) * 4;
  static constexpr int kRingFloats = STAGES * (kAStage + kBStage);
  static constexpr int kSmemBytes = kRingFloats * 4 + 2 * STAGES * 8 + 16;
  static_assert(STAGES % KG == 0, "a ring slot always serves the same k group");
  static_assert(KG * BM * BN <= kRingFloats, "the groups' partial tiles fit in the ring");
  static_assert(BK % 4 == 0, "A is k-chunked by 4");
  static_assert(ALAY == kAKChunk || ALAY == kAKMajor, "A's shared-memory layout");
};

template <int WM, int WN, int KG, int BK, int STAGES, int ALAY>
__global__ void __launch_bounds__(WarpkCfg<WM, WN, KG, BK, STAGES, ALAY>::kThreads, 1)
    sgemm_warpk_kernel(const __grid_constant__ SgemmParams p,
                       const __grid_constant__ CUtensorMap tmA,
                       const __grid_constant__ CUtensorMap tmB) {
  using Cfg = WarpkCfg<WM, WN, KG, BK, STAGES, ALAY>;
  constexpr int BM = Cfg::BM, BN = Cfg::BN, TN = Cfg::TN;
  extern __shared__ __align__(1024) unsigned char smem[];
  float* sA = reinterpret_cast<float*>(smem);          // [STAGES][BK/4][BM][4] or [STAGES][BK][BM]
  float* sB = sA + STAGES * Cfg::kAStage;              // [STAGES][BK][BN]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sA + Cfg::kRingFloats);
  const uint32_t full0 = smem_addr(bars);
  const uint32_t empty0 = smem_addr(bars + STAGES);
  volatile int* failed = reinterpret_cast<volatile int*>(bars + 2 * STAGES);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  pdl_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, Cfg::kGroupWarps);
    }
    *failed = 0;
    fence_mbar_init();
    fence_proxy_async_smem();
  }
  __syncthreads();
  pdl_wait();  // global memory only once the previous grid has completed

  int bt, tm, tn;
  tile_coords(p, (int)blockIdx.x, bt, tm, tn);
  const int m0 = tm * BM, n0 = tn * BN;
  const int k_tiles = p.k_tiles;

  // ---------------------------------------------------------------- producer
  if (warp == 0) {
    if (lane != 0) return;
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    int stage = 0, issued = 0;
    uint32_t phase = 0;
    for (int kt = 0; kt < k_tiles; ++kt) {
      if (p.debug_stop_ktile >= 0 && issued >= p.debug_stop_ktile) break;
      if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, p.wait_limit_ns, p.status,
                     kStatusTimeoutEmpty))
        break;
      const uint32_t fb = full0 + 8 * stage;
      mbar_arrive_expect_tx(fb, Cfg::kStageBytes);
      if constexpr (ALAY == kAKChunk)  // view {4, M, K/4, batch}
        tma_load_4d(smem_addr(sA + stage * Cfg::kAStage), &tmA, 0, m0, kt * (BK / 4), bt, fb);
      else  // A stored K x M: {M, K, batch}
        tma_load_3d(smem_addr(sA + stage * Cfg::kAStage), &tmA, m0, kt * BK, bt, fb);
      tma_load_3d(smem_addr(sB + stage * Cfg::kBStage), &tmB, n0, kt * BK, bt, fb);
      ++issued;
      if (++stage == STAGES) stage = 0, phase ^= 1u;
    }
    // leave only after every copy this thread started has landed
    for (int d = 0, pending = min(issued, STAGES); d < pending; ++d) {
      if (--stage < 0) stage = STAGES - 1, phase ^= 1u;
      if (!mbar_wait(full0 + 8 * stage, phase, p.wait_limit_ns, p.status, kStatusTimeoutDrain))
        break;
    }
    return;
  }

  // --------------------------------------------------------------- consumers
  const int cw = warp - 1;
  const int g = cw / Cfg::kGroupWarps;  // k group
  const int wm = cw % Cfg::kGroupWarps % WM, wn = cw % Cfg::kGroupWarps / WM;  // warp tile
  const int tr = lane >> 3, tc = lane & 7;
  // Thread rows: wm*32 + tr + 4i with A k-chunked (the 4 thread rows of a
  // warp read 4 consecutive 16-byte vectors), wm*32 + 4tr + (i & 3) + 16(i >> 2)
  // with A transposed (one 16-byte load gives 4 rows at one k).  Thread
  // columns 4tc + 32(j >> 2) + (j & 3).
  const int a_off = ALAY == kAKChunk ? (wm * 32 + tr) * 4 : wm * 32 + 4 * tr;
  const int b_off = wn * 64 + 4 * tc;
  float acc[8][TN];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

  for (int kt = g; kt < k_tiles; kt += KG) {
    const int stage = kt % STAGES;
    const uint32_t phase = (uint32_t)(kt / STAGES) & 1u;
    const bool landed =
        mbar_wait(full0 + 8 * stage, phase, p.wait_limit_ns, p.status, kStatusTimeoutFull);
    if (!__all_sync(0xffffffffu, landed)) {  // the whole warp gives up together
      if (lane == 0) *failed = 1;
      break;
    }
    const float* As = sA + stage * Cfg::kAStage + a_off;
    const float* Bs = sB + stage * Cfg::kBStage + b_off;
    if constexpr (ALAY == kAKMajor) {
#pragma unroll
      for (int k = 0; k < BK; ++k) {
        const float4 a0 = *reinterpret_cast<const float4*>(As + k * BM);
        const float4 a1 = *reinterpret_cast<const float4*>(As + k * BM + 16);
        const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
        float b[TN];
#pragma unroll
        for (int j4 = 0; j4 < TN / 4; ++j4) {
          const float4 v = *reinterpret_cast<const float4*>(Bs + k * BN + 32 * j4);
          b[4 * j4 + 0] = v.x, b[4 * j4 + 1] = v.y, b[4 * j4 + 2] = v.z, b[4 * j4 + 3] = v.w;
        }
        outer_product<5, TN>(acc, a, b);
      }
    } else {
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
          const float4 v = *reinterpret_cast<const float4*>(Bs + (4 * q + kk) * BN + 32 * j4);
          b[4 * j4 + 0] = v.x, b[4 * j4 + 1] = v.y, b[4 * j4 + 2] = v.z, b[4 * j4 + 3] = v.w;
        }
        float a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          a[i] = kk == 0 ? a4[i].x : kk == 1 ? a4[i].y : kk == 2 ? a4[i].z : a4[i].w;
        outer_product<5, TN>(acc, a, b);
      }
    }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * stage);
  }

  // Every consumer is past the ring (and every copy has landed) after this;
  // on a timeout anywhere, C is left alone.
  asm volatile("bar.sync 1, %0;" ::"n"(Cfg::kConsumers) : "memory");
  if (*failed) return;
  float* part = sA;  // [KG][BM][BN]: group g's partial tile
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = ALAY == kAKChunk ? wm * 32 + tr + 4 * i
                                   : wm * 32 + 4 * tr + (i & 3) + 16 * (i >> 2);
    float* row = part + (g * BM + r) * BN + b_off;
#pragma unroll
    for (int j4 = 0; j4 < TN / 4; ++j4)
      *reinterpret_cast<float4*>(row + 32 * j4) =
          make_float4(acc[i][4 * j4], acc[i][4 * j4 + 1], acc[i][4 * j4 + 2], acc[i][4 * j4 + 3]);
  }
  asm volatile("bar.sync 1, %0;" ::"n"(Cfg::kConsumers) : "memory");

  // Sum the groups' partial tiles in group order and write C: each thread takes
  // float4 positions e = t, t + kConsumers, ... of the tile (row e / (BN/4)).
  constexpr int kPos = BM * BN / 4;
  constexpr int kPer = (kPos + Cfg::kConsumers - 1) / Cfg::kConsumers;
  const int t = threadIdx.x - 32;
  float* Cb = p.C + (long long)bt * p.strideC;
  const float alpha = p.alpha, beta = p.beta;
  float4 cv[kPer];
  if (beta != 0.f && p.c_vec4) {  // every C vector this thread needs, in flight together
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int e = t + u * Cfg::kConsumers;
      const int gr = m0 + e / (BN / 4), gc = n0 + 4 * (e % (BN / 4));
      if (e < kPos && gr < p.M && gc + 3 < p.N)
        cv[u] = *reinterpret_cast<const float4*>(Cb + (long long)gr * p.ldc + gc);
    }
  }
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    const int e = t + u * Cfg::kConsumers;
    const int gr = m0 + e / (BN / 4), gc = n0 + 4 * (e % (BN / 4));
    if (e >= kPos || gr >= p.M || gc >= p.N) continue;
    float4 s = *reinterpret_cast<const float4*>(part + 4 * e);
#pragma unroll
    for (int q = 1; q < KG; ++q) {
      const float4 v = *reinterpret_cast<const float4*>(part + q * BM * BN + 4 * e);
      s.x += v.x, s.y += v.y, s.z += v.z, s.w += v.w;
    }
    float* crow = Cb + (long long)gr * p.ldc;
    if (p.c_vec4 && gc + 3 < p.N) {
      float4 o;
      if (beta != 0.f) {
        o = make_float4(fmaf(alpha, s.x, beta * cv[u].x), fmaf(alpha, s.y, beta * cv[u].y),
                        fmaf(alpha, s.z, beta * cv[u].z), fmaf(alpha, s.w, beta * cv[u].w));
      } else {
        o = make_float4(alpha * s.x, alpha * s.y, alpha * s.z, alpha * s.w);
      }
      *reinterpret_cast<float4*>(crow + gc) = o;
    } else {
      const float sv[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (gc + q < p.N) {
          float* o = crow + gc + q;
          *o = (beta != 0.f) ? fmaf(alpha, sv[q], beta * *o) : alpha * sv[q];
        }
    }
  }
}

// One CTA per output tile (of every problem of a batch).
template <int WM, int WN, int KG, int BK, int STAGES, int ALAY>
cudaError_t launch_warpk(const SgemmParams& p, const CUtensorMap* tmA, const CUtensorMap* tmB,
                         int /*num_sms*/, cudaStream_t stream) {
  using Cfg = WarpkCfg<WM, WN, KG, BK, STAGES, ALAY>;
  auto kern = sgemm_warpk_kernel<WM, WN, KG, BK, STAGES, ALAY>;
  static std::atomic<int> opted[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return cudaErrorInvalidDevice;
  if (!opted[dev].load(std::memory_order_acquire)) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
    if (e != cudaSuccess) return e;
    opted[dev].store(1, std::memory_order_release);
  }
  const long long tiles = (long long)p.tiles_m * p.tiles_n * p.batch;
  if (tiles <= 0 || tiles > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  SgemmParams pc = p;
  CUtensorMap a = *tmA, b = *tmB;
  void* args[] = {&pc, &a, &b};
  return launch_pdl(reinterpret_cast<const void*>(kern), dim3((unsigned)tiles),
                    dim3(Cfg::kThreads), args, Cfg::kSmemBytes, stream);
}

#define B2G_WARPK_PLAN(NAME, WM, WN, KG, BK, ST, ALAY, PRE)                                     \
  Plan {                                                                                         \
    NAME, WarpkCfg<WM, WN, KG, BK, ST, ALAY>::BM, WarpkCfg<WM, WN, KG, BK, ST, ALAY>::BN, BK,    \
        ST, WarpkCfg<WM, WN, KG, BK, ST, ALAY>::TN, ALAY, kFeedTMA,                              \
        WarpkCfg<WM, WN, KG, BK, ST, ALAY>::kThreads,                                            \
        WarpkCfg<WM, WN, KG, BK, ST, ALAY>::kSmemBytes, &launch_warpk<WM, WN, KG, BK, ST, ALAY>, \
        PRE, nullptr                                                                             \
  }

// Fields: name, warp tiles WM x WN (BM = 32 WM, BN = 64 WN), k groups KG, BK,
// stages, A's layout in shared memory, what runs before the kernel (as for
// the FFMA plans: 0 nothing, 2 both operands packed aligned with A
// transposed, 3 B^T (and A) transposed with 16-byte vectors).  No occupancy
// function: the host then gives these plans no split tail.
//   wk_   row-major A, k-chunked (aligned operands)
//   wkT_  A stored K x M (op(A) = A^T, aligned operands)
//   wkP_  any operands, packed first
//   wkR_  op(B) = B^T on aligned operands, transposed first
const Plan kPlansWarpk[] = {
    B2G_WARPK_PLAN("wk_32x64x32_g8", 1, 1, 8, 32, 8, kAKChunk, 0),
    B2G_WARPK_PLAN("wk_64x64x32_g4", 2, 1, 4, 32, 8, kAKChunk, 0),
    B2G_WARPK_PLAN("wk_64x128x32_g2", 2, 2, 2, 32, 8, kAKChunk, 0),
    B2G_WARPK_PLAN("wkT_32x64x32_g8", 1, 1, 8, 32, 8, kAKMajor, 0),
    B2G_WARPK_PLAN("wkT_64x64x32_g4", 2, 1, 4, 32, 8, kAKMajor, 0),
    B2G_WARPK_PLAN("wkT_64x128x32_g2", 2, 2, 2, 32, 8, kAKMajor, 0),
    B2G_WARPK_PLAN("wkP_32x64x32_g8", 1, 1, 8, 32, 8, kAKMajor, 2),
    B2G_WARPK_PLAN("wkP_64x64x32_g4", 2, 1, 4, 32, 8, kAKMajor, 2),
    B2G_WARPK_PLAN("wkP_64x128x32_g2", 2, 2, 2, 32, 8, kAKMajor, 2),
    B2G_WARPK_PLAN("wkR_32x64x32_g8", 1, 1, 8, 32, 8, kAKMajor, 3),
    B2G_WARPK_PLAN("wkR_64x64x32_g4", 2, 1, 4, 32, 8, kAKMajor, 3),
    B2G_WARPK_PLAN("wkR_64x128x32_g2", 2, 2, 2, 32, 8, kAKMajor, 3),
};
const int kNumPlansWarpk = sizeof(kPlansWarpk) / sizeof(kPlansWarpk[0]);

}  // namespace b2g
