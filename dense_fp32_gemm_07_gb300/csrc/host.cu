// host.cu -- the C ABI (include/b2g_sgemm.h): argument checks, the quick
// returns, plan choice from the tune table, bulk-tensor descriptors, launch.
//
// Quick returns follow the reference-BLAS convention (the pages are silent):
// M == 0 or N == 0 launches nothing; K == 0 or alpha == 0 only scales C by beta
// (beta == 0 writes zeros without reading C).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/b2g_sgemm.h"
#include "plan_registry.h"
#include "ptx.cuh"
#include "sgemm_params.h"
#include "tf32x3.h"
#include "transpose.h"
#include "tune_table.h"

namespace b2g {

// The device status word every kernel may flag (timeouts).  One per device
// context; the host passes its address to each kernel.
__device__ unsigned int g_status_word;

// C = beta * C over an M x N window with leading dimension ldc (beta == 0 writes
// zeros without reading C).  Used when the product term vanishes.
__global__ void scale_c_kernel(int M, int N, float beta, float* __restrict__ C, long long ldc,
                               int batch, long long strideC) {
  pdl_launch_dependents();
  pdl_wait();
  const long long per = (long long)M * N;
  const long long total = per * batch;
  for (long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long b = idx / per, r = idx - b * per;
    const long long i = r / N, j = r - i * N;
    float* q = C + b * strideC + i * ldc + j;
    *q = (beta == 0.f) ? 0.f : beta * *q;
  }
}

// Y = (P0 + P1) + Y, then Y += b * X when X is given, over an M x N window of
// row-major matrices that share the leading dimension ld (a multiple of 4, all
// bases 16-byte aligned: float4 throughout).  Rows go to blockIdx.y, float4
// columns to the threads of blockIdx.x.
__global__ void combine_rows_kernel(int M, int N4, long long ld, const float* __restrict__ P0,
                                    const float* __restrict__ P1, float b,
                                    const float* __restrict__ X, float* __restrict__ Y) {
  pdl_launch_dependents();
  pdl_wait();
  for (int i = blockIdx.y; i < M; i += gridDim.y) {
    const long long row = (long long)i * ld;
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < N4; j += gridDim.x * blockDim.x) {
      const long long o = row + 4LL * j;
      const float4 p0 = *reinterpret_cast<const float4*>(P0 + o);
      const float4 p1 = *reinterpret_cast<const float4*>(P1 + o);
      float4* yp = reinterpret_cast<float4*>(Y + o);
      float4 y = *yp;
      y.x = (p0.x + p1.x) + y.x, y.y = (p0.y + p1.y) + y.y;
      y.z = (p0.z + p1.z) + y.z, y.w = (p0.w + p1.w) + y.w;
      if (X) {
        const float4 x = *reinterpret_cast<const float4*>(X + o);
        y.x = fmaf(b, x.x, y.x), y.y = fmaf(b, x.y, y.y);
        y.z = fmaf(b, x.z, y.z), y.w = fmaf(b, x.w, y.w);
      }
      *yp = y;
    }
  }
}

namespace {

struct DeviceState {
  bool init = false;
  int err = 0;
  int sms = 0;
  unsigned int* status = nullptr;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];
std::atomic<unsigned long long> g_wait_limit_ns{2000000000ull};
std::atomic<int> g_debug_stop{-1};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_encode_init = false;

int device_state(DeviceState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return B2G_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.init) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      return B2G_ERR_DEVICE;  // not cached: a later call may succeed
    }
    if (major != 10 || minor != 3) {
      d.err = B2G_ERR_DEVICE;
    } else if (cudaGetSymbolAddress(reinterpret_cast<void**>(&d.status), g_status_word) !=
               cudaSuccess) {
      d.err = B2G_ERR_CUDA;
    }
    d.init = true;
  }
  if (d.err) return d.err;
  *out = &d;
  return 0;
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode_init) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    g_encode_init = true;
  }
  return g_encode;
}

// Library-owned workspace, one per device, for calls that do not bring their
// own.  Its users on different streams are ordered through an event recorded
// after each use, so a stream never overwrites a buffer another stream may
// still read.  It is allocated (stream-ordered) on first need and grown when a
// larger call comes; it is never used while the stream is being captured.
struct AutoWorkspace {
  std::mutex mu;
  void* ptr = nullptr;
  size_t bytes = 0;
  cudaEvent_t done = nullptr;
  bool used = false;
};
AutoWorkspace g_ws[kMaxDevices];

// Lock the device's workspace and make it at least `bytes` long, ordered on
// `st`; returns nullptr (lock released) when it cannot be had.  On success the
// caller enqueues its work and then calls ws_release().
void* ws_acquire(int dev, cudaStream_t st, size_t bytes) {
  AutoWorkspace& w = g_ws[dev];
  w.mu.lock();
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
    w.mu.unlock();
    return nullptr;
  }
  if (!w.done && cudaEventCreateWithFlags(&w.done, cudaEventDisableTiming) != cudaSuccess) {
    w.done = nullptr;
    w.mu.unlock();
    return nullptr;
  }
  if (w.used && cudaStreamWaitEvent(st, w.done, 0) != cudaSuccess) {
    w.mu.unlock();
    return nullptr;
  }
  if (bytes > w.bytes) {
    const size_t grain = size_t(2) << 20;
    const size_t want = (bytes + grain - 1) / grain * grain;
    void* np = nullptr;
    if (cudaMallocAsync(&np, want, st) != cudaSuccess) {
      cudaGetLastError();
      w.mu.unlock();
      return nullptr;
    }
    if (w.ptr) cudaFreeAsync(w.ptr, st);
    w.ptr = np;
    w.bytes = want;
  }
  return w.ptr;
}

void ws_release(int dev, cudaStream_t st) {
  AutoWorkspace& w = g_ws[dev];
  if (cudaEventRecord(w.done, st) == cudaSuccess) w.used = true;
  w.mu.unlock();
}

// Every compiled plan, indexed in this order.
struct PlanGroup {
  const Plan* plans;
  const int* count;
};
const PlanGroup kGroups[] = {
    {kPlansTMA, &kNumPlansTMA},         {kPlansT, &kNumPlansT},
    {kPlansT64x128, &kNumPlansT64x128}, {kPlansT128x64, &kNumPlansT128x64},
    {kPlansT128x64k32, &kNumPlansT128x64k32},
    {kPlansT64x128k32, &kNumPlansT64x128k32},
    {kPlansT128x128, &kNumPlansT128x128}, {kPlansGeneral, &kNumPlansGeneral},
    {kPlansSkinny, &kNumPlansSkinny},     {kPlansSkinnyTma, &kNumPlansSkinnyTma},
    {kPlansCs, &kNumPlansCs},           {kPlansTmaO5, &kNumPlansTmaO5},
    {kPlansWarpk, &kNumPlansWarpk},
};

int num_plans() {
  int n = 0;
  for (const PlanGroup& g : kGroups) n += *g.count;
  return n;
}

const Plan* plan_at(int i) {
  if (i < 0) return nullptr;
  for (const PlanGroup& g : kGroups) {
    if (i < *g.count) return &g.plans[i];
    i -= *g.count;
  }
  return nullptr;
}

int plan_index(const char* name) {
  for (int i = 0; i < num_plans(); ++i)
    if (std::strcmp(plan_at(i)->name, name) == 0) return i;
  return -1;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool is_skinny(const Plan& pl) { return pl.feed == kFeedSkinny || pl.feed == kFeedSkinnyTMA; }

constexpr int kHostPanelsMax = 16;  // row panels of b2g_sgemm_host

struct Call {
  int transA, transB, M, N, K;
  float alpha, beta;
  const float* A;
  int lda;
  const float* B;
  int ldb;
  float* C;
  int ldc;
  int batch = 1;  // independent problems, operands advancing by the strides (elements)
  long long strideA = 0, strideB = 0, strideC = 0;
};

// 0 when the arguments are valid, else the B2G_ERR_* code.
int validate(const Call& c) {
  if (c.M < 0 || c.N < 0 || c.K < 0 || c.batch < 0) return B2G_ERR_INVALID_DIM;
  if (c.strideA < 0 || c.strideB < 0 || c.strideC < 0) return B2G_ERR_INVALID_LD;
  const int a_cols = c.transA ? c.M : c.K;
  const int b_cols = c.transB ? c.K : c.N;
  if (c.lda < (a_cols > 1 ? a_cols : 1) || c.ldb < (b_cols > 1 ? b_cols : 1) ||
      c.ldc < (c.N > 1 ? c.N : 1))
    return B2G_ERR_INVALID_LD;
  if (c.M == 0 || c.N == 0 || c.batch == 0) return 0;
  if (c.C == nullptr) return B2G_ERR_NULL;
  if (c.K > 0 && c.alpha != 0.f && (c.A == nullptr || c.B == nullptr)) return B2G_ERR_NULL;
  return 0;
}

bool needs_gemm(const Call& c) {
  return c.M > 0 && c.N > 0 && c.K > 0 && c.batch > 0 && c.alpha != 0.f;
}

int operand_class(const Call& c) {
  const bool ab_aligned = aligned16(c.A) && aligned16(c.B) && c.lda % 4 == 0 && c.ldb % 4 == 0 &&
                          (c.batch <= 1 || (c.strideA % 4 == 0 && c.strideB % 4 == 0));
  if (!ab_aligned) return kClassGeneral;
  if (c.transB) return c.K % 4 == 0 ? kClassFastTransB : kClassGeneral;
  if (c.transA) return kClassFastTransA;
  return c.K % 4 == 0 ? kClassFast : kClassGeneral;
}

bool plan_accepts(const Plan& pl, const Call& c) {
  if (pl.feed == kFeedCpAsync) return true;
  const int cls = operand_class(c);
  if (is_skinny(pl))
    return cls == kClassFast && c.M <= pl.BM && c.N % 4 == 0 && c.batch <= 65535;
  if (pl.pretranspose == 2) return true;  // packing accepts any operands
  if (pl.pretranspose == 1) return cls == kClassFast;
  if (pl.pretranspose == 3) return cls == kClassFastTransB;
  if (pl.feed == kFeedTMATrans || pl.alayout == kAKChunk) return cls == kClassFast;
  return cls == kClassFastTransA;
}

// The tune table's plan; `fallback` receives the plan to use when the chosen
// one needs a workspace that cannot be had (the same plan when it needs none).
int tail_split(const Plan& pl, const Call& c, int* first);
double tile_shape_score(const Plan& pl, const Call& c);

// The packed 128 x 64 plans and their 64 x 128 twins run at the same rate on
// large products; which one a call gets depends on padding and wave fill.
const char* const kTileTwins[][2] = {
    {"pre_128x64x32_s3_o5", "pre_64x128x32_s3_o5"},
    {"tmaT_128x64x32_s3_o5", "tmaT_64x128x32_s3_o5"},
    {"pack_128x64x32_s3_o5", "pack_64x128x32_s3_o5"},
    {"pret_128x64x32_s3_o5", "pret_64x128x32_s3_o5"},
};

// The one-launch small-problem plans (wk_*: one CTA per output tile, its k
// range split between the CTA's warps) against the split-tail plan that the
// next rule names, by a model fitted to GB300 timings of back-to-back calls:
// a wk call takes 2.0 + waves x (2.4 + BM x BN x K x 4.6e-6 x (1 + 0.1 x
// log2(K / 1024) above K = 1024)) us (waves of one CTA per SM; each wave pays
// its CTAs' start, first copies and reduction),
// the split-tail plan 7.4 + (M N K of the whole call) x 3.7e-8 us, and a wk
// plan is taken when its estimate is 3% lower (near a tie the wk plan's
// second wave made it the slower one with operands out of L2: the ragged
// 1000 x 1025 x 777, packed first, 50.9 us against 47.4).  Measured (us; split tail /
// 32 x 64 / 64 x 64 tiles, 16-k stages): 128^3 10.4 / 8.4 / 7.2, 256^3 10.2 / 7.2
// / 8.1, 384^3 9.9 / 7.9 / 10.5, 512^3 12.4 / 9.2 / 13.2, 768^3 23.7 / 24.0 /
// 18.6, 1024^3 47.6 / 59.2 / 47.0; strided batches (split tail / the wk plan
// the model picks): 128 x 128^3 14.6 / 27.2, 64 x 256^3 48.4 / 53.2,
// 16 x 384^3 35.6 / 41.0, 4 x 512^3 29.6 / 26.2, 2 x 768^3 40.4 / 36.8;
// 1000 x 1024 x 776 (split tail / wk 64 x 64) 42.2 / 37.0, with A stored
// K x M 38.7 / 33.9, with B stored N x K 42.8 / 39.1.
// Returns the plan of the family `rule_plan` names (wk_, wkT_, wkP_, wkR_:
// the same kernel for each operand class) with the smaller estimate (the
// larger tile on a tie: fewer waves), or -1 when the split-tail plan should
// run (many waves of small tiles, or few tiles over a long k range such as
// 128 x 128 x 32768).  A family's packing or transposing pass is the same as
// its split-tail counterpart's, so the estimates leave it out.
int warpk_choice(const Call& c, const char* rule_plan) {
  int sms = 152;
  DeviceState* d = nullptr;
  if (device_state(&d) == 0) sms = d->sms;
  const double b = c.batch > 0 ? c.batch : 1;
  double best = 0.97 * (7.4 + (double)c.M * c.N * (double)c.K * b * 3.7e-8);
  int pick = -1;
  // a CTA's FP32 pipe keeps less busy over a long k range (1-wave timings:
  // 4.6e-6 us per multiply-add of a CTA up to K = 1024, 5.5e-6 at K = 4096)
  const double long_k = c.K > 1024 ? 1.0 + 0.1 * std::log2((double)c.K / 1024.0) : 1.0;
  const char* us = std::strchr(rule_plan, '_');
  const size_t fam = us ? (size_t)(us - rule_plan) : 0;
  for (const char* tile : {"_32x64x32_g8", "_64x64x32_g4", "_64x128x32_g2"}) {
    char name[32];
    if (fam == 0 || fam + std::strlen(tile) >= sizeof(name)) break;
    std::memcpy(name, rule_plan, fam);
    std::strcpy(name + fam, tile);
    const int i = plan_index(name);
    if (i < 0 || !plan_accepts(*plan_at(i), c)) continue;
    const Plan& pl = *plan_at(i);
    const double tiles = (double)((c.M + pl.BM - 1) / pl.BM) * ((c.N + pl.BN - 1) / pl.BN) * b;
    const double waves = std::ceil(tiles / sms);
    const double t = 2.0 + waves * (2.4 + pl.BM * pl.BN * (double)c.K * 4.6e-6 * long_k);
    if (t <= best) best = t, pick = i;
  }
  return pick;
}

int select_plan(const Call& c, int* fallback = nullptr) {
  const int cls = operand_class(c);
  // The work of the whole call: a batch of products amortises a
  // transpose-first plan like one large product (one launch each for all),
  // once each product has ~5e7 multiply-adds (measured: 32 x 512^3 171.6 us
  // against 203.1 on the k-chunked split-tail plan; 64 x 256^3 66.7 against
  // 60.1).
  const double per = (double)c.M * c.N * c.K;
  const double mnk = c.batch > 1 && per >= 5.0e7 ? per * c.batch : per;
  for (const TuneRule& r : kTuneTable) {
    if (r.cls == cls && c.M >= r.m_min && c.M <= r.m_max && c.N >= r.n_min && c.N <= r.n_max &&
        mnk >= r.mnk_min && mnk < r.mnk_max) {
      int i = plan_index(r.plan);
      if (std::strncmp(r.plan, "wk", 2) == 0) {  // a wk family's plan, or the next rule
        i = warpk_choice(c, r.plan);
        if (i < 0) continue;
      }
      if (i >= 0 && plan_accepts(*plan_at(i), c)) {
        if (fallback) {
          const int f = r.fallback ? plan_index(r.fallback) : i;
          *fallback = f >= 0 ? f : i;
        }
        for (const auto& tw : kTileTwins) {  // the other tile shape, when clearly better
          if (strcmp(r.plan, tw[0]) != 0) continue;
          const int j = plan_index(tw[1]);
          if (j >= 0 && plan_accepts(*plan_at(j), c) &&
              tile_shape_score(*plan_at(j), c) > 1.03 * tile_shape_score(*plan_at(i), c))
            i = j;
        }
        return i;
      }
    }
  }
  const int g = plan_index("gen_128x128x16_s4");
  if (fallback) *fallback = g;
  return g;
}

long long pre_ld(int M) { return ((long long)M + 3) / 4 * 4; }

// SMs and resident CTAs per SM of plan `pl` on the current device (152 and 4
// when no device answers, as on a machine without a GPU).
void plan_capacity(const Plan& pl, int* sms, int* occ) {
  *sms = 152, *occ = 4;
  DeviceState* d = nullptr;
  if (device_state(&d) == 0) {
    *sms = d->sms;
    const int o = pl.occupancy ? pl.occupancy() : 0;
    if (o > 0) *occ = o;
  }
}

// Split-K factor of the skinny plans: as many k splits per 128-column slab as
// fill every resident CTA slot once (one wave), at least 64 k per split; *kc
// receives the k extent of one split (a multiple of 16).
int skinny_splits(const Plan& pl, const Call& c, int* kc) {
  int sms = 0, occ = 0;
  plan_capacity(pl, &sms, &occ);
  const long long slabs = (c.N + 127) / 128 * (c.batch > 0 ? c.batch : 1);
  long long S = (long long)sms * occ / slabs;
  long long smax = c.K / 64 > 1 ? c.K / 64 : 1;
  if (pl.feed == kFeedSkinnyTMA && smax > 8) smax = 8;  // the k slabs of a slab form one cluster
  if (S > smax) S = smax;
  if (S < 1) S = 1;
  long long k = (c.K + S - 1) / S;
  const long long granule = pl.feed == kFeedSkinnyTMA ? pl.BK : 16;  // whole stages per split
  k = (k + granule - 1) / granule * granule;
  *kc = (int)k;
  return (int)((c.K + k - 1) / k);
}

// Split tail of an FFMA plan: with T output tiles and G = SMs x resident
// CTAs, T = q*G + r.  When 0 < r, the last r tiles are each cut into S = G / r
// k slices (at most one slice per CTA, at least 64 k per slice), so the
// persistent grid's last round keeps every CTA busy instead of r of them.
// Returns S (1: no split) and the first split tile in *first.
// 64-k slices: 512^3 (32 tiles on 456 slots) 14.7 -> 17.1 TFLOP/s against
// 128-k slices; 32 k gained nothing more (17.25)
constexpr int kMinSliceK = 64;

// Estimated time (us) of a persistent FFMA grid whose work units are
// `first` whole tiles and then (tiles - first) tiles cut into S k slices,
// unit u going to CTA u mod G and CTA b to SM b mod sms (so SM 0 carries the
// most).  An SM's CTAs run side by side until the shortest is done; each
// phase runs at the FP32 pipe efficiency of the consumer warps still active
// (12 or more 0.88, 8 0.85, 4 0.40) and every unit pays one k tile of
// overhead (its fill and epilogue).  A split adds its reduction: the slices
// written and read back, C read and written, at 5.5 TB/s, plus 2 us.
// Fitted to 20 GB300 timings of square products from 1152^3 to 4096^3 with
// chosen splits (3% root-mean-square error).
double tail_time_us(const Plan& pl, long long tiles, long long kt, int sms, int occ,
                    long long first, long long S, bool read_c) {
  const long long G = (long long)sms * occ;
  const long long f = S > 1 ? first : tiles;
  const long long ns = S > 1 ? (tiles - first) * S : 0;
  const long long slice = (kt + S - 1) / S;
  double loads[8];
  const int n = occ < 8 ? occ : 8;
  for (int i = 0; i < n; ++i) {
    const long long b = (long long)i * sms;
    const long long whole = b < f ? (f - b + G - 1) / G : 0;
    const long long sl = b < ns ? (ns - b + G - 1) / G : 0;
    loads[i] = (double)(whole * (kt + 1) + sl * (slice + 1));
  }
  std::sort(loads, loads + n);
  const int cw = pl.threads / 32 - 1;  // consumer warps per CTA
  double t = 0.0, prev = 0.0;
  for (int i = 0; i < n; ++i) {
    const int active = n - i, w = active * cw;
    const double e = w >= 12 ? 0.88 : w >= 8 ? 0.85 : w >= 4 ? 0.40 : 0.20;
    t += active * (loads[i] - prev) / e;
    prev = loads[i];
  }
  t *= (double)pl.BM * pl.BN * pl.BK / (128.0 * 2070.0);
  if (S > 1)
    t += (double)(tiles - first) * pl.BM * pl.BN * 4.0 * (2.0 * S + 1.0 + (read_c ? 1.0 : 0.0)) /
             5.5e6 +
         2.0;
  return t;
}

// The split: the rule above, unless the balance model expects another split
// (all of the last two or three rounds' tiles cut, or more slices) to be at
// least 3% faster.  Measured (us, rule -> chosen): 1152^3 70.8 -> 63.1 (all
// 162 tiles in 4 slices), 1664^3 178.7 -> 157.8 (338 tiles in 4 slices, no
// split before: 34 SMs ran three tiles, the rest two), 2560^3 546.8 -> 513.7
// (the 344 tiles after the first round in 2 slices); 1408^3 and 3072^3, where
// the model's alternatives measured slower (116.1 and 876.3 against 104.7
// and 863.0), keep the rule's choice.
int tail_split(const Plan& pl, const Call& c, int* first) {
  *first = 0;
  if (is_skinny(pl) || !pl.occupancy || pl.cluster_max) return 1;
  const long long tiles =
      (long long)((c.M + pl.BM - 1) / pl.BM) * ((c.N + pl.BN - 1) / pl.BN) * c.batch;
  int sms = 0, occ = 0;
  plan_capacity(pl, &sms, &occ);
  const long long G = (long long)sms * occ;
  if (tiles <= 0 || G <= 0) return 1;
  const long long q = tiles / G, r = tiles - q * G;
  if (r == 0) return 1;
  const long long smax = c.K / kMinSliceK;
  long long S = G / r;
  if (S > smax) S = smax;
  long long f = q * G;
  if (S < 2) S = 1, f = 0;
  const long long kt = (c.K + pl.BK - 1) / pl.BK;
  const bool read_c = c.beta != 0.f;
  const double rule = tail_time_us(pl, tiles, kt, sms, occ, f, S, read_c);
  double best = 0.97 * rule;
  for (long long qq = q >= 2 ? q - 2 : 0; qq <= q; ++qq) {
    if (qq * G >= tiles) continue;
    for (long long s = 1; s <= smax && s <= 16; ++s) {
      if (s == 1 && qq != q) continue;  // no split: one candidate
      const double t = tail_time_us(pl, tiles, kt, sms, occ, qq * G, s, read_c);
      if (t < best) best = t, S = s, f = s > 1 ? qq * G : 0;
    }
  }
  if (S < 2) return 1;
  *first = (int)f;
  return (int)S;
}

// k slices per tile of a cluster-split plan: as many as fill the resident CTA
// slots once (S = slots / tiles), at most the plan's largest cluster, and at
// least two k stages per slice.
int cs_splits(const Plan& pl, const Call& c) {
  const long long tiles =
      (long long)((c.M + pl.BM - 1) / pl.BM) * ((c.N + pl.BN - 1) / pl.BN) * c.batch;
  int sms = 0, occ = 0;
  plan_capacity(pl, &sms, &occ);
  long long S = tiles > 0 ? (long long)sms * occ / tiles : 1;
  const long long k_tiles = (c.K + pl.BK - 1) / pl.BK;
  if (S > pl.cluster_max) S = pl.cluster_max;
  if (S > k_tiles / 2) S = k_tiles / 2;
  if (S < 1) S = 1;
  return (int)S;
}

// Expected share of the FFMA pipe's work that is useful for plan pl's tile
// shape: the wave fill of its persistent grid (whole rounds of tiles, the last
// round shortened to 1/S by the split tail) over the padding of M and N up to
// whole tiles.  Measured, 128 x 64 vs 64 x 128 tiles at K = 4096: M = 64
// 0.49 vs 0.98 (28.6 vs 43.0 TFLOP/s), M = 448 0.49 vs 0.98 (34.0 vs 64.2),
// M = 1088 0.90 vs 0.99 (61.1 vs 66.9), M = 192 x N = 11008 0.57 vs 0.57
// (39.2 vs 39.2).
double tile_shape_score(const Plan& pl, const Call& c) {
  const long long tm = (c.M + pl.BM - 1) / pl.BM, tn = (c.N + pl.BN - 1) / pl.BN;
  const double pad = (double)(tm * pl.BM) * (double)(tn * pl.BN) / ((double)c.M * c.N);
  const long long tiles = tm * tn * (c.batch > 0 ? c.batch : 1);
  int sms = 0, occ = 0;
  plan_capacity(pl, &sms, &occ);
  const double G = (double)sms * occ;
  int first = 0;
  const int S = tail_split(pl, c, &first);
  const long long q = (long long)(tiles / G), r = tiles - (long long)(q * G);
  const double rounds = (double)q + (r > 0 ? (S > 1 ? 1.0 / S : 1.0) : 0.0);
  const double fill = rounds > 0 ? (double)tiles / G / rounds : 0.0;
  return fill / pad;
}

// Bytes of the split tail's partial sums (0 without a split) and where they
// start in the workspace (after what the plan itself needs, 256-byte aligned).
size_t tail_bytes(const Plan& pl, const Call& c, int S, int first) {
  if (S <= 1) return 0;
  const long long tiles =
      (long long)((c.M + pl.BM - 1) / pl.BM) * ((c.N + pl.BN - 1) / pl.BN) * c.batch;
  return (size_t)(tiles - first) * S * pl.BM * pl.BN * sizeof(float);
}
size_t tail_offset(size_t base) { return (base + 255) / 256 * 256; }

// Workspace bytes plan `pl` cannot do without for this call (0 when none).
size_t plan_base_bytes(const Plan& pl, const Call& c) {
  const size_t nb = (size_t)(c.batch > 0 ? c.batch : 0);
  if (pl.pretranspose == 1) return nb * (size_t)c.K * (size_t)pre_ld(c.M) * sizeof(float);
  if (pl.pretranspose == 2)
    return nb * (size_t)c.K * (size_t)(pre_ld(c.M) + pre_ld(c.N)) * sizeof(float);
  if (pl.pretranspose == 3)  // B^T transposed, and A unless it comes stored K x M
    return nb * (size_t)c.K * (size_t)((c.transA ? 0 : pre_ld(c.M)) + pre_ld(c.N)) * sizeof(float);
  if (pl.feed == kFeedSkinny) {  // partial sums per k slab (the cluster plans keep them on chip)
    int kc = 0;
    const int S = skinny_splits(pl, c, &kc);
    return S > 1 ? nb * (size_t)S * c.M * c.N * sizeof(float) : 0;
  }
  return 0;
}

// Workspace bytes plan `pl` wants for this call: its own need plus room for
// the split tail's partial sums.
size_t plan_work_bytes(const Plan& pl, const Call& c) {
  const size_t base = plan_base_bytes(pl, c);
  int first = 0;
  const int S = tail_split(pl, c, &first);
  const size_t t = tail_bytes(pl, c, S, first);
  return t ? tail_offset(base) + t : base;
}



// Row-major {inner, outer} matrices, `batch` of them `batch_stride_elems`
// apart: a 3-D view {inner, outer, batch} with boxes {box_inner, box_outer, 1}.
int encode_2d(CUtensorMap* m, const float* base, long long inner, long long outer,
              long long row_stride_elems, int box_inner, int box_outer, int batch = 1,
              long long batch_stride_elems = 0) {
  auto enc = encoder();
  if (!enc) return B2G_ERR_TENSOR_MAP;
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)outer, (cuuint64_t)batch};
  cuuint64_t strides[2] = {(cuuint64_t)row_stride_elems * 4,
                           batch > 1 ? (cuuint64_t)batch_stride_elems * 4 : 16};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)box_outer, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : B2G_ERR_TENSOR_MAP;
}

// 2-D row-major tensor {inner, outer} with boxes of 32 x box_outer FP32
// elements (128 bytes) landing with the 128-byte swizzle: the K-major operand
// layout the tensor cores read.
int encode_2d_sw128(CUtensorMap* m, const float* base, long long inner, long long outer,
                    long long row_stride_elems, int box_outer) {
  auto enc = encoder();
  if (!enc) return B2G_ERR_TENSOR_MAP;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)row_stride_elems * 4};
  cuuint32_t box[2] = {32, (cuuint32_t)box_outer};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : B2G_ERR_TENSOR_MAP;
}

// Row-major A (M x K, lda) seen as a 4-D tensor {4, M, K/4, batch}: element
// (e, r, q, b) is A_b[r][4q + e].  A box {4, BM, BK/4, 1} lands in shared memory
// as [BK/4][BM][4].
int encode_a_kchunk(CUtensorMap* m, const float* A, int M, int K, int lda, int BM, int BK,
                    int batch = 1, long long batch_stride_elems = 0) {
  auto enc = encoder();
  if (!enc) return B2G_ERR_TENSOR_MAP;
  cuuint64_t dims[4] = {4, (cuuint64_t)M, (cuuint64_t)(K / 4), (cuuint64_t)batch};
  cuuint64_t strides[3] = {(cuuint64_t)lda * 4, 16,
                           batch > 1 ? (cuuint64_t)batch_stride_elems * 4 : 16};
  cuuint32_t box[4] = {4, (cuuint32_t)BM, (cuuint32_t)(BK / 4), 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float*>(A), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : B2G_ERR_TENSOR_MAP;
}

int launch_scale(const Call& c, const DeviceState& d, cudaStream_t st) {
  const long long total = (long long)c.M * c.N * c.batch;
  long long blocks = (total + 255) / 256;
  const long long cap = (long long)d.sms * 8;
  if (blocks > cap) blocks = cap;
  long long ldc = c.ldc, strideC = c.strideC;
  int batch = c.batch;
  void* args[] = {(void*)&c.M, (void*)&c.N, (void*)&c.beta, (void*)&c.C, &ldc, &batch, &strideC};
  cudaError_t e = launch_pdl(reinterpret_cast<const void*>(&scale_c_kernel),
                             dim3((unsigned)blocks), dim3(256), args, 0, st);
  return e == cudaSuccess ? 0 : B2G_ERR_LAUNCH;
}

// Launch one GEMM.  `user_ws` (may be null) is a caller-provided workspace of
// `user_ws_bytes`; without one, plans that need a workspace take the device's
// library-owned one, and fall back to a plan that needs none when it cannot be
// had.  A forced plan that needs a workspace fails with B2G_ERR_UNSUPPORTED
// when none can be had.
int run(const Call& c, int forced_plan, void* stream, void* user_ws = nullptr,
        size_t user_ws_bytes = 0, bool allow_auto_ws = true) {
  int rc = validate(c);
  if (rc) return rc;
  if (c.M == 0 || c.N == 0 || c.batch == 0) return 0;
  if (forced_plan >= num_plans()) return B2G_ERR_INVALID_PLAN;
  DeviceState* d = nullptr;
  rc = device_state(&d);
  if (rc) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (!needs_gemm(c)) return launch_scale(c, *d, st);

  int fallback = -1;
  int pi = forced_plan >= 0 ? forced_plan : select_plan(c, &fallback);
  const Plan* pl = plan_at(pi);
  if (!pl) return B2G_ERR_INVALID_PLAN;
  if (!plan_accepts(*pl, c)) return B2G_ERR_UNSUPPORTED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return B2G_ERR_DEVICE;
  float* ws = nullptr;
  bool auto_ws = false;
  const size_t base = plan_base_bytes(*pl, c);
  int tail_first = 0;
  int tail_S = tail_split(*pl, c, &tail_first);
  const size_t tail = tail_bytes(*pl, c, tail_S, tail_first);
  const size_t need = tail ? tail_offset(base) + tail : base;
  if (need) {
    if (user_ws && aligned16(user_ws) && user_ws_bytes >= need) {
      ws = static_cast<float*>(user_ws);
    } else if (user_ws && aligned16(user_ws) && base && user_ws_bytes >= base) {
      ws = static_cast<float*>(user_ws);  // room for the plan, not for the split tail
      tail_S = 1;
    } else if (allow_auto_ws) {
      ws = static_cast<float*>(ws_acquire(dev, st, need));
      auto_ws = ws != nullptr;
    }
    if (!ws) tail_S = 1;
    if (!ws && pl->pretranspose) {
      if (forced_plan >= 0 || fallback < 0) return B2G_ERR_UNSUPPORTED;
      pi = fallback;
      pl = plan_at(pi);
      if (!pl || !plan_accepts(*pl, c) || pl->pretranspose) return B2G_ERR_UNSUPPORTED;
    }
    // a skinny plan without a workspace runs unsplit
  }

  SgemmParams p;
  p.M = c.M, p.N = c.N, p.K = c.K;
  p.alpha = c.alpha, p.beta = c.beta;
  p.A = c.A, p.lda = c.lda, p.B = c.B, p.ldb = c.ldb, p.C = c.C, p.ldc = c.ldc;
  p.transA = c.transA, p.transB = c.transB;
  p.batch = c.batch, p.strideA = c.strideA, p.strideB = c.strideB, p.strideC = c.strideC;
  p.c_vec4 = aligned16(c.C) && c.ldc % 4 == 0 && (c.batch <= 1 || c.strideC % 4 == 0);
  p.tiles_m = (c.M + pl->BM - 1) / pl->BM;
  p.tiles_n = (c.N + pl->BN - 1) / pl->BN;
  if ((long long)p.tiles_m * p.tiles_n * c.batch >= 0x7fffffffLL) {
    if (auto_ws) ws_release(dev, st);
    return B2G_ERR_INVALID_DIM;  // more output tiles than the tile index can address
  }
  p.group_m = 8;
  p.k_tiles = (c.K + pl->BK - 1) / pl->BK;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.debug_stop_ktile = g_debug_stop.load();
  p.status = d->status;
  p.work = nullptr, p.splits = 1, p.kc = c.K;
  p.tail_first = 0, p.tail_splits = 1;
  if (pl->feed == kFeedSkinnyTMA) {  // split k slabs meet in a cluster: no workspace
    p.splits = skinny_splits(*pl, c, &p.kc);
  } else if (pl->feed == kFeedSkinny && ws) {
    p.splits = skinny_splits(*pl, c, &p.kc);
    p.work = ws;
  } else if (pl->cluster_max) {  // k slices summed inside clusters: no workspace
    p.tail_first = 0, p.tail_splits = cs_splits(*pl, c);
  } else if (ws && tail_S > 1) {
    p.tail_first = tail_first, p.tail_splits = tail_S;
    p.work = ws + tail_offset(base) / sizeof(float);
  }

  cudaError_t e = cudaSuccess;
  if (ws && pl->pretranspose == 1) {  // At = A^T, then the kernel reads A stored K x M
    const long long ldat = pre_ld(c.M), sat = (long long)c.K * ldat;
    e = launch_transpose_a(c.A, c.M, c.K, c.lda, ws, ldat, st, c.batch, c.strideA, sat);
    p.A = ws, p.lda = ldat, p.transA = 1, p.strideA = sat;
  } else if (ws && pl->pretranspose == 2) {  // At = op(A)^T and Bp = op(B), both aligned
    const long long ldat = pre_ld(c.M), ldbp = pre_ld(c.N);
    const long long sat = (long long)c.K * ldat, sbp = (long long)c.K * ldbp;
    float* At = ws;
    float* Bp = ws + (size_t)c.batch * sat;
    e = launch_pack2(pack_job(c.A, c.lda, c.transA ? 0 : 1, c.K, c.M, At, ldat, c.strideA, sat),
                     pack_job(c.B, c.ldb, c.transB ? 1 : 0, c.K, c.N, Bp, ldbp, c.strideB, sbp),
                     st, c.batch);
    p.A = At, p.lda = ldat, p.transA = 1, p.strideA = sat;
    p.B = Bp, p.ldb = ldbp, p.transB = 0, p.strideB = sbp;
  } else if (ws && pl->pretranspose == 3) {
    // B stored N x K -> Bp (K x ldbp), and row-major A -> At (K x ldat), both
    // with 16-byte vectors; A stored K x M is read in place
    const long long ldbp = pre_ld(c.N), sbp = (long long)c.K * ldbp;
    float* Bp = ws;
    if (!c.transA) {
      const long long ldat = pre_ld(c.M), sat = (long long)c.K * ldat;
      float* At = ws;
      Bp = ws + (size_t)c.batch * sat;
      e = launch_transpose_a(c.A, c.M, c.K, c.lda, At, ldat, st, c.batch, c.strideA, sat);
      p.A = At, p.lda = ldat, p.transA = 1, p.strideA = sat;
    }
    if (e == cudaSuccess)
      e = launch_transpose_a(c.B, c.N, c.K, c.ldb, Bp, ldbp, st, c.batch, c.strideB, sbp);
    p.B = Bp, p.ldb = ldbp, p.transB = 0, p.strideB = sbp;
  }

  CUtensorMap tmA, tmB;
  const CUtensorMap* pA = nullptr;
  const CUtensorMap* pB = nullptr;
  if (e == cudaSuccess && pl->feed == kFeedSkinnyTMA) {
    // A {K, M, batch} in boxes of 32 k x BM rows; B {N, K, batch} in boxes of
    // 128 columns x 32 k
    rc = encode_2d(&tmA, p.A, c.K, c.M, p.lda, pl->BK, pl->BM, c.batch, p.strideA);
    if (!rc) rc = encode_2d(&tmB, p.B, c.N, c.K, p.ldb, pl->BN, pl->BK, c.batch, p.strideB);
    pA = &tmA, pB = &tmB;
  } else if (e == cudaSuccess && pl->feed != kFeedCpAsync && pl->feed != kFeedSkinny) {
    if (pl->feed != kFeedTMA || pl->alayout == kAKChunk)
      rc = encode_a_kchunk(&tmA, p.A, c.M, c.K, (int)p.lda, pl->BM, pl->BK, c.batch, p.strideA);
    else  // A stored K x M
      rc = encode_2d(&tmA, p.A, c.M, c.K, p.lda, pl->BM, pl->BK, c.batch, p.strideA);
    if (!rc) rc = encode_2d(&tmB, p.B, c.N, c.K, p.ldb, pl->BN, pl->BK, c.batch, p.strideB);
    pA = &tmA, pB = &tmB;
  }
  if (e == cudaSuccess && !rc) e = pl->launch(p, pA, pB, d->sms, st);
  if (e == cudaSuccess && !rc && p.tail_splits > 1 && !pl->cluster_max)
    e = launch_tail_reduce(p, pl->BM, pl->BN, st);
  if (auto_ws) ws_release(dev, st);
  if (rc) return rc;
  return e == cudaSuccess ? 0 : B2G_ERR_LAUNCH;
}

// ------------------------------------------------------------ host operands
//
// b2g_sgemm_host: A, B and C live in host memory; the host link (about 210 GB/s
// in, 190 GB/s out on GB300) is much slower than the GEMM, so the copies are
// overlapped with it:
//  * K is cut into chunks (for K >= 2048: three growing chunks, K/8, 3K/8 and
//    K/2, 16-aligned); the copy stream sends B's rows and A's columns of chunk
//    0, then of chunk 1, then of chunk 2, then C.  The caller's stream
//    multiplies each chunk as soon as it has landed, into a product of its
//    own (P0, P1, D: every GEMM runs with beta 0 and never reads C, which
//    saves the epilogue's waits for C; at 4096 x 4096 x 1536 a beta-1 pass
//    takes 782 us against 752).
//  * The last chunk runs in row panels of about 1024 rows, the last of them
//    cut into 3/4 and 1/4: each panel is combined, D = (P0 + P1) + D + beta * C,
//    and goes back to the host on a second copy stream while the next panel
//    multiplies.
// So the GEMM starts after 1/8 of A and B have arrived, C's copy hides behind
// the first chunks, and only the last, short panel's return is exposed.  With
// K < 2048 there is one chunk and C goes in with A, panel by panel, straight
// into D.  Chunked sums are rounded once per chunk, which the FP32 bound
// covers.  Device copies are packed with rows padded to a multiple of 4 floats.
struct HostPath {
  std::mutex mu;
  bool init = false;
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, done = nullptr, c_in = nullptr, c_out = nullptr;
  cudaEvent_t chunk[kHostPanelsMax] = {}, panel_in[kHostPanelsMax] = {},
              gemm[kHostPanelsMax] = {};
  void* buf = nullptr;
  size_t bytes = 0;
  bool used = false;
};
HostPath g_hostpath[kMaxDevices];

int hostpath_init(HostPath& h) {
  if (h.init) return 0;
  if (cudaStreamCreateWithFlags(&h.h2d, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&h.d2h, cudaStreamNonBlocking) != cudaSuccess)
    return B2G_ERR_CUDA;
  cudaEvent_t* evs[] = {&h.start, &h.done, &h.c_in, &h.c_out};
  for (cudaEvent_t* e : evs)
    if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return B2G_ERR_CUDA;
  for (int i = 0; i < kHostPanelsMax; ++i)
    if (cudaEventCreateWithFlags(&h.chunk[i], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h.panel_in[i], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&h.gemm[i], cudaEventDisableTiming) != cudaSuccess)
      return B2G_ERR_CUDA;
  h.init = true;
  return 0;
}

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

int run_host(const Call& c, void* stream) {
  int rc = validate(c);
  if (rc) return rc;
  if (c.M == 0 || c.N == 0) return 0;
  DeviceState* d = nullptr;
  rc = device_state(&d);
  if (rc) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return B2G_ERR_DEVICE;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
    return B2G_ERR_UNSUPPORTED;  // allocations and host copies stay out of graphs

  const bool gemm = needs_gemm(c);
  const bool read_c = c.beta != 0.f;
  const size_t M = (size_t)c.M, N = (size_t)c.N, K = (size_t)c.K;
  const size_t kp = (K + 3) / 4 * 4, np = (N + 3) / 4 * 4;  // padded row lengths (floats)
  // K chunks (16-aligned boundaries kb[0] = 0 < ... < kb[chunks] = K) and row
  // panels of the last chunk.  The chunks grow, K/8, 3K/8, K/2: the first copy
  // is all the GEMM waits for, and each chunk's GEMM outlasts the next chunk's
  // copy (at 4096^3, 2.49 ms a call against 2.63 with four equal chunks)
  int kb[4] = {0, c.K, c.K, c.K};
  int chunks = 1;
  if (gemm && c.K >= 2048) {
    kb[1] = c.K / 8 / 16 * 16, kb[2] = c.K / 2 / 16 * 16, kb[3] = c.K;
    chunks = 3;
  }
  // Row panels of the last chunk, rows pb[i] .. pb[i+1]-1: about 1024 rows
  // each (at 4096 columns, 512 tiles: one round of the persistent grid plus a
  // split tail).  With K chunks (all of A and C already copied in), the last
  // panel is cut into 3/4 and 1/4 (multiples of 128 rows) so that the return
  // left exposed after the last GEMM is a quarter as long; each earlier
  // panel's return hides behind the next panel's GEMM.  With one chunk each
  // panel first brings its own rows of A and C in.
  int pb[kHostPanelsMax + 1];
  int panels = 0;
  pb[0] = 0;
  {
    int n = c.M / 1024;  // at most kHostPanelsMax - 1, leaving room for the cut
    n = n < 1 ? 1 : n > kHostPanelsMax - 1 ? kHostPanelsMax - 1 : n;
    const int rows = ((c.M + n - 1) / n + 127) / 128 * 128;
    for (int r = rows; r < c.M; r += rows) pb[++panels] = r;
    const int base = pb[panels], last = c.M - base;
    if (chunks > 1 && last >= 512) {
      const int cut = base + (last * 3 / 4 + 127) / 128 * 128;
      if (cut < c.M) pb[++panels] = cut;
    }
    pb[++panels] = c.M;
  }
  const bool separate_c = chunks > 1 && read_c;  // C kept apart, added at the end

  const size_t a_bytes = gemm ? round256(M * kp * 4) : 0;
  const size_t b_bytes = gemm ? round256(K * np * 4) : 0;
  const size_t d_bytes = round256(M * np * 4);
  const size_t p_bytes = chunks > 1 ? 2 * d_bytes : 0;  // P0, P1: the first chunks' products
  const size_t need = a_bytes + b_bytes + d_bytes + p_bytes + (separate_c ? d_bytes : 0);

  HostPath& h = g_hostpath[dev];
  std::lock_guard<std::mutex> lk(h.mu);
  rc = hostpath_init(h);
  if (rc) return rc;
  // this call's copies start after the caller's earlier work and after the
  // previous host-operand call (whatever its stream) has finished with the buffer
  if (cudaEventRecord(h.start, st) != cudaSuccess) return B2G_ERR_CUDA;
  if (cudaStreamWaitEvent(h.h2d, h.start, 0) != cudaSuccess) return B2G_ERR_CUDA;
  if (h.used && cudaStreamWaitEvent(h.h2d, h.done, 0) != cudaSuccess) return B2G_ERR_CUDA;
  if (h.bytes < need) {
    if (h.buf) {
      if (h.used && cudaStreamWaitEvent(st, h.done, 0) != cudaSuccess) return B2G_ERR_CUDA;
      cudaFreeAsync(h.buf, st);
      h.buf = nullptr, h.bytes = 0;
    }
    if (cudaMallocAsync(&h.buf, need, st) != cudaSuccess) return B2G_ERR_CUDA;
    h.bytes = need;
    if (cudaEventRecord(h.start, st) != cudaSuccess) return B2G_ERR_CUDA;
    if (cudaStreamWaitEvent(h.h2d, h.start, 0) != cudaSuccess) return B2G_ERR_CUDA;
  }
  char* base = static_cast<char*>(h.buf);
  float* dA = reinterpret_cast<float*>(base);
  float* dB = reinterpret_cast<float*>(base + a_bytes);
  float* dD = reinterpret_cast<float*>(base + a_bytes + b_bytes);
  float* dP0 = reinterpret_cast<float*>(base + a_bytes + b_bytes + d_bytes);
  float* dP1 = reinterpret_cast<float*>(base + a_bytes + b_bytes + 2 * d_bytes);
  float* dC = separate_c ? reinterpret_cast<float*>(base + a_bytes + b_bytes + d_bytes + p_bytes)
                         : dD;

  auto ok = [](cudaError_t e) { return e == cudaSuccess ? 0 : B2G_ERR_CUDA; };
  const int lda_d = (int)(kp > 0 ? kp : 1);
  // copy stream: chunks of B's rows and A's columns, then C
  if (chunks > 1) {
    for (int j = 0; j < chunks && !rc; ++j) {
      const int k0 = kb[j], k1 = kb[j + 1];
      rc = ok(cudaMemcpy2DAsync(dB + (size_t)k0 * np, np * 4, c.B + (size_t)k0 * c.ldb,
                                (size_t)c.ldb * 4, N * 4, (size_t)(k1 - k0),
                                cudaMemcpyHostToDevice, h.h2d));
      if (!rc)
        rc = ok(cudaMemcpy2DAsync(dA + k0, kp * 4, c.A + k0, (size_t)c.lda * 4,
                                  (size_t)(k1 - k0) * 4, M, cudaMemcpyHostToDevice, h.h2d));
      if (!rc) rc = ok(cudaEventRecord(h.chunk[j], h.h2d));
    }
    if (!rc && separate_c) {
      rc = ok(cudaMemcpy2DAsync(dC, np * 4, c.C, (size_t)c.ldc * 4, N * 4, M,
                                cudaMemcpyHostToDevice, h.h2d));
      if (!rc) rc = ok(cudaEventRecord(h.c_in, h.h2d));
    }
    // all chunks but the last, over all rows, each into its own product
    for (int j = 0; j + 1 < chunks && !rc; ++j) {
      const int k0 = kb[j], k1 = kb[j + 1];
      rc = ok(cudaStreamWaitEvent(st, h.chunk[j], 0));
      if (!rc) {
        Call pc{0, 0, c.M, c.N, k1 - k0, c.alpha, 0.f, dA + k0, lda_d,
                dB + (size_t)k0 * np, (int)np, j == 0 ? dP0 : dP1, (int)np};
        rc = run(pc, -1, st);
      }
    }
    if (!rc) rc = ok(cudaStreamWaitEvent(st, h.chunk[chunks - 1], 0));
    if (!rc && separate_c) rc = ok(cudaStreamWaitEvent(st, h.c_in, 0));
  } else if (gemm) {
    rc = ok(cudaMemcpy2DAsync(dB, np * 4, c.B, (size_t)c.ldb * 4, N * 4, K,
                              cudaMemcpyHostToDevice, h.h2d));
    if (!rc) rc = ok(cudaEventRecord(h.chunk[0], h.h2d));
    if (!rc) rc = ok(cudaStreamWaitEvent(st, h.chunk[0], 0));
  }
  // the last chunk (or the only one), panel by panel, then back to the host
  const int kl0 = kb[chunks - 1];
  for (int i = 0; i < panels && !rc; ++i) {
    const size_t r0 = (size_t)pb[i];
    const size_t rn = (size_t)(pb[i + 1] - pb[i]);
    if (chunks == 1) {  // A's and C's rows of this panel come now
      if (gemm)
        rc = ok(cudaMemcpy2DAsync(dA + r0 * kp, kp * 4, c.A + r0 * c.lda, (size_t)c.lda * 4,
                                  K * 4, rn, cudaMemcpyHostToDevice, h.h2d));
      if (!rc && read_c)
        rc = ok(cudaMemcpy2DAsync(dD + r0 * np, np * 4, c.C + r0 * c.ldc, (size_t)c.ldc * 4,
                                  N * 4, rn, cudaMemcpyHostToDevice, h.h2d));
      if (!rc) rc = ok(cudaEventRecord(h.panel_in[i], h.h2d));
      if (!rc) rc = ok(cudaStreamWaitEvent(st, h.panel_in[i], 0));
    }
    if (!rc) {
      const float beta = chunks == 1 ? c.beta : 0.f;
      Call pc{0, 0, (int)rn, c.N, c.K - kl0, c.alpha, beta, dA + r0 * kp + kl0, lda_d,
              dB + (size_t)kl0 * np, (int)np, dD + r0 * np, (int)np};
      rc = run(pc, -1, st);
    }
    if (!rc && chunks > 1) {  // D = (P0 + P1) + D + beta * C over the panel
      int n4 = (int)(np / 4), rn_i = (int)rn;
      const unsigned bx = (unsigned)((n4 + 255) / 256);
      unsigned by = (unsigned)rn;
      const unsigned cap = (unsigned)d->sms * 8 / bx;
      if (by > cap) by = cap > 0 ? cap : 1;
      long long ld = (long long)np;
      const float* p0 = dP0 + r0 * np;
      const float* p1 = dP1 + r0 * np;
      const float* x = separate_c ? dC + r0 * np : nullptr;
      float* y = dD + r0 * np;
      float beta = c.beta;
      void* args[] = {&rn_i, &n4, &ld, (void*)&p0, (void*)&p1, &beta, (void*)&x, &y};
      rc = ok(launch_pdl(reinterpret_cast<const void*>(&combine_rows_kernel), dim3(bx, by),
                         dim3(256), args, 0, st));
    }
    if (!rc) rc = ok(cudaEventRecord(h.gemm[i], st));
    if (!rc) rc = ok(cudaStreamWaitEvent(h.d2h, h.gemm[i], 0));
    if (!rc)
      rc = ok(cudaMemcpy2DAsync(c.C + r0 * c.ldc, (size_t)c.ldc * 4, dD + r0 * np, np * 4,
                                N * 4, rn, cudaMemcpyDeviceToHost, h.d2h));
  }
  // join: the caller's stream holds the whole call; later calls wait for it
  if (!rc) rc = ok(cudaEventRecord(h.c_out, h.d2h));
  if (!rc) rc = ok(cudaStreamWaitEvent(st, h.c_out, 0));
  if (!rc) rc = ok(cudaEventRecord(h.done, st));
  if (!rc) h.used = true;
  return rc;
}

// The 3xTF32 tensor-core path: split the operands into a workspace, then the
// tcgen05 kernel.  Row-major, no op() flags; A 16-byte aligned with lda and K
// multiples of 4 (B is read element by element by its split kernel).
size_t tf32x3_bytes(const Call& c) {
  return 2 * ((size_t)c.M * c.K + (size_t)c.N * c.K) * sizeof(float);
}

// variant: 0 one CTA per 128 x 128 tile, 1 a CTA pair per 256 x 128 tile,
// 2 a CTA pair per 256 x 256 tile.
// Measured on GB300 (TFLOP/s of FP32 results, variants 0 / 1 / 2): 1536^3
// 172.7 / 164.0 / 114.1, 2048^3 184.4 / 179.1 / 215.6, 3072^3 219.8 / 224.7 /
// 281.1, 4096^3 234.9 / 240.2 / 305.0, 8192^3 266.5 / 267.7 / 351.9: the
// 256 x 256 pair (twice the work per MMA instruction) from about 1800^3 up,
// one CTA per 128 x 128 tile below.
int tc_default_variant(const Call& c) {
  return ((double)c.M * c.N * c.K >= 6.0e9 && c.M >= 512 && c.N >= 512) ? 2 : 0;
}

int run_tf32x3(const Call& c, void* stream, int variant) {
  int rc = validate(c);
  if (rc) return rc;
  if (c.M == 0 || c.N == 0) return 0;
  DeviceState* d = nullptr;
  rc = device_state(&d);
  if (rc) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (!needs_gemm(c)) return launch_scale(c, *d, st);
  if (c.transA || c.transB || !aligned16(c.A) || c.lda % 4 || c.K % 4) return B2G_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return B2G_ERR_DEVICE;

  Tf32x3Params p;
  p.M = c.M, p.N = c.N, p.K = c.K;
  p.alpha = c.alpha, p.beta = c.beta;
  p.C = c.C, p.ldc = c.ldc;
  p.c_vec4 = aligned16(c.C) && c.ldc % 4 == 0;
  const int pn = variant == 2 ? 256 : 128;            // a pair's N
  const int bbox = variant >= 1 ? pn / 2 : kTcBN;     // a pair's CTA stages half of B's columns
  const int tile_m = variant >= 1 ? 2 * kTcBM : kTcBM;
  const int tile_n = variant >= 1 ? pn : kTcBN;
  p.tiles_m = (c.M + tile_m - 1) / tile_m;
  p.tiles_n = (c.N + tile_n - 1) / tile_n;
  p.group_m = 8;
  p.k_tiles = (c.K + kTcBK - 1) / kTcBK;
  p.wait_limit_ns = g_wait_limit_ns.load();
  p.debug_stop_ktile = g_debug_stop.load();
  p.status = d->status;
  p.work = nullptr, p.tail_first = 0, p.tail_splits = 1;
  // Split tail of the pair kernels: T tiles over G resident pairs, T = q*G + r;
  // the last r tiles in S = G / r k slices (at least 16 k tiles each).
  size_t tail_bytes = 0;
  if (variant >= 1) {
    const long long T = (long long)p.tiles_m * p.tiles_n;
    const long long G = tf32x3_pair_capacity(pn, d->sms);
    if (G > 0 && T % G) {
      const long long q = T / G, r = T - q * G;
      long long S = G / r;
      if (S > p.k_tiles / 16) S = p.k_tiles / 16;
      if (S >= 2) {
        p.tail_first = (int)(q * G), p.tail_splits = (int)S;
        tail_bytes = (size_t)r * S * (2 * kTcBM) * pn * sizeof(float);
      }
    }
  }
  const size_t split_bytes = (tf32x3_bytes(c) + 255) / 256 * 256;
  float* ws = static_cast<float*>(ws_acquire(dev, st, split_bytes + tail_bytes));
  if (!ws) return B2G_ERR_UNSUPPORTED;  // capturing, or the workspace cannot be had
  float* Ahi = ws;
  float* Alo = Ahi + (size_t)c.M * c.K;
  float* Bhi = Alo + (size_t)c.M * c.K;
  float* Blo = Bhi + (size_t)c.N * c.K;
  if (tail_bytes) p.work = ws + split_bytes / sizeof(float);
  cudaError_t e =
      launch_split_ab(c.A, c.M, c.K, c.lda, Ahi, Alo, c.B, c.N, c.ldb, Bhi, Blo, d->sms, st);
  CUtensorMap maps[4];
  if (e == cudaSuccess) {
    rc = encode_2d_sw128(&maps[0], Ahi, c.K, c.M, c.K, kTcBM);
    if (!rc) rc = encode_2d_sw128(&maps[1], Alo, c.K, c.M, c.K, kTcBM);
    if (!rc) rc = encode_2d_sw128(&maps[2], Bhi, c.K, c.N, c.K, bbox);
    if (!rc) rc = encode_2d_sw128(&maps[3], Blo, c.K, c.N, c.K, bbox);
  }
  if (e == cudaSuccess && !rc) {
    e = variant >= 1 ? launch_tf32x3_pair(p, maps, pn, d->sms, st)
                     : launch_tf32x3(p, maps, d->sms, st);
    if (e == cudaSuccess && p.tail_splits > 1) e = launch_tf32x3_tail_reduce(p, pn, st);
  }
  ws_release(dev, st);
  if (rc) return rc;
  return e == cudaSuccess ? 0 : B2G_ERR_LAUNCH;
}

}  // namespace

int sgemm_min_workspace_bytes(int M, int N, int K, float alpha, const float* A, int lda,
                              const float* B, int ldb, const float* C, int ldc, size_t* bytes) {
  if (!bytes) return B2G_ERR_NULL;
  Call c{0, 0, M, N, K, alpha, 0.f, A, lda, B, ldb, const_cast<float*>(C), ldc};
  const int rc = validate(c);
  if (rc) return rc;
  *bytes = 0;
  if (needs_gemm(c)) {
    const Plan* pl = plan_at(select_plan(c));
    if (pl) *bytes = plan_base_bytes(*pl, c);
  }
  return 0;
}

}  // namespace b2g

using namespace b2g;

extern "C" {

int b2g_sgemm(int M, int N, int K, float alpha, const float* A, int lda, const float* B, int ldb,
              float beta, float* C, int ldc, void* stream) {
  return run(Call{0, 0, M, N, K, alpha, beta, A, lda, B, ldb, C, ldc}, -1, stream);
}

int b2g_sgemm_ex(int transA, int transB, int M, int N, int K, float alpha, const float* A, int lda,
                 const float* B, int ldb, float beta, float* C, int ldc, void* stream) {
  return run(Call{transA != 0, transB != 0, M, N, K, alpha, beta, A, lda, B, ldb, C, ldc}, -1,
             stream);
}

// Column-major C = op(A) op(B) is row-major C^T = op(B)^T op(A)^T on the same
// memory: swap the operands, their op() flags and M with N.
int b2g_sgemm_colmajor(int transA, int transB, int M, int N, int K, float alpha, const float* A,
                       int lda, const float* B, int ldb, float beta, float* C, int ldc,
                       void* stream) {
  return run(Call{transB != 0, transA != 0, N, M, K, alpha, beta, B, ldb, A, lda, C, ldc}, -1,
             stream);
}

int b2g_sgemm_with_plan(int plan, int transA, int transB, int M, int N, int K, float alpha,
                        const float* A, int lda, const float* B, int ldb, float beta, float* C,
                        int ldc, void* stream) {
  if (plan < 0 || plan >= num_plans()) return B2G_ERR_INVALID_PLAN;
  return run(Call{transA != 0, transB != 0, M, N, K, alpha, beta, A, lda, B, ldb, C, ldc}, plan,
             stream);
}

int b2g_sgemm_strided_batched(int transA, int transB, int M, int N, int K, float alpha,
                              const float* A, int lda, long long strideA, const float* B, int ldb,
                              long long strideB, float beta, float* C, int ldc,
                              long long strideC, int batch, void* stream) {
  Call c{transA != 0, transB != 0, M, N, K, alpha, beta, A, lda, B, ldb, C, ldc};
  c.batch = batch, c.strideA = strideA, c.strideB = strideB, c.strideC = strideC;
  return run(c, -1, stream);
}

int b2g_sgemm_3xtf32(int M, int N, int K, float alpha, const float* A, int lda, const float* B,
                     int ldb, float beta, float* C, int ldc, void* stream) {
  const Call c{0, 0, M, N, K, alpha, beta, A, lda, B, ldb, C, ldc};
  return run_tf32x3(c, stream, tc_default_variant(c));
}

int b2g_sgemm_3xtf32_variant(int variant, int M, int N, int K, float alpha, const float* A,
                             int lda, const float* B, int ldb, float beta, float* C, int ldc,
                             void* stream) {
  if (variant < 0 || variant > 2) return B2G_ERR_INVALID_PLAN;
  return run_tf32x3(Call{0, 0, M, N, K, alpha, beta, A, lda, B, ldb, C, ldc}, stream, variant);
}

int b2g_sgemm_ws(int transA, int transB, int M, int N, int K, float alpha, const float* A, int lda,
                 const float* B, int ldb, float beta, float* C, int ldc, void* workspace,
                 size_t workspace_bytes, void* stream) {
  return run(Call{transA != 0, transB != 0, M, N, K, alpha, beta, A, lda, B, ldb, C, ldc}, -1,
             stream, workspace, workspace_bytes, false);
}

int b2g_sgemm_workspace_size(int transA, int transB, int M, int N, int K, float alpha,
                             const float* A, int lda, const float* B, int ldb, const float* C,
                             int ldc, size_t* bytes) {
  if (!bytes) return B2G_ERR_NULL;
  Call c{transA != 0, transB != 0, M, N, K, alpha, 0.f, A, lda, B, ldb, const_cast<float*>(C), ldc};
  const int rc = validate(c);
  if (rc) return rc;
  *bytes = 0;
  if (needs_gemm(c)) {
    const Plan* pl = plan_at(select_plan(c));
    if (pl) *bytes = plan_work_bytes(*pl, c);
  }
  return 0;
}

int b2g_sgemm_launch_count(int transA, int transB, int M, int N, int K, float alpha,
                           const float* A, int lda, const float* B, int ldb, const float* C,
                           int ldc, int* launches) {
  if (!launches) return B2G_ERR_NULL;
  Call c{transA != 0, transB != 0, M, N, K, alpha, 0.f, A, lda, B, ldb, const_cast<float*>(C), ldc};
  const int rc = validate(c);
  if (rc) return rc;
  *launches = 0;
  if (M == 0 || N == 0) return 0;
  if (!needs_gemm(c)) {
    *launches = 1;  // C = beta * C
    return 0;
  }
  const Plan* pl = plan_at(select_plan(c));
  if (!pl) return B2G_ERR_INVALID_PLAN;
  // a transpose, or one launch packing both operands, or a transpose per operand
  int n = 1 + (pl->pretranspose == 3 ? (c.transA ? 1 : 2) : pl->pretranspose ? 1 : 0);
  if (pl->feed == kFeedSkinny) {
    int kc = 0;
    if (skinny_splits(*pl, c, &kc) > 1) n += 1;  // the split-K reduction
  } else if (pl->feed == kFeedSkinnyTMA || pl->cluster_max) {
    // the split-K sums are added inside the kernel's clusters
  } else {
    int first = 0;
    if (tail_split(*pl, c, &first) > 1) n += 1;  // the split tail's reduction
  }
  *launches = n;
  return 0;
}

int b2g_sgemm_host(int M, int N, int K, float alpha, const float* A, int lda, const float* B,
                   int ldb, float beta, float* C, int ldc, void* stream) {
  return run_host(Call{0, 0, M, N, K, alpha, beta, A, lda, B, ldb, C, ldc}, stream);
}

int b2g_release_workspaces(void) {
  int rc = 0;
  for (int dev = 0; dev < kMaxDevices; ++dev) {
    AutoWorkspace& w = g_ws[dev];
    std::lock_guard<std::mutex> lk(w.mu);
    if (!w.ptr) continue;
    int cur = 0;
    cudaGetDevice(&cur);
    if (cudaSetDevice(dev) != cudaSuccess) {
      rc = B2G_ERR_CUDA;
      continue;
    }
    if (w.done) cudaEventSynchronize(w.done);
    if (cudaFree(w.ptr) != cudaSuccess) rc = B2G_ERR_CUDA;
    w.ptr = nullptr;
    w.bytes = 0;
    cudaSetDevice(cur);
  }
  for (int dev = 0; dev < kMaxDevices; ++dev) {  // the host-operand staging buffers
    HostPath& h = g_hostpath[dev];
    std::lock_guard<std::mutex> lk(h.mu);
    if (!h.buf) continue;
    int cur = 0;
    cudaGetDevice(&cur);
    if (cudaSetDevice(dev) != cudaSuccess) {
      rc = B2G_ERR_CUDA;
      continue;
    }
    if (h.used) cudaEventSynchronize(h.done);
    if (cudaFree(h.buf) != cudaSuccess) rc = B2G_ERR_CUDA;
    h.buf = nullptr;
    h.bytes = 0;
    cudaSetDevice(cur);
  }
  return rc;
}

int b2g_sgemm_select_plan(int transA, int transB, int M, int N, int K, float alpha, const float* A,
                          int lda, const float* B, int ldb, const float* C, int ldc) {
  Call c{transA != 0, transB != 0, M, N, K, alpha, 0.f, A, lda, B, ldb, const_cast<float*>(C), ldc};
  const int rc = validate(c);
  if (rc) return rc;
  if (!needs_gemm(c)) return num_plans();
  return select_plan(c);
}

int b2g_plan_count(void) { return num_plans(); }

const char* b2g_plan_name(int plan) {
  const Plan* p = plan_at(plan);
  return p ? p->name : nullptr;
}

int b2g_plan_info(int plan, int* info) {
  const Plan* p = plan_at(plan);
  if (!p) return B2G_ERR_INVALID_PLAN;
  if (!info) return B2G_ERR_NULL;
  const int v[9] = {p->BM, p->BN, p->BK, p->stages, p->TN, p->alayout, p->feed, p->threads,
                    p->smem_bytes};
  for (int i = 0; i < 9; ++i) info[i] = v[i];
  return 0;
}

int b2g_status(void* stream, unsigned int* flags, int clear) {
  if (!flags) return B2G_ERR_NULL;
  DeviceState* d = nullptr;
  const int rc = device_state(&d);
  if (rc) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  unsigned int v = 0;
  if (cudaMemcpyAsync(&v, d->status, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return B2G_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return B2G_ERR_CUDA;
  if (clear && v) {
    if (cudaMemsetAsync(d->status, 0, sizeof(unsigned int), st) != cudaSuccess) return B2G_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return B2G_ERR_CUDA;
  }
  *flags = v;
  return v ? B2G_ERR_TIMEOUT : 0;
}

int b2g_sgemm_debug_status(void* stream) {
  unsigned int flags = 0;
  const int rc = b2g_status(stream, &flags, 0);
  if (rc && rc != B2G_ERR_TIMEOUT) return rc;
  return (int)(flags & 0x7fffffffu);
}

int b2g_set_wait_limit_ns(unsigned long long ns) {
  if (ns == 0) return B2G_ERR_INVALID_DIM;
  g_wait_limit_ns.store(ns);
  return 0;
}

int b2g_debug_stop_after(int n) {
  g_debug_stop.store(n < 0 ? -1 : n);
  return 0;
}

const char* b2g_strerror(int code) {
  switch (code) {
    case B2G_OK: return "ok";
    case B2G_ERR_INVALID_DIM: return "invalid dimension (M, N or K < 0)";
    case B2G_ERR_INVALID_LD: return "invalid leading dimension";
    case B2G_ERR_NULL: return "null pointer for an operand that must be read or written";
    case B2G_ERR_LAUNCH: return "kernel launch failed";
    case B2G_ERR_DEVICE: return "no usable sm_103 device is current";
    case B2G_ERR_UNSUPPORTED: return "the requested plan cannot take these operands";
    case B2G_ERR_INVALID_PLAN: return "plan index out of range";
    case B2G_ERR_TENSOR_MAP: return "bulk-tensor descriptor rejected by the driver";
    case B2G_ERR_CUDA: return "CUDA runtime call failed";
    case B2G_ERR_TIMEOUT: return "a kernel's bounded wait ran out (see b2g_status flags)";
    case B2G_ERR_SCRATCH_LIMIT:
      return "the call needs more scratch than b2g_sgemm_noalloc's fixed array holds";
    default: return "unknown error code";
  }
}

const char* b2g_version(void) { return "b2g_sgemm 0.1 (sm_103a)"; }

}  // extern "C"
