// sgemm_params.h -- what the host passes to every SGEMM kernel, and the plan
// descriptor the tune table is made of.  Shared by the C-ABI layer and the
// kernel translation units; holds no arithmetic.  The list of compiled plan
// tables and the host-side launchers live in plan_registry.h.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

namespace b2g {

struct SgemmParams {
  int M, N, K;
  float alpha, beta;
  const float* A;
  long long lda;
  const float* B;
  long long ldb;
  float* C;
  long long ldc;
  int transA;   // A stored K x M (op(A) = A^T); general feed only
  int transB;   // B stored N x K (op(B) = B^T); general feed only
  int c_vec4;   // C 16-byte aligned and ldc % 4 == 0: float4 epilogue allowed
  int tiles_m, tiles_n, group_m, k_tiles;
  unsigned long long wait_limit_ns;  // bound on every mbarrier wait
  int debug_stop_ktile;              // < 0 normally; >= 0 stops the producer (timeout test)
  unsigned int* status;              // device status word (timeout flags)
  int batch;                         // independent problems (strided batched); 1 otherwise
  long long strideA, strideB, strideC;  // elements between consecutive problems
  float* work;                       // partial sums (skinny split-K, FFMA split tail), or null
  int splits;                        // split-K factor (skinny plans); 1 = no split
  int kc;                            // k extent of one split (skinny plans)
  // FFMA plans' split tail: output tiles tail_first .. tiles-1 are each cut
  // into tail_splits k slices (tail_splits == 1: none).  A slice writes its raw
  // BM x BN sums to work + (slice unit index) * BM * BN; launch_tail_reduce
  // then adds each tile's slices in order and applies the epilogue.
  int tail_first;
  int tail_splits;
  // 1 when the grid leaves resident CTA slots free: the kernel then does not
  // let the next grid launch early, since an early grid's CTAs would be placed
  // into those free slots unevenly (some SMs three, others none); they are
  // placed once this grid's CTAs exit.  Set by the launcher.
  int pdl_late;
};

// How A is laid out in one shared-memory stage.
enum ALayout : int {
  kAKChunk = 0,  // [BK/4][BM][4]: a row's 4 consecutive k in one 16-byte vector
  kAKMajor = 1,  // [BK][BM]: transposed, a column's m values contiguous
};

// How stages are filled.
enum Feed : int {
  kFeedTMA = 0,      // one elected thread issues bulk-tensor copies (aligned operands)
  kFeedCpAsync = 1,  // producer warps issue 4-byte cp.async with zero fill (any layout)
  kFeedTMATrans = 2,  // bulk-tensor copies; A lands k-chunked in a staging slot and the
                      // consumer warps rewrite it transposed ([BK][BM]) a few stages ahead
  kFeedSkinny = 3,    // skinny-M split-K kernel: B streamed from global, A staged per k slab
  kFeedSkinnyTMA = 4,  // skinny-M split-K kernel: B and A in bulk-tensor stages
};

constexpr int kMaxDevices = 64;

// Launch one plan's kernel on `stream` with a persistent grid of at most
// num_sms x (CTAs resident per SM) CTAs.  Returns the launch's CUDA error.
using LaunchFn = cudaError_t (*)(const SgemmParams& p, const CUtensorMap* tmA,
                                 const CUtensorMap* tmB, int num_sms, cudaStream_t stream);

struct Plan {
  const char* name;
  int BM, BN, BK, stages, TN;
  int alayout;  // ALayout
  int feed;     // Feed
  int threads;  // CTA size (consumer warps + producer warps)
  int smem_bytes;
  LaunchFn launch;
  int pretranspose;  // 1: row-major A is first transposed into a workspace, then this
                     // plan's kernel (which reads A stored K x M) runs on it; 2: both
                     // operands are packed into a workspace first (A^T and B, aligned,
                     // from any alignment, leading dimension or op() flags); 3: B stored
                     // N x K (op(B) = B^T) is transposed into the workspace, and A too
                     // unless it comes stored K x M (aligned operands, 16-byte vectors)
  int (*occupancy)();  // CTAs of this plan resident per SM on the current device (0 on
                       // failure); the host sizes split-K and split tails by it
  int cluster_max = 0;  // > 0: cluster-split kernel, one CTA per (tile, k slice), at most
                        // this many k slices of a tile summed inside one cluster
};

}  // namespace b2g
