// noalloc.cu -- b2g_sgemm_noalloc: the SGEMM for callers that must not have the
// library allocate device memory.
//
// Some applications reserve their device memory once at start-up (a framework's
// caching allocator, a serving process with a fixed memory budget, code that
// must not risk an allocation failing or synchronising the device halfway
// through a run) and forbid libraries to call cudaMalloc or cudaMallocAsync
// afterwards.  b2g_sgemm may allocate its workspace on first need and
// b2g_sgemm_ws needs the caller to find one; this entry point instead keeps its
// scratch in a fixed array that every GPU loading the library holds until the
// process exits, and allocates nothing itself.
//
// The scratch receives A^T (K x round_up(M, 4) floats) for the plans that
// transpose A first; the transpose writes every element the GEMM later reads
// (padding columns included), so nothing has to be cleared between calls.
// All calls share the one array per device: calls whose work overlaps on the
// GPU (different streams without ordering between them) race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/b2g_sgemm.h"
#include "plan_registry.h"
#include "sgemm_params.h"

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;  // 64 MiB per device

// The scratch itself.  In host code this name is only a stand-in for the
// device symbol; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) float g_noalloc_scratch[kScratchBytes / sizeof(float)];

std::mutex g_scratch_mu;
float* g_scratch_addr[b2g::kMaxDevices];  // device address of the array, per device

// Device address of the array on the current device (looked up on the first
// call there), or an error code.
int scratch_address(float** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= b2g::kMaxDevices)
    return B2G_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return B2G_ERR_CUDA;
    g_scratch_addr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_addr[dev];
  return 0;
}

}  // namespace

extern "C" int b2g_sgemm_noalloc(int M, int N, int K, float alpha, const float* A, int lda,
                                 const float* B, int ldb, float beta, float* C, int ldc,
                                 void* stream) {
  // `need` is what the plan cannot do without (A^T for the transposing plans);
  // `want` adds the split tail's partial sums, which take the array's
  // remaining room when they fit (the plan runs without the split otherwise).
  size_t need = 0, want = 0;
  int rc = b2g::sgemm_min_workspace_bytes(M, N, K, alpha, A, lda, B, ldb, C, ldc, &need);
  if (!rc) rc = b2g_sgemm_workspace_size(0, 0, M, N, K, alpha, A, lda, B, ldb, C, ldc, &want);
  if (rc) return rc;
  if (need > kScratchBytes) return B2G_ERR_SCRATCH_LIMIT;
  float* scratch = nullptr;
  size_t give = 0;
  if (want > 0) {
    rc = scratch_address(&scratch);
    if (rc) return rc;
    give = want < kScratchBytes ? want : kScratchBytes;
  }
  return b2g_sgemm_ws(0, 0, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, scratch, give, stream);
}
