/*
 * b2g_sgemm.h -- C ABI of the GB300 (sm_103a) FP32 SGEMM library.
 *
 * The operation (GEMM 优化之路 / CUDA 进阶手册, section 问题定义与性能上限):
 *
 *     C = alpha * op(A) * op(B) + beta * C
 *
 * with op(A) an M x K matrix, op(B) K x N and C M x N, all FP32 and ROW-MAJOR:
 * element (i, k) of a stored matrix X with leading dimension ldX sits at
 * X[i * ldX + k].  op(X) is X, or X transposed when the trans flag is set (the
 * optimisation guide on gsyq.cn, section 6.4 step 8, lists A^T*B and A*B^T as
 * the cases a complete GEMM handles).  Every product and sum is an FP32
 * multiply-add (no reduced-precision arithmetic).
 *
 * Ownership and ordering
 *   - A, B and C are DEVICE pointers owned by the caller; the library never
 *     allocates, frees or keeps them.  C must not overlap A or B.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Calls are
 *     asynchronous: they enqueue work on `stream` and return; the result is
 *     ordered on that stream.  No call synchronises the host except
 *     b2g_status().
 *   - The calls are thread-safe.  Only sm_103 devices are supported.
 *
 * Return values: 0 on success, a negative B2G_ERR_* code otherwise.  Nothing is
 * printed, nothing throws, nothing exits.  b2g_strerror() names a code.
 */
#ifndef B2G_SGEMM_H
#define B2G_SGEMM_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

#define B2G_OK 0
#define B2G_ERR_INVALID_DIM (-1)  /* M, N or K < 0 */
#define B2G_ERR_INVALID_LD (-2)   /* a leading dimension smaller than its row width (min 1) */
#define B2G_ERR_NULL (-3)         /* a pointer the call must dereference is NULL */
#define B2G_ERR_LAUNCH (-4)       /* the kernel launch failed (cudaLaunchKernel's error) */
#define B2G_ERR_DEVICE (-5)       /* no current device, or it is not sm_103 */
#define B2G_ERR_UNSUPPORTED (-6)  /* the forced plan cannot run these operands */
#define B2G_ERR_INVALID_PLAN (-7) /* plan index out of range */
#define B2G_ERR_TENSOR_MAP (-8)   /* the driver refused a bulk-tensor descriptor */
#define B2G_ERR_CUDA (-9)         /* another CUDA runtime call failed */
#define B2G_ERR_TIMEOUT (-10)     /* b2g_status(): a kernel's bounded wait ran out */
#define B2G_ERR_SCRATCH_LIMIT (-11) /* b2g_sgemm_noalloc: more scratch than its fixed array */

/*
 * Row-major SGEMM, C = alpha*A*B + beta*C.
 *   M, N, K  >= 0.  M == 0 or N == 0: nothing is launched, returns 0.
 *   A        device, M x K, lda >= max(1, K).  Not read when K == 0 or alpha == 0.
 *   B        device, K x N, ldb >= max(1, N).  Not read when K == 0 or alpha == 0.
 *   C        device, M x N, ldc >= max(1, N).  Read only when beta != 0 (beta == 0
 *            makes C write-only, so NaN/Inf already in C do not propagate).
 *   stream   cudaStream_t or NULL.
 * Any alignment and any leading dimension are accepted; 16-byte aligned
 * operands with lda, ldb, ldc and K multiples of 4 take the bulk-tensor fed
 * kernels, everything else the 4-byte-fed kernel.  The plan comes from the
 * library's shape-keyed tune table.
 *
 * Workspace: for large aligned problems the fastest plan first writes A^T
 * (K x round_up(M, 4) floats) into a workspace.  This entry point uses a
 * library-owned workspace, one per device, allocated stream-ordered
 * (cudaMallocAsync) the first time a call needs it and grown when a later call
 * needs more; calls on different streams that share it are ordered by an event
 * the library records after each use.  While `stream` is being captured into a
 * CUDA graph, or when the allocation fails, the call takes a plan that needs no
 * workspace instead.  b2g_sgemm_ws lets the caller supply the workspace and
 * never allocates; b2g_release_workspaces frees the library-owned ones.
 *
 * Split tail: a persistent grid of G CTAs over T output tiles, T = q*G + r
 * with 0 < r < G, would keep only r CTAs busy in its last round.  The last r
 * tiles are then cut into S = G / r k slices (at least 64 k each) whose
 * partial sums go to the workspace, after A^T, and a second kernel adds each
 * tile's slices in slice order and applies the epilogue.  The summation order
 * is fixed for given arguments, so results stay reproducible run to run; the
 * result bound is unchanged.  Without a workspace the tiles run whole.
 */
int b2g_sgemm(int M, int N, int K, float alpha, const float* A, int lda, const float* B, int ldb,
              float beta, float* C, int ldc, void* stream);

/*
 * As b2g_sgemm with op() flags.  transA != 0: A is stored K x M (lda >= max(1, M))
 * and op(A) = A^T.  transB != 0: B is stored N x K (ldb >= max(1, K)) and
 * op(B) = B^T.  C is always M x N row-major.
 */
int b2g_sgemm_ex(int transA, int transB, int M, int N, int K, float alpha, const float* A, int lda,
                 const float* B, int ldb, float beta, float* C, int ldc, void* stream);

/*
 * The same product for COLUMN-major operands, with BLAS's argument
 * conventions: C is M x N column-major (element (i, j) at C[i + j*ldc],
 * ldc >= max(1, M)); transA == 0: A is M x K column-major, lda >= max(1, M);
 * transA != 0: A is stored K x M column-major (lda >= max(1, K)) and
 * op(A) = A^T; likewise B (K x N, ldb >= max(1, K); or stored N x K,
 * ldb >= max(1, N), when transB != 0).
 *
 * A column-major matrix is the row-major transpose of the same memory, and
 * C = op(A) op(B) holds exactly when C^T = op(B)^T op(A)^T ("GEMM 优化之路",
 * 完整代码: the identity by which the page drives column-major cuBLAS with
 * row-major data).  So this call is b2g_sgemm_ex(transB, transA, N, M, K,
 * alpha, B, ldb, A, lda, beta, C, ldc, stream): the same plans, kernels,
 * workspace behaviour and error bound, with the roles of the two operands
 * swapped.  Error codes as b2g_sgemm_ex (a leading dimension below the bounds
 * above is B2G_ERR_INVALID_LD).
 */
int b2g_sgemm_colmajor(int transA, int transB, int M, int N, int K, float alpha, const float* A,
                       int lda, const float* B, int ldb, float beta, float* C, int ldc,
                       void* stream);

/*
 * `batch` independent products C_b = alpha * op(A_b) * op(B_b) + beta * C_b,
 * b = 0 .. batch-1, with A_b = A + b*strideA, B_b = B + b*strideB and
 * C_b = C + b*strideC (strides in elements, >= 0; C_b must not overlap each
 * other).  Same layout rules, plans and workspace behaviour as b2g_sgemm_ex
 * (workspace scaled by batch); one launch covers the whole batch (the batch
 * index is the outermost coordinate of the tile scheduler).  batch == 0 does
 * nothing; batch < 0 is B2G_ERR_INVALID_DIM, a negative stride
 * B2G_ERR_INVALID_LD.  Batched GEMM is not on the pages; it shares their kernel.
 */
int b2g_sgemm_strided_batched(int transA, int transB, int M, int N, int K, float alpha,
                              const float* A, int lda, long long strideA, const float* B, int ldb,
                              long long strideB, float beta, float* C, int ldc,
                              long long strideC, int batch, void* stream);

/*
 * As b2g_sgemm_ex with a caller-owned device workspace of workspace_bytes
 * (16-byte aligned).  Never allocates.  With at least what
 * b2g_sgemm_workspace_size reports, the tune table's plan runs with its split
 * tail; with less, but room for A^T (K x round_up(M, 4) floats) when the plan
 * transposes A first, it runs without the split tail; with less than that, or
 * a NULL workspace, a plan that needs none runs instead (slower, same result
 * bound).  The caller orders reuse of the workspace across streams.
 */
int b2g_sgemm_ws(int transA, int transB, int M, int N, int K, float alpha, const float* A, int lda,
                 const float* B, int ldb, float beta, float* C, int ldc, void* workspace,
                 size_t workspace_bytes, void* stream);

/*
 * b2g_sgemm on HOST operands: A, B and C are host pointers (same row-major
 * layout and leading-dimension rules as b2g_sgemm; page-locked memory from
 * cudaHostAlloc / cudaHostRegister gives full copy speed, pageable memory
 * works more slowly).  The copies overlap the multiplication: for K >= 2048
 * the library copies A's columns and B's rows in three growing K chunks
 * (K/8, 3K/8, K/2) and then C on its own copy stream, while `stream`
 * multiplies each chunk, as soon as it has arrived, into a device product of
 * its own; the last chunk runs in row panels of about 1024 rows (multiples of
 * 128 rows, at most 16 panels), the last panel cut into 3/4 and 1/4 when it
 * has 512 rows or more; each finished panel is added up, (P0 + P1) + P2 +
 * beta * C, and goes back to the host on a second copy stream while the next
 * one multiplies, so that only the last, short return is exposed.  For
 * K < 2048 it copies B, then A and C in the same row panels (no cut), and
 * multiplies each panel as it arrives.  Every step is ordered after earlier
 * work on `stream`, and the call's last copy is joined back into `stream`.
 * Sums split over K chunks are rounded once per chunk, within the same error
 * bound.  C holds the result once `stream` has completed the call's work (for
 * instance after cudaStreamSynchronize(stream)); until then the host buffers
 * must stay valid and unmodified.  Device staging (A, B and C with rows padded
 * to a multiple of 4 floats, and for K >= 2048 two more M x N products) is a
 * library-owned buffer per device, grown when needed and
 * freed by b2g_release_workspaces; calls on different streams are ordered one
 * after the other.  Same return codes as b2g_sgemm, plus B2G_ERR_UNSUPPORTED
 * while `stream` is being captured into a graph and B2G_ERR_CUDA when a copy
 * or the allocation fails.  Not on the pages: it serves callers whose data
 * live in host memory.
 */
int b2g_sgemm_host(int M, int N, int K, float alpha, const float* A, int lda, const float* B,
                   int ldb, float beta, float* C, int ldc, void* stream);

/*
 * Workspace bytes the tune table's plan wants for these arguments (0 when it
 * needs none), stored in *bytes: A^T or the packed operands when the plan
 * writes them, then (256-byte aligned) the split tail's partial sums, one
 * BM x BN block of floats per k slice of every split tile (at most 16 slices
 * a tile; 224 tiles x 2 slices at 4096^3, 338 x 4 at 1664^3).  The split
 * depends on the current device's SM count and occupancy.  Returns 0, a B2G_ERR_* code for invalid
 * arguments, or B2G_ERR_NULL when bytes is NULL.  Launches nothing.
 */
int b2g_sgemm_workspace_size(int transA, int transB, int M, int N, int K, float alpha,
                             const float* A, int lda, const float* B, int ldb, const float* C,
                             int ldc, size_t* bytes);

/*
 * Number of kernel launches that one b2g_sgemm_ex call with these arguments
 * makes when the workspace can be had, stored in *launches: 0 when M or N is
 * 0, 1 when only C is scaled, else the GEMM kernel plus the plan's prepasses
 * (1 transpose, or 1 launch packing both operands) plus 1 when a split-K or split-tail
 * reduction follows.  Depends on the current device like the split itself.
 * Returns 0, a B2G_ERR_* code for invalid arguments, or B2G_ERR_NULL when
 * launches is NULL.  Launches nothing.
 */
int b2g_sgemm_launch_count(int transA, int transB, int M, int N, int K, float alpha,
                           const float* A, int lda, const float* B, int ldb, const float* C,
                           int ldc, int* launches);

/*
 * Free the library-owned workspaces (and the staging buffers of
 * b2g_sgemm_host) of all devices, after waiting for the work that used them.  Later calls allocate again when needed.  Returns 0 or
 * B2G_ERR_CUDA.
 */
int b2g_release_workspaces(void);

/*
 * Row-major SGEMM (same arguments and result bound as b2g_sgemm) for callers
 * that must not have the library allocate device memory -- for instance an
 * application whose allocator reserved device memory at start-up and forbids
 * later cudaMalloc / cudaMallocAsync calls.  It never allocates: its scratch
 * (A^T for the plans that transpose A first, then the split tail's partial
 * sums when they fit) is a fixed 64 MiB array that every device loading the
 * library holds until the process exits.
 *   - A call is rejected with B2G_ERR_SCRATCH_LIMIT, launching nothing, when
 *     the scratch its tune-table plan cannot do without exceeds 64 MiB
 *     (16,777,216 floats).  That scratch is: A^T, K x round_up(M, 4) floats,
 *     for the plans that transpose A first (aligned operands, M*N*K >= 1e9);
 *     A^T plus an aligned copy of B, K x (round_up(M, 4) + round_up(N, 4))
 *     floats, for the packing plans (a misaligned pointer, lda or ldb not a
 *     multiple of 4, or K % 4 != 0, with M*N*K >= 5e7); the k slabs' partial
 *     sums, S x M x N floats with S <= K / 64, for the skinny split-K plans
 *     with M <= 32 and N < 2048 (at most about 20 MB on a 152-SM GPU);
 *     nothing otherwise.  The split tail's partial
 *     sums are optional: they use the room left, else the plan runs without
 *     its split.  Use b2g_sgemm_ws with your own buffer for rejected calls.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before capturing any stream.
 *   - The array is shared by every call on a device and keeps the last call's
 *     contents; each call rewrites all of the scratch it reads, so nothing
 *     needs clearing, but calls that overlap on the GPU (different streams with
 *     no ordering between them) race on it.
 * No counterpart on the pages: it serves callers, not the method.
 */
int b2g_sgemm_noalloc(int M, int N, int K, float alpha, const float* A, int lda, const float* B,
                      int ldb, float beta, float* C, int ldc, void* stream);

/*
 * As b2g_sgemm_ex, but run plan `plan` (0 <= plan < b2g_plan_count()) instead of
 * the tune table's choice.  Returns B2G_ERR_UNSUPPORTED when that plan cannot
 * take these operands (alignment, op() flags) or needs a workspace that cannot
 * be had (it uses the library-owned one).  For tests and tuning sweeps.
 */
int b2g_sgemm_with_plan(int plan, int transA, int transB, int M, int N, int K, float alpha,
                        const float* A, int lda, const float* B, int ldb, float beta, float* C,
                        int ldc, void* stream);

/*
 * The plan index the tune table picks for these arguments (nothing is
 * launched), or a negative B2G_ERR_* code for invalid arguments.  Calls that
 * need no GEMM kernel (K == 0 or alpha == 0: C = beta*C only; M == 0 or N == 0:
 * nothing) return b2g_plan_count(), one past the last plan.
 */
int b2g_sgemm_select_plan(int transA, int transB, int M, int N, int K, float alpha, const float* A,
                          int lda, const float* B, int ldb, const float* C, int ldc);

/* Number of GEMM plans compiled into the library. */
int b2g_plan_count(void);

/* Name of plan `plan` ("tma_128x128x16_s6", ...), or NULL when out of range. */
const char* b2g_plan_name(int plan);

/*
 * Plan parameters written to info[0..8]: BM, BN, BK, stages, TN (per-thread
 * columns; rows are 8), A layout (0 = k-chunked, 1 = transposed), feed
 * (0 = bulk-tensor, 1 = 4-byte cp.async), threads per CTA, dynamic shared bytes.
 * Returns 0 or B2G_ERR_INVALID_PLAN / B2G_ERR_NULL.
 */
int b2g_plan_info(int plan, int* info);

/*
 * Read the device status word that kernels set when a bounded wait runs out.
 * Synchronises `stream`, then stores the flags in *flags (0 = none; bit 0 a
 * consumer timed out waiting for data, bit 1 a producer timed out waiting for
 * a free stage, bit 2 a producer timed out waiting for its own copies, bit 3
 * the tensor-core path timed out waiting for its MMAs).  clear != 0 resets the
 * word.  Returns 0, B2G_ERR_TIMEOUT when a flag is set, or B2G_ERR_CUDA.
 */
int b2g_status(void* stream, unsigned int* flags, int clear);

/*
 * The same status word as a return value, without clearing it: synchronises
 * `stream`, then returns the flags (0 when no bounded wait has run out since
 * the word was last cleared, else the bit set described at b2g_status), or a
 * negative B2G_ERR_* code when the current device is unusable or the word
 * cannot be read.  Exported in every build (the word is only written when a
 * wait gives up, so reading it costs the normal path nothing).  After a
 * reported timeout the C of the call that timed out is undefined: tiles whose
 * consumers gave up were not written, and a split tail may have added partial
 * sums that were never finished.
 */
int b2g_sgemm_debug_status(void* stream);

/*
 * Upper bound, in nanoseconds of GPU wall time, on every mbarrier wait inside
 * the kernels (default 2e9 = 2 s).  A wait that runs past it sets a status flag
 * and its kernel returns early instead of hanging.  Returns 0, or
 * B2G_ERR_INVALID_DIM for 0.
 */
int b2g_set_wait_limit_ns(unsigned long long ns);

/*
 * Failure-injection hook for tests of the bounded waits: with n >= 0 the
 * producer of every subsequently launched GEMM kernel stops after issuing n
 * stages, so the consumers' waits run out; n < 0 (the default) turns it off.
 * Only meaningful on tiny problems with a short wait limit.  Returns 0.
 */
int b2g_debug_stop_after(int n);

/*
 * Row-major SGEMM on the 5th-generation tensor cores with the 3xTF32 split --
 * a separate path from the FFMA entry points above, reported apart.  TF32 keeps
 * a 10-bit mantissa (the handbook, section 接下来的优化方向, 使用 Tensor Core);
 * each operand x is split into hi = x rounded to TF32 and lo = x - hi (exact in
 * FP32), and alpha*(A_lo*B_hi + A_hi*B_lo + A_hi*B_hi) + beta*C is accumulated
 * in FP32 (tcgen05.mma kind::tf32, accumulator in tensor memory).  The dropped
 * A_lo*B_lo term and the rounding of lo are below 2^-21 |a||b| per product, so
 * results stay inside the same elementwise bound the FFMA path is tested
 * against for the shapes the tests cover.
 *   Same arguments as b2g_sgemm.  Requires A 16-byte aligned and lda, K
 *   multiples of 4 (else B2G_ERR_UNSUPPORTED); B and C may have any alignment.  Needs a workspace of
 *   2*(M*K + N*K) floats for the split operands, taken from the library-owned
 *   per-device workspace (see b2g_sgemm); while `stream` is being captured, or
 *   when that workspace cannot be had, it returns B2G_ERR_UNSUPPORTED.
 */
int b2g_sgemm_3xtf32(int M, int N, int K, float alpha, const float* A, int lda, const float* B,
                     int ldb, float beta, float* C, int ldc, void* stream);

/*
 * b2g_sgemm_3xtf32 with a chosen tensor-core kernel: variant 0 runs one CTA
 * per 128 x 128 output tile; variant 1 runs a CTA pair (a cluster of two CTAs
 * on two SMs) per 256 x 128 tile with tcgen05.mma.cta_group::2, each CTA
 * staging half of A's rows and half of B's columns; variant 2 is the CTA pair
 * on 256 x 256 tiles.  Same arguments, result
 * bound and errors as b2g_sgemm_3xtf32, which runs variant 2 from 6e9
 * multiply-adds (M*N*K) up with M and N at least 512, and variant 0 otherwise;
 * any other variant is B2G_ERR_INVALID_PLAN.  For tests and comparisons.
 */
int b2g_sgemm_3xtf32_variant(int variant, int M, int N, int K, float alpha, const float* A,
                             int lda, const float* B, int ldb, float beta, float* C, int ldc,
                             void* stream);

/* Static string for a B2G_* code. */
const char* b2g_strerror(int code);

/* Library version string. */
const char* b2g_version(void);

#ifdef __cplusplus
}
#endif

#endif /* B2G_SGEMM_H */
