"""Python binding of the GB300 FP32 SGEMM C ABI (include/b2g_sgemm.h).

Argument marshalling only: every step of the GEMM runs in the CUDA library
``libb2g_sgemm.so``; torch supplies device memory and the current stream.  The
library must be built first (``dense_fp32_gemm_07_gb300.build.build()``); there
is no fallback when it is missing.

Low-level names mirror the C ABI one to one (``b2g_sgemm``, ``b2g_sgemm_ex``,
``b2g_sgemm_with_plan``, ...) and take raw device pointers; ``sgemm`` is the
tensor-level convenience: ``C <- alpha * op(A) @ op(B) + beta * C`` in place;
``sgemm_colmajor`` is the same for column-major tensors.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libb2g_sgemm.so")

B2G_OK = 0
B2G_ERR_INVALID_DIM = -1
B2G_ERR_INVALID_LD = -2
B2G_ERR_NULL = -3
B2G_ERR_LAUNCH = -4
B2G_ERR_DEVICE = -5
B2G_ERR_UNSUPPORTED = -6
B2G_ERR_INVALID_PLAN = -7
B2G_ERR_TENSOR_MAP = -8
B2G_ERR_CUDA = -9
B2G_ERR_TIMEOUT = -10
B2G_ERR_SCRATCH_LIMIT = -11

# every symbol include/b2g_sgemm.h declares
EXPORTS = (
    "b2g_sgemm", "b2g_sgemm_ex", "b2g_sgemm_colmajor", "b2g_sgemm_with_plan",
    "b2g_sgemm_select_plan",
    "b2g_sgemm_ws", "b2g_sgemm_workspace_size", "b2g_sgemm_launch_count", "b2g_sgemm_host",
    "b2g_release_workspaces", "b2g_sgemm_noalloc",
    "b2g_sgemm_3xtf32", "b2g_sgemm_3xtf32_variant", "b2g_sgemm_strided_batched",
    "b2g_plan_count", "b2g_plan_name", "b2g_plan_info", "b2g_status", "b2g_sgemm_debug_status",
    "b2g_set_wait_limit_ns",
    "b2g_debug_stop_after", "b2g_strerror", "b2g_version",
)

_lock = threading.Lock()
_lib = None


class B2GError(RuntimeError):
    def __init__(self, code: int):
        self.code = code
        super().__init__(f"b2g error {code}: {b2g_strerror(code)}")


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built; run dense_fp32_gemm_07_gb300.build.build() "
                "(or __graft_entry__.build()) first")
        lib = ctypes.CDLL(LIB_PATH)
        i, f, vp, u64 = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_ulonglong
        gemm = [i, i, i, f, vp, i, vp, i, f, vp, i, vp]
        lib.b2g_sgemm.argtypes = gemm
        lib.b2g_sgemm_ex.argtypes = [i, i] + gemm
        lib.b2g_sgemm_colmajor.argtypes = [i, i] + gemm
        lib.b2g_sgemm_with_plan.argtypes = [i, i, i] + gemm
        lib.b2g_sgemm_select_plan.argtypes = [i, i, i, i, i, f, vp, i, vp, i, vp, i]
        lib.b2g_sgemm_ws.argtypes = [i, i, i, i, i, f, vp, i, vp, i, f, vp, i, vp, ctypes.c_size_t,
                                     vp]
        lib.b2g_sgemm_workspace_size.argtypes = [i, i, i, i, i, f, vp, i, vp, i, vp, i,
                                                 ctypes.POINTER(ctypes.c_size_t)]
        lib.b2g_sgemm_launch_count.argtypes = [i, i, i, i, i, f, vp, i, vp, i, vp, i,
                                               ctypes.POINTER(ctypes.c_int)]
        lib.b2g_release_workspaces.argtypes = []
        lib.b2g_sgemm_noalloc.argtypes = gemm
        lib.b2g_sgemm_host.argtypes = gemm
        lib.b2g_sgemm_3xtf32.argtypes = gemm
        lib.b2g_sgemm_3xtf32_variant.argtypes = [i] + gemm
        ll = ctypes.c_longlong
        lib.b2g_sgemm_strided_batched.argtypes = [i, i, i, i, i, f, vp, i, ll, vp, i, ll, f, vp,
                                                  i, ll, i, vp]
        lib.b2g_plan_count.argtypes = []
        lib.b2g_plan_name.argtypes = [i]
        lib.b2g_plan_name.restype = ctypes.c_char_p
        lib.b2g_plan_info.argtypes = [i, ctypes.POINTER(ctypes.c_int)]
        lib.b2g_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint), i]
        lib.b2g_sgemm_debug_status.argtypes = [vp]
        lib.b2g_set_wait_limit_ns.argtypes = [u64]
        lib.b2g_debug_stop_after.argtypes = [i]
        lib.b2g_strerror.argtypes = [i]
        lib.b2g_strerror.restype = ctypes.c_char_p
        lib.b2g_version.argtypes = []
        lib.b2g_version.restype = ctypes.c_char_p
        for name in EXPORTS:
            if not hasattr(lib, name):
                raise RuntimeError(f"{LIB_PATH} does not export {name}")
        _lib = lib
        return lib


def library():
    """The loaded ctypes library (raises when it has not been built)."""
    return _load()


# --- one-to-one wrappers of the C ABI -------------------------------------------

def b2g_sgemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> int:
    return _load().b2g_sgemm(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def b2g_sgemm_ex(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> int:
    return _load().b2g_sgemm_ex(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                                stream)


def b2g_sgemm_colmajor(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                       stream=0) -> int:
    return _load().b2g_sgemm_colmajor(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C,
                                      ldc, stream)


def b2g_sgemm_with_plan(plan, transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                        stream=0) -> int:
    return _load().b2g_sgemm_with_plan(plan, transA, transB, M, N, K, alpha, A, lda, B, ldb,
                                       beta, C, ldc, stream)


def b2g_sgemm_select_plan(transA, transB, M, N, K, alpha, A, lda, B, ldb, C, ldc) -> int:
    return _load().b2g_sgemm_select_plan(transA, transB, M, N, K, alpha, A, lda, B, ldb, C, ldc)


def b2g_sgemm_ws(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, workspace,
                 workspace_bytes, stream=0) -> int:
    return _load().b2g_sgemm_ws(transA, transB, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                                workspace, workspace_bytes, stream)


def b2g_sgemm_workspace_size(transA, transB, M, N, K, alpha, A, lda, B, ldb, C, ldc):
    """(rc, bytes) for the tune table's plan."""
    n = ctypes.c_size_t(0)
    rc = _load().b2g_sgemm_workspace_size(transA, transB, M, N, K, alpha, A, lda, B, ldb, C, ldc,
                                          ctypes.byref(n))
    return rc, n.value


def b2g_sgemm_launch_count(transA, transB, M, N, K, alpha, A, lda, B, ldb, C, ldc):
    """(rc, kernel launches one b2g_sgemm_ex call with these arguments makes)."""
    n = ctypes.c_int(0)
    rc = _load().b2g_sgemm_launch_count(transA, transB, M, N, K, alpha, A, lda, B, ldb, C, ldc,
                                        ctypes.byref(n))
    return rc, n.value


def b2g_release_workspaces() -> int:
    return _load().b2g_release_workspaces()


def b2g_sgemm_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> int:
    """The SGEMM for callers that cannot let the library allocate device memory
    (its scratch is a fixed per-device array; see include/b2g_sgemm.h)."""
    return _load().b2g_sgemm_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def b2g_sgemm_3xtf32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> int:
    return _load().b2g_sgemm_3xtf32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def b2g_sgemm_host(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=0) -> int:
    return _load().b2g_sgemm_host(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream)


def _host_ld(x, name):
    """Leading dimension (elements) of a row-major host float32 array or tensor."""
    import numpy as np

    if isinstance(x, np.ndarray):
        if x.dtype != np.float32 or x.ndim != 2 or (x.shape[1] > 1 and x.strides[1] != 4):
            raise ValueError(f"{name}: 2-D float32 array with unit column stride expected")
        return max(x.strides[0] // 4, 1), x.ctypes.data
    if x.device.type != "cpu" or x.dtype.is_floating_point is False or x.element_size() != 4:
        raise ValueError(f"{name}: CPU float32 tensor expected")
    if x.dim() != 2 or (x.shape[1] > 1 and x.stride(1) != 1):
        raise ValueError(f"{name}: 2-D tensor with unit column stride expected")
    return max(x.stride(0), 1), x.data_ptr()


def sgemm_host(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None, sync: bool = True):
    """C <- alpha * A @ B + beta * C for HOST float32 arrays or CPU tensors
    (page-locked ones copy fastest); see b2g_sgemm_host in include/b2g_sgemm.h.
    With sync (default) the call waits for the stream, so C holds the result
    on return."""
    lda, pa = _host_ld(A, "A")
    ldb, pb = _host_ld(B, "B")
    ldc, pc = _host_ld(C, "C")
    M, K = A.shape
    Kb, N = B.shape
    if Kb != K or tuple(C.shape) != (M, N):
        raise ValueError("shape mismatch")
    h = _stream_handle(stream)
    rc = b2g_sgemm_host(M, N, K, float(alpha), pa, lda, pb, ldb, float(beta), pc, ldc, h)
    if rc:
        raise B2GError(rc)
    if sync:
        import torch

        s = torch.cuda.current_stream() if stream is None else stream
        s.synchronize() if hasattr(s, "synchronize") else torch.cuda.synchronize()
    return C


def b2g_sgemm_3xtf32_variant(variant, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc,
                             stream=0) -> int:
    return _load().b2g_sgemm_3xtf32_variant(variant, M, N, K, alpha, A, lda, B, ldb, beta, C,
                                            ldc, stream)


def sgemm_3xtf32(A, B, C, alpha: float = 1.0, beta: float = 0.0, stream=None,
                 variant: Optional[int] = None):
    """C <- alpha * A @ B + beta * C on the tensor cores (3xTF32 split); see
    b2g_sgemm_3xtf32 in include/b2g_sgemm.h.  variant: None for the default
    kernel, 0 (one CTA per 128 x 128 tile), 1 (a CTA pair per 256 x 128 tile)
    or 2 (a CTA pair per 256 x 256 tile)."""
    M, K, lda = _check(A, "A")
    Kb, N, ldb = _check(B, "B")
    Mc, Nc, ldc = _check(C, "C")
    if Kb != K or Mc != M or Nc != N:
        raise ValueError(f"shape mismatch: A {M}x{K}, B {Kb}x{N}, C {Mc}x{Nc}")
    args = (M, N, K, float(alpha), A.data_ptr(), lda, B.data_ptr(), ldb, float(beta),
            C.data_ptr(), ldc, _stream_handle(stream))
    rc = b2g_sgemm_3xtf32(*args) if variant is None else b2g_sgemm_3xtf32_variant(variant, *args)
    if rc:
        raise B2GError(rc)
    return C


def b2g_sgemm_strided_batched(transA, transB, M, N, K, alpha, A, lda, strideA, B, ldb, strideB,
                              beta, C, ldc, strideC, batch, stream=0) -> int:
    return _load().b2g_sgemm_strided_batched(transA, transB, M, N, K, alpha, A, lda, strideA, B,
                                             ldb, strideB, beta, C, ldc, strideC, batch, stream)


def sgemm_batched(A, B, C, alpha: float = 1.0, beta: float = 0.0, transA: bool = False,
                  transB: bool = False, stream=None):
    """C[b] <- alpha * op(A[b]) @ op(B[b]) + beta * C[b] for 3-D float32 CUDA
    tensors (batch first; each matrix row-major with unit column stride)."""
    import torch

    for t, name in ((A, "A"), (B, "B"), (C, "C")):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or t.dim() != 3 or not t.is_cuda:
            raise TypeError(f"{name} must be a 3-D float32 CUDA tensor")
        if t.size(2) > 1 and t.stride(2) != 1:
            raise ValueError(f"{name} must have unit column stride")
    batch = A.size(0)
    if B.size(0) != batch or C.size(0) != batch:
        raise ValueError("batch sizes differ")
    M, K = (A.size(2), A.size(1)) if transA else (A.size(1), A.size(2))
    Kb, N = (B.size(2), B.size(1)) if transB else (B.size(1), B.size(2))
    if Kb != K or tuple(C.shape[1:]) != (M, N):
        raise ValueError("shape mismatch")

    def ld(t):
        return max(1, t.stride(1)) if t.size(1) > 1 else max(1, t.size(2))

    rc = b2g_sgemm_strided_batched(int(transA), int(transB), M, N, K, float(alpha), A.data_ptr(),
                                   ld(A), A.stride(0), B.data_ptr(), ld(B), B.stride(0),
                                   float(beta), C.data_ptr(), ld(C), C.stride(0), batch,
                                   _stream_handle(stream))
    if rc:
        raise B2GError(rc)
    return C


def b2g_plan_count() -> int:
    return _load().b2g_plan_count()


def b2g_plan_name(plan: int) -> Optional[str]:
    r = _load().b2g_plan_name(plan)
    return r.decode() if r is not None else None


def b2g_plan_info(plan: int) -> dict:
    buf = (ctypes.c_int * 9)()
    rc = _load().b2g_plan_info(plan, buf)
    if rc:
        raise B2GError(rc)
    keys = ("BM", "BN", "BK", "stages", "TN", "alayout", "feed", "threads", "smem_bytes")
    return dict(zip(keys, list(buf)))


def b2g_status(stream=0, clear: bool = True):
    """(rc, flags): synchronises `stream` and reads the kernels' status word."""
    flags = ctypes.c_uint(0)
    rc = _load().b2g_status(stream, ctypes.byref(flags), int(clear))
    return rc, flags.value


def b2g_sgemm_debug_status(stream=0) -> int:
    """Timeout flags of the status word (>= 0, not cleared) or a negative code;
    synchronises `stream`."""
    return _load().b2g_sgemm_debug_status(stream)


def b2g_set_wait_limit_ns(ns: int) -> int:
    return _load().b2g_set_wait_limit_ns(int(ns))


def b2g_debug_stop_after(n: int) -> int:
    return _load().b2g_debug_stop_after(int(n))


def b2g_strerror(code: int) -> str:
    return _load().b2g_strerror(code).decode()


def b2g_version() -> str:
    return _load().b2g_version().decode()


# --- tensor-level convenience ----------------------------------------------------

_torch = None


def _t():
    """torch, imported on first use (the C-ABI wrappers above need no torch)."""
    global _torch
    if _torch is None:
        import torch

        _torch = torch
    return _torch


def _stream_handle(stream) -> int:
    if stream is None:
        torch = _t()
        # the current stream's handle without building a Stream object (2.8 us
        # a call through torch.cuda.current_stream(), 0.1 us this way)
        raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        if raw is not None:
            return raw(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _check(t, name):
    """(rows, cols, leading dimension) of a row-major float32 CUDA matrix."""
    torch = _t()
    if not isinstance(t, torch.Tensor) or t.dtype is not torch.float32 or t.dim() != 2:
        raise TypeError(f"{name} must be a 2-D torch.float32 tensor")
    if not t.is_cuda:
        raise TypeError(f"{name} must be on a CUDA device")
    r, c = t.shape
    s0, s1 = t.stride()
    if c > 1 and s1 != 1:
        raise ValueError(f"{name} must have unit column stride (row-major rows)")
    return r, c, (max(1, s0) if r > 1 else max(1, c))


def sgemm(A, B, C, alpha: float = 1.0, beta: float = 0.0, transA: bool = False,
          transB: bool = False, plan: Optional[int] = None, stream=None):
    """C <- alpha * op(A) @ op(B) + beta * C on the current (or given) stream.

    A, B, C are 2-D float32 CUDA tensors with unit column stride; their row
    stride is the leading dimension.  op(A) is A.T when transA (A stored K x M),
    likewise for B.  Returns C.  Raises B2GError on a library error code.
    """
    ra, ca, lda = _check(A, "A")
    rb, cb, ldb = _check(B, "B")
    rc_, cc, ldc = _check(C, "C")
    M, K = (ca, ra) if transA else (ra, ca)
    Kb, N = (cb, rb) if transB else (rb, cb)
    if Kb != K or rc_ != M or cc != N:
        raise ValueError(f"shape mismatch: op(A) {M}x{K}, op(B) {Kb}x{N}, C {rc_}x{cc}")
    lib = _lib or _load()
    args = (M, N, K, float(alpha), A.data_ptr(), lda, B.data_ptr(), ldb, float(beta),
            C.data_ptr(), ldc, _stream_handle(stream))
    if plan is None:
        rc = lib.b2g_sgemm_ex(int(transA), int(transB), *args)
    else:
        rc = lib.b2g_sgemm_with_plan(int(plan), int(transA), int(transB), *args)
    if rc:
        raise B2GError(rc)
    return C


def _check_colmajor(t, name):
    import torch

    if not isinstance(t, torch.Tensor) or t.dtype != torch.float32 or t.dim() != 2:
        raise TypeError(f"{name} must be a 2-D torch.float32 tensor")
    if not t.is_cuda:
        raise TypeError(f"{name} must be on a CUDA device")
    if t.size(0) > 1 and t.stride(0) != 1:
        raise ValueError(f"{name} must have unit row stride (column-major columns)")
    return max(1, t.stride(1)) if t.size(1) > 1 else max(1, t.size(0))


def sgemm_colmajor(A, B, C, alpha: float = 1.0, beta: float = 0.0, transA: bool = False,
                   transB: bool = False, stream=None):
    """C <- alpha * op(A) @ op(B) + beta * C for column-major tensors.

    A, B, C are 2-D float32 CUDA tensors with unit row stride (for instance
    ``X.t()`` of a contiguous tensor); their column stride is the leading
    dimension.  op(A) is A.T when transA, likewise for B.  Runs
    ``b2g_sgemm_colmajor``; returns C.  Raises B2GError on a library error.
    """
    lda, ldb = _check_colmajor(A, "A"), _check_colmajor(B, "B")
    ldc = _check_colmajor(C, "C")
    M, K = (A.size(1), A.size(0)) if transA else (A.size(0), A.size(1))
    Kb, N = (B.size(1), B.size(0)) if transB else (B.size(0), B.size(1))
    if Kb != K or tuple(C.shape) != (M, N):
        raise ValueError(f"shape mismatch: op(A) {M}x{K}, op(B) {Kb}x{N}, C {tuple(C.shape)}")
    rc = b2g_sgemm_colmajor(int(transA), int(transB), M, N, K, float(alpha), A.data_ptr(), lda,
                            B.data_ptr(), ldb, float(beta), C.data_ptr(), ldc,
                            _stream_handle(stream))
    if rc:
        raise B2GError(rc)
    return C


def plans():
    """Names of the compiled plans, by index."""
    return [b2g_plan_name(i) for i in range(b2g_plan_count())]
