"""CPU oracle for row-major FP32 SGEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the bench's CPU-baseline and
reference legs may import this package.  The CUDA library never uses it.

The arithmetic lives in ``sgemm_oracle.c`` (plain C, double accumulation,
i-k-j loop order); this module only compiles it with gcc and marshals numpy
arrays through ctypes.  Parity of every function here is pinned by
``tests/test_oracle_pins.py`` (identity, all-ones, alpha/beta closed forms,
small-integer exactness, exact-rational brute force, transpose identity,
linearity, padded leading dimensions, multiply-add count).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sgemm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_sgemm.so")
_lock = threading.Lock()
_lib = None

# -ffp-contract=off: every double product/sum is rounded as written, on x86 and
# Arm alike (no fused multiply-add contraction).
CFLAGS = ["-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared", "-std=c11"]


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc + OpenMP); returns its path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, dbl, vp, ci = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
            lib.oracle_sgemm.restype = i64
            lib.oracle_sgemm.argtypes = [ci, ci, ci, ci, ci, dbl, vp, i64, vp, i64, dbl, vp, i64,
                                         vp, vp, ci]
            lib.oracle_sgemm_entries.restype = i64
            lib.oracle_sgemm_entries.argtypes = [ci, ci, ci, ci, ci, dbl, vp, i64, vp, i64, dbl,
                                                 vp, i64, i64, vp, vp, vp, vp, ci]
            lib.oracle_max_threads.restype = ci
            _lib = lib
    return _lib


def _f32(x: Optional[np.ndarray]) -> Optional[np.ndarray]:
    if x is None:
        return None
    if x.dtype != np.float32 or x.ndim != 2 or (x.size and x.shape[1] > 1 and x.strides[1] != 4):
        raise TypeError("oracle operands must be 2-D float32 arrays with unit column stride")
    return x


def _ptr(x: Optional[np.ndarray]):
    return None if x is None else x.ctypes.data


def _shape(A, B, transA, transB):
    M, K = (A.shape[1], A.shape[0]) if transA else (A.shape[0], A.shape[1])
    K2, N = (B.shape[1], B.shape[0]) if transB else (B.shape[0], B.shape[1])
    if K != K2:
        raise ValueError(f"inner dimensions differ: {K} vs {K2}")
    return M, N, K


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def sgemm(A: np.ndarray, B: np.ndarray, C: Optional[np.ndarray], alpha: float, beta: float,
          transA: bool = False, transB: bool = False, threads: int = 0,
          M: Optional[int] = None, N: Optional[int] = None, K: Optional[int] = None
          ) -> Tuple[np.ndarray, np.ndarray, int]:
    """Reference ``alpha*op(A)@op(B) + beta*C`` in float64.

    A, B, C are 2-D float32 arrays whose row stride is the leading dimension;
    the logical sizes default to the array shapes and may be given explicitly
    (for padded leading dimensions the arrays are wider than the logical
    matrix).  Returns ``(ref, bound, fmas)``: the M x N double result, the
    elementwise FP32 error budget, and the number of multiply-adds done.
    """
    A, B, C = _f32(A), _f32(B), _f32(C)
    if M is None or N is None or K is None:
        m0, n0, k0 = _shape(A, B, transA, transB)
        M = m0 if M is None else M
        N = n0 if N is None else N
        K = k0 if K is None else K
    lda, ldb = A.strides[0] // 4, B.strides[0] // 4
    ldc = C.strides[0] // 4 if C is not None else N
    if beta != 0.0 and C is None:
        raise ValueError("beta != 0 needs C")
    ref = np.empty((M, N), dtype=np.float64)
    bound = np.empty((M, N), dtype=np.float64)
    fmas = _load().oracle_sgemm(int(transA), int(transB), M, N, K, float(alpha), _ptr(A), lda,
                                _ptr(B), ldb, float(beta), _ptr(C), ldc, _ptr(ref), _ptr(bound),
                                int(threads))
    return ref, bound, int(fmas)


def sgemm_entries(A: np.ndarray, B: np.ndarray, C: Optional[np.ndarray], alpha: float,
                  beta: float, rows: np.ndarray, cols: np.ndarray, K: Optional[int] = None,
                  transA: bool = False, transB: bool = False, threads: int = 0
                  ) -> Tuple[np.ndarray, np.ndarray, int]:
    """Reference values and error budgets for the entries (rows[t], cols[t]) only."""
    A, B, C = _f32(A), _f32(B), _f32(C)
    if K is None:
        K = _shape(A, B, transA, transB)[2]
    rows = np.ascontiguousarray(rows, dtype=np.int64).ravel()
    cols = np.ascontiguousarray(cols, dtype=np.int64).ravel()
    if rows.shape != cols.shape:
        raise ValueError(f"rows and cols differ in length: {rows.size} vs {cols.size}")
    lda, ldb = A.strides[0] // 4, B.strides[0] // 4
    ldc = C.strides[0] // 4 if C is not None else 0
    ref = np.empty(rows.shape[0], dtype=np.float64)
    bound = np.empty(rows.shape[0], dtype=np.float64)
    fmas = _load().oracle_sgemm_entries(int(transA), int(transB), 0, 0, K, float(alpha),
                                        _ptr(A), lda, _ptr(B), ldb, float(beta), _ptr(C), ldc,
                                        rows.shape[0], _ptr(rows), _ptr(cols), _ptr(ref),
                                        _ptr(bound), int(threads))
    return ref, bound, int(fmas)


def violations(got: np.ndarray, ref: np.ndarray, bound: np.ndarray) -> np.ndarray:
    """Boolean mask of entries outside the elementwise FP32 error budget.

    An entry passes when ``|got - ref| <= bound``; NaN/Inf in ``got`` fail
    unless ``ref`` holds the same non-finite value.
    """
    got = np.asarray(got, dtype=np.float64)
    with np.errstate(invalid="ignore"):
        err = np.abs(got - ref)
        bad = ~(err <= bound)
        same_nonfinite = ~np.isfinite(ref) & ((got == ref) | (np.isnan(got) & np.isnan(ref)))
    return bad & ~same_nonfinite
