"""Shared helpers of the GPU parity tests: device buffers with guard bands,
calls through the C ABI, and the elementwise check against the oracle."""
from __future__ import annotations

import numpy as np

import oracle

SENTINEL = np.float32(np.nan)

# Full-size workloads checked by several test files: their inputs and oracle
# result are computed once per test process (the 4096^3 oracle takes ~4 s on
# 16 cores, 8192 x 11008 x 4096 ~22 s) and kept for the later files.
_SHARED = ("square4096", "mlp8192x11008x4096")
_REF_CACHE = {}


def workload_reference(name):
    """(workload, A, B, C, ref, bound) for a named workload: the seeded inputs
    and the oracle's result and error budget for EVERY output element."""
    import workloads

    hit = _REF_CACHE.get(name)
    if hit is not None:
        return hit
    w = workloads.WORKLOADS[name]
    A, B, C = w.make()
    ref, bound, _ = oracle.sgemm(A, B, C, w.alpha, w.beta, M=w.M, N=w.N, K=w.K)
    out = (w, A, B, C, ref, bound)
    if name in _SHARED:
        _REF_CACHE[name] = out
    return out


def env():
    import torch

    if not torch.cuda.is_available():
        raise RuntimeError("GPU tests need a CUDA device")
    from dense_fp32_gemm_07_gb300 import build

    build.build()
    import dense_fp32_gemm_07_gb300 as b2g

    b2g.library()
    return torch, b2g


def to_device(torch, host: np.ndarray, rows: int, cols: int, ld: int, extra_rows: int = 0,
              misalign: int = 0, fill=SENTINEL):
    """Copy the logical rows x cols block of `host` into a fresh device buffer
    with leading dimension `ld`, `extra_rows` guard rows below, every padding
    element set to `fill`, and the base shifted by `misalign` floats.
    Returns (view, flat_buffer)."""
    total = (rows + extra_rows) * ld + misalign
    flat = torch.full((max(total, 1),), float(fill), dtype=torch.float32, device="cuda")
    if rows and cols:
        blk = torch.from_numpy(np.ascontiguousarray(host[:rows, :cols])).to("cuda")
        view = flat[misalign:misalign + rows * ld].view(rows, ld)[:, :cols]
        view.copy_(blk)
    view = torch.as_strided(flat, (rows, cols), (ld, 1), misalign)
    return view, flat


def gemm(b2g, torch, A, B, C, alpha, beta, transA=False, transB=False, plan=None,
         lds=None, misalign=(0, 0, 0), guard=True):
    """Run one SGEMM on device copies; return (result M x N, rc, guard_ok)."""
    M = A.shape[1] if transA else A.shape[0]
    K = A.shape[0] if transA else A.shape[1]
    N = B.shape[0] if transB else B.shape[1]
    lda, ldb, ldc = lds or (A.shape[1], B.shape[1], N)
    dA, _ = to_device(torch, A, A.shape[0], A.shape[1], max(lda, 1), misalign=misalign[0])
    dB, _ = to_device(torch, B, B.shape[0], B.shape[1], max(ldb, 1), misalign=misalign[1])
    dC, flatC = to_device(torch, C, M, N, max(ldc, 1), extra_rows=2 if guard else 0,
                          misalign=misalign[2])
    before = flatC.clone()
    s = torch.cuda.current_stream().cuda_stream
    args = (M, N, K, float(alpha), dA.data_ptr(), max(lda, 1), dB.data_ptr(), max(ldb, 1),
            float(beta), dC.data_ptr(), max(ldc, 1), s)
    if plan is None:
        rc = b2g.b2g_sgemm_ex(int(transA), int(transB), *args)
    else:
        rc = b2g.b2g_sgemm_with_plan(plan, int(transA), int(transB), *args)
    torch.cuda.synchronize()
    got = dC.cpu().numpy() if rc == 0 else None
    guard_ok = True
    if rc == 0 and guard:
        # everything outside the logical M x N window must be bit-identical
        mask = torch.ones_like(flatC, dtype=torch.bool)
        win = torch.as_strided(mask, (M, N), (max(ldc, 1), 1), misalign[2])
        win.fill_(False)
        a = flatC.view(torch.int32)[mask]
        b = before.view(torch.int32)[mask]
        guard_ok = bool(torch.equal(a, b))
    return got, rc, guard_ok


def check(got, ref, bound, what=""):
    bad = oracle.violations(got, ref, bound)
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} entries outside the FP32 bound; first "
            + ", ".join(f"{tuple(i)} got {got[tuple(i)]!r} ref {ref[tuple(i)]!r} "
                        f"bound {bound[tuple(i)]:.3g}" for i in idx))
    with np.errstate(invalid="ignore", divide="ignore"):
        ratio = np.abs(got.astype(np.float64) - ref) / bound
    return float(np.nanmax(ratio)) if ratio.size else 0.0


def sample_entries(M, N, tile=128, per_tile=3, seed=0):
    """Entries covering every tile x tile block: its two corners plus random
    interior points, and the matrix's last row and column."""
    rng = np.random.default_rng(seed)
    rows, cols = [], []
    for i0 in range(0, M, tile):
        for j0 in range(0, N, tile):
            i1, j1 = min(M, i0 + tile) - 1, min(N, j0 + tile) - 1
            rows += [i0, i1]
            cols += [j0, j1]
            rows += list(rng.integers(i0, i1 + 1, size=per_tile))
            cols += list(rng.integers(j0, j1 + 1, size=per_tile))
    rows += [M - 1] * 8 + list(rng.integers(0, M, size=8))
    cols += list(rng.integers(0, N, size=8)) + [N - 1] * 8
    return np.array(rows, dtype=np.int64), np.array(cols, dtype=np.int64)
