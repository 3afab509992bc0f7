"""b2g_sgemm_noalloc, the entry point for callers that cannot let the library
allocate device memory (its scratch is a fixed per-device array).

Called through the C ABI twice in a row with different inputs -- so scratch
left over from the first call cannot pass for the second -- and compared with
b2g_sgemm, the regular entry point, and with the oracle, within the FP32 bound
the other GPU tests use.  This file is collected last on purpose: the other
tests have run by the time it can fail.  It also passes alone in a fresh
process.
"""
import ctypes

import numpy as np
import pytest

import oracle
from gpu_helpers import check, env

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tb():
    return env()


def _run(torch, fn, A, B, C, alpha, beta):
    M, K = A.shape
    N = B.shape[1]
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (A, B, C))
    s = torch.cuda.current_stream().cuda_stream
    rc = fn(M, N, K, ctypes.c_float(alpha), ctypes.c_void_p(dA.data_ptr()), K,
            ctypes.c_void_p(dB.data_ptr()), N, ctypes.c_float(beta),
            ctypes.c_void_p(dC.data_ptr()), N, ctypes.c_void_p(s))
    torch.cuda.synchronize()
    return rc, dC.cpu().numpy()


def test_noalloc_matches_regular_entry_point_twice(tb):
    torch, b2g = tb
    lib = b2g.library()  # the C ABI through ctypes
    M, N, K = 1030, 1500, 1400  # large enough that the plan uses the scratch
    rc, need = b2g.b2g_sgemm_workspace_size(0, 0, M, N, K, 1.0, 1 << 20, K, 1 << 20, N,
                                            1 << 20, N)
    assert rc == 0 and 0 < need <= 64 << 20
    for call, seed in enumerate((7, 8)):
        rng = np.random.default_rng(seed)
        A = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
        B = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
        C = rng.uniform(-1, 1, size=(M, N)).astype(np.float32)
        alpha, beta = (1.0, 0.5) if call == 0 else (-0.75, 1.25)
        rc, got = _run(torch, lib.b2g_sgemm_noalloc, A, B, C, alpha, beta)
        assert rc == 0, b2g.b2g_strerror(rc)
        rc, regular = _run(torch, lib.b2g_sgemm, A, B, C, alpha, beta)
        assert rc == 0
        ref, bound, _ = oracle.sgemm(A, B, C, alpha, beta)
        check(got, ref, bound, f"noalloc call {call}")
        assert (np.abs(got.astype(np.float64) - regular) <= bound).all(), f"call {call}"


def _rejects(torch, b2g, lib, M, N, K, lda):
    """Call b2g_sgemm_noalloc on real device operands (so that a call which is
    wrongly let through reads valid memory and fails an assertion instead of a
    GPU access); it must refuse and leave C untouched."""
    dA = torch.zeros((M, lda), device="cuda")
    dB = torch.zeros((K, N), device="cuda")
    C = torch.full((M, N), 3.0, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    rc = lib.b2g_sgemm_noalloc(M, N, K, ctypes.c_float(1.0), ctypes.c_void_p(dA.data_ptr()), lda,
                               ctypes.c_void_p(dB.data_ptr()), N, ctypes.c_float(0.0),
                               ctypes.c_void_p(C.data_ptr()), N, ctypes.c_void_p(s))
    torch.cuda.synchronize()
    assert rc == b2g.B2G_ERR_SCRATCH_LIMIT, b2g.b2g_strerror(rc)
    assert bool((C == 3.0).all())  # nothing was launched


def test_noalloc_rejects_more_than_its_scratch(tb):
    """A transpose-first plan whose A^T (4096 x 8192 floats, 128 MiB) is larger
    than the fixed array."""
    torch, b2g = tb
    lib = b2g.library()
    M, N, K = 8192, 64, 4096
    name = b2g.b2g_plan_name(b2g.b2g_sgemm_select_plan(0, 0, M, N, K, 1.0, 1 << 20, K, 1 << 20,
                                                        N, 1 << 20, N))
    assert name.startswith("pre_"), name
    _rejects(torch, b2g, lib, M, N, K, K)


def test_noalloc_rejects_packed_operands_past_its_scratch(tb):
    """K % 4 != 0 takes a packing plan, whose scratch holds A^T and an aligned
    copy of B: here A^T alone (33.5 MB) would fit, A^T plus B (167 MB) does not."""
    torch, b2g = tb
    lib = b2g.library()
    M, N, K = 2048, 8192, 4095
    name = b2g.b2g_plan_name(b2g.b2g_sgemm_select_plan(0, 0, M, N, K, 1.0, 1 << 20, K, 1 << 20,
                                                        N, 1 << 20, N))
    assert name.startswith("pack_"), name
    assert K * ((M + 3) // 4 * 4) * 4 < 64 << 20 < K * (M + N) * 4
    _rejects(torch, b2g, lib, M, N, K, K)


def test_noalloc_runs_a_packing_plan(tb):
    """Odd leading dimensions (the ragged workload's layout) take a packing
    plan whose scratch fits: the result matches b2g_sgemm and the oracle."""
    torch, b2g = tb
    lib = b2g.library()
    M, N, K = 1000, 1025, 777
    rng = np.random.default_rng(11)
    A = rng.standard_normal((M, K)).astype(np.float32)
    B = rng.standard_normal((K, N)).astype(np.float32)
    C = rng.standard_normal((M, N)).astype(np.float32)
    ref, bound, _ = oracle.sgemm(A, B, C, 0.75, -1.25)
    rc, got = _run(torch, lib.b2g_sgemm_noalloc, A, B, C, 0.75, -1.25)
    assert rc == 0, b2g.b2g_strerror(rc)
    check(got, ref, bound, "noalloc packing plan")
    rc, regular = _run(torch, lib.b2g_sgemm, A, B, C, 0.75, -1.25)
    assert rc == 0
    assert (np.abs(got.astype(np.float64) - regular) <= bound).all()
