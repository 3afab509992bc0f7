"""b2g_sgemm_host: operands in host memory (page-locked and pageable), copied
to the device in row panels overlapped with the panel GEMMs, result copied
back.  Every result is checked against the oracle's FP32 bound."""
import numpy as np
import pytest

import oracle
from gpu_helpers import check, env, workload_reference

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tb():
    return env()


def _inputs(seed, M, N, K, lda=None, ldc=None):
    rng = np.random.default_rng(seed)
    A = rng.uniform(-1, 1, size=(M, lda or K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
    C = rng.uniform(-1, 1, size=(M, ldc or N)).astype(np.float32)
    return A, B, C


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("shape", [(200, 161, 92), (1000, 1025, 777), (2500, 300, 260),
                                   (4100, 260, 300)])
def test_host_operands(tb, shape, pinned):
    torch, b2g = tb
    M, N, K = shape
    A, B, C = _inputs(M + N + K, M, N, K)
    ref, bound, _ = oracle.sgemm(A, B, C, 0.75, -1.25)
    if pinned:
        hA, hB, hC = (torch.from_numpy(x).pin_memory() for x in (A, B, C))
    else:
        hA, hB, hC = A.copy(), B.copy(), C.copy()
    b2g.sgemm_host(hA, hB, hC, 0.75, -1.25)
    got = hC.numpy() if pinned else hC
    check(got, ref, bound, f"host {shape} pinned={pinned}")


def test_padded_leading_dims_untouched(tb):
    """Logical windows of wider host arrays: padding columns are neither read
    into the result nor written."""
    torch, b2g = tb
    M, N, K = 300, 170, 130
    A, B, C = _inputs(4, M, N, K, lda=141, ldc=181)
    C[:, N:] = 7.0
    ref, bound, _ = oracle.sgemm(A[:, :K], B, C[:, :N], 1.5, 0.5)
    hC = C.copy()
    rc = b2g.b2g_sgemm_host(M, N, K, 1.5, A.ctypes.data, 141, B.ctypes.data, N, 0.5,
                            hC.ctypes.data, 181, torch.cuda.current_stream().cuda_stream)
    assert rc == 0
    torch.cuda.synchronize()
    check(hC[:, :N], ref, bound, "padded")
    assert (hC[:, N:] == 7.0).all()


def test_beta_zero_does_not_read_c_and_scale_only(tb):
    torch, b2g = tb
    M, N, K = 2100, 200, 64
    A, B, _ = _inputs(5, M, N, K)
    C = np.full((M, N), np.nan, np.float32)  # beta == 0: C is write-only
    ref, bound, _ = oracle.sgemm(A, B, None, 1.0, 0.0)
    b2g.sgemm_host(A, B, C, 1.0, 0.0)
    check(C, ref, bound, "beta 0")
    C2 = np.full((M, N), 2.0, np.float32)
    b2g.sgemm_host(A, B, C2, 0.0, 3.0)  # alpha == 0: C = beta * C
    assert (C2 == 6.0).all()


def test_consecutive_calls_and_stream_order(tb):
    """Two calls in a row with different data reuse the staging buffer."""
    torch, b2g = tb
    for seed in (10, 11):
        A, B, C = _inputs(seed, 1500, 700, 900)
        ref, bound, _ = oracle.sgemm(A, B, C, 1.0, 1.0)
        hA, hB, hC = (torch.from_numpy(x).pin_memory() for x in (A, B, C))
        b2g.sgemm_host(hA, hB, hC, 1.0, 1.0)
        check(hC.numpy(), ref, bound, f"call {seed}")


def test_square4096_full(tb):
    """The bench's e2e workload through b2g_sgemm_host (three K chunks, the
    last in row panels), every output element against the oracle."""
    torch, b2g = tb
    w, A, B, C, ref, bound = workload_reference("square4096")
    hA, hB, hC = (torch.from_numpy(x).pin_memory() for x in (A, B, C))
    b2g.sgemm_host(hA, hB, hC, w.alpha, w.beta)
    check(hC.numpy(), ref, bound, "square4096 host")


@pytest.mark.parametrize("shape,beta", [((1100, 300, 2100), 0.5), ((2100, 300, 2052), -1.0),
                                        ((600, 1030, 2050), 0.0)])
def test_k_chunked_schedule(tb, shape, beta):
    """K >= 2048: three growing K chunks (K/8, 3K/8, K/2 rounded down to 16),
    the last in row panels; ragged K (K % 4 != 0 included), two panels, and
    beta = 0 (C not copied in).  Every element against the oracle."""
    torch, b2g = tb
    M, N, K = shape
    A, B, C = _inputs(M * 3 + K, M, N, K)
    ref, bound, _ = oracle.sgemm(A, B, C, 0.75, beta)
    hA, hB, hC = (torch.from_numpy(x).pin_memory() for x in (A, B, C))
    b2g.sgemm_host(hA, hB, hC, 0.75, beta)
    check(hC.numpy(), ref, bound, f"host chunked {shape} beta={beta}")


def test_k_chunked_beta_zero_does_not_read_c(tb):
    """K >= 2048 with beta = 0: the chunks' products and the panel kernel
    never read C, so NaN in C does not reach the result."""
    torch, b2g = tb
    M, N, K = 1300, 516, 2048
    A, B, _ = _inputs(12, M, N, K)
    C = np.full((M, N), np.nan, np.float32)
    ref, bound, _ = oracle.sgemm(A, B, None, -0.5, 0.0)
    hA, hB, hC = (torch.from_numpy(x).pin_memory() for x in (A, B, C))
    b2g.sgemm_host(hA, hB, hC, -0.5, 0.0)
    check(hC.numpy(), ref, bound, "host chunked beta 0, NaN C")
