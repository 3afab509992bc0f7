"""The 3xTF32 tensor-core path (b2g_sgemm_3xtf32) against the oracle, within
the same elementwise FP32 bound as the FFMA path, for both tensor-core kernels:
variant 0 (one CTA per 128 x 128 tile), variant 1 (a CTA pair per 256 x 128
tile, tcgen05.mma.cta_group::2) and variant 2 (a CTA pair per 256 x 256 tile)."""

import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import check, env, workload_reference

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tb():
    return env()


VARIANTS = [0, 1, 2]


def run3(torch, b2g, A, B, C, alpha, beta, variant=None):
    M, K = A.shape
    N = B.shape[1]
    dA, dB, dC = (torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (A, B, C))
    s = torch.cuda.current_stream().cuda_stream
    args = (M, N, K, alpha, dA.data_ptr(), K, dB.data_ptr(), N, beta, dC.data_ptr(), N, s)
    if variant is None:
        rc = b2g.b2g_sgemm_3xtf32(*args)
    else:
        rc = b2g.b2g_sgemm_3xtf32_variant(variant, *args)
    torch.cuda.synchronize()
    return rc, (dC.cpu().numpy() if rc == 0 else None)


@pytest.mark.parametrize("shape", [(128, 128, 32), (128, 128, 64), (256, 128, 32), (128, 256, 96),
                                   (1, 1, 4), (5, 7, 8), (37, 45, 52), (130, 257, 68),
                                   (300, 200, 1024), (257, 129, 96), (513, 384, 64)])
@pytest.mark.parametrize("variant", VARIANTS)
def test_shapes_within_bound(tb, shape, variant):
    torch, b2g = tb
    M, N, K = shape
    rng = np.random.default_rng(M + 3 * N + 7 * K)
    A = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
    C = rng.uniform(-1, 1, size=(M, N)).astype(np.float32)
    ref, bound, _ = oracle.sgemm(A, B, C, 0.75, -1.25)
    rc, got = run3(torch, b2g, A, B, C, 0.75, -1.25, variant)
    assert rc == 0, b2g.b2g_strerror(rc)
    check(got, ref, bound, f"3xtf32 {shape} variant {variant}")


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("shape", [(200, 160, 512), (600, 520, 2048)])
def test_small_integers_bit_exact(tb, variant, shape):
    """Integers up to 2^10 are TF32 values (lo = 0) and every partial sum stays
    below 2^24, so the tensor-core result must be exact -- also when the last
    tiles are split along k (K = 2048 on the CTA-pair kernels)."""
    torch, b2g = tb
    rng = np.random.default_rng(5)
    M, N, K = shape
    A = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    B = rng.integers(-3, 4, size=(K, N)).astype(np.float32)
    C = rng.integers(-3, 4, size=(M, N)).astype(np.float32)
    ref, _, _ = oracle.sgemm(A, B, C, 2.0, -1.0)
    rc, got = run3(torch, b2g, A, B, C, 2.0, -1.0, variant)
    assert rc == 0
    assert np.array_equal(got.astype(np.float64), ref)


@pytest.mark.parametrize("name", ["square512", "sweep128", "sweep1024", "skinny16x4096x4096"])
@pytest.mark.parametrize("variant", VARIANTS)
def test_workloads_full(tb, name, variant):
    torch, b2g = tb
    w = workloads.WORKLOADS[name]
    A, B, C = w.make()
    ref, bound, _ = oracle.sgemm(A, B, C, w.alpha, w.beta)
    rc, got = run3(torch, b2g, A, B, C, w.alpha, w.beta, variant)
    assert rc == 0
    check(got, ref, bound, name)


@pytest.mark.parametrize("name", ["square4096", "mlp8192x11008x4096"])
@pytest.mark.parametrize("variant", [None] + VARIANTS)
def test_workloads_full_size(tb, name, variant):
    """Full-size workloads on every kernel variant and on the default choice
    (the 256 x 256 CTA pair with its split tail at these sizes), every output
    element against the oracle."""
    torch, b2g = tb
    w, A, B, C, ref, bound = workload_reference(name)
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (A, B, C))
    b2g.sgemm_3xtf32(dA, dB, dC, w.alpha, w.beta, variant=variant)
    torch.cuda.synchronize()
    check(dC.cpu().numpy(), ref, bound, f"{name} variant {variant}")


def test_unsupported_operands(tb):
    torch, b2g = tb
    w = workloads.WORKLOADS["ragged1000x1025x777"]  # lda = 777: not a multiple of 4
    A, B, C = (torch.from_numpy(x).cuda() for x in w.make())
    s = torch.cuda.current_stream().cuda_stream
    rc = b2g.b2g_sgemm_3xtf32(w.M, w.N, w.K, w.alpha, A.data_ptr(), 777, B.data_ptr(), 1025,
                              w.beta, C.data_ptr(), 1025, s)
    assert rc == b2g.B2G_ERR_UNSUPPORTED


@pytest.mark.parametrize("variant", VARIANTS)
def test_nonfinite_and_beta_zero(tb, variant):
    torch, b2g = tb
    rng = np.random.default_rng(9)
    A = rng.uniform(-1, 1, size=(130, 64)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(64, 140)).astype(np.float32)
    A[100, 0] = np.nan
    C = np.full((130, 140), np.nan, np.float32)  # beta == 0: C must not be read
    ref, bound, _ = oracle.sgemm(A, B, C, 1.0, 0.0)
    rc, got = run3(torch, b2g, A, B, C, 1.0, 0.0, variant)
    assert rc == 0
    check(got, ref, bound, "nonfinite")
    assert np.isnan(got[100]).all() and np.isfinite(np.delete(got, 100, axis=0)).all()


@pytest.mark.parametrize("variant", VARIANTS)
def test_wait_runs_out_and_context_survives(tb, variant):
    torch, b2g = tb
    rng = np.random.default_rng(0)
    A = rng.uniform(-1, 1, size=(128, 128)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(128, 128)).astype(np.float32)
    C = np.zeros((128, 128), np.float32)
    s = torch.cuda.current_stream().cuda_stream
    b2g.b2g_status(s, clear=True)
    try:
        b2g.b2g_set_wait_limit_ns(20_000_000)
        b2g.b2g_debug_stop_after(1)  # 128 / 32 = 4 stages needed, 1 issued
        rc, _ = run3(torch, b2g, A, B, C, 1.0, 0.0, variant)
        assert rc == 0
        rc, flags = b2g.b2g_status(s, clear=True)
        assert rc == b2g.B2G_ERR_TIMEOUT and flags, f"{flags:#x}"
    finally:
        b2g.b2g_debug_stop_after(-1)
        b2g.b2g_set_wait_limit_ns(2_000_000_000)
    ref, bound, _ = oracle.sgemm(A, B, C, 1.0, 0.0)
    rc, got = run3(torch, b2g, A, B, C, 1.0, 0.0, variant)
    assert rc == 0
    check(got, ref, bound, "after timeout")


def test_unknown_variant(tb):
    torch, b2g = tb
    C = torch.zeros(4, 4, device="cuda")
    rc = b2g.b2g_sgemm_3xtf32_variant(3, 4, 4, 4, 1.0, C.data_ptr(), 4, C.data_ptr(), 4, 0.0,
                                      C.data_ptr(), 4, 0)
    assert rc == b2g.B2G_ERR_INVALID_PLAN
