"""The one-launch small-problem plans (wk_*: the k tiles of an output tile
split between the warps of its CTA, the warps' partial tiles added in shared
memory) against the oracle: ragged edges, rings that wrap many times, k
groups left without work, beta = 0 with C unread, and run-to-run bitwise
reproducibility."""
import numpy as np
import pytest

import oracle
from gpu_helpers import check, env, gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tb():
    return env()


def _wk(b2g):
    names = b2g.plans()
    ids = [i for i, n in enumerate(names) if n.startswith("wk_")]
    assert ids
    return ids


# k tiles of 16: K = 16 (one group busy), 260 (16 tiles + a ragged tail: the
# ring's 16 slots just wrap), 1000, 4096 (the ring wraps 16 times)
# (N and K multiples of 4: the operands' rows must be 16-byte aligned)
SHAPES = [(1, 4, 16), (31, 68, 260), (64, 64, 64), (100, 200, 1000), (33, 68, 4096),
          (257, 132, 260), (512, 512, 512), (96, 320, 2048)]


@pytest.mark.parametrize("shape", SHAPES)
def test_warpk_plans(tb, shape):
    torch, b2g = tb
    M, N, K = shape
    rng = np.random.default_rng(M * 11 + N * 5 + K)
    A = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
    C = rng.uniform(-1, 1, size=(M, N)).astype(np.float32)
    ref, bound, _ = oracle.sgemm(A, B, C, 0.75, -1.25)
    for plan in _wk(b2g):
        got, rc, guard = gemm(b2g, torch, A, B, C, 0.75, -1.25, plan=plan)
        assert rc == 0 and guard, (b2g.plans()[plan], b2g.b2g_strerror(rc))
        check(got, ref, bound, f"{b2g.plans()[plan]} {shape}")


def test_warpk_padded_and_unaligned_c(tb):
    """Padded leading dimensions, and C whose rows are not 16-byte aligned
    (the epilogue's scalar path)."""
    torch, b2g = tb
    M, N, K = 70, 132, 300
    rng = np.random.default_rng(5)
    A = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
    C = rng.uniform(-1, 1, size=(M, N)).astype(np.float32)
    ref, bound, _ = oracle.sgemm(A, B, C, 1.5, 0.5)
    for plan in _wk(b2g):
        # A and B rows stay 16-byte aligned (the bulk-tensor feed needs it); C's do not
        for lds, mis in [((K + 4, N + 8, N + 10), (0, 0, 0)), ((K, N, N + 1), (0, 0, 3))]:
            got, rc, guard = gemm(b2g, torch, A, B, C, 1.5, 0.5, plan=plan, lds=lds,
                                  misalign=mis)
            assert rc == 0 and guard, (plan, lds, mis)
            check(got, ref, bound, f"{b2g.plans()[plan]} lds {lds} misalign {mis}")


def test_warpk_beta_zero_does_not_read_c(tb):
    torch, b2g = tb
    M, N, K = 96, 192, 512
    rng = np.random.default_rng(6)
    A = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
    C = np.full((M, N), np.nan, dtype=np.float32)
    ref, bound, _ = oracle.sgemm(A, B, np.zeros_like(C), 2.0, 0.0)
    for plan in _wk(b2g):
        got, rc, _ = gemm(b2g, torch, A, B, C, 2.0, 0.0, plan=plan)
        assert rc == 0
        check(got, ref, bound, b2g.plans()[plan])


def test_warpk_integers_exact_and_reproducible(tb):
    """Small integers: every partial sum is exact, so the result equals the
    oracle's bit for bit; two runs agree bit for bit on real-valued inputs."""
    torch, b2g = tb
    M, N, K = 64, 128, 1024
    rng = np.random.default_rng(7)
    A = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    B = rng.integers(-3, 4, size=(K, N)).astype(np.float32)
    C = rng.integers(-3, 4, size=(M, N)).astype(np.float32)
    ref, _, _ = oracle.sgemm(A, B, C, 1.0, -2.0)
    Ar = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    Br = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
    for plan in _wk(b2g):
        got, rc, _ = gemm(b2g, torch, A, B, C, 1.0, -2.0, plan=plan)
        assert rc == 0 and np.array_equal(got.astype(np.float64), ref)
        r1, _, _ = gemm(b2g, torch, Ar, Br, C, 0.5, 0.25, plan=plan)
        r2, _, _ = gemm(b2g, torch, Ar, Br, C, 0.5, 0.25, plan=plan)
        assert np.array_equal(r1.view(np.int32), r2.view(np.int32))


def test_warpk_refuses_unaligned_operands(tb):
    """The bulk-tensor feed needs aligned A and B with K % 4 == 0."""
    torch, b2g = tb
    A = np.ones((8, 6), np.float32)
    B = np.ones((6, 8), np.float32)
    C = np.zeros((8, 8), np.float32)
    for plan in _wk(b2g):
        _, rc, _ = gemm(b2g, torch, A, B, C, 1.0, 0.0, plan=plan)
        assert rc == b2g.B2G_ERR_UNSUPPORTED
