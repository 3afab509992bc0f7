"""The split tail of the FFMA plans: when the last round of the persistent
grid would keep only some CTAs busy, the last tiles are cut into k slices
whose partial sums a second kernel adds in slice order before the epilogue.
Every result is checked against the oracle's FP32 bound; integer inputs
(exact partial sums) must match exactly, and the fixed summation order must
give bitwise-identical results run to run."""
import numpy as np
import pytest

import oracle
from gpu_helpers import check, env, gemm

pytestmark = pytest.mark.gpu

FAKE = 1 << 20


@pytest.fixture(scope="module")
def tb():
    return env()


def ffma_plans(b2g):
    return [n for n in b2g.plans() if not n.startswith("skinny")]


def launches(b2g, M, N, K, lda=None):
    rc, n = b2g.b2g_sgemm_launch_count(0, 0, M, N, K, 1.0, FAKE, lda or K, FAKE, N, FAKE, N)
    assert rc == 0
    return n


def test_split_engages_on_these_shapes(tb):
    _, b2g = tb
    # table plans: the GEMM kernel, plus a transpose for pre_ plans, plus the tail
    assert launches(b2g, 300, 260, 1000) == 2
    assert launches(b2g, 1030, 1500, 1400) == 3
    assert launches(b2g, 4096, 4096, 4096) == 3
    assert launches(b2g, 300, 260, 100) == 1  # under 128 k: no split


@pytest.mark.parametrize("trans", [(False, False), (True, False), (False, True)])
def test_every_plan_split_ragged(tb, trans):
    """A few tiles and 1000 k (ragged last k tile): every plan splits the
    tiles into k slices (up to 15 of at least 64 k)."""
    torch, b2g = tb
    M, N, K = 300, 260, 1000
    rng = np.random.default_rng(11)
    tA, tB = trans
    A = rng.uniform(-1, 1, size=(K, M) if tA else (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(N, K) if tB else (K, N)).astype(np.float32)
    C = rng.uniform(-1, 1, size=(M, N)).astype(np.float32)
    ref, bound, _ = oracle.sgemm(A, B, C, 1.25, -0.5, transA=tA, transB=tB)
    ran = 0
    for name in ffma_plans(b2g):
        pi = b2g.plans().index(name)
        got, rc, guard_ok = gemm(b2g, torch, A, B, C, 1.25, -0.5, transA=tA, transB=tB, plan=pi)
        if rc == b2g.B2G_ERR_UNSUPPORTED:
            continue
        assert rc == 0, (name, b2g.b2g_strerror(rc))
        assert guard_ok, name
        check(got, ref, bound, name)
        ran += 1
    assert ran > 0


def test_small_integers_exact(tb):
    torch, b2g = tb
    rng = np.random.default_rng(3)
    M, N, K = 300, 260, 1000
    A = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    B = rng.integers(-3, 4, size=(K, N)).astype(np.float32)
    C = rng.integers(-3, 4, size=(M, N)).astype(np.float32)
    ref, _, _ = oracle.sgemm(A, B, C, 2.0, -1.0)
    got, rc, _ = gemm(b2g, torch, A, B, C, 2.0, -1.0)
    assert rc == 0
    assert np.array_equal(got.astype(np.float64), ref)


def test_bitwise_reproducible(tb):
    torch, b2g = tb
    M, N, K = 1030, 1500, 1400
    rng = np.random.default_rng(5)
    A = torch.from_numpy(rng.uniform(-1, 1, size=(M, K)).astype(np.float32)).cuda()
    B = torch.from_numpy(rng.uniform(-1, 1, size=(K, N)).astype(np.float32)).cuda()
    C0 = torch.from_numpy(rng.uniform(-1, 1, size=(M, N)).astype(np.float32)).cuda()
    outs = []
    for _ in range(3):
        C = C0.clone()
        b2g.sgemm(A, B, C, 1.0, 0.5)
        torch.cuda.synchronize()
        outs.append(C.view(torch.int32).cpu())
    assert all(torch.equal(outs[0], o) for o in outs[1:])


def test_batched_split(tb):
    torch, b2g = tb
    batch, M, N, K = 3, 200, 170, 900
    rng = np.random.default_rng(9)
    A = rng.uniform(-1, 1, size=(batch, M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(batch, K, N)).astype(np.float32)
    C = rng.uniform(-1, 1, size=(batch, M, N)).astype(np.float32)
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (A, B, C))
    b2g.sgemm_batched(dA, dB, dC, 0.5, 1.5)
    torch.cuda.synchronize()
    got = dC.cpu().numpy()
    for b in range(batch):
        ref, bound, _ = oracle.sgemm(A[b], B[b], C[b], 0.5, 1.5)
        check(got[b], ref, bound, f"problem {b}")


@pytest.mark.parametrize("lds,mis", [((1000, 260, 261), (0, 0, 0)), ((1000, 260, 260), (0, 0, 1))])
def test_split_tail_unaligned_c(tb, lds, mis):
    """C whose rows are not 16-byte aligned (odd ldc, or a base one float off):
    the split tail's reduction then moves C element by element; same bound,
    beta != 0 so C is read."""
    torch, b2g = tb
    M, N, K = 300, 260, 1000
    rng = np.random.default_rng(17)
    A = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
    C = rng.uniform(-1, 1, size=(M, N)).astype(np.float32)
    ref, bound, _ = oracle.sgemm(A, B, C, 0.5, 1.5)
    assert launches(b2g, M, N, K) == 2  # the GEMM and the split tail's reduction
    got, rc, guard = gemm(b2g, torch, A, B, C, 0.5, 1.5, lds=lds, misalign=mis)
    assert rc == 0 and guard
    check(got, ref, bound, f"ldc {lds[2]} misalign {mis}")
