"""Seeded random calls through the tune table: shapes, op() flags, padded or
odd leading dimensions, misaligned bases and alpha/beta drawn at random, so
that every plan family the table reaches (the one-launch wk families, the
split-tail plans with their transposes and packing, the 4-byte feed, the
skinny plans) is met on shapes nobody picked by hand.  Every output element is
checked against the oracle, and everything outside C must stay untouched."""
import numpy as np
import pytest

import oracle
from gpu_helpers import check, env, gemm

pytestmark = pytest.mark.gpu

FAKE = 1 << 20


@pytest.fixture(scope="module")
def tb():
    return env()


def _case(seed):
    """Operand class by seed (aligned row-major, A stored K x M, B stored N x K,
    anything else), then random sizes, leading dimensions and scalars."""
    rng = np.random.default_rng(1000 + seed)
    cls = seed % 4
    size = int(rng.choice([64, 300, 800, 1300]))
    M, N, K = (int(rng.integers(max(1, size // 3), size + 1)) for _ in range(3))
    if rng.random() < 0.15:
        M = int(rng.integers(1, 33))  # skinny
    transA = cls == 1 or (cls == 2 and rng.random() < 0.5)
    transB = cls == 2
    if cls < 3:  # 16-byte-vector eligible: K, N (and M for A stored K x M) % 4 == 0
        K, N = (K + 3) // 4 * 4, (N + 3) // 4 * 4
        M = (M + 3) // 4 * 4 if transA else M
        pad = [int(rng.choice([0, 4, 8])) for _ in range(2)] + [int(rng.choice([0, 1, 4]))]
        mis = (0, 0, int(rng.choice([0, 1])))
    else:
        pad = [int(rng.choice([0, 1, 3, 4])) for _ in range(3)]
        mis = tuple(int(rng.choice([0, 1])) for _ in range(3))
    alpha = float(rng.choice([1.0, -0.5, 2.0]))
    beta = float(rng.choice([0.0, 1.0, -1.25]))
    return M, N, K, transA, transB, pad, mis, alpha, beta


@pytest.mark.parametrize("seed", range(60))
def test_random_call(tb, seed):
    torch, b2g = tb
    M, N, K, transA, transB, pad, mis, alpha, beta = _case(seed)
    rng = np.random.default_rng(seed)
    A = rng.uniform(-1, 1, size=(K, M) if transA else (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(N, K) if transB else (K, N)).astype(np.float32)
    C = rng.uniform(-1, 1, size=(M, N)).astype(np.float32)
    lds = (A.shape[1] + pad[0], B.shape[1] + pad[1], N + pad[2])
    ref, bound, _ = oracle.sgemm(A, B, C, alpha, beta, transA=transA, transB=transB)
    plan = b2g.b2g_plan_name(b2g.b2g_sgemm_select_plan(
        int(transA), int(transB), M, N, K, alpha, FAKE + 4 * mis[0], lds[0],
        FAKE + 4 * mis[1], lds[1], FAKE + 4 * mis[2], lds[2]))
    got, rc, guard = gemm(b2g, torch, A, B, C, alpha, beta, transA, transB, lds=lds,
                          misalign=mis)
    what = f"seed {seed}: {M}x{N}x{K} op {transA},{transB} lds {lds} mis {mis} plan {plan}"
    assert rc == 0, (what, b2g.b2g_strerror(rc))
    assert guard, what
    check(got, ref, bound, what)
