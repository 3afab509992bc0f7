"""Pins for the CPU oracle: facts fixed by the pages and by the mathematics.

Each check is independent of the oracle's own code path (closed forms, exact
integer or rational arithmetic in Python, structural identities), chosen so
that a dropped term, a wrong sign, a swapped index or a transposed operand in
the oracle fails at least one of them.  The definition being pinned is
C = alpha*A*B + beta*C with row-major A (M x K), B (K x N), C (M x N)
(GEMM 优化之路, section 问题定义与性能上限).
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U = 2.0 ** -24


def _rng(seed):
    return np.random.default_rng(seed)


def _rand(rng, shape):
    return rng.uniform(-1, 1, size=shape).astype(np.float32)


# --- golden values printed on the pages --------------------------------------

def test_page_flop_and_traffic_figures():
    """2MNK, minimum traffic and arithmetic intensity at 4096^3 match the pages."""
    with open(os.path.join(GOLDEN, "page_figures.json")) as f:
        entries = json.load(f)["entries"]
    for e in entries:
        w = workloads.Workload("g", e["M"], e["N"], e["K"], 1.0,
                               0.5 if e.get("beta_nonzero", True) else 0.0, 0, "u11", "u11")
        if e["name"].startswith("flops"):
            got = w.flops()
        elif e["name"].startswith("bytes"):
            got = w.min_bytes()
        else:
            got = w.flops() / w.min_bytes()
        assert abs(got - e["value"]) <= e["rel"] * e["value"], (e["name"], got, e["cite"])


def test_hand_worked_example(oracle_mod):
    with open(os.path.join(GOLDEN, "hand_example.json")) as f:
        g = json.load(f)
    A = np.array(g["A"], np.float32)
    B = np.array(g["B"], np.float32)
    C = np.array(g["C"], np.float32)
    ref, bound, fmas = oracle_mod.sgemm(A, B, C, g["alpha"], g["beta"])
    assert np.array_equal(ref, np.array(g["expected"]))
    assert fmas == g["M"] * g["N"] * g["K"]


# --- multiply-add count (2MNK FLOPs) -----------------------------------------

@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (17, 9, 33), (64, 1, 5)])
def test_fma_count_is_mnk(oracle_mod, M, N, K):
    rng = _rng(M * 100 + N * 10 + K)
    A, B = _rand(rng, (M, K)), _rand(rng, (K, N))
    _, _, fmas = oracle_mod.sgemm(A, B, None, 1.0, 0.0)
    assert 2 * fmas == 2 * M * N * K
    _, _, fmas0 = oracle_mod.sgemm(A, B, None, 0.0, 0.0)
    assert fmas0 == 0  # alpha == 0: A and B are not read


# --- identity / all-ones / alpha-beta closed forms ---------------------------

@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (0.75, -1.25), (-2.0, 0.5)])
def test_identity_left(oracle_mod, alpha, beta):
    """A = I (M = K): result is alpha*B + beta*C, every product exact."""
    rng = _rng(1)
    n, N = 13, 10
    A = np.eye(n, dtype=np.float32)
    B, C = _rand(rng, (n, N)), _rand(rng, (n, N))
    ref, _, _ = oracle_mod.sgemm(A, B, C, alpha, beta)
    expect = alpha * B.astype(np.float64) + (beta * C.astype(np.float64) if beta else 0.0)
    assert np.array_equal(ref, expect)


@pytest.mark.parametrize("alpha,beta", [(1.0, 0.0), (0.75, -1.25)])
def test_identity_right(oracle_mod, alpha, beta):
    """B = I (K = N): result is alpha*A + beta*C."""
    rng = _rng(2)
    M, n = 9, 12
    A, C = _rand(rng, (M, n)), _rand(rng, (M, n))
    B = np.eye(n, dtype=np.float32)
    ref, _, _ = oracle_mod.sgemm(A, B, C, alpha, beta)
    expect = alpha * A.astype(np.float64) + (beta * C.astype(np.float64) if beta else 0.0)
    assert np.array_equal(ref, expect)


@pytest.mark.parametrize("K", [1, 7, 100, 1025])
def test_all_ones(oracle_mod, K):
    """A = B = 1: every entry is alpha*K + beta*C_ij exactly."""
    rng = _rng(K)
    M, N = 6, 11
    A = np.ones((M, K), np.float32)
    B = np.ones((K, N), np.float32)
    C = _rand(rng, (M, N))
    alpha, beta = 0.75, -1.25
    ref, bound, _ = oracle_mod.sgemm(A, B, C, alpha, beta)
    c = C.astype(np.float64)
    assert np.array_equal(ref, alpha * K + beta * c)
    # |A||B| summed is exactly K, so the error budget is fixed too
    assert np.allclose(bound, 2 * K * U * (abs(alpha) * K + np.abs(beta * c)) + 1e-6, rtol=1e-15)


def test_alpha_zero_gives_beta_c(oracle_mod):
    rng = _rng(3)
    A = np.full((5, 4), np.nan, np.float32)  # alpha == 0: A and B must not be read
    B = np.full((4, 6), np.inf, np.float32)
    C = _rand(rng, (5, 6))
    ref, _, _ = oracle_mod.sgemm(A, B, C, 0.0, -1.5)
    assert np.array_equal(ref, -1.5 * C.astype(np.float64))


def test_beta_zero_does_not_read_c(oracle_mod):
    rng = _rng(4)
    A, B = _rand(rng, (7, 5)), _rand(rng, (5, 3))
    C = np.full((7, 3), np.nan, np.float32)
    ref, bound, _ = oracle_mod.sgemm(A, B, C, 1.0, 0.0)
    assert np.isfinite(ref).all() and np.isfinite(bound).all()


def test_k_zero(oracle_mod):
    A = np.zeros((4, 0), np.float32)
    B = np.zeros((0, 3), np.float32)
    C = np.arange(12, dtype=np.float32).reshape(4, 3)
    ref, bound, fmas = oracle_mod.sgemm(A, B, C, 2.0, 0.5, K=0, M=4, N=3)
    assert fmas == 0 and np.array_equal(ref, 0.5 * C.astype(np.float64))
    assert np.allclose(bound, 1e-6)


# --- exact arithmetic brute force ---------------------------------------------

@pytest.mark.parametrize("seed", range(4))
def test_small_integer_exactness(oracle_mod, seed):
    """Entries in {-3..3}: every partial sum is an integer below 2**24, so the
    oracle must equal exact integer arithmetic done in Python."""
    rng = _rng(10 + seed)
    M, N, K = rng.integers(1, 40, size=3)
    Ai = rng.integers(-3, 4, size=(M, K))
    Bi = rng.integers(-3, 4, size=(K, N))
    Ci = rng.integers(-3, 4, size=(M, N))
    exact = [[2 * sum(int(Ai[i, k]) * int(Bi[k, j]) for k in range(K)) - 3 * int(Ci[i, j])
              for j in range(N)] for i in range(M)]
    ref, _, _ = oracle_mod.sgemm(Ai.astype(np.float32), Bi.astype(np.float32),
                                 Ci.astype(np.float32), 2.0, -3.0)
    assert np.array_equal(ref, np.array(exact, dtype=np.float64))


@pytest.mark.parametrize("transA,transB", [(False, False), (True, False), (False, True), (True, True)])
@pytest.mark.parametrize("seed", range(3))
def test_fraction_brute_force(oracle_mod, transA, transB, seed):
    """Tiny shapes, padded leading dimensions, both op() flags: compare with exact
    rationals.  The double-accumulated oracle must sit within K double roundings
    of the exact value, and its error budget must use the exact |A||B| sum."""
    rng = _rng(100 + seed + 7 * transA + 13 * transB)
    M, N, K = (int(x) for x in rng.integers(1, 8, size=3))
    pa, pb, pc = (int(x) for x in rng.integers(0, 3, size=3))
    a_rows, a_cols = (K, M) if transA else (M, K)
    b_rows, b_cols = (N, K) if transB else (K, N)
    Astore = _rand(rng, (a_rows, a_cols + pa))
    Bstore = _rand(rng, (b_rows, b_cols + pb))
    Cstore = _rand(rng, (M, N + pc))
    alpha, beta = float(np.float32(rng.uniform(-2, 2))), float(np.float32(rng.uniform(-2, 2)))
    ref, bound, fmas = oracle_mod.sgemm(Astore, Bstore, Cstore, alpha, beta, transA=transA,
                                        transB=transB, M=M, N=N, K=K)
    assert fmas == M * N * K

    def a(i, k):
        return Fraction(float(Astore[k, i] if transA else Astore[i, k]))

    def b(k, j):
        return Fraction(float(Bstore[j, k] if transB else Bstore[k, j]))

    for i in range(M):
        for j in range(N):
            dot = sum((a(i, k) * b(k, j) for k in range(K)), Fraction(0))
            mag = sum((abs(a(i, k)) * abs(b(k, j)) for k in range(K)), Fraction(0))
            c = Fraction(float(Cstore[i, j]))
            exact = Fraction(alpha) * dot + Fraction(beta) * c
            scale = abs(Fraction(alpha)) * mag + abs(Fraction(beta) * c)
            tol = (K + 3) * 2.0 ** -53 * float(scale)
            assert abs(Fraction(ref[i, j]) - exact) <= Fraction(tol), (i, j)
            b_exact = 2 * K * U * float(scale) + 1e-6
            assert abs(bound[i, j] - b_exact) <= 1e-12 * b_exact


# --- structural identities ------------------------------------------------------

def test_transpose_identity(oracle_mod):
    """(A B)^T = B^T A^T: the same k-ordered double sums, so bitwise equal."""
    rng = _rng(5)
    M, N, K = 23, 17, 31
    A, B, C = _rand(rng, (M, K)), _rand(rng, (K, N)), _rand(rng, (M, N))
    ref, _, _ = oracle_mod.sgemm(A, B, C, 0.5, 2.0)
    refT, _, _ = oracle_mod.sgemm(np.ascontiguousarray(B.T), np.ascontiguousarray(A.T),
                                  np.ascontiguousarray(C.T), 0.5, 2.0)
    assert np.array_equal(ref, refT.T)
    # op() flags on the stored transposes give the same matrix
    refF, _, _ = oracle_mod.sgemm(np.ascontiguousarray(A.T), np.ascontiguousarray(B.T), C, 0.5,
                                  2.0, transA=True, transB=True)
    assert np.array_equal(ref, refF)


def test_linearity_in_alpha(oracle_mod):
    rng = _rng(6)
    A, B = _rand(rng, (9, 40)), _rand(rng, (40, 8))
    r1, _, _ = oracle_mod.sgemm(A, B, None, 0.5, 0.0)
    r2, _, _ = oracle_mod.sgemm(A, B, None, 0.25, 0.0)
    r3, _, _ = oracle_mod.sgemm(A, B, None, 0.75, 0.0)
    # powers-of-two scalings of the same double sum: exact
    assert np.array_equal(r1 + r2, r3)
    r4, _, _ = oracle_mod.sgemm(A, B, None, -1.0, 0.0)
    r5, _, _ = oracle_mod.sgemm(A, B, None, 1.0, 0.0)
    assert np.array_equal(r4, -r5)


def test_padded_leading_dims(oracle_mod):
    rng = _rng(7)
    M, N, K = 19, 21, 13
    Ap, Bp, Cp = _rand(rng, (M, K + 5)), _rand(rng, (K, N + 3)), _rand(rng, (M, N + 9))
    ref_p, bnd_p, _ = oracle_mod.sgemm(Ap, Bp, Cp, 1.5, -0.5, M=M, N=N, K=K)
    A, B, C = (np.ascontiguousarray(Ap[:, :K]), np.ascontiguousarray(Bp[:, :N]),
               np.ascontiguousarray(Cp[:, :N]))
    ref, bnd, _ = oracle_mod.sgemm(A, B, C, 1.5, -0.5)
    assert np.array_equal(ref_p, ref) and np.array_equal(bnd_p, bnd)


def test_row_independence_and_threads(oracle_mod):
    """Rows are independent sums: any thread count gives identical bits."""
    rng = _rng(8)
    A, B, C = _rand(rng, (37, 50)), _rand(rng, (50, 29)), _rand(rng, (37, 29))
    r1, b1, _ = oracle_mod.sgemm(A, B, C, 1.0, 1.0, threads=1)
    r4, b4, _ = oracle_mod.sgemm(A, B, C, 1.0, 1.0, threads=4)
    assert np.array_equal(r1, r4) and np.array_equal(b1, b4)
    # a single row computed alone equals that row of the full product
    r_row, _, _ = oracle_mod.sgemm(A[5:6], B, C[5:6], 1.0, 1.0)
    assert np.array_equal(r_row[0], r1[5])


@pytest.mark.parametrize("transA,transB", [(False, False), (True, True)])
def test_entries_match_full(oracle_mod, transA, transB):
    rng = _rng(9)
    M, N, K = 33, 47, 29
    A = _rand(rng, (K, M) if transA else (M, K))
    B = _rand(rng, (N, K) if transB else (K, N))
    C = _rand(rng, (M, N))
    ref, bound, _ = oracle_mod.sgemm(A, B, C, -0.75, 1.25, transA=transA, transB=transB)
    rows = rng.integers(0, M, size=200)
    cols = rng.integers(0, N, size=200)
    er, eb, fmas = oracle_mod.sgemm_entries(A, B, C, -0.75, 1.25, rows, cols, transA=transA,
                                            transB=transB)
    assert fmas == 200 * K
    assert np.array_equal(er, ref[rows, cols]) and np.array_equal(eb, bound[rows, cols])


def test_violations_mask(oracle_mod):
    ref = np.array([1.0, 2.0, np.inf, np.nan])
    bound = np.array([0.1, 0.1, 0.1, 0.1])
    got = np.array([1.05, 2.2, np.inf, np.nan])
    assert oracle_mod.violations(got, ref, bound).tolist() == [False, True, False, False]
    assert oracle_mod.violations(np.array([np.nan]), np.array([1.0]), np.array([1.0])).tolist() == [True]
