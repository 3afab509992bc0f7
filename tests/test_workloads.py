"""The seeded input recipe: determinism, ranges, moments and the named shapes."""
import numpy as np

import workloads


def test_counter_based_and_deterministic():
    a = workloads.uniform_pm1(1, workloads.STREAM_A, 1000)
    b = workloads.uniform_pm1(1, workloads.STREAM_A, 1000)
    assert np.array_equal(a, b)
    # element i does not depend on how many were drawn
    assert np.array_equal(workloads.uniform_pm1(1, workloads.STREAM_A, 10), a[:10])
    bits = workloads.raw_bits(1, workloads.STREAM_A, 500, 20)
    assert np.array_equal(bits, workloads.raw_bits(1, workloads.STREAM_A, 0, 520)[500:])
    # streams and seeds differ
    assert not np.array_equal(a, workloads.uniform_pm1(1, workloads.STREAM_B, 1000))
    assert not np.array_equal(a, workloads.uniform_pm1(2, workloads.STREAM_A, 1000))


def test_splitmix_reference_value():
    # SplitMix64 finaliser of 0x9E3779B97F4A7C15 (first output of splitmix64 seeded 0)
    z = workloads._mix64(np.array([0x9E3779B97F4A7C15], dtype=np.uint64))[0]
    assert int(z) == 0xE220A8397B1DCDAF


def test_uniform_range_and_moments():
    u = workloads.uniform_pm1(3, workloads.STREAM_B, 1 << 20)
    assert u.dtype == np.float32 and u.min() >= -1.0 and u.max() < 1.0
    assert abs(u.mean()) < 5e-3 and abs(u.var() - 1.0 / 3.0) < 5e-3
    # exact multiples of 2**-23
    assert np.array_equal(u.astype(np.float64) * 2 ** 23, np.round(u.astype(np.float64) * 2 ** 23))


def test_normal_moments():
    z = workloads.normal(2, workloads.STREAM_A, 1 << 20 | 1, 0.0, 1.0)
    assert z.shape == ((1 << 20) + 1,) and np.isfinite(z).all()
    assert abs(z.mean()) < 5e-3 and abs(z.std() - 1.0) < 5e-3
    s = workloads.normal(4, workloads.STREAM_A, 1 << 18, 0.0, 0.02)
    assert abs(s.std() - 0.02) < 5e-4


def test_named_workloads():
    w = workloads.WORKLOADS
    h = w[workloads.HEADLINE]
    assert (h.M, h.N, h.K, h.alpha, h.beta, h.seed) == (4096, 4096, 4096, 1.0, 0.5, 1)
    r = w["ragged1000x1025x777"]
    assert r.lds == (777, 1025, 1025) and (r.alpha, r.beta) == (0.75, -1.25)
    A, B, C = r.make()
    assert A.shape == (1000, 777) and B.shape == (777, 1025) and C.shape == (1000, 1025)
    s = w["square512"]
    A, B, C = s.make()
    assert not C.any() and s.beta == 0.0
    sk = w["skinny16x4096x4096"]
    assert (sk.M, sk.N, sk.K, sk.beta) == (16, 4096, 4096, 1.0)
    assert sk.min_bytes() == 4.0 * (16 * 4096 + 4096 * 4096 + 2 * 16 * 4096)
    for n in workloads.SWEEP_SIZES:
        assert w[f"sweep{n}"].flops() == 2.0 * n ** 3
