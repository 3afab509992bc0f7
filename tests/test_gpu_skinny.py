"""Skinny M (M <= 32): the split-K plans (B from global memory, skinny_m*, and
B and A in bulk-tensor stages, skinnyT_m*) against the oracle, with the
partial sums in a workspace (split) and without one (one CTA per column slab)."""
import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import check, env, gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tb():
    return env()


SHAPES = [(1, 4, 4), (16, 4096, 4096), (7, 132, 100), (16, 128, 64), (17, 260, 1000),
          (32, 512, 4096), (3, 1000, 2052), (31, 4, 516)]


@pytest.mark.parametrize("shape", SHAPES)
def test_skinny_plans(tb, shape):
    torch, b2g = tb
    M, N, K = shape
    rng = np.random.default_rng(M * 13 + N + K)
    A = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
    C = rng.uniform(-1, 1, size=(M, N)).astype(np.float32)
    ref, bound, _ = oracle.sgemm(A, B, C, 0.5, 2.0)
    names = b2g.plans()
    ran = 0
    for name in [n for n in names if n.startswith("skinny")]:
        got, rc, guard = gemm(b2g, torch, A, B, C, 0.5, 2.0, plan=names.index(name))
        if rc == b2g.B2G_ERR_UNSUPPORTED:
            assert M > int(name.split("_m")[1])
            continue
        assert rc == 0 and guard, name
        check(got, ref, bound, f"{name} {shape}")
        ran += 1
    assert ran >= 1


def test_unsplit_without_workspace_matches(tb):
    """b2g_sgemm_ws with no workspace runs the skinny plan unsplit."""
    torch, b2g = tb
    M, N, K = 16, 1024, 2048
    rng = np.random.default_rng(3)
    A = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
    C = rng.uniform(-1, 1, size=(M, N)).astype(np.float32)
    ref, bound, _ = oracle.sgemm(A, B, C, 1.0, -1.0)
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (A, B, C))
    s = torch.cuda.current_stream().cuda_stream
    rc = b2g.b2g_sgemm_ws(0, 0, M, N, K, 1.0, dA.data_ptr(), K, dB.data_ptr(), N, -1.0,
                          dC.data_ptr(), N, None, 0, s)
    assert rc == 0
    torch.cuda.synchronize()
    check(dC.cpu().numpy(), ref, bound, "unsplit")


def test_padded_lds_and_unaligned_c(tb):
    torch, b2g = tb
    M, N, K = 20, 256, 512
    rng = np.random.default_rng(4)
    A = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
    C = rng.uniform(-1, 1, size=(M, N)).astype(np.float32)
    ref, bound, _ = oracle.sgemm(A, B, C, 1.0, 0.25)
    for lds, mis in [((K + 4, N + 8, N + 3), (0, 0, 0)), ((K, N, N), (0, 0, 1))]:
        got, rc, guard = gemm(b2g, torch, A, B, C, 1.0, 0.25, lds=lds, misalign=mis)
        assert rc == 0 and guard, (lds, mis)
        check(got, ref, bound, f"lds {lds} misalign {mis}")


def test_integers_bit_exact(tb):
    torch, b2g = tb
    M, N, K = 16, 512, 3000
    rng = np.random.default_rng(6)
    A = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    B = rng.integers(-3, 4, size=(K, N)).astype(np.float32)
    C = rng.integers(-3, 4, size=(M, N)).astype(np.float32)
    ref, _, _ = oracle.sgemm(A, B, C, 2.0, -1.0)
    K4 = (K + 3) // 4 * 4
    got, rc, _ = gemm(b2g, torch, A, B, C, 2.0, -1.0, lds=(K4, N, N))
    assert rc == 0
    assert np.array_equal(got.astype(np.float64), ref)


def test_skinny_workload_is_table_plan(tb):
    torch, b2g = tb
    w = workloads.WORKLOADS["skinny16x4096x4096"]
    assert b2g.b2g_plan_name(b2g.b2g_sgemm_select_plan(
        0, 0, w.M, w.N, w.K, w.alpha, 1 << 20, w.K, 1 << 20, w.N, 1 << 20, w.N)).startswith(
            "skinny")
