"""The cluster-split plans (cs8_/cs16_): one CTA per (output tile, k slice),
the k slices of a tile in one thread-block cluster, their sums added through
distributed shared memory in slice order and the epilogue applied by the CTA
that adds them.  Every result against the oracle's FP32 bound, integer inputs
bit for bit, the fixed slice order bitwise-reproducible run to run, C untouched
outside its window."""
import numpy as np
import pytest

import oracle
from gpu_helpers import check, env, gemm

pytestmark = pytest.mark.gpu

CS_PLANS = ["cs8_64x128x16_s6_o2", "cs16_64x128x16_s6_o2"]


@pytest.fixture(scope="module")
def tb():
    return env()


# (M, N, K) with N and K multiples of 4 (the bulk-tensor operand class these
# plans take): one tile with 2..16 slices, ragged tiles on every side, K not
# a multiple of the 16-k stage, many tiles (few slices each), K too short to
# split (one slice: no cluster)
SHAPES = [(64, 128, 256), (60, 100, 1000), (130, 260, 512), (512, 512, 512), (200, 332, 96),
          (1000, 1020, 64), (33, 44, 20), (256, 256, 2048), (700, 900, 300)]


def test_cluster_split_refuses_other_operands(tb):
    """An odd leading dimension is outside these plans' operand class."""
    torch, b2g = tb
    A = np.zeros((130, 512), np.float32)
    B = np.zeros((512, 257), np.float32)
    C = np.zeros((130, 257), np.float32)
    for name in CS_PLANS:
        _, rc, _ = gemm(b2g, torch, A, B, C, 1.0, 0.0, plan=b2g.plans().index(name))
        assert rc == b2g.B2G_ERR_UNSUPPORTED


@pytest.mark.parametrize("plan_name", CS_PLANS)
@pytest.mark.parametrize("shape", SHAPES)
def test_cluster_split_within_bound(tb, plan_name, shape):
    torch, b2g = tb
    M, N, K = shape
    rng = np.random.default_rng(M * 5 + N * 3 + K)
    A = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
    C = rng.uniform(-1, 1, size=(M, N)).astype(np.float32)
    ref, bound, _ = oracle.sgemm(A, B, C, 0.75, -1.25)
    plan = b2g.plans().index(plan_name)
    got, rc, guard = gemm(b2g, torch, A, B, C, 0.75, -1.25, plan=plan)
    assert rc == 0, b2g.b2g_strerror(rc)
    assert guard, "wrote outside C's window"
    check(got, ref, bound, f"{plan_name} {shape}")


@pytest.mark.parametrize("plan_name", CS_PLANS)
def test_cluster_split_integers_exact(tb, plan_name):
    torch, b2g = tb
    rng = np.random.default_rng(21)
    M, N, K = 300, 260, 1000
    A = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    B = rng.integers(-3, 4, size=(K, N)).astype(np.float32)
    C = rng.integers(-3, 4, size=(M, N)).astype(np.float32)
    ref, _, _ = oracle.sgemm(A, B, C, 2.0, -1.0)
    got, rc, _ = gemm(b2g, torch, A, B, C, 2.0, -1.0, plan=b2g.plans().index(plan_name))
    assert rc == 0
    assert np.array_equal(got.astype(np.float64), ref)


@pytest.mark.parametrize("plan_name", CS_PLANS)
def test_cluster_split_beta_zero_does_not_read_c(tb, plan_name):
    torch, b2g = tb
    rng = np.random.default_rng(22)
    A = rng.uniform(-1, 1, size=(190, 512)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(512, 252)).astype(np.float32)
    C = np.full((190, 252), np.nan, np.float32)
    ref, bound, _ = oracle.sgemm(A, B, C, 1.0, 0.0)
    got, rc, _ = gemm(b2g, torch, A, B, C, 1.0, 0.0, plan=b2g.plans().index(plan_name))
    assert rc == 0 and np.isfinite(got).all()
    check(got, ref, bound, plan_name)


@pytest.mark.parametrize("plan_name", CS_PLANS)
def test_cluster_split_bitwise_reproducible(tb, plan_name):
    torch, b2g = tb
    M, N, K = 512, 512, 512
    rng = np.random.default_rng(23)
    A = torch.from_numpy(rng.uniform(-1, 1, size=(M, K)).astype(np.float32)).cuda()
    B = torch.from_numpy(rng.uniform(-1, 1, size=(K, N)).astype(np.float32)).cuda()
    C0 = torch.from_numpy(rng.uniform(-1, 1, size=(M, N)).astype(np.float32)).cuda()
    plan = b2g.plans().index(plan_name)
    outs = []
    for _ in range(3):
        C = C0.clone()
        b2g.sgemm(A, B, C, 1.0, 0.5, plan=plan)
        torch.cuda.synchronize()
        outs.append(C.view(torch.int32).cpu())
    assert all(torch.equal(outs[0], o) for o in outs[1:])


def test_cluster_split_one_launch(tb):
    """A cluster-split plan is one kernel launch: no reduction kernel."""
    _, b2g = tb
    for name in CS_PLANS:
        assert b2g.b2g_plan_name(b2g.plans().index(name)) == name
    # the table's choice for small aligned problems is checked in
    # test_abi_host; here the forced plan must need no workspace
    rc, need = b2g.b2g_sgemm_workspace_size(0, 0, 512, 512, 512, 1.0, 1 << 20, 512, 1 << 20, 512,
                                            1 << 20, 512)
    assert rc == 0
