"""Shapes whose split tail the balance model chooses instead of the plain rule
(every tile cut into k slices, or the tiles after the first rounds): every
output element against the oracle, small integers bit-exact, and run-to-run
bitwise reproducibility.  The split the host picks is read back through the
workspace size, so a change of the model shows up here."""
import numpy as np
import pytest

import oracle
from gpu_helpers import check, env, gemm

pytestmark = pytest.mark.gpu

FAKE = 1 << 20


@pytest.fixture(scope="module")
def tb():
    return env()


def _split_bytes(b2g, M, N, K):
    rc, need = b2g.b2g_sgemm_workspace_size(0, 0, M, N, K, 1.0, FAKE, K, FAKE, N, FAKE, N)
    assert rc == 0
    return need


# (M, N, K): every tile in slices (1152^3, 1664^3, 1100 x 1700 x 2000,
# 4096 x 640 x 4096) or the tiles after the first round (2560^3)
SHAPES = [(1152, 1152, 1152), (1664, 1664, 1664), (1100, 1700, 2000), (4096, 640, 4096),
          (2560, 2560, 2560)]


@pytest.mark.parametrize("shape", SHAPES)
def test_balanced_split_full_output(tb, shape):
    torch, b2g = tb
    M, N, K = shape
    rng = np.random.default_rng(M + 3 * N + 7 * K)
    A = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
    C = rng.uniform(-1, 1, size=(M, N)).astype(np.float32)
    ref, bound, _ = oracle.sgemm(A, B, C, 1.25, -0.75)
    name = b2g.b2g_plan_name(b2g.b2g_sgemm_select_plan(0, 0, M, N, K, 1.25, FAKE, K, FAKE, N,
                                                        FAKE, N))
    # the transposing plan's own workspace is A^T; anything more is the split
    at = K * ((M + 3) // 4 * 4) * 4
    need = _split_bytes(b2g, M, N, K)
    assert name.startswith("pre_") and need > at, (name, need, at)
    got, rc, guard = gemm(b2g, torch, A, B, C, 1.25, -0.75)
    assert rc == 0 and guard
    check(got, ref, bound, f"{shape} {name}")


def test_balanced_split_integers_exact_and_reproducible(tb):
    torch, b2g = tb
    M, N, K = 1664, 1664, 1664
    rng = np.random.default_rng(21)
    A = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    B = rng.integers(-3, 4, size=(K, N)).astype(np.float32)
    C = rng.integers(-3, 4, size=(M, N)).astype(np.float32)
    ref, _, _ = oracle.sgemm(A, B, C, 1.0, 2.0)
    got, rc, _ = gemm(b2g, torch, A, B, C, 1.0, 2.0)
    assert rc == 0 and np.array_equal(got.astype(np.float64), ref)
    Ar = torch.from_numpy(rng.uniform(-1, 1, size=(M, K)).astype(np.float32)).cuda()
    Br = torch.from_numpy(rng.uniform(-1, 1, size=(K, N)).astype(np.float32)).cuda()
    C0 = torch.from_numpy(rng.uniform(-1, 1, size=(M, N)).astype(np.float32)).cuda()
    outs = []
    for _ in range(3):
        Cc = C0.clone()
        b2g.sgemm(Ar, Br, Cc, 0.5, 0.5)
        torch.cuda.synchronize()
        outs.append(Cc.view(torch.int32).cpu())
    assert all(torch.equal(outs[0], o) for o in outs[1:])
