"""Calls chained on one stream with no host synchronisation in between.

Every kernel of the library is launched as a programmatic dependent of the
grid before it on the stream and waits for that grid before touching global
memory.  These tests pin the two orders that wait must keep: a call that reads
what the previous call wrote (read after write), and a call that overwrites an
operand the previous call is still reading (write after read).  Each chain
mixes plans with different kernel sequences (transpose + GEMM + split-tail
reduction, the cluster kernel for skinny M, packed operands, the 3xTF32
kernels), and every result is checked against the oracle computed in the same
order on the host.
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import check, env

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tb():
    return env()


def _dev(torch, x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def _ref(A, B, C, alpha, beta):
    ref, bound, _ = oracle.sgemm(np.ascontiguousarray(A), np.ascontiguousarray(B),
                                 None if C is None else np.ascontiguousarray(C), alpha, beta)
    return ref, bound


def test_read_after_write_chain(tb):
    """C1 = A B (1536^3, transpose-first plan with split tail); C2 = C1[:16] W
    (skinny cluster kernel reads C1's first rows); C3 = C1 V + C3 (odd shape,
    packed operands): each call starts while the previous may be draining."""
    torch, b2g = tb
    rng = np.random.default_rng(31)
    n = 1536
    A = rng.uniform(-1, 1, (n, n)).astype(np.float32)
    B = rng.uniform(-1, 1, (n, n)).astype(np.float32)
    W = rng.uniform(-1, 1, (n, 4096)).astype(np.float32)
    V = rng.uniform(-1, 1, (n, 1001)).astype(np.float32)
    C3 = rng.uniform(-1, 1, (n, 1001)).astype(np.float32)
    dA, dB, dW, dV, dC3 = (_dev(torch, x) for x in (A, B, W, V, C3))
    dC1 = torch.empty((n, n), device="cuda")
    dC2 = torch.zeros((16, 4096), device="cuda")
    b2g.sgemm(dA, dB, dC1, 1.0, 0.0)
    b2g.sgemm(dC1[:16], dW, dC2, 0.5, 0.0)
    b2g.sgemm(dC1, dV, dC3, 1.0, 1.0)
    torch.cuda.synchronize()
    got1 = dC1.cpu().numpy()
    ref1, bound1 = _ref(A, B, None, 1.0, 0.0)
    check(got1, ref1, bound1, "C1")
    # later calls are checked against the oracle on the GPU's C1 (its own
    # rounding is already within bound)
    ref2, bound2 = _ref(got1[:16], W, None, 0.5, 0.0)
    check(dC2.cpu().numpy(), ref2, bound2, "C2 = C1[:16] W")
    ref3, bound3 = _ref(got1, V, C3, 1.0, 1.0)
    check(dC3.cpu().numpy(), ref3, bound3, "C3 = C1 V + C3")


def test_skinny_reads_b_the_previous_kernel_writes(tb):
    """The skinny cluster kernel fetches its first stages of B into L2 before
    it waits for the previous grid.  Here that grid writes the very B it reads
    (a GEMM writes W2 = X Y; the skinny call reads W2), and then a second
    skinny call reads the first one's output as its B: both must see the
    finished values, not lines fetched while they were being written."""
    torch, b2g = tb
    rng = np.random.default_rng(34)
    X = rng.uniform(-1, 1, (1024, 256)).astype(np.float32)
    Y = rng.uniform(-1, 1, (256, 4096)).astype(np.float32)
    A16 = rng.uniform(-1, 1, (16, 1024)).astype(np.float32)
    A8 = rng.uniform(-1, 1, (8, 16)).astype(np.float32)
    dX, dY, dA16, dA8 = (_dev(torch, x) for x in (X, Y, A16, A8))
    dW2 = torch.full((1024, 4096), float("nan"), device="cuda")
    dC4 = torch.zeros((16, 4096), device="cuda")
    dC5 = torch.zeros((8, 4096), device="cuda")
    torch.cuda.synchronize()
    b2g.sgemm(dX, dY, dW2, 1.0, 0.0)     # writes B of the next call
    b2g.sgemm(dA16, dW2, dC4, 1.0, 0.0)  # skinny: B = W2
    b2g.sgemm(dA8, dC4, dC5, 1.0, 0.0)   # skinny (K = 16): B = the previous output
    torch.cuda.synchronize()
    got_w = dW2.cpu().numpy()
    refw, boundw = _ref(X, Y, None, 1.0, 0.0)
    check(got_w, refw, boundw, "W2 = X Y")
    got4 = dC4.cpu().numpy()
    ref4, bound4 = _ref(A16, got_w, None, 1.0, 0.0)
    check(got4, ref4, bound4, "C4 = A16 W2")
    ref5, bound5 = _ref(A8, got4, None, 1.0, 0.0)
    check(dC5.cpu().numpy(), ref5, bound5, "C5 = A8 C4")
    for name, (M, N, K) in {"C4": (16, 4096, 1024), "C5": (8, 4096, 16)}.items():
        plan = b2g.b2g_plan_name(b2g.b2g_sgemm_select_plan(0, 0, M, N, K, 1.0, 1 << 20, K,
                                                           1 << 20, N, 1 << 20, N))
        assert plan.startswith("skinnyT"), (name, plan)


def test_write_after_read_chain(tb):
    """Call 1 reads A and B; call 2 writes into A's and B's storage at once.
    Call 1's result must be the product of the original A and B."""
    torch, b2g = tb
    rng = np.random.default_rng(32)
    n = 2048
    A = rng.uniform(-1, 1, (n, n)).astype(np.float32)
    B = rng.uniform(-1, 1, (n, n)).astype(np.float32)
    X = rng.uniform(-1, 1, (n, 512)).astype(np.float32)
    Y = rng.uniform(-1, 1, (512, n)).astype(np.float32)
    dA, dB, dX, dY = (_dev(torch, x) for x in (A, B, X, Y))
    dC = torch.empty((n, n), device="cuda")
    b2g.sgemm(dA, dB, dC, 1.0, 0.0)          # reads A, B
    b2g.sgemm(dX, dY, dA, 1.0, 0.0)          # overwrites A
    b2g.sgemm_3xtf32(dX, dY, dB, 2.0, 0.0)   # overwrites B (tensor-core path)
    torch.cuda.synchronize()
    ref, bound = _ref(A, B, None, 1.0, 0.0)
    check(dC.cpu().numpy(), ref, bound, "C = A B before A and B were overwritten")
    refa, bounda = _ref(X, Y, None, 1.0, 0.0)
    check(dA.cpu().numpy(), refa, bounda, "A <- X Y")
    refb, boundb = _ref(X, Y, None, 2.0, 0.0)
    check(dB.cpu().numpy(), refb, boundb, "B <- 2 X Y (3xTF32)")


def test_long_chain_accumulates(tb):
    """Forty dependent calls C <- C W + C0 (alternating FFMA and 3xTF32),
    small enough that launch latency, not the GEMMs, sets the pace: each call
    must see the previous call's C."""
    torch, b2g = tb
    rng = np.random.default_rng(33)
    n = 256
    W = (rng.uniform(-1, 1, (n, n)) / n).astype(np.float32)
    C0 = rng.uniform(-1, 1, (n, n)).astype(np.float32)
    dW, dC0 = _dev(torch, W), _dev(torch, C0)
    dC = dC0.clone()
    tmp = torch.empty_like(dC)
    host = C0.astype(np.float64)
    for i in range(40):
        tmp.copy_(dC0)  # a torch kernel between our kernels (no dependent launch)
        if i % 2:
            b2g.sgemm_3xtf32(dC, dW, tmp, 1.0, 1.0)
        else:
            b2g.sgemm(dC, dW, tmp, 1.0, 1.0)
        dC, tmp = tmp, dC
        host = host @ W.astype(np.float64) + C0
    torch.cuda.synchronize()
    got = dC.cpu().numpy().astype(np.float64)
    # forty roundings of a contraction with |W| row sums <= 1: a loose but
    # order-revealing bound (a skipped or stale step is off by O(1))
    err = np.abs(got - host).max()
    assert err < 1e-3, err
