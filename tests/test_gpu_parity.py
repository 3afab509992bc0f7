"""GPU parity: the CUDA library through its C ABI against the CPU oracle, element
by element, within the FP32 bound
    |C_gpu - C_ref| <= 2*K*2^-24*(|alpha|*(|A||B|)_ij + |beta*C_ij|) + 1e-6
(the standard forward-error bound of a K-term FP32 dot product plus the
epilogue's roundings; the optimisation guide on gsyq.cn, section 6.1, notes
that summation order makes exact equality the wrong test, and this bound
allows every order).  Integer-valued inputs whose sums are exact in FP32 must
match bit for bit.
"""
import numpy as np
import pytest

import oracle
import workloads
from gpu_helpers import check, env, gemm, workload_reference

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tb():
    return env()


FULL = ["square512", "ragged1000x1025x777", "sweep128", "sweep256", "sweep512", "sweep1024",
        "skinny16x4096x4096"]
FULL_SIZE = ["square4096", "sweep2048", "sweep4096", "sweep8192", "mlp8192x11008x4096"]


@pytest.mark.parametrize("name", FULL)
def test_workload_full(tb, name):
    torch, b2g = tb
    w = workloads.WORKLOADS[name]
    A, B, C = w.make()
    ref, bound, _ = oracle.sgemm(A, B, C, w.alpha, w.beta, M=w.M, N=w.N, K=w.K)
    got, rc, guard = gemm(b2g, torch, A, B, C, w.alpha, w.beta, lds=w.lds)
    assert rc == 0, b2g.b2g_strerror(rc)
    assert guard, "wrote outside C's M x N window"
    check(got, ref, bound, name)


@pytest.mark.parametrize("name", FULL_SIZE)
def test_workload_full_size(tb, name):
    """The large workloads in the launch configuration the bench times (the
    tune table's plan with its transpose and split tail, device-resident
    contiguous operands), every output element against the oracle."""
    torch, b2g = tb
    w, A, B, C, ref, bound = workload_reference(name)
    dA = torch.from_numpy(A).cuda()
    dB = torch.from_numpy(B).cuda()
    dC = torch.from_numpy(C).cuda()
    b2g.sgemm(dA, dB, dC, w.alpha, w.beta)
    torch.cuda.synchronize()
    check(dC.cpu().numpy(), ref, bound, name)


SHAPES = [(1, 1, 4), (1, 37, 8), (37, 1, 12), (5, 7, 3), (37, 45, 52), (130, 257, 68),
          (129, 128, 20), (256, 256, 16), (200, 333, 100)]


def _plans(b2g):
    return list(range(b2g.b2g_plan_count()))


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("trans", [(False, False), (True, False), (False, True), (True, True)])
def test_every_plan_ragged(tb, shape, trans):
    """Every compiled plan on shapes spanning several tiles with ragged tails;
    plans that cannot take the operands must say so (B2G_ERR_UNSUPPORTED)."""
    torch, b2g = tb
    M, N, K = shape
    transA, transB = trans
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    A = rng.uniform(-1, 1, size=(K, M) if transA else (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(N, K) if transB else (K, N)).astype(np.float32)
    C = rng.uniform(-1, 1, size=(M, N)).astype(np.float32)
    ref, bound, _ = oracle.sgemm(A, B, C, 0.75, -1.25, transA=transA, transB=transB)
    ran = 0
    for plan in [None] + _plans(b2g):
        got, rc, guard = gemm(b2g, torch, A, B, C, 0.75, -1.25, transA, transB, plan=plan)
        if rc == b2g.B2G_ERR_UNSUPPORTED:
            continue
        assert rc == 0, (plan, b2g.b2g_strerror(rc))
        assert guard, f"plan {plan} wrote outside C"
        check(got, ref, bound, f"plan {plan} {shape} {trans}")
        ran += 1
    assert ran >= 2


@pytest.mark.parametrize("K", [4, 64, 1000])
def test_small_integers_bit_exact(tb, K):
    """Entries in {-3..3} with |partial sums| < 2^24: every FP32 operation is
    exact, so every plan must reproduce the oracle bit for bit."""
    torch, b2g = tb
    rng = np.random.default_rng(K)
    M, N = 150, 140
    A = rng.integers(-3, 4, size=(M, K)).astype(np.float32)
    B = rng.integers(-3, 4, size=(K, N)).astype(np.float32)
    C = rng.integers(-3, 4, size=(M, N)).astype(np.float32)
    ref, _, _ = oracle.sgemm(A, B, C, 2.0, -1.0)
    for plan in [None] + _plans(b2g):
        got, rc, _ = gemm(b2g, torch, A, B, C, 2.0, -1.0, plan=plan)
        if rc == b2g.B2G_ERR_UNSUPPORTED:
            continue
        assert rc == 0
        assert np.array_equal(got.astype(np.float64), ref), f"plan {plan}"


def test_beta_zero_does_not_read_c(tb):
    torch, b2g = tb
    rng = np.random.default_rng(1)
    A = rng.uniform(-1, 1, size=(96, 64)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(64, 80)).astype(np.float32)
    C = np.full((96, 80), np.nan, np.float32)
    ref, bound, _ = oracle.sgemm(A, B, C, 1.0, 0.0)
    for plan in [None] + _plans(b2g):
        got, rc, _ = gemm(b2g, torch, A, B, C, 1.0, 0.0, plan=plan)
        if rc == b2g.B2G_ERR_UNSUPPORTED:
            continue
        assert np.isfinite(got).all(), f"plan {plan} read C"
        check(got, ref, bound, f"plan {plan}")


@pytest.mark.parametrize("alpha,K", [(0.0, 64), (1.5, 0)])
def test_product_term_vanishes(tb, alpha, K):
    """alpha == 0 or K == 0: C = beta*C, A and B not read (here they are NaN)."""
    torch, b2g = tb
    rng = np.random.default_rng(2)
    A = np.full((33, K), np.nan, np.float32)
    B = np.full((K, 65), np.nan, np.float32)
    C = rng.uniform(-1, 1, size=(33, 65)).astype(np.float32)
    for beta in (0.0, -0.5):
        got, rc, guard = gemm(b2g, torch, A, B, C, alpha, beta, lds=(max(K, 1), 65, 65))
        assert rc == 0 and guard
        assert np.array_equal(got, (np.float32(beta) * C) if beta else np.zeros_like(C))


def test_padded_leading_dims_and_guards(tb):
    torch, b2g = tb
    rng = np.random.default_rng(3)
    M, N, K = 150, 131, 75
    A = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
    C = rng.uniform(-1, 1, size=(M, N)).astype(np.float32)
    ref, bound, _ = oracle.sgemm(A, B, C, -1.0, 2.0)
    for lds in [(80, 136, 136), (K + 1, N + 3, N + 5), (128, 256, 132)]:
        got, rc, guard = gemm(b2g, torch, A, B, C, -1.0, 2.0, lds=lds)
        assert rc == 0 and guard, lds
        check(got, ref, bound, f"lds {lds}")


@pytest.mark.parametrize("mis", [(1, 0, 0), (0, 1, 0), (0, 0, 1), (3, 2, 1)])
def test_misaligned_operands(tb, mis):
    """Base pointers off the 16-byte grid take the 4-byte feed and stay exact."""
    torch, b2g = tb
    rng = np.random.default_rng(4)
    M, N, K = 140, 136, 64
    A = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
    C = rng.uniform(-1, 1, size=(M, N)).astype(np.float32)
    ref, bound, _ = oracle.sgemm(A, B, C, 1.0, 1.0)
    got, rc, guard = gemm(b2g, torch, A, B, C, 1.0, 1.0, misalign=mis)
    assert rc == 0 and guard
    check(got, ref, bound, f"misalign {mis}")


def test_ieee_denormals_not_flushed(tb):
    """2^-70 * 2^-70 = 2^-140 is an FP32 subnormal; a flush-to-zero build would
    return 0."""
    torch, b2g = tb
    A = np.full((64, 4), 2.0 ** -70, np.float32)
    B = np.zeros((4, 64), np.float32)
    B[0, :] = 2.0 ** -70
    C = np.zeros((64, 64), np.float32)
    for plan in [None] + _plans(b2g):
        got, rc, _ = gemm(b2g, torch, A, B, C, 1.0, 0.0, plan=plan)
        if rc == b2g.B2G_ERR_UNSUPPORTED:
            continue
        assert (got == np.float32(2.0 ** -140)).all(), f"plan {plan}"


def test_nonfinite_inputs_propagate(tb):
    torch, b2g = tb
    rng = np.random.default_rng(5)
    A = rng.uniform(-1, 1, size=(130, 40)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(40, 140)).astype(np.float32)
    A[7, 3] = np.inf
    A[100, 0] = np.nan
    C = np.zeros((130, 140), np.float32)
    ref, bound, _ = oracle.sgemm(A, B, C, 1.0, 0.0)
    got, rc, _ = gemm(b2g, torch, A, B, C, 1.0, 0.0)
    assert rc == 0
    check(got, ref, bound, "nonfinite")
    assert np.isnan(got[100]).all()


def test_bitwise_deterministic(tb):
    torch, b2g = tb
    w = workloads.WORKLOADS["square512"]
    A, B, C = w.make()
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    outs = []
    for _ in range(3):
        dC = torch.from_numpy(C).cuda()
        b2g.sgemm(dA, dB, dC, 1.0, 0.5)
        outs.append(dC.cpu())
    assert torch.equal(outs[0].view(torch.int32), outs[1].view(torch.int32))
    assert torch.equal(outs[0].view(torch.int32), outs[2].view(torch.int32))


def test_side_stream_ordering(tb):
    """A call on a non-default stream is ordered after that stream's copies."""
    torch, b2g = tb
    rng = np.random.default_rng(6)
    A = rng.uniform(-1, 1, size=(256, 128)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(128, 256)).astype(np.float32)
    ref, bound, _ = oracle.sgemm(A, B, None, 1.0, 0.0)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        dA = torch.from_numpy(A).pin_memory().cuda(non_blocking=True)
        dB = torch.from_numpy(B).pin_memory().cuda(non_blocking=True)
        dC = torch.empty(256, 256, device="cuda")
        b2g.sgemm(dA, dB, dC, 1.0, 0.0)
        out = dC.cpu()
    check(out.numpy(), ref, bound, "side stream")


def test_status_word_clean(tb):
    torch, b2g = tb
    rc, flags = b2g.b2g_status(torch.cuda.current_stream().cuda_stream)
    assert rc == 0 and flags == 0


@pytest.mark.parametrize("trans", [(False, True), (True, True), (True, False)])
def test_square4096_transposed_operands_full(tb, trans):
    """The headline product with A and/or B handed over transposed (A stored
    K x M, B stored N x K): the same result, every element against the oracle.
    op(B) = B^T takes the plan that transposes B^T (and A) with 16-byte
    vectors before the GEMM."""
    torch, b2g = tb
    transA, transB = trans
    w, A, B, C, ref, bound = workload_reference("square4096")
    dA = torch.from_numpy(np.ascontiguousarray(A.T) if transA else A).cuda()
    dB = torch.from_numpy(np.ascontiguousarray(B.T) if transB else B).cuda()
    dC = torch.from_numpy(C).cuda()
    plan = b2g.b2g_plan_name(b2g.b2g_sgemm_select_plan(
        int(transA), int(transB), w.M, w.N, w.K, w.alpha, dA.data_ptr(), dA.stride(0),
        dB.data_ptr(), dB.stride(0), dC.data_ptr(), w.N))
    assert plan.startswith("pret_" if transB else "tmaT_"), plan
    b2g.sgemm(dA, dB, dC, w.alpha, w.beta, transA=transA, transB=transB)
    torch.cuda.synchronize()
    check(dC.cpu().numpy(), ref, bound, f"square4096 trans {trans}")


@pytest.mark.parametrize("shape", [(600, 520, 1024), (1000, 1028, 776), (64, 4096, 512),
                                   (1100, 1028, 1024)])
@pytest.mark.parametrize("transA", [False, True])
def test_transposed_b_plans(tb, shape, transA):
    """op(B) = B^T on aligned operands above 5e7 multiply-adds: B^T (and A)
    transposed first, then the one-launch wkR_ plans below about 1e9
    multiply-adds or the pret_ plans (both tile shapes, split tail included)."""
    torch, b2g = tb
    M, N, K = shape
    rng = np.random.default_rng(M + N + K + transA)
    A = rng.uniform(-1, 1, size=(K, M) if transA else (M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(N, K)).astype(np.float32)
    C = rng.uniform(-1, 1, size=(M, N)).astype(np.float32)
    ref, bound, _ = oracle.sgemm(A, B, C, 0.5, 1.5, transA=transA, transB=True)
    plan = b2g.b2g_plan_name(b2g.b2g_sgemm_select_plan(int(transA), 1, M, N, K, 0.5, 1 << 20,
                                                        A.shape[1], 1 << 20, K, 1 << 20, N))
    assert plan.startswith("pret_" if M * N * K >= 1.0e9 else ("pret_", "wkR_")), plan
    got, rc, guard = gemm(b2g, torch, A, B, C, 0.5, 1.5, transA, True)
    assert rc == 0 and guard
    check(got, ref, bound, f"{shape} transA={transA} {plan}")
