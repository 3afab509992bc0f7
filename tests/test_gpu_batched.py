"""Strided-batched SGEMM: every problem of the batch against the oracle,
across the plan families the tune table reaches (k-chunked, pre-transposed,
packed, B^T transposed first, skinny split-K) and with padded strides and op()
flags."""
import numpy as np
import pytest

import oracle
from gpu_helpers import check, env

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tb():
    return env()


def run_batched(torch, b2g, As, Bs, Cs, alpha, beta, transA=False, transB=False, pad=0):
    """Pack the per-problem host matrices into one device buffer each, `pad`
    extra elements between consecutive problems; returns the results."""
    batch = len(As)

    def stack(mats):
        rows, cols = mats[0].shape
        stride = rows * cols + pad
        buf = torch.full((batch * stride + 1,), float("nan"), device="cuda")
        for b, m in enumerate(mats):
            buf[b * stride:b * stride + rows * cols].copy_(torch.from_numpy(m.ravel()))
        return buf, stride, cols

    dA, sA, lda = stack(As)
    dB, sB, ldb = stack(Bs)
    dC, sC, ldc = stack(Cs)
    M = As[0].shape[1] if transA else As[0].shape[0]
    K = As[0].shape[0] if transA else As[0].shape[1]
    N = Bs[0].shape[0] if transB else Bs[0].shape[1]
    rc = b2g.b2g_sgemm_strided_batched(int(transA), int(transB), M, N, K, alpha, dA.data_ptr(),
                                       lda, sA, dB.data_ptr(), ldb, sB, beta, dC.data_ptr(), ldc,
                                       sC, batch, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    out = dC.cpu().numpy()
    return rc, [out[b * sC:b * sC + M * N].reshape(M, N) for b in range(batch)], out, sC


CASES = [
    # (M, N, K, batch, transA, transB, pad)
    (130, 257, 68, 3, False, False, 0),
    (256, 256, 64, 4, False, False, 0),
    (256, 256, 64, 3, False, False, 4),
    (200, 160, 96, 2, True, False, 0),
    (200, 160, 96, 2, False, True, 0),
    (16, 512, 256, 5, False, False, 0),     # skinny split-K
    (1024, 1024, 2048, 2, False, False, 0),  # pre-transposed A (workspace x batch)
    (1000, 1025, 777, 2, False, False, 0),   # packed operands
    (400, 384, 512, 3, False, True, 0),      # op(B) = B^T: B^T and A transposed first
    (400, 384, 512, 3, True, True, 4),       # the same with A stored K x M, padded strides
    (64, 64, 64, 1, False, False, 0),
]


@pytest.mark.parametrize("case", CASES)
def test_batched_matches_oracle(tb, case):
    torch, b2g = tb
    M, N, K, batch, tA, tB, pad = case
    rng = np.random.default_rng(M + N + K + batch)
    As = [rng.uniform(-1, 1, size=(K, M) if tA else (M, K)).astype(np.float32) for _ in range(batch)]
    Bs = [rng.uniform(-1, 1, size=(N, K) if tB else (K, N)).astype(np.float32) for _ in range(batch)]
    Cs = [rng.uniform(-1, 1, size=(M, N)).astype(np.float32) for _ in range(batch)]
    rc, outs, flat, sC = run_batched(torch, b2g, As, Bs, Cs, 0.75, -0.5, tA, tB, pad)
    assert rc == 0, b2g.b2g_strerror(rc)
    for b in range(batch):
        ref, bound, _ = oracle.sgemm(As[b], Bs[b], Cs[b], 0.75, -0.5, transA=tA, transB=tB)
        check(outs[b], ref, bound, f"{case} problem {b}")
    if pad:  # the gaps between problems are untouched
        for b in range(batch):
            gap = flat[b * sC + M * N:(b + 1) * sC]
            assert np.isnan(gap).all()


def test_batch_zero_and_invalid(tb):
    torch, b2g = tb
    C = torch.full((4, 4), 5.0, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    p = C.data_ptr()
    assert b2g.b2g_sgemm_strided_batched(0, 0, 4, 4, 4, 1.0, p, 4, 16, p, 4, 16, 0.0, p, 4, 16, 0,
                                         s) == 0
    assert b2g.b2g_sgemm_strided_batched(0, 0, 4, 4, 4, 1.0, p, 4, 16, p, 4, 16, 0.0, p, 4, 16, -1,
                                         s) == b2g.B2G_ERR_INVALID_DIM
    assert b2g.b2g_sgemm_strided_batched(0, 0, 4, 4, 4, 1.0, p, 4, -16, p, 4, 16, 0.0, p, 4, 16, 2,
                                         s) == b2g.B2G_ERR_INVALID_LD
    torch.cuda.synchronize()
    assert bool((C == 5.0).all())


def test_tensor_api(tb):
    torch, b2g = tb
    rng = np.random.default_rng(11)
    A = rng.uniform(-1, 1, size=(3, 70, 40)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(3, 40, 90)).astype(np.float32)
    C = np.zeros((3, 70, 90), np.float32)
    dC = torch.from_numpy(C).cuda()
    b2g.sgemm_batched(torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda(), dC, 1.0, 0.0)
    got = dC.cpu().numpy()
    for b in range(3):
        ref, bound, _ = oracle.sgemm(A[b], B[b], None, 1.0, 0.0)
        check(got[b], ref, bound, f"tensor api {b}")


@pytest.mark.parametrize("M,N,K", [(16, 16, 16), (17, 19, 13)])
def test_batch_past_grid_z_limit(tb, M, N, K):
    """70000 problems (more than the 65535 a grid's z extent holds): the plans
    that put the batch in z refuse, the table's choice walks the batch in its
    tile scheduler.  Sampled problems, both sides of 65535, against the oracle."""
    torch, b2g = tb
    batch = 70000
    rng = np.random.default_rng(M * N * K)
    A = rng.uniform(-1, 1, (batch, M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, (batch, K, N)).astype(np.float32)
    C = rng.uniform(-1, 1, (batch, M, N)).astype(np.float32)
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (A, B, C))
    rc = b2g.b2g_sgemm_strided_batched(0, 0, M, N, K, 0.5, dA.data_ptr(), K, M * K, dB.data_ptr(),
                                       N, K * N, 2.0, dC.data_ptr(), N, M * N, batch,
                                       torch.cuda.current_stream().cuda_stream)
    assert rc == 0, b2g.b2g_strerror(rc)
    torch.cuda.synchronize()
    out = dC.cpu().numpy()
    picks = sorted(set([0, 1, 65534, 65535, 65536, 65537, batch - 1] +
                       list(rng.integers(0, batch, 40))))
    for b in picks:
        ref, bound, _ = oracle.sgemm(A[b], B[b], C[b], 0.5, 2.0)
        check(out[b], ref, bound, f"problem {b} of {batch}")
