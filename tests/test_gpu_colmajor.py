"""Column-major operands through b2g_sgemm_colmajor.

"GEMM 优化之路" (完整代码) drives column-major cuBLAS with row-major data through
the identity C = AB <=> C^T = B^T A^T; the library offers the same identity
the other way round.  The oracle is handed the logical op(A), op(B) and C as
row-major copies, so it checks the operand swap independently of how the
library performs it.  The storage padding of C (rows ldc > M of every
column) must be bit-identical afterwards.
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import check, env

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tb():
    return env()


def colmajor(rng, rows, cols, ld):
    """Storage of a rows x cols column-major matrix with leading dimension ld:
    a (cols, ld) row-major array whose [:, :rows].T is the matrix."""
    return rng.uniform(-1, 1, size=(cols, ld)).astype(np.float32)


# (M, N, K, pad): leading dimensions are the stored row counts + pad
CASES = [
    (300, 260, 1000, 3),   # ragged tiles, split tail, odd leading dimensions
    (1000, 1025, 777, 0),  # ragged, K % 4 != 0
    (1024, 768, 512, 0),   # aligned: no-transpose column-major is the fast class
    (2048, 16, 1024, 0),   # N = 16 column-major is M = 16 row-major: the skinny plans
]


def run_colmajor(torch, b2g, tA, tB, M, N, K, pad, alpha, beta, seed):
    rng = np.random.default_rng(seed)
    ar, ac = (K, M) if tA else (M, K)  # stored shape of A
    br, bc = (N, K) if tB else (K, N)  # stored shape of B
    lda, ldb, ldc = ar + pad, br + pad, M + pad
    SA, SB, SC = colmajor(rng, ar, ac, lda), colmajor(rng, br, bc, ldb), colmajor(rng, M, N, ldc)
    A_st, B_st = SA[:, :ar].T, SB[:, :br].T
    opA = A_st.T if tA else A_st
    opB = B_st.T if tB else B_st
    ref, bound, _ = oracle.sgemm(np.ascontiguousarray(opA), np.ascontiguousarray(opB),
                                 np.ascontiguousarray(SC[:, :M].T), alpha, beta)
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (SA, SB, SC))
    s = torch.cuda.current_stream().cuda_stream
    rc = b2g.b2g_sgemm_colmajor(tA, tB, M, N, K, alpha, dA.data_ptr(), lda, dB.data_ptr(), ldb,
                                beta, dC.data_ptr(), ldc, s)
    torch.cuda.synchronize()
    assert rc == 0, b2g.b2g_strerror(rc)
    return SC, dC.cpu().numpy(), ref, bound, (dA, lda, dB, ldb, ldc)


@pytest.mark.parametrize("tB", [0, 1])
@pytest.mark.parametrize("tA", [0, 1])
@pytest.mark.parametrize("M,N,K,pad", CASES)
def test_colmajor_matches_oracle(tb, M, N, K, pad, tA, tB):
    torch, b2g = tb
    SC, out, ref, bound, _ = run_colmajor(torch, b2g, tA, tB, M, N, K, pad, 0.75, -1.5,
                                          seed=M * 7 + N * 3 + K + 10 * tA + 20 * tB)
    check(out[:, :M].T, ref, bound, f"column-major tA={tA} tB={tB} {M}x{N}x{K}")
    assert np.array_equal(out[:, M:].view(np.int32), SC[:, M:].view(np.int32))


@pytest.mark.parametrize("tA,tB", [(0, 0), (1, 1)])
def test_colmajor_is_the_swapped_row_major_call(tb, tA, tB):
    """Same plan, same kernels: bitwise the row-major call on the transposes."""
    torch, b2g = tb
    M, N, K = 700, 520, 900
    SC, out, _, _, (dA, lda, dB, ldb, ldc) = run_colmajor(torch, b2g, tA, tB, M, N, K, 1, 1.25,
                                                          0.5, seed=5)
    dC2 = torch.from_numpy(SC).cuda()
    s = torch.cuda.current_stream().cuda_stream
    rc = b2g.b2g_sgemm_ex(tB, tA, N, M, K, 1.25, dB.data_ptr(), ldb, dA.data_ptr(), lda, 0.5,
                          dC2.data_ptr(), ldc, s)
    torch.cuda.synchronize()
    assert rc == 0
    assert np.array_equal(out.view(np.int32), dC2.cpu().numpy().view(np.int32))


def test_tensor_level_colmajor(tb):
    """sgemm_colmajor on transposed views of contiguous tensors (unit row
    stride); a row-major tensor is refused."""
    torch, b2g = tb
    M, N, K = 513, 257, 300
    rng = np.random.default_rng(9)
    SA, SB, SC = colmajor(rng, M, K, M), colmajor(rng, K, N, K), colmajor(rng, M, N, M)
    ref, bound, _ = oracle.sgemm(np.ascontiguousarray(SA.T), np.ascontiguousarray(SB.T),
                                 np.ascontiguousarray(SC.T), 2.0, 0.25)
    A, B = torch.from_numpy(SA).cuda().t(), torch.from_numpy(SB).cuda().t()
    C = torch.from_numpy(SC).cuda().t()
    assert A.shape == (M, K) and A.stride() == (1, M)
    out = b2g.sgemm_colmajor(A, B, C, alpha=2.0, beta=0.25)
    torch.cuda.synchronize()
    check(out.cpu().numpy(), ref, bound, "tensor-level column-major")
    with pytest.raises(ValueError):
        b2g.sgemm_colmajor(A.contiguous(), B, C)
