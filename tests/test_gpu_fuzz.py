"""Seeded random cases through the public entry points, each checked against
the oracle element by element.

The cases mix what the fixed-shape tests take one at a time: sizes from 1 to
several hundred (skinny M with N past the cluster plan's threshold, and long
K, mixed in), op() flags, leading dimensions padded past the operand widths,
base pointers one float off 16-byte alignment, alpha and beta including 0 (C
is filled with NaN when beta is 0: it must not be read), and strided batches
whose strides leave gaps.  Every single-product case also checks that no
float outside C's M x N window changed.  The seeds are fixed, so a failure
names a reproducible case.
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import check, env, gemm

pytestmark = pytest.mark.gpu

ALPHAS = (1.0, -0.5, 0.0, 2.5)
BETAS = (0.0, 1.0, -1.25)


@pytest.fixture(scope="module")
def tb():
    return env()


def _sizes(rng):
    kind = int(rng.integers(0, 4))
    if kind == 0:  # skinny M, N around the cluster plan's 2048-column threshold
        return (int(rng.integers(1, 33)), int(rng.choice([4, 132, 1028, 2048, 2052])),
                int(rng.integers(1, 3000)))
    if kind == 1:  # long K on a small output
        return int(rng.integers(1, 200)), int(rng.integers(1, 200)), int(rng.integers(1000, 5000))
    m, n, k = np.exp(rng.uniform(0.0, np.log(700.0), 3)).astype(int) + 1
    return int(m), int(n), int(k)


def _stored(rng, rows, cols):
    return rng.standard_normal((rows, cols)).astype(np.float32)


@pytest.mark.parametrize("seed", range(96))
def test_random_case(tb, seed):
    torch, b2g = tb
    rng = np.random.default_rng(1000 + seed)
    M, N, K = _sizes(rng)
    transA, transB = bool(rng.integers(0, 2)), bool(rng.integers(0, 2))
    A = _stored(rng, *((K, M) if transA else (M, K)))
    B = _stored(rng, *((N, K) if transB else (K, N)))
    alpha = float(rng.choice(ALPHAS))
    beta = float(rng.choice(BETAS))
    C = _stored(rng, M, N)
    if beta == 0.0:
        C[:] = np.nan
    pads = rng.choice([0, 0, 1, 3, 4], size=3)
    lds = (A.shape[1] + int(pads[0]), B.shape[1] + int(pads[1]), N + int(pads[2]))
    mis = tuple(int(x) for x in rng.choice([0, 0, 1], size=3))
    what = (f"seed {seed}: {M}x{N}x{K} transA={transA} transB={transB} alpha={alpha} "
            f"beta={beta} lds={lds} misalign={mis}")
    got, rc, guard = gemm(b2g, torch, A, B, C, alpha, beta, transA=transA, transB=transB,
                          lds=lds, misalign=mis)
    assert rc == 0, f"{what}: {b2g.b2g_strerror(rc)}"
    assert guard, f"{what}: a float outside C's window changed"
    ref, bound, _ = oracle.sgemm(A, B, C, alpha, beta, transA=transA, transB=transB)
    check(got, ref, bound, what)


@pytest.mark.parametrize("seed", range(24))
def test_random_strided_batch(tb, seed):
    torch, b2g = tb
    rng = np.random.default_rng(2000 + seed)
    batch = int(rng.integers(2, 6))
    M, N, K = (int(x) for x in rng.integers(1, 300, size=3))
    transA, transB = bool(rng.integers(0, 2)), bool(rng.integers(0, 2))
    ra, ca = (K, M) if transA else (M, K)
    rb, cb = (N, K) if transB else (K, N)
    lda, ldb, ldc = (c + int(rng.choice([0, 0, 2, 4])) for c in (ca, cb, N))
    sA, sB, sC = (r * ld + int(rng.choice([0, 4, 7])) for r, ld in ((ra, lda), (rb, ldb), (M, ldc)))
    alpha = float(rng.choice(ALPHAS))
    beta = float(rng.choice(BETAS))
    As = [_stored(rng, ra, ca) for _ in range(batch)]
    Bs = [_stored(rng, rb, cb) for _ in range(batch)]
    Cs = [_stored(rng, M, N) for _ in range(batch)]

    def flat(mats, ld, stride):
        buf = np.full(batch * stride, np.nan, np.float32)
        for b, x in enumerate(mats):
            for r in range(x.shape[0]):
                buf[b * stride + r * ld:b * stride + r * ld + x.shape[1]] = x[r]
        return torch.from_numpy(buf).cuda()

    dA, dB, dC = flat(As, lda, sA), flat(Bs, ldb, sB), flat(Cs, ldc, sC)
    before = dC.clone()
    s = torch.cuda.current_stream().cuda_stream
    rc = b2g.b2g_sgemm_strided_batched(int(transA), int(transB), M, N, K, alpha, dA.data_ptr(),
                                       lda, sA, dB.data_ptr(), ldb, sB, beta, dC.data_ptr(), ldc,
                                       sC, batch, s)
    what = (f"seed {seed}: batch {batch} of {M}x{N}x{K} transA={transA} transB={transB} "
            f"alpha={alpha} beta={beta} lds=({lda},{ldb},{ldc}) strides=({sA},{sB},{sC})")
    assert rc == 0, f"{what}: {b2g.b2g_strerror(rc)}"
    torch.cuda.synchronize()
    out = dC.cpu().numpy()
    keep = np.ones(out.size, bool)
    for b in range(batch):
        got = np.stack([out[b * sC + r * ldc:b * sC + r * ldc + N] for r in range(M)])
        for r in range(M):
            keep[b * sC + r * ldc:b * sC + r * ldc + N] = False
        ref, bound, _ = oracle.sgemm(As[b], Bs[b], Cs[b], alpha, beta, transA=transA,
                                     transB=transB)
        check(got, ref, bound, f"{what}, problem {b}")
    prev = before.cpu().numpy()
    assert np.array_equal(out[keep].view(np.uint32), prev[keep].view(np.uint32)), \
        f"{what}: a float outside the C windows changed"


@pytest.mark.parametrize("seed", range(24))
def test_random_tf32x3(tb, seed):
    """The 3xTF32 path (every kernel variant) on random ragged shapes: row-major
    operands with K and lda multiples of 4, its documented domain."""
    torch, b2g = tb
    rng = np.random.default_rng(3000 + seed)
    M, N = (int(x) for x in rng.integers(1, 700, size=2))
    K = 4 * int(rng.integers(1, 400))
    variant = seed % 3
    lda = K + 4 * int(rng.integers(0, 3))
    ldb, ldc = N + int(rng.integers(0, 5)), N + int(rng.integers(0, 5))
    alpha = float(rng.choice(ALPHAS))
    beta = float(rng.choice(BETAS))
    A, B, C = _stored(rng, M, K), _stored(rng, K, N), _stored(rng, M, N)
    dA = torch.full((M, lda), float("nan"), device="cuda")
    dA[:, :K] = torch.from_numpy(A).cuda()
    dB = torch.full((K, ldb), float("nan"), device="cuda")
    dB[:, :N] = torch.from_numpy(B).cuda()
    dC = torch.full((M + 1, ldc), float("nan"), device="cuda")
    dC[:M, :N] = torch.from_numpy(C).cuda()
    before = dC.clone()
    s = torch.cuda.current_stream().cuda_stream
    rc = b2g.b2g_sgemm_3xtf32_variant(variant, M, N, K, alpha, dA.data_ptr(), lda, dB.data_ptr(),
                                      ldb, beta, dC.data_ptr(), ldc, s)
    what = f"seed {seed}: variant {variant} {M}x{N}x{K} lds=({lda},{ldb},{ldc}) {alpha} {beta}"
    assert rc == 0, f"{what}: {b2g.b2g_strerror(rc)}"
    torch.cuda.synchronize()
    out, prev = dC.cpu().numpy(), before.cpu().numpy()
    ref, bound, _ = oracle.sgemm(A, B, C, alpha, beta)
    check(out[:M, :N], ref, bound, what)
    outside = np.ones(out.shape, bool)
    outside[:M, :N] = False
    assert np.array_equal(out[outside].view(np.uint32), prev[outside].view(np.uint32)), what


@pytest.mark.parametrize("seed", range(8))
def test_random_host_operands(tb, seed):
    """b2g_sgemm_host on random shapes on both sides of its 2048-k chunking
    threshold, from page-locked and from pageable host memory."""
    torch, b2g = tb
    rng = np.random.default_rng(4000 + seed)
    M, N = (int(x) for x in rng.integers(1, 600, size=2))
    K = int(rng.integers(2048, 3000)) if seed % 2 else int(rng.integers(1, 2048))
    alpha = float(rng.choice(ALPHAS))
    beta = float(rng.choice(BETAS))
    A, B, C = _stored(rng, M, K), _stored(rng, K, N), _stored(rng, M, N)
    pinned = seed % 4 < 2
    hA, hB, hC = (torch.from_numpy(x.copy()) for x in (A, B, C))
    if pinned:
        hA, hB, hC = hA.pin_memory(), hB.pin_memory(), hC.pin_memory()
    b2g.sgemm_host(hA, hB, hC, alpha, beta)
    ref, bound, _ = oracle.sgemm(A, B, C, alpha, beta)
    check(hC.numpy(), ref, bound, f"seed {seed}: {M}x{N}x{K} pinned={pinned} {alpha} {beta}")
