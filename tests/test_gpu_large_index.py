"""Operands with more than 2^31 elements: 64-bit offsets in every kernel.

Each test puts one operand past 2^31 elements (8.6 GB of FP32) so that any
32-bit index arithmetic in a kernel would address the wrong element:
  * B of a skinny product (16 x 16384 x 131200, the cluster kernel),
  * C of a transpose-first product (66000 x 32768 x 64, C read with beta),
  * A of a transpose-first product with split tail (66000 x 64 x 32768),
  * A of the 3xTF32 path (66000 x 256 x 32768, split kernels + CTA pairs).
Inputs are small multiples of 1/4 given by a formula of (row, column), so
every partial sum is exact in FP32 whatever the summation order: the GPU must
match the oracle bit for bit.  The device fills each operand from the formula;
the oracle gets host copies, from the same formula, of only the rows and
columns the sampled entries need (`oracle.sgemm_entries` on those
sub-matrices), so nothing on the oracle side comes from the GPU.
"""
import numpy as np
import pytest

import oracle
from gpu_helpers import env

pytestmark = pytest.mark.gpu

GIB = 1 << 30


@pytest.fixture(scope="module")
def tb():
    torch, b2g = env()
    free, _ = torch.cuda.mem_get_info()
    if free < 48 * GIB:
        pytest.skip(f"needs 48 GiB of free device memory, {free / GIB:.0f} GiB free")
    return torch, b2g


def host_vals(rows, cols, a, b):
    """((a*i + b*j) mod 9 - 4) / 4 for i in rows, j in cols (float32, exact)."""
    i = np.asarray(rows, np.int64)[:, None] * a
    j = np.asarray(cols, np.int64)[None, :] * b
    return ((((i + j) % 9) - 4) * 0.25).astype(np.float32)


def dev_fill(torch, R, Cn, a, b):
    """The same values as host_vals over all R x Cn, built on the device in row
    blocks (int32 arithmetic: a*i + b*j stays far below 2^31 here)."""
    t = torch.empty((R, Cn), dtype=torch.float32, device="cuda")
    j = torch.arange(Cn, dtype=torch.int32, device="cuda")[None, :] * b
    step = max(1, (1 << 26) // Cn)
    for r0 in range(0, R, step):
        r1 = min(R, r0 + step)
        i = torch.arange(r0, r1, dtype=torch.int32, device="cuda")[:, None] * a
        t[r0:r1] = (((i + j) % 9) - 4).to(torch.float32) * 0.25
    return t


def sample(M, N, rng, extra_rows=(), n=40):
    """(rows, cols) of the entries to check, paired: n random entries, the two
    corners, and each extra row at a random column."""
    extra_rows = list(extra_rows)
    rows = list(rng.integers(0, M, n)) + [0, M - 1] + extra_rows
    cols = list(rng.integers(0, N, n)) + [0, N - 1] + list(rng.integers(0, N, len(extra_rows)))
    return np.array(rows, np.int64), np.array(cols, np.int64)


def check_entries(torch, dC, A_sub, B_sub, C_sub, rows, cols, alpha, beta):
    """Oracle on the sub-matrices; GPU entries read straight from dC."""
    assert rows.shape == cols.shape
    ru, ri = np.unique(rows, return_inverse=True)
    cu, ci = np.unique(cols, return_inverse=True)
    ref, bound, _ = oracle.sgemm_entries(A_sub, B_sub, C_sub, alpha, beta, ri, ci)
    r_t = torch.from_numpy(rows).cuda()
    c_t = torch.from_numpy(cols).cuda()
    got = dC[r_t, c_t].cpu().numpy()
    assert np.all(np.isfinite(got))
    assert np.array_equal(got.astype(np.float64), ref), (
        f"{int((got != ref).sum())} of {got.size} sampled entries differ; first "
        f"{[(int(rows[k]), int(cols[k]), float(got[k]), float(ref[k])) for k in np.flatnonzero(got != ref)[:3]]}")


def _done(torch, b2g):
    """After the test has dropped its tensors: free the library's workspaces
    and the allocator's cache before the next 8.6 GB operand."""
    b2g.b2g_release_workspaces()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_skinny_b_past_2g(tb):
    torch, b2g = tb
    M, N, K = 16, 16384, 131200  # B: 2.15e9 elements
    assert K * N > 2**31
    rng = np.random.default_rng(41)
    dA = dev_fill(torch, M, K, 3, 5)
    dB = dev_fill(torch, K, N, 7, 11)
    dC = dev_fill(torch, M, N, 13, 1)
    rows, cols = sample(M, N, rng, extra_rows=range(M))
    b2g.sgemm(dA, dB, dC, 1.0, 0.5)
    torch.cuda.synchronize()
    cu = np.unique(cols)
    A_sub = host_vals(np.arange(M), np.arange(K), 3, 5)
    B_sub = host_vals(np.arange(K), cu, 7, 11)
    C_sub = host_vals(np.arange(M), cu, 13, 1)
    check_entries(torch, dC, A_sub, B_sub, C_sub, rows, cols, 1.0, 0.5)
    del dA, dB, dC
    _done(torch, b2g)


def test_transpose_first_c_past_2g(tb):
    torch, b2g = tb
    M, N, K = 66000, 32768, 64  # C: 2.16e9 elements, read (beta != 0) and written
    assert M * N > 2**31
    rng = np.random.default_rng(42)
    dA = dev_fill(torch, M, K, 3, 5)
    dB = dev_fill(torch, K, N, 7, 11)
    dC = dev_fill(torch, M, N, 13, 1)
    rows, cols = sample(M, N, rng, extra_rows=(65535, 65536, 65537, 65999))
    b2g.sgemm(dA, dB, dC, 1.0, 0.5)
    torch.cuda.synchronize()
    ru, cu = np.unique(rows), np.unique(cols)
    check_entries(torch, dC, host_vals(ru, np.arange(K), 3, 5), host_vals(np.arange(K), cu, 7, 11),
                  host_vals(ru, cu, 13, 1), rows, cols, 1.0, 0.5)
    del dA, dB, dC
    _done(torch, b2g)


def test_transpose_first_a_past_2g_split_tail(tb):
    torch, b2g = tb
    M, N, K = 66000, 64, 32768  # A: 2.16e9 elements; its transpose another 8.6 GB
    assert M * K > 2**31
    rc, launches = b2g.b2g_sgemm_launch_count(0, 0, M, N, K, 1.0, 1 << 20, K, 1 << 20, N,
                                              1 << 20, N)
    assert rc == 0 and launches == 3  # transpose, GEMM, split-tail reduction
    rng = np.random.default_rng(43)
    dA = dev_fill(torch, M, K, 3, 5)
    dB = dev_fill(torch, K, N, 7, 11)
    dC = dev_fill(torch, M, N, 13, 1)
    rows, cols = sample(M, N, rng, extra_rows=(65535, 65536, 65537, 65999))
    b2g.sgemm(dA, dB, dC, 1.0, -1.0)
    torch.cuda.synchronize()
    ru, cu = np.unique(rows), np.unique(cols)
    check_entries(torch, dC, host_vals(ru, np.arange(K), 3, 5), host_vals(np.arange(K), cu, 7, 11),
                  host_vals(ru, cu, 13, 1), rows, cols, 1.0, -1.0)
    del dA, dB, dC
    _done(torch, b2g)


def test_3xtf32_a_past_2g(tb):
    torch, b2g = tb
    M, N, K = 66000, 256, 32768  # A: 2.16e9 elements; its hi and lo parts 17 GB
    rng = np.random.default_rng(44)
    dA = dev_fill(torch, M, K, 3, 5)
    dB = dev_fill(torch, K, N, 7, 11)
    dC = dev_fill(torch, M, N, 13, 1)
    rows, cols = sample(M, N, rng, extra_rows=(65535, 65536, 65537, 65999))
    b2g.sgemm_3xtf32(dA, dB, dC, 1.0, 0.5)
    torch.cuda.synchronize()
    ru, cu = np.unique(rows), np.unique(cols)
    # quarter-integers are exact in TF32: the split's low parts are zero and
    # every product and sum is exact, as on the FFMA path
    check_entries(torch, dC, host_vals(ru, np.arange(K), 3, 5), host_vals(np.arange(K), cu, 7, 11),
                  host_vals(ru, cu, 13, 1), rows, cols, 1.0, 0.5)
    del dA, dB, dC
    _done(torch, b2g)
