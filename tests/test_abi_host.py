"""The C-ABI library loads, exports every symbol the header declares, and its
host-side logic (argument checks, quick returns, plan choice) behaves as the
header states.  None of these calls reaches a kernel, so they run without a GPU.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "b2g_sgemm.h")


@pytest.fixture(scope="module")
def b2g():
    from dense_fp32_gemm_07_gb300 import build

    build.build()
    import dense_fp32_gemm_07_gb300 as pkg

    pkg.library()
    return pkg


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(b2g_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(b2g):
    names = declared_functions()
    assert len(names) >= 12
    lib = ctypes.CDLL(b2g.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(b2g.EXPORTS) == names


def test_error_codes_match_header(b2g):
    text = open(HEADER).read()
    for name, val in re.findall(r"#define (B2G_\w+) \(?(-?\d+)\)?", text):
        assert getattr(b2g, name) == int(val), name
        assert b2g.b2g_strerror(int(val)) != "unknown error code"


def test_version_and_plans(b2g):
    assert "sm_103a" in b2g.b2g_version()
    names = b2g.plans()
    assert len(names) == b2g.b2g_plan_count() >= 4 and len(set(names)) == len(names)
    for i, n in enumerate(names):
        info = b2g.b2g_plan_info(i)
        assert info["BM"] > 0 and info["BN"] > 0 and info["BK"] % 4 == 0
        assert info["threads"] % 32 == 0 and info["smem_bytes"] <= 227 * 1024
        assert n.startswith(("tma", "gen", "pre", "pack", "skinny", "cs", "wk"))
    assert b2g.b2g_plan_name(len(names)) is None
    with pytest.raises(b2g.B2GError):
        b2g.b2g_plan_info(-1)


FAKE = 0x100000  # a 16-byte aligned address; never dereferenced by these calls


@pytest.mark.parametrize("args,code", [
    ((-1, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4), -1),
    ((4, -1, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4), -1),
    ((4, 4, -1, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4), -1),
    ((4, 4, 8, 1.0, FAKE, 7, FAKE, 4, 0.0, FAKE, 4), -2),   # lda < K
    ((4, 4, 8, 1.0, FAKE, 8, FAKE, 3, 0.0, FAKE, 4), -2),   # ldb < N
    ((4, 4, 8, 1.0, FAKE, 8, FAKE, 4, 0.0, FAKE, 3), -2),   # ldc < N
    ((4, 4, 0, 1.0, FAKE, 0, FAKE, 4, 0.0, FAKE, 4), -2),   # lda >= max(1, K)
    ((4, 4, 8, 1.0, FAKE, 8, FAKE, 4, 0.0, None, 4), -3),   # C null
    ((4, 4, 8, 1.0, None, 8, FAKE, 4, 0.0, FAKE, 4), -3),   # A null and read
    ((4, 4, 8, 1.0, FAKE, 8, None, 4, 0.0, FAKE, 4), -3),   # B null and read
])
def test_invalid_arguments(b2g, args, code):
    assert b2g.b2g_sgemm(*args, 0) == code
    assert b2g.b2g_sgemm_select_plan(0, 0, *args[:8], args[9], args[10]) == code


def test_quick_returns_touch_nothing(b2g):
    # M == 0 or N == 0: valid, nothing launched (so no device needed)
    assert b2g.b2g_sgemm(0, 4, 4, 1.0, None, 4, None, 4, 0.0, None, 4, 0) == 0
    assert b2g.b2g_sgemm(4, 0, 4, 1.0, None, 4, None, 1, 0.0, None, 1, 0) == 0
    n = b2g.b2g_plan_count()
    # alpha == 0 or K == 0: A and B not needed, beta-scale only
    assert b2g.b2g_sgemm_select_plan(0, 0, 4, 4, 8, 0.0, None, 8, None, 4, FAKE, 4) == n
    assert b2g.b2g_sgemm_select_plan(0, 0, 4, 4, 0, 1.0, None, 1, None, 4, FAKE, 4) == n


def test_transposed_leading_dims(b2g):
    # transA: A stored K x M -> lda >= M ; transB: B stored N x K -> ldb >= K
    assert b2g.b2g_sgemm_select_plan(1, 0, 16, 8, 4, 1.0, FAKE, 15, FAKE, 8, FAKE, 8) == -2
    assert b2g.b2g_sgemm_select_plan(1, 0, 16, 8, 4, 1.0, FAKE, 16, FAKE, 8, FAKE, 8) >= 0
    assert b2g.b2g_sgemm_select_plan(0, 1, 16, 8, 4, 1.0, FAKE, 4, FAKE, 3, FAKE, 8) == -2
    assert b2g.b2g_sgemm_select_plan(0, 1, 16, 8, 4, 1.0, FAKE, 4, FAKE, 4, FAKE, 8) >= 0


def _plan(b2g, *a):
    return b2g.b2g_plan_name(b2g.b2g_sgemm_select_plan(*a))


def test_tune_table_classes(b2g):
    # aligned, ld % 4 == 0, K % 4 == 0 -> bulk-tensor plans; large ones pre-transpose A
    assert _plan(b2g, 0, 0, 4096, 4096, 4096, 1.0, FAKE, 4096, FAKE, 4096, FAKE, 4096).startswith("pre_")
    assert _plan(b2g, 0, 0, 16, 4096, 4096, 1.0, FAKE, 4096, FAKE, 4096, FAKE, 4096) == "skinnyT_m16"
    assert _plan(b2g, 0, 0, 32, 4096, 4096, 1.0, FAKE, 4096, FAKE, 4096, FAKE, 4096) == "skinnyT_m32"
    assert _plan(b2g, 0, 0, 16, 1024, 8192, 1.0, FAKE, 8192, FAKE, 1024, FAKE, 1024) == "skinny_m16"
    # skinny M with N % 4 != 0 takes a tiled plan
    assert _plan(b2g, 0, 0, 16, 4095, 4096, 1.0, FAKE, 4096, FAKE, 4096, FAKE, 4096).startswith("tma_")
    # small products: one launch, the k range split between a CTA's warps;
    # few tiles over a long k range keep the split-tail plan
    assert _plan(b2g, 0, 0, 64, 64, 64, 1.0, FAKE, 64, FAKE, 64, FAKE, 64) == "wk_32x64x32_g8"
    assert _plan(b2g, 0, 0, 512, 512, 512, 1.0, FAKE, 512, FAKE, 512, FAKE, 512) == "wk_32x64x32_g8"
    assert _plan(b2g, 0, 0, 768, 768, 768, 1.0, FAKE, 768, FAKE, 768, FAKE, 768) == "wk_64x64x32_g4"
    assert _plan(b2g, 0, 0, 128, 128, 32768, 1.0, FAKE, 32768, FAKE, 128, FAKE, 128).startswith("tma_")
    # odd leading dimension -> operands packed into the workspace first
    assert _plan(b2g, 0, 0, 1000, 1025, 777, 0.75, FAKE, 777, FAKE, 1025, FAKE, 1025).startswith(
        ("pack_", "wkP_"))
    # misaligned base pointer -> packed (small: then the one-launch wk kernel)
    assert _plan(b2g, 0, 0, 512, 512, 512, 1.0, FAKE + 4, 512, FAKE, 512, FAKE, 512) == "wkP_32x64x32_g8"
    assert _plan(b2g, 0, 0, 2048, 2048, 2048, 1.0, FAKE + 4, 2048, FAKE, 2048, FAKE, 2048).startswith("pack_")
    # K not a multiple of 4 -> packed
    assert _plan(b2g, 0, 0, 512, 512, 510, 1.0, FAKE, 512, FAKE, 512, FAKE, 512).startswith("wkP_")
    # small general problems -> packed, then the one-launch wk kernel (the
    # 4-byte feed is the fallback without a workspace)
    assert _plan(b2g, 0, 0, 64, 64, 63, 1.0, FAKE, 64, FAKE, 64, FAKE, 64).startswith("wkP_")
    # op(A) = A^T aligned -> transposed-layout bulk-tensor plan; op(B) = B^T
    # aligned -> B^T (and A) transposed with 16-byte vectors, then that plan
    # (small products of each class on the one-launch wk kernel)
    assert _plan(b2g, 1, 0, 512, 512, 512, 1.0, FAKE, 512, FAKE, 512, FAKE, 512) == "wkT_32x64x32_g8"
    assert _plan(b2g, 1, 0, 4096, 4096, 4096, 1.0, FAKE, 4096, FAKE, 4096, FAKE, 4096).startswith("tmaT_")
    assert _plan(b2g, 0, 1, 512, 512, 512, 1.0, FAKE, 512, FAKE, 512, FAKE, 512) == "wkR_32x64x32_g8"
    assert _plan(b2g, 1, 1, 512, 512, 512, 1.0, FAKE, 512, FAKE, 512, FAKE, 512) == "wkR_32x64x32_g8"
    assert _plan(b2g, 0, 1, 4096, 4096, 4096, 1.0, FAKE, 4096, FAKE, 4096, FAKE, 4096).startswith("pret_")
    # op(B) = B^T with K % 4 != 0 or an odd leading dimension -> packed
    assert _plan(b2g, 0, 1, 512, 512, 510, 1.0, FAKE, 512, FAKE, 510, FAKE, 512).startswith("wkP_")
    assert _plan(b2g, 0, 1, 512, 512, 512, 1.0, FAKE, 512, FAKE, 513, FAKE, 512).startswith("wkP_")
    assert _plan(b2g, 0, 1, 2048, 2048, 2048, 1.0, FAKE, 2048, FAKE, 2049, FAKE, 2048).startswith("pack_")
    # small op(B) = B^T calls -> one packing launch, then the wk kernel
    assert _plan(b2g, 0, 1, 64, 64, 64, 1.0, FAKE, 64, FAKE, 64, FAKE, 64).startswith("wkP_")


# With no device answering, the host sizes splits for 152 SMs x 4 resident CTAs.
NO_DEVICE_SLOTS = 152 * 4


def _tail_time(tiles, kt, sms, occ, first, S, BM, BN, BK, cw, read_c):
    """The host's estimate of a persistent grid's time (us) for a split."""
    G = sms * occ
    f = first if S > 1 else tiles
    ns = (tiles - first) * S if S > 1 else 0
    sl = -(-kt // S)
    loads = []
    for i in range(min(occ, 8)):
        b = i * sms
        whole = (f - b + G - 1) // G if b < f else 0
        nsl = (ns - b + G - 1) // G if b < ns else 0
        loads.append(float(whole * (kt + 1) + nsl * (sl + 1)))
    loads.sort()
    t, prev, n = 0.0, 0.0, len(loads)
    for i, L in enumerate(loads):
        w = (n - i) * cw
        e = 0.88 if w >= 12 else 0.85 if w >= 8 else 0.40 if w >= 4 else 0.20
        t += (n - i) * (L - prev) / e
        prev = L
    t *= BM * BN * BK / (128.0 * 2070.0)
    if S > 1:
        t += (tiles - first) * BM * BN * 4.0 * (2.0 * S + 1.0 + (1.0 if read_c else 0.0)) / 5.5e6 + 2.0
    return t


def split_tail(M, N, K, BM, BN, slots=NO_DEVICE_SLOTS, BK=32, cw=4, read_c=True, sms=152):
    """(first split tile, slices) of the split-tail rule: T tiles over G slots,
    T = q*G + r; the last r tiles get S = G // r slices of at least 64 k, unless
    the balance model finds a split at least 3% faster."""
    T = -(-M // BM) * -(-N // BN)
    q, r = divmod(T, slots)
    if r == 0:
        return 0, 1
    occ = slots // sms
    smax = K // 64
    S = min(slots // r, smax)
    f = q * slots
    if S < 2:
        S, f = 1, 0
    kt = -(-K // BK)
    best = 0.97 * _tail_time(T, kt, sms, occ, f, S, BM, BN, BK, cw, read_c)
    for qq in range(max(0, q - 2), q + 1):
        if qq * slots >= T:
            continue
        for s in range(1, min(smax, 16) + 1):
            if s == 1 and qq != q:
                continue
            t = _tail_time(T, kt, sms, occ, qq * slots, s, BM, BN, BK, cw, read_c)
            if t < best:
                best, S, f = t, s, (qq * slots if s > 1 else 0)
    return (f, S) if S >= 2 else (0, 1)


def want_bytes(base, M, N, K, BM, BN):
    first, S = split_tail(M, N, K, BM, BN)
    if S == 1:
        return base
    T = -(-M // BM) * -(-N // BN)
    return -(-base // 256) * 256 + (T - first) * S * BM * BN * 4


def plan_tile(b2g, M, N, K, lda, ldb, ldc):
    pi = b2g.b2g_sgemm_select_plan(0, 0, M, N, K, 1.0, FAKE, lda, FAKE, ldb, FAKE, ldc)
    info = b2g.b2g_plan_info(pi)
    return info["BM"], info["BN"]


def test_split_tail_rule_examples():
    # 4096^3 on 128 x 64 tiles: 2048 = 3 * 608 + 224 -> the last 224 tiles in 2 slices
    assert split_tail(4096, 4096, 4096, 128, 64) == (1824, 2)
    assert split_tail(4096, 4096, 4096, 128, 64, slots=456) == (1824, 2)
    # 2048^3 on 64 x 128 tiles over 456 slots: 512 = 456 + 56 -> 8 slices
    assert split_tail(2048, 2048, 2048, 64, 128, slots=456) == (456, 8)
    # whole waves or too little k: no split
    assert split_tail(64 * 608, 128, 4096, 64, 128) == (0, 1)
    assert split_tail(4096, 4096, 127, 128, 64) == (0, 1)
    # too many tiles left for 2 slices each, but SMs unevenly loaded (320
    # tiles: some SMs run 3, the others 2): the balance model cuts every tile
    assert split_tail(4096, 640, 4096, 128, 64) == (0, 5)
    assert split_tail(4096, 640, 4096, 128, 64, slots=456) == (0, 4)
    # measured on GB300 (456 slots): 1664^3 178.7 -> 157.8 us with every tile in
    # 4 slices, 2560^3 546.8 -> 513.7 with the tiles after the first round in
    # 2; 1408^3 and 3072^3 (alternatives measured slower) keep no split
    assert split_tail(1664, 1664, 1664, 128, 64, slots=456) == (0, 4)
    assert split_tail(2560, 2560, 2560, 128, 64, slots=456) == (456, 2)
    assert split_tail(1408, 1408, 1408, 128, 64, slots=456) == (0, 1)
    assert split_tail(3072, 3072, 3072, 128, 64, slots=456) == (0, 1)
    assert split_tail(8192, 11008, 4096, 128, 64, slots=456) == (10944, 7)


def test_workspace_size_query(b2g):
    BM, BN = plan_tile(b2g, 4096, 4096, 4096, 4096, 4096, 4096)
    rc, n = b2g.b2g_sgemm_workspace_size(0, 0, 4096, 4096, 4096, 1.0, FAKE, 4096, FAKE, 4096,
                                         FAKE, 4096)
    # A^T (K x round_up(M, 4) floats), then the split tail's partial sums
    assert rc == 0 and n == want_bytes(4096 * 4096 * 4, 4096, 4096, 4096, BM, BN)
    assert n > 4096 * 4096 * 4
    BM, BN = plan_tile(b2g, 1001, 4096, 4096, 4096, 4096, 4096)
    rc, n = b2g.b2g_sgemm_workspace_size(0, 0, 1001, 4096, 4096, 1.0, FAKE, 4096, FAKE, 4096,
                                         FAKE, 4096)
    assert rc == 0 and n == want_bytes(4096 * 1004 * 4, 1001, 4096, 4096, BM, BN)
    rc, n = b2g.b2g_sgemm_workspace_size(0, 0, 64, 64, 64, 1.0, FAKE, 64, FAKE, 64, FAKE, 64)
    assert rc == 0 and n == 0  # one tile, 64 k: nothing to split
    # skinny, N >= 2048: the k slabs add up inside clusters, no workspace
    rc, n = b2g.b2g_sgemm_workspace_size(0, 0, 16, 4096, 4096, 1.0, FAKE, 4096, FAKE, 4096,
                                         FAKE, 4096)
    assert rc == 0 and n == 0
    # skinny, small N: split-K partial sums, S x M x N floats for some S > 1
    rc, n = b2g.b2g_sgemm_workspace_size(0, 0, 16, 1024, 8192, 1.0, FAKE, 8192, FAKE, 1024,
                                         FAKE, 1024)
    assert rc == 0 and n > 0 and n % (16 * 1024 * 4) == 0
    rc, n = b2g.b2g_sgemm_workspace_size(0, 0, 64, 64, 64, 1.0, FAKE, 63, FAKE, 64, FAKE, 64)
    assert rc == -2
    # packing: A^T (K x round_up(M, 4)) and B (K x round_up(N, 4)), then the
    # tail (none for the one-launch wk plans)
    BM, BN = plan_tile(b2g, 1000, 1025, 777, 777, 1025, 1025)
    rc, n = b2g.b2g_sgemm_workspace_size(0, 0, 1000, 1025, 777, 1.0, FAKE, 777, FAKE, 1025,
                                         FAKE, 1025)
    name = b2g.b2g_plan_name(b2g.b2g_sgemm_select_plan(0, 0, 1000, 1025, 777, 1.0, FAKE, 777,
                                                        FAKE, 1025, FAKE, 1025))
    base = 777 * (1000 + 1028) * 4
    assert rc == 0 and n == (base if name.startswith("wk") else
                             want_bytes(base, 1000, 1025, 777, BM, BN))
    assert b2g.b2g_release_workspaces() == 0  # nothing allocated yet: no CUDA call needed


def test_launch_count_query(b2g):
    def count(M, N, K, alpha=1.0, lda=None, ldb=None, ldc=None):
        lda, ldb, ldc = lda or max(K, 1), ldb or max(N, 1), ldc or max(N, 1)
        rc, n = b2g.b2g_sgemm_launch_count(0, 0, M, N, K, alpha, FAKE, lda, FAKE, ldb, FAKE,
                                           ldc)
        assert rc == 0
        return n

    assert count(0, 64, 64) == 0 and count(64, 0, 64) == 0
    assert count(64, 64, 64, alpha=0.0) == 1 and count(64, 64, 0) == 1  # C = beta * C
    assert count(64, 64, 64) == 1                    # one tile, one kernel
    assert count(4096, 4096, 4096) == 3              # transpose, GEMM, tail reduction
    assert count(16, 4096, 4096) == 1                # skinny, split-K summed in clusters
    assert count(16, 1024, 8192) == 2                # skinny split-K and its reduction
    assert count(1000, 1025, 777, lda=777) == 2      # one packing launch, one-launch wk GEMM
    assert count(4096, 4096, 4095, lda=4095) == 3    # one packing launch, GEMM, tail
    rc, _ = b2g.b2g_sgemm_launch_count(0, 0, 64, 64, 64, 1.0, FAKE, 63, FAKE, 64, FAKE, 64)
    assert rc == -2
    # op(B) = B^T at 4096^3: transposes of A and of B^T, GEMM, tail reduction;
    # with A stored K x M only B^T is transposed
    for tA, n in ((0, 4), (1, 3)):
        rc, got = b2g.b2g_sgemm_launch_count(tA, 1, 4096, 4096, 4096, 1.0, FAKE, 4096, FAKE, 4096,
                                             FAKE, 4096)
        assert rc == 0 and got == n, (tA, got)


def test_workspace_of_transposed_b(b2g):
    """pret_ plans: B^T transposed (K x round_up(N, 4)), plus A^T unless A
    comes stored K x M, then the split tail's room."""
    M, N, K = 4096, 4092, 4096
    for tA in (0, 1):
        pi = b2g.b2g_sgemm_select_plan(tA, 1, M, N, K, 1.0, FAKE, 4096, FAKE, 4096, FAKE, N)
        info = b2g.b2g_plan_info(pi)
        assert b2g.b2g_plan_name(pi).startswith("pret_")
        rc, n = b2g.b2g_sgemm_workspace_size(tA, 1, M, N, K, 1.0, FAKE, 4096, FAKE, 4096, FAKE, N)
        base = K * ((0 if tA else M) + N) * 4
        assert rc == 0 and n == want_bytes(base, M, N, K, info["BM"], info["BN"]), (tA, n)


def test_forced_plan_range(b2g):
    n = b2g.b2g_plan_count()
    args = (0, 0, 4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4, 0)
    assert b2g.b2g_sgemm_with_plan(n, *args) == -7
    assert b2g.b2g_sgemm_with_plan(-1, *args) == -7


def test_wait_limit_and_debug_hook(b2g):
    assert b2g.b2g_set_wait_limit_ns(0) == -1
    assert b2g.b2g_set_wait_limit_ns(2_000_000_000) == 0
    assert b2g.b2g_debug_stop_after(-5) == 0


def test_no_gpu_means_loud_failure(b2g):
    """Without a usable sm_103 device a real call fails with a code; nothing
    falls back to the CPU."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc = b2g.b2g_sgemm(4, 4, 4, 1.0, FAKE, 4, FAKE, 4, 0.0, FAKE, 4, 0)
    assert rc == b2g.B2G_ERR_DEVICE


def test_debug_status_without_device(b2g):
    """b2g_sgemm_debug_status returns the status word's flags (>= 0) or a
    negative code; with no usable device it is the device error, never a
    flag value."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert b2g.b2g_sgemm_debug_status(0) == b2g.B2G_ERR_DEVICE
    lib = ctypes.CDLL(b2g.LIB_PATH)
    lib.b2g_sgemm_debug_status.argtypes = [ctypes.c_void_p]
    assert lib.b2g_sgemm_debug_status(None) == b2g.B2G_ERR_DEVICE


def test_tensor_api_rejects_cpu_tensors(b2g):
    import torch

    a = torch.zeros(4, 4)
    with pytest.raises(TypeError):
        b2g.sgemm(a, a, a)


def test_host_operand_argument_checks(b2g):
    """b2g_sgemm_host checks its arguments before touching a device."""
    args = lambda M, N, K, lda, ldb, ldc, C=FAKE: (M, N, K, 1.0, FAKE, lda, FAKE, ldb, 0.0, C,
                                                   ldc, 0)
    assert b2g.b2g_sgemm_host(*args(-1, 4, 4, 4, 4, 4)) == -1
    assert b2g.b2g_sgemm_host(*args(4, 4, 4, 3, 4, 4)) == -2
    assert b2g.b2g_sgemm_host(*args(4, 4, 4, 4, 4, 4, C=None)) == -3
    assert b2g.b2g_sgemm_host(*args(0, 4, 4, 4, 4, 4)) == 0  # nothing to do, no device needed


@pytest.mark.parametrize("tA,tB,M,N,K,lda,ldb,ldc,code", [
    (0, 0, 16, 8, 4, 16, 4, 16, 0),     # A M x K (lda >= M), B K x N (ldb >= K), C ldc >= M
    (0, 0, 16, 8, 4, 15, 4, 16, -2),    # lda < M
    (0, 0, 16, 8, 4, 16, 3, 16, -2),    # ldb < K
    (0, 0, 16, 8, 4, 16, 4, 15, -2),    # ldc < M
    (1, 0, 16, 8, 4, 4, 4, 16, 0),      # A stored K x M: lda >= K
    (1, 0, 16, 8, 4, 3, 4, 16, -2),
    (0, 1, 16, 8, 4, 16, 8, 16, 0),     # B stored N x K: ldb >= N
    (0, 1, 16, 8, 4, 16, 7, 16, -2),
    (0, 0, -1, 8, 4, 16, 4, 16, -1),
    (0, 0, 16, 8, 4, 16, 4, 16, "Cnull"),
])
def test_colmajor_leading_dims(b2g, tA, tB, M, N, K, lda, ldb, ldc, code):
    """b2g_sgemm_colmajor checks BLAS's column-major bounds: the row-major call
    it becomes has M and N, A and B and their op() flags swapped.  A valid case
    would launch a kernel, so it is checked through the row-major plan choice
    and through the M = 0 quick return (which still checks every argument)."""
    if code == "Cnull":
        assert b2g.b2g_sgemm_colmajor(tA, tB, M, N, K, 1.0, FAKE, lda, FAKE, ldb, 0.0, None, ldc,
                                      0) == -3
        return
    if code:
        assert b2g.b2g_sgemm_colmajor(tA, tB, M, N, K, 1.0, FAKE, lda, FAKE, ldb, 0.0, FAKE, ldc,
                                      0) == code
    else:
        # the same leading dimensions are valid; the row-major view selects a plan
        assert b2g.b2g_sgemm_select_plan(tB, tA, N, M, K, 1.0, FAKE, ldb, FAKE, lda, FAKE,
                                         ldc) >= 0
        assert b2g.b2g_sgemm_colmajor(tA, tB, 0, N, K, 1.0, None, lda, None, ldb, 0.0, None,
                                      ldc, 0) == 0


def test_build_rejects_register_spills():
    """build.spills() finds ptxas's spill report per function, so a kernel that
    starts spilling fails the build; the current build has none."""
    from dense_fp32_gemm_07_gb300 import build

    log = ("ptxas info    : Function properties for _Z3fooPf\n"
           "    0 bytes stack frame, 0 bytes spill stores, 0 bytes spill loads\n"
           "ptxas info    : Function properties for _Z3barPf\n"
           "    32 bytes stack frame, 36 bytes spill stores, 44 bytes spill loads\n")
    assert build.spills(log) == [("_Z3barPf", 36, 44)]
    build.build()
    for src in build.sources():
        path = os.path.join(build.BUILD, f"ptxas_{src[:-3]}.log")
        if os.path.exists(path):
            assert build.spills(open(path).read()) == [], src
