"""Failure detection without a GPU fault: every mbarrier wait in the kernels is
bounded.  Here the producer is told (through the library's test hook) to stop
after one stage, so the consumers' waits run out; the kernel must record the
timeout in the status word and return, and the context must stay usable."""
import numpy as np
import pytest

import oracle
from gpu_helpers import check, env, gemm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tb():
    return env()


@pytest.mark.parametrize("plan_name,M,N,K", [
    ("tma_64x128x16_s6_o2", 64, 64, 64),
    ("tma_64x128x16_s6_o5", 64, 64, 64),      # packed, k-chunked A
    ("wk_32x64x32_g8", 64, 64, 64),           # the small-problem plans: k split between warps
    ("wk_64x64x32_g4", 64, 64, 64),
    ("tmaX_64x128x16_s6_o1", 64, 64, 64),
    ("gen_64x64x16_s4", 64, 64, 64),
    ("pre_128x64x32_s3_o5", 64, 64, 128),   # packed kernels, both tile shapes
    ("pre_64x128x32_s3_o5", 64, 64, 128),
    ("skinnyT_m16", 16, 512, 1024),         # k slabs summed in a cluster of 8 CTAs
    ("cs8_64x128x16_s6_o2", 64, 128, 256),  # one tile's 8 k slices in one cluster
    ("cs16_64x128x16_s6_o2", 128, 256, 512),  # four clusters of 16 k slices
])
def test_wait_runs_out_and_context_survives(tb, plan_name, M, N, K):
    torch, b2g = tb
    plan = b2g.plans().index(plan_name)
    stream = torch.cuda.current_stream().cuda_stream
    rng = np.random.default_rng(0)
    A = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
    C = np.zeros((M, N), np.float32)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.from_numpy(C).cuda()
    b2g.b2g_status(stream, clear=True)
    try:
        assert b2g.b2g_set_wait_limit_ns(20_000_000) == 0  # 20 ms
        b2g.b2g_debug_stop_after(1)  # at least 2 stages needed per CTA, only 1 issued
        rc = b2g.b2g_sgemm_with_plan(plan, 0, 0, M, N, K, 1.0, dA.data_ptr(), K,
                                     dB.data_ptr(), N, 0.0, dC.data_ptr(), N, stream)
        assert rc == 0
        # the debug read returns the same flags and leaves them set
        dbg = b2g.b2g_sgemm_debug_status(stream)
        assert dbg > 0 and dbg & 1, f"debug status {dbg}"
        rc, flags = b2g.b2g_status(stream, clear=True)
        assert rc == b2g.B2G_ERR_TIMEOUT
        assert flags & 1, f"consumer timeout flag missing: {flags:#x}"
        assert flags == dbg
        assert b2g.b2g_sgemm_debug_status(stream) == 0
    finally:
        b2g.b2g_debug_stop_after(-1)
        b2g.b2g_set_wait_limit_ns(2_000_000_000)
    # the status word is clear again and a normal call is correct
    rc, flags = b2g.b2g_status(stream, clear=True)
    assert rc == 0 and flags == 0
    ref, bound, _ = oracle.sgemm(A, B, C, 1.0, 0.0)
    got, rc, guard = gemm(b2g, torch, A, B, C, 1.0, 0.0, plan=plan)
    assert rc == 0 and guard
    check(got, ref, bound, plan_name)


@pytest.mark.parametrize("variant", [0, 2])
def test_tensor_core_wait_runs_out(tb, variant):
    """The 3xTF32 kernels (one CTA; a CTA pair with remote arrivals): the copy
    issuer stops after one stage, the MMA issuer's wait runs out, the epilogue's
    wait for the accumulator runs out, and every thread of both CTAs still
    reaches the teardown barrier before tensor memory is freed."""
    torch, b2g = tb
    M = N = K = 512
    stream = torch.cuda.current_stream().cuda_stream
    rng = np.random.default_rng(1)
    A = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.zeros((M, N), device="cuda")
    args = (M, N, K, 1.0, dA.data_ptr(), K, dB.data_ptr(), N, 0.0, dC.data_ptr(), N, stream)
    b2g.b2g_status(stream, clear=True)
    try:
        assert b2g.b2g_set_wait_limit_ns(20_000_000) == 0
        b2g.b2g_debug_stop_after(1)
        assert b2g.b2g_sgemm_3xtf32_variant(variant, *args) == 0
        rc, flags = b2g.b2g_status(stream, clear=True)
        assert rc == b2g.B2G_ERR_TIMEOUT and flags != 0, f"{flags:#x}"
    finally:
        b2g.b2g_debug_stop_after(-1)
        b2g.b2g_set_wait_limit_ns(2_000_000_000)
    rc, flags = b2g.b2g_status(stream, clear=True)
    assert rc == 0 and flags == 0
    assert b2g.b2g_sgemm_3xtf32_variant(variant, *args) == 0
    torch.cuda.synchronize()
    ref, bound, _ = oracle.sgemm(A, B, None, 1.0, 0.0)
    check(dC.cpu().numpy(), ref, bound, f"3xTF32 variant {variant} after a timeout")
