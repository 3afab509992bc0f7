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


@pytest.mark.parametrize("plan_name", ["tma_64x128x16_s6_o2", "tmaX_64x128x16_s6_o1",
                                       "gen_64x64x16_s4"])
def test_wait_runs_out_and_context_survives(tb, plan_name):
    torch, b2g = tb
    plan = b2g.plans().index(plan_name)
    stream = torch.cuda.current_stream().cuda_stream
    rng = np.random.default_rng(0)
    A = rng.uniform(-1, 1, size=(64, 64)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(64, 64)).astype(np.float32)
    C = np.zeros((64, 64), np.float32)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.from_numpy(C).cuda()
    b2g.b2g_status(stream, clear=True)
    try:
        assert b2g.b2g_set_wait_limit_ns(20_000_000) == 0  # 20 ms
        b2g.b2g_debug_stop_after(1)  # 64 / 16 = 4 stages needed, only 1 issued
        rc = b2g.b2g_sgemm_with_plan(plan, 0, 0, 64, 64, 64, 1.0, dA.data_ptr(), 64,
                                     dB.data_ptr(), 64, 0.0, dC.data_ptr(), 64, stream)
        assert rc == 0
        rc, flags = b2g.b2g_status(stream, clear=True)
        assert rc == b2g.B2G_ERR_TIMEOUT
        assert flags & 1, f"consumer timeout flag missing: {flags:#x}"
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
