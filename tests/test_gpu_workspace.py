"""Plans that transpose A into a workspace first: caller-owned workspace,
too-small workspace (a plan without one runs instead), the library-owned
workspace shared by two streams, and graph capture (no allocation while
capturing).  Every result is checked against the oracle's FP32 bound."""
import numpy as np
import pytest

import oracle
from gpu_helpers import check, env

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tb():
    return env()


def _inputs(seed, M, N, K):
    rng = np.random.default_rng(seed)
    A = rng.uniform(-1, 1, size=(M, K)).astype(np.float32)
    B = rng.uniform(-1, 1, size=(K, N)).astype(np.float32)
    C = rng.uniform(-1, 1, size=(M, N)).astype(np.float32)
    return A, B, C


# M*N*K at or above the size where the tune table pre-transposes A
SHAPE = (1030, 1500, 1400)


def test_table_picks_pretranspose(tb):
    torch, b2g = tb
    M, N, K = SHAPE
    name = b2g.b2g_plan_name(b2g.b2g_sgemm_select_plan(0, 0, M, N, K, 1.0, 1 << 20, K, 1 << 20, N,
                                                        1 << 20, N))
    assert name.startswith("pre_")


@pytest.mark.parametrize("ws_kind", ["exact", "large", "at_only", "small", "none"])
def test_caller_workspace(tb, ws_kind):
    """exact / large: the plan with its split tail; at_only (room for A^T, not
    for the partial sums): the same plan without the split; small / none: a
    plan that needs no workspace."""
    torch, b2g = tb
    M, N, K = SHAPE
    A, B, C = _inputs(1, M, N, K)
    ref, bound, _ = oracle.sgemm(A, B, C, 0.75, -0.5)
    rc, need = b2g.b2g_sgemm_workspace_size(0, 0, M, N, K, 0.75, 1 << 20, K, 1 << 20, N, 1 << 20, N)
    at = K * ((M + 3) // 4 * 4) * 4
    assert rc == 0 and need >= at
    nbytes = {"exact": need, "large": need + 4096, "at_only": at, "small": at - 16,
              "none": 0}[ws_kind]
    ws = torch.empty(max(nbytes, 4) // 4, dtype=torch.float32, device="cuda")
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.from_numpy(C).cuda()
    s = torch.cuda.current_stream().cuda_stream
    rc = b2g.b2g_sgemm_ws(0, 0, M, N, K, 0.75, dA.data_ptr(), K, dB.data_ptr(), N, -0.5,
                          dC.data_ptr(), N, ws.data_ptr() if nbytes else None, nbytes, s)
    assert rc == 0
    check(dC.cpu().numpy(), ref, bound, ws_kind)


def test_library_workspace_two_streams(tb):
    """Two streams, different problems, no synchronisation between the calls:
    the shared library workspace must not mix them up."""
    torch, b2g = tb
    M, N, K = SHAPE
    probs = [_inputs(10 + i, M, N, K) for i in range(2)]
    refs = [oracle.sgemm(A, B, C, 1.0, 1.0)[:2] for A, B, C in probs]
    dev = [tuple(torch.from_numpy(x).cuda() for x in p) for p in probs]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    hostC = [torch.from_numpy(p[2]).pin_memory() for p in probs]
    for rep in range(3):
        for i, ((dA, dB, dC), st) in enumerate(zip(dev, streams)):
            with torch.cuda.stream(st):
                if rep:
                    dC.copy_(hostC[i], non_blocking=True)
                b2g.sgemm(dA, dB, dC, 1.0, 1.0)
        torch.cuda.synchronize()
        for (dA, dB, dC), (ref, bound) in zip(dev, refs):
            check(dC.cpu().numpy(), ref, bound, f"two streams, round {rep}")


def test_graph_capture_takes_plan_without_workspace(tb):
    torch, b2g = tb
    M, N, K = SHAPE
    A, B, C = _inputs(20, M, N, K)
    ref, bound, _ = oracle.sgemm(A, B, C, 1.0, 0.0)
    dA, dB = torch.from_numpy(A).cuda(), torch.from_numpy(B).cuda()
    dC = torch.zeros(M, N, device="cuda")
    b2g.sgemm(dA, dB, dC, 1.0, 0.0)  # first use of both plans outside the capture
    s = torch.cuda.current_stream().cuda_stream
    assert b2g.b2g_sgemm_ws(0, 0, M, N, K, 1.0, dA.data_ptr(), K, dB.data_ptr(), N, 0.0,
                            dC.data_ptr(), N, None, 0, s) == 0
    torch.cuda.synchronize()
    dC.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        b2g.sgemm(dA, dB, dC, 1.0, 0.0)
    g.replay()
    torch.cuda.synchronize()
    check(dC.cpu().numpy(), ref, bound, "graph replay")


def test_release_and_reuse(tb):
    torch, b2g = tb
    assert b2g.b2g_release_workspaces() == 0
    M, N, K = SHAPE
    A, B, C = _inputs(30, M, N, K)
    ref, bound, _ = oracle.sgemm(A, B, C, 1.0, 0.5)
    dA, dB, dC = (torch.from_numpy(x).cuda() for x in (A, B, C))
    b2g.sgemm(dA, dB, dC, 1.0, 0.5)
    torch.cuda.synchronize()
    check(dC.cpu().numpy(), ref, bound, "after release")
