"""b2g_sgemm_launch_count against the kernels a call really launches.

The bench reports gpu_launches from b2g_sgemm_launch_count.  Here one call is
captured into a CUDA graph (driver API through ctypes) and its kernel nodes
are counted, for each family of plans: transpose first + split tail, packed
operands + split tail, the skinny cluster kernel, the streaming skinny kernel
+ split-K reduction, one plain kernel, and the beta-only scaling kernel.  The
call passes a workspace of b2g_sgemm_workspace_size bytes (b2g_sgemm_ws), so
the plan and its splits are the ones an ordinary call takes.
"""
import ctypes

import numpy as np
import pytest

from gpu_helpers import env

pytestmark = pytest.mark.gpu

CU_STREAM_CAPTURE_MODE_RELAXED = 2
CU_GRAPH_NODE_TYPE_KERNEL = 0


@pytest.fixture(scope="module")
def tb():
    torch, b2g = env()
    cu = ctypes.CDLL("libcuda.so.1")
    return torch, b2g, cu


def _kernel_nodes(cu, stream_handle, fn):
    s = ctypes.c_void_p(stream_handle)
    assert cu.cuStreamBeginCapture_v2(s, CU_STREAM_CAPTURE_MODE_RELAXED) == 0
    try:
        fn()
    finally:
        graph = ctypes.c_void_p()
        rc_end = cu.cuStreamEndCapture(s, ctypes.byref(graph))
    assert rc_end == 0
    n = ctypes.c_size_t(0)
    assert cu.cuGraphGetNodes(graph, None, ctypes.byref(n)) == 0
    nodes = (ctypes.c_void_p * max(1, n.value))()
    assert cu.cuGraphGetNodes(graph, nodes, ctypes.byref(n)) == 0
    kernels = 0
    for i in range(n.value):
        t = ctypes.c_int(-1)
        assert cu.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(t)) == 0
        kernels += t.value == CU_GRAPH_NODE_TYPE_KERNEL
    cu.cuGraphDestroy(graph)
    return kernels, n.value


@pytest.mark.parametrize("M,N,K,lda,alpha,beta", [
    (2048, 2048, 2048, 2048, 1.0, 0.5),   # transpose-first, split tail
    (2000, 2000, 2001, 2001, 1.0, 0.5),   # packed operands (K % 4 != 0), split tail
    (1000, 1025, 777, 777, 0.75, -1.25),  # packed operands (odd lda), split tail
    (512, 512, 510, 510, 1.0, 0.5),       # packed operands (K % 4 != 0), one-launch wk GEMM
    (16, 4096, 4096, 4096, 1.0, 1.0),     # skinny, k slabs summed in the cluster
    (16, 1024, 8192, 8192, 1.0, 1.0),     # skinny, streaming kernel + split-K reduction
    (256, 256, 64, 64, 1.0, 0.0),         # one kernel, no split (64 k)
    (512, 512, 512, 512, 0.0, 2.0),       # alpha == 0: C scaled only
])
def test_reported_launches_match(tb, M, N, K, lda, alpha, beta):
    torch, b2g, cu = tb
    rng = np.random.default_rng(M + N + K)
    A = torch.from_numpy(rng.uniform(-1, 1, (M, lda)).astype(np.float32)).cuda()
    B = torch.from_numpy(rng.uniform(-1, 1, (K, N)).astype(np.float32)).cuda()
    C = torch.from_numpy(rng.uniform(-1, 1, (M, N)).astype(np.float32)).cuda()
    args = (0, 0, M, N, K, alpha, A.data_ptr(), lda, B.data_ptr(), N)
    rc, expected = b2g.b2g_sgemm_launch_count(*args, C.data_ptr(), N)
    assert rc == 0
    rc, need = b2g.b2g_sgemm_workspace_size(*args, C.data_ptr(), N)
    assert rc == 0
    ws = torch.empty(max(16, need), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    def call():
        assert b2g.b2g_sgemm_ws(*args, beta, C.data_ptr(), N, ws.data_ptr(), need,
                                stream.cuda_stream) == 0

    got, nodes = _kernel_nodes(cu, stream.cuda_stream, call)
    assert got == expected, (expected, got, nodes)


@pytest.mark.parametrize("transA,expected_transposes", [(0, 2), (1, 1)])
def test_reported_launches_match_transposed_b(tb, transA, expected_transposes):
    """op(B) = B^T at 2048^3: one transpose per operand not in the kernel's
    layout, the GEMM and its split-tail reduction."""
    torch, b2g, cu = tb
    M = N = K = 2048
    rng = np.random.default_rng(7 + transA)
    A = torch.from_numpy(rng.uniform(-1, 1, (M, K)).astype(np.float32)).cuda()
    B = torch.from_numpy(rng.uniform(-1, 1, (N, K)).astype(np.float32)).cuda()
    C = torch.from_numpy(rng.uniform(-1, 1, (M, N)).astype(np.float32)).cuda()
    args = (transA, 1, M, N, K, 1.0, A.data_ptr(), 2048, B.data_ptr(), 2048)
    rc, expected = b2g.b2g_sgemm_launch_count(*args, C.data_ptr(), N)
    assert rc == 0 and expected == expected_transposes + 2
    rc, need = b2g.b2g_sgemm_workspace_size(*args, C.data_ptr(), N)
    assert rc == 0
    ws = torch.empty(max(16, need), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()

    def call():
        assert b2g.b2g_sgemm_ws(*args, 0.5, C.data_ptr(), N, ws.data_ptr(), need,
                                stream.cuda_stream) == 0

    got, nodes = _kernel_nodes(cu, stream.cuda_stream, call)
    assert got == expected, (expected, got, nodes)
