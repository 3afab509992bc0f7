"""Concurrent calls from several host threads, each on its own stream.

The library keeps per-device state that calls share: the library-owned
workspace (ordered across streams by an event recorded after each use), the
host-operand staging buffers, the plans' one-time configuration.  ctypes
releases the GIL during a call, so these threads enter the C library at the
same time.  Every call's result is checked against the oracle afterwards.
"""
import threading

import numpy as np
import pytest

import oracle
from gpu_helpers import check, env

pytestmark = pytest.mark.gpu

# (M, N, K, lda pad): transpose-first (workspace), packed (workspace), skinny
# cluster, one-kernel small plan
SHAPES = [(1536, 1280, 1024, 0), (700, 515, 333, 1), (16, 4096, 2048, 0), (300, 260, 96, 0)]


@pytest.fixture(scope="module")
def tb():
    return env()


def test_threads_on_separate_streams(tb):
    torch, b2g = tb
    rng = np.random.default_rng(51)
    jobs = []
    for t in range(4):
        for i, (M, N, K, pad) in enumerate(SHAPES):
            lda = K + pad
            A = rng.uniform(-1, 1, (M, lda)).astype(np.float32)
            B = rng.uniform(-1, 1, (K, N)).astype(np.float32)
            C = rng.uniform(-1, 1, (M, N)).astype(np.float32)
            jobs.append((t, i, A, B, C, M, N, K, lda))
    dev = {id(j): tuple(torch.from_numpy(x).cuda() for x in (j[2], j[3], j[4])) for j in jobs}
    torch.cuda.synchronize()
    errors = []
    start = threading.Barrier(4)

    def worker(t):
        try:
            stream = torch.cuda.Stream()
            start.wait()
            for rep in range(3):  # each job three times: C <- 0.5 A B + 0.25 C, three times
                for j in jobs:
                    if j[0] != t:
                        continue
                    _, i, _, _, _, M, N, K, lda = j
                    dA, dB, dC = dev[id(j)]
                    if i == 0 and rep == 1:  # the tensor-core path once, same update
                        rc = b2g.b2g_sgemm_3xtf32(M, N, K, 0.5, dA.data_ptr(), lda, dB.data_ptr(),
                                                  N, 0.25, dC.data_ptr(), N, stream.cuda_stream)
                    else:
                        rc = b2g.b2g_sgemm(M, N, K, 0.5, dA.data_ptr(), lda, dB.data_ptr(), N,
                                           0.25, dC.data_ptr(), N, stream.cuda_stream)
                    if rc:
                        errors.append((t, i, rep, rc))
            stream.synchronize()
        except Exception as e:  # reported below, on the main thread
            errors.append((t, repr(e)))

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join(120)
    assert not any(th.is_alive() for th in threads)
    assert not errors, errors
    torch.cuda.synchronize()
    for j in jobs:
        t, i, A, B, C, M, N, K, lda = j
        ref = C.astype(np.float64)
        bound = np.zeros_like(ref)
        Cin = C
        for _ in range(3):  # the oracle applied three times, each on the previous result
            r, b, _ = oracle.sgemm(A[:, :K], B, Cin, 0.5, 0.25)
            # the next update starts from the GPU's FP32 value of this step: take the
            # oracle's own result rounded to FP32 and carry its bound forward
            bound = np.abs(0.25) * bound + b
            ref = r
            Cin = r.astype(np.float32)
        check(dev[id(j)][2].cpu().numpy(), ref, bound + 1e-6 * np.abs(ref), f"thread {t} job {i}")
