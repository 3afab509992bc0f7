"""The bench's host-side helpers, on CPU: the peak formulas, the e2e check
against the oracle (it must pass a correct result and reject a wrong one),
the oracle's rate on a row block, and the recorded-traffic lookup."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads  # noqa: E402


def test_peaks_from_unit_counts():
    # 152 SMs x 128 FP32 lanes x 2 FLOP x 2070 MHz
    assert bench.fp32_peak_tflops(152, 2070.0) == pytest.approx(80.54784)
    # 152 SMs x 4096 dense TF32 FLOP/clk x 2070 MHz
    assert bench.tf32_peak_tflops(152, 2070.0) == pytest.approx(1288.76544)
    # scales with SMs and clock
    assert bench.fp32_peak_tflops(76, 1035.0) == pytest.approx(80.54784 / 4)


def test_max_clock_has_a_fallback():
    mhz, basis = bench.max_sm_mhz(0)
    assert mhz > 0 and isinstance(basis, str)


def _small():
    return workloads.Workload("e2e_small", 300, 260, 200, 0.75, -0.5, 9, "u11", "u11")


def test_e2e_check_passes_the_oracle_and_rejects_a_wrong_result(oracle_mod):
    w = _small()
    A, B, C = w.make()
    ref, _, _ = oracle_mod.sgemm(A, B, C, w.alpha, w.beta)
    good = ref.astype(np.float32)
    assert bench.e2e_check(w, A, B, C, good) > w.M // 256 * 3
    bad = good.copy()
    bad[0, 0] += 1.0  # a corner the check always samples
    with pytest.raises(RuntimeError):
        bench.e2e_check(w, A, B, C, bad)


def test_oracle_rate_reports_cores_and_rows(oracle_mod):
    w = _small()
    A, B, C = w.make()
    r = bench.oracle_rate(w, A, B, C, 0.05)
    assert r["gflops"] > 0 and r["cores"] == oracle_mod.max_threads()
    assert 1 <= r["rows"] <= w.M


def test_recorded_traffic_follows_the_kernel_sources():
    """The committed DRAM-traffic record is used only while the kernel's
    sources hash as they did when it was taken."""
    plan = "tmaT_128x64x32_s3_o5"
    got = bench.recorded_traffic(plan)
    assert got is None or got > 0
    assert bench.recorded_traffic("no_such_plan") is None
