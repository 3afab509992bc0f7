"""Time the oracle on every workload with this host's cores -- TEST
INFRASTRUCTURE ONLY (a CPU baseline beside the GPU numbers, never a target).

    python -m oracle.timing [--budget SECONDS]

For each workload the oracle (double accumulation, OpenMP over rows, all
cores) runs on a leading block of rows sized to take about --budget seconds
(the whole problem when that is less), and the multiply-add rate of that
block is reported as GFLOP/s (2 FLOP per multiply-add).  512^3 is timed once
more on one core.  The ragged workload keeps its odd leading dimension.
"""
from __future__ import annotations

import argparse
import time

import oracle
import workloads


def time_rows(w, A, B, C, rows: int, threads: int = 0) -> float:
    t0 = time.perf_counter()
    oracle.sgemm(A[:rows], B, C[:rows], w.alpha, w.beta, threads=threads, M=rows, N=w.N, K=w.K)
    return time.perf_counter() - t0


def measure(w, budget: float, threads: int = 0):
    A, B, C = w.make()
    probe = min(w.M, 8)
    per_row = max(time_rows(w, A, B, C, probe, threads) / probe, 1e-7)
    rows = int(max(probe, min(w.M, budget / per_row)))
    dt = time_rows(w, A, B, C, rows, threads)
    return rows, dt, 2.0 * rows * w.N * w.K / dt / 1e9


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--budget", type=float, default=3.0, help="seconds per workload (about)")
    args = ap.parse_args()
    cores = oracle.max_threads()
    print(f"oracle threads: {cores}")
    print(f"{'workload':24s} {'rows timed':>12s} {'seconds':>8s} {'GFLOP/s':>9s}")
    for name, w in workloads.WORKLOADS.items():
        rows, dt, gflops = measure(w, args.budget)
        print(f"{name:24s} {rows:>5d}/{w.M:<6d} {dt:8.2f} {gflops:9.2f}", flush=True)
    w = workloads.WORKLOADS["square512"]
    rows, dt, gflops = measure(w, args.budget, threads=1)
    print(f"{'square512 (1 core)':24s} {rows:>5d}/{w.M:<6d} {dt:8.2f} {gflops:9.2f}", flush=True)


if __name__ == "__main__":
    main()
