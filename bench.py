"""Benchmark of the FP32 SGEMM hot path: one JSON line on stdout (rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one C = alpha*A*B + beta*C over the 4096^3 headline workload
(alpha = 1, beta = 0.5, A, B, C uniform[-1, 1) from seed 1), inputs resident in
device memory.  The three operands (192 MiB) exceed the 129 MB L2, so no flush
runs between steps.  Under torchrun every rank runs its own replica of the
problem (the GEMM needs no exchange between GPUs): weak scaling, no collective
on the data path, timing is the max over ranks.

`e2e` is the same metric with the operands in page-locked host memory, through
b2g_sgemm_host: every step copies A, B and C to the device (row panels of A and
C overlapped with the panel GEMMs), multiplies, and copies C back.

`skinny` reports the 16 x 4096 x 4096 workload (alpha = beta = 1), which HBM
bounds, as GB/s of algorithmic bytes against the measured copy bandwidth; its
calls rotate through four operand sets so that each finds its operands out of
L2.

`--impl reference` times the CPU oracle (double i-k-j loops, all host cores)
on a bounded row sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads  # noqa: E402

METRIC = "SGEMM TFLOPS (2MNK/t) at M=N=K=4096; % of GB300 FP32 vector peak"
UNIT = "TFLOP/s"
# FP32 vector peak from unit counts: 152 SMs x 128 FP32 lanes x 2 FLOP per FMA
# x clock.  The contract's peak uses the maximum SM clock (2070 MHz).
SMS, LANES, MAX_MHZ = 152, 128, 2070.0
L2_BYTES = 129e6
# device code of the dominant kernel: a change here voids the recorded traffic
# The recorded traffic is valid while these headers and the translation unit
# that compiles the plan's kernel are unchanged.
KERNEL_HEADERS = ("csrc/sgemm_ffma.cuh", "csrc/ptx.cuh", "csrc/sgemm_params.h")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic_square4096.txt")


def tf32_peak_tflops():
    """Dense TF32 tensor peak: the measured bf16 GEMM peak x the nominal TF32/bf16
    ratio (1.1 / 2.25 PFLOP/s); the recipe's 1.9 PFLOP/s bf16 when no
    measurement is present."""
    basis = "fallback bf16 1900 TFLOP/s"
    bf16 = 1900.0
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            bf16 = float(json.load(f)["bf16_tflops"])
            basis = f"measured bf16 {bf16:.1f} TFLOP/s"
    except (OSError, KeyError, ValueError):
        pass
    return bf16 * 1.1 / 2.25, basis + " x 1.1/2.25 (nominal TF32/bf16)"


def hbm_peak_gbs():
    """HBM bandwidth: the measured copy bandwidth, else the recipe's fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            v = float(json.load(f)["hbm_gbs"])
            return v, f"measured copy {v:.1f} GB/s"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback 6800 GB/s"


def fp32_peak_tflops(mhz: float) -> float:
    return SMS * LANES * 2 * mhz * 1e6 / 1e12


def kernel_unit(plan: str) -> str:
    """The csrc/*.cu file that defines `plan` in a plan table (B2G_..._PLAN(...)
    entry) and so compiles its kernel; other files may name the plan."""
    import re

    csrc = os.path.join(ROOT, "dense_fp32_gemm_07_gb300", "csrc")
    pat = re.compile(r'B2G_\w*PLAN\w*\(\s*"' + re.escape(plan) + '"')
    for f in sorted(os.listdir(csrc)):
        if f.endswith(".cu"):
            with open(os.path.join(csrc, f)) as fh:
                if pat.search(fh.read()):
                    return "csrc/" + f
    raise KeyError(plan)


def kernel_sources_hash(plan: str) -> str:
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "dense_fp32_gemm_07_gb300")
    for rel in KERNEL_HEADERS + (kernel_unit(plan),):
        with open(os.path.join(pkg, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(plan: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel sources or the plan changed since it was taken."""
    try:
        kv = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("plan") != plan or kv.get("kernel_sources_sha256") != kernel_sources_hash(plan):
            return None
        return float(kv["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock/throttle sampling in the background while the GPU works."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"b2g_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 8:
                    try:
                        rows.append((float(parts[0]), float(parts[1]), parts[2], parts[4:8]))
                    except ValueError:
                        pass
        if not rows:
            return None
        # samples taken while the GEMM loop ran: clock above idle floor
        load = [r for r in rows if r[0] > 0.5 * r[1]] or rows
        reasons = set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in load:
            for n, v in zip(names, r[3]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(r[0] for r in load),
                "sm_max_mhz": max(r[1] for r in load), "samples": len(load),
                "reasons": sorted(reasons)}


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, world: int, device=None) -> float:
    """The largest value of x over all ranks; every rank receives it (a device
    tensor for NCCL, a host tensor for gloo)."""
    if world <= 1:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, ms: float) -> float:
    """Whole-job rate in units per second: the units every rank processed in a
    step, over the slowest rank's time per step (ms)."""
    return world * units_per_rank / (ms * 1e-3)


def run_reference(args, w):
    """The CPU oracle on host cores: each step computes a bounded block of rows."""
    import numpy as np

    import oracle

    rank, world, _ = dist_env()
    if rank != 0:
        return
    A, B, C = w.make()
    threads = oracle.max_threads()
    # size the row block from a short calibration so the whole run stays short
    t0 = time.perf_counter()
    oracle.sgemm(A[:8], B, C[:8], w.alpha, w.beta)
    per_row = max((time.perf_counter() - t0) / 8, 1e-6)
    # the whole --warmup W --steps K run takes about 90 s of CPU time
    per_step = min(2.0, 90.0 / (args.warmup + args.steps))
    rows = int(max(1, min(w.M, per_step / per_row)))
    times = []
    for i in range(args.warmup + args.steps):
        r0 = (i * rows) % max(1, w.M - rows + 1)
        t0 = time.perf_counter()
        oracle.sgemm(A[r0:r0 + rows], B, C[r0:r0 + rows], w.alpha, w.beta)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
    t = sum(times) / len(times)
    value = 2.0 * rows * w.N * w.K / t / 1e12
    sample = (f"{rows} rows of the {w.M}x{w.N}x{w.K} problem per step "
              f"({rows}x{w.N}x{w.K} multiply-adds, double accumulation)")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "alpha": w.alpha,
                   "beta": w.beta, "seed": w.seed, "rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(w):
    """The oracle as it stands, all host cores, a bounded row block (~10 s)."""
    import oracle

    A, B, C = w.make()
    t0 = time.perf_counter()
    oracle.sgemm(A[:8], B, C[:8], w.alpha, w.beta)
    per_row = max((time.perf_counter() - t0) / 8, 1e-6)
    rows = int(max(8, min(w.M, 10.0 / per_row)))
    t0 = time.perf_counter()
    oracle.sgemm(A[:rows], B, C[:rows], w.alpha, w.beta)
    dt = time.perf_counter() - t0
    return {"value": 2.0 * rows * w.N * w.K / dt / 1e12, "unit": UNIT,
            "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"rows 0..{rows - 1} of the {w.M}x{w.N}x{w.K} problem "
                      f"({rows}x{w.N}x{w.K} multiply-adds, double accumulation), {dt:.1f} s"}


def run_ours(args, w):
    import numpy as np
    import torch

    import dense_fp32_gemm_07_gb300 as b2g
    from dense_fp32_gemm_07_gb300 import build

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    build.build()
    b2g.library()
    dev = torch.device("cuda", torch.cuda.current_device())

    A, B, C = w.make()
    hA, hB, hC = (torch.from_numpy(x).pin_memory() for x in (A, B, C))
    dA, dB, dC = (x.to(dev) for x in (hA, hB, hC))
    stream = torch.cuda.current_stream()
    plan = b2g.b2g_plan_name(b2g.b2g_sgemm_select_plan(
        0, 0, w.M, w.N, w.K, w.alpha, dA.data_ptr(), w.K, dB.data_ptr(), w.N, dC.data_ptr(), w.N))

    def step():
        b2g.sgemm(dA, dB, dC, w.alpha, w.beta, stream=stream)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    # warm-up: at least W steps and about half a second of load
    t_end = time.perf_counter() + 0.5
    n = 0
    while n < args.warmup or time.perf_counter() < t_end:
        step()
        n += 1
        if n % 20 == 0:
            torch.cuda.synchronize()
    barrier()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        step()
    ev1.record(stream)
    barrier()
    clocks = sampler.stop()
    ms = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world, dev)
    value = job_throughput(w.flops(), world, ms) / 1e12
    rc, launches_per_step = b2g.b2g_sgemm_launch_count(0, 0, w.M, w.N, w.K, w.alpha,
                                                       dA.data_ptr(), w.K, dB.data_ptr(), w.N,
                                                       dC.data_ptr(), w.N)
    if rc:
        raise b2g.B2GError(rc)

    # The dominant kernel alone, timed live the same way: for a plan that first
    # transposes A, its GEMM kernel is the transposed-layout plan of the same
    # name run on a pre-transposed copy of A (torch makes the copy: plumbing).
    # When the plan splits its last tiles, the call also runs the small tail
    # reduction, which this time includes: the figure is then conservative.
    kernel_plan = plan.replace("pre_", "tmaT_", 1) if plan.startswith("pre_") else plan
    kplan = b2g.plans().index(kernel_plan)
    kA = dA.t().contiguous() if plan.startswith("pre_") else dA
    trans = plan.startswith("pre_")

    def kernel_only():
        b2g.sgemm(kA, dB, dC, w.alpha, w.beta, transA=trans, plan=kplan, stream=stream)

    for _ in range(3):
        kernel_only()
    barrier()
    ev0.record(stream)
    for _ in range(args.steps):
        kernel_only()
    ev1.record(stream)
    barrier()
    kernel_ms = ev0.elapsed_time(ev1) / args.steps
    kernel_launches = launches_per_step - (1 if plan.startswith("pre_") else 0)
    del kA

    # The 3xTF32 tensor-core path, reported apart from the FFMA headline: the
    # same call shape through b2g_sgemm_3xtf32 (split kernels + tcgen05 GEMM).
    def tc_step():
        b2g.sgemm_3xtf32(dA, dB, dC, w.alpha, w.beta, stream=stream)

    for _ in range(3):
        tc_step()
    barrier()
    ev0.record(stream)
    for _ in range(args.steps):
        tc_step()
    ev1.record(stream)
    barrier()
    tc_ms = ev0.elapsed_time(ev1) / args.steps

    # The skinny workload (M = 16), bound by HBM: reported as GB/s of
    # algorithmic bytes against the copy bandwidth.  Its operands (67.9 MB) fit
    # in L2, so the timed calls rotate through four device copies of them
    # (272 MB): at least 200 MB of other operands pass through L2 between two
    # uses of a set.  beta = 1 accumulates into each set's C.
    sk = workloads.WORKLOADS["skinny16x4096x4096"]
    sk_host = sk.make()
    sk_sets = [tuple(torch.from_numpy(x).to(dev) for x in sk_host) for _ in range(4)]
    sk_plan = b2g.b2g_plan_name(b2g.b2g_sgemm_select_plan(
        0, 0, sk.M, sk.N, sk.K, sk.alpha, sk_sets[0][0].data_ptr(), sk.K,
        sk_sets[0][1].data_ptr(), sk.N, sk_sets[0][2].data_ptr(), sk.N))
    _, sk_launches = b2g.b2g_sgemm_launch_count(
        0, 0, sk.M, sk.N, sk.K, sk.alpha, sk_sets[0][0].data_ptr(), sk.K,
        sk_sets[0][1].data_ptr(), sk.N, sk_sets[0][2].data_ptr(), sk.N)

    def sk_step(i):
        a_, b_, c_ = sk_sets[i % len(sk_sets)]
        b2g.sgemm(a_, b_, c_, sk.alpha, sk.beta, stream=stream)

    sk_calls = max(40, min(4 * args.steps, 400))
    for i in range(8):
        sk_step(i)
    barrier()
    ev0.record(stream)
    for i in range(sk_calls):
        sk_step(i)
    ev1.record(stream)
    barrier()
    sk_ms = ev0.elapsed_time(ev1) / sk_calls
    del sk_sets

    # end to end through the public API with host buffers: b2g_sgemm_host
    # copies A, B and C from page-locked host memory, multiplies (row panels
    # overlapped with the copies) and copies C back, every step; C is updated
    # in place, so each step starts from the previous step's C
    e2e_steps = max(3, min(args.steps, 20))
    out = hC

    def e2e_step():
        b2g.sgemm_host(hA, hB, hC, w.alpha, w.beta, stream=stream, sync=False)

    for _ in range(2):
        e2e_step()
    barrier()
    ev0.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    ev1.record(stream)
    barrier()
    e2e_ms = max_over_ranks(ev0.elapsed_time(ev1) / e2e_steps, world, dev)
    # the result of the last step is still correct (spot check of one row)
    got = out[w.M // 2].numpy()
    if not np.isfinite(got).all():
        raise RuntimeError("non-finite output in the e2e check")

    rc, flags = b2g.b2g_status(stream.cuda_stream)
    if rc or flags:
        raise RuntimeError(f"kernel status word {flags:#x}")

    if rank == 0:
        achieved = w.flops() / (kernel_ms * 1e-3) / 1e12
        peak = fp32_peak_tflops(MAX_MHZ)
        traffic = recorded_traffic(kernel_plan)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": w.name, "M": w.M, "N": w.N, "K": w.K, "alpha": w.alpha,
                       "beta": w.beta, "seed": w.seed, "plan": plan,
                       "l2": "operands 201 MB > 129 MB L2, no flush between steps",
                       "parallelism": "replicas" if world > 1 else "single"},
            "roofline": {"bound": "alu", "achieved": achieved, "peak": peak, "unit": UNIT,
                         "frac": achieved / peak, "traffic": traffic,
                         "kernel": kernel_plan + (" + tail reduction" if kernel_launches > 1
                                                  else ""),
                         "kernel_ms": kernel_ms, "kernel_launches": kernel_launches,
                         "step_frac": value / world / peak,
                         "peak_basis": "152 SMs x 128 FP32 FMA/clk x 2 x 2070 MHz (derived)",
                         "frac_at_sampled_clock": (achieved / fp32_peak_tflops(clocks["sm_mhz"])
                                                   if clocks else None)},
            "e2e": {"value": job_throughput(w.flops(), world, e2e_ms) / 1e12, "unit": UNIT,
                    "h2d_bytes_per_step": int(hA.numel() + hB.numel() + hC.numel()) * 4,
                    "d2h_bytes_per_step": int(out.numel()) * 4},
            "gpu_launches": args.steps * launches_per_step,
            "clocks": clocks,
        }
        tpeak, tbasis = tf32_peak_tflops()
        tc_tensor = 3 * w.flops() / (tc_ms * 1e-3) / 1e12  # three TF32 products per term
        line["tf32x3"] = {
            "value": w.flops() / (tc_ms * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": tc_ms,
            "launches_per_step": 4, "path": "b2g_sgemm_3xtf32 (2 split kernels + tcgen05 GEMM on CTA pairs, 256 x 256 tiles + split-tail reduction)",
            "accuracy": "same elementwise FP32 bound as the FFMA path",
            "roofline": {"bound": "tensor", "achieved": tc_tensor, "peak": tpeak, "unit": UNIT,
                         "frac": tc_tensor / tpeak, "peak_basis": tbasis},
        }
        hpeak, hbasis = hbm_peak_gbs()
        sk_gbs = sk.min_bytes() / (sk_ms * 1e-3) / 1e9
        line["skinny"] = {
            "workload": sk.name, "M": sk.M, "N": sk.N, "K": sk.K, "alpha": sk.alpha,
            "beta": sk.beta, "plan": sk_plan, "launches_per_call": sk_launches,
            "us_per_call": sk_ms * 1e3, "tflops": sk.flops() / (sk_ms * 1e-3) / 1e12,
            "l2": "4 operand sets rotated (272 MB), 67.9 MB each",
            "roofline": {"bound": "hbm", "achieved": sk_gbs, "peak": hpeak, "unit": "GB/s",
                         "frac": sk_gbs / hpeak, "algorithmic_bytes": sk.min_bytes(),
                         "peak_basis": hbasis},
        }
        if not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(w)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=("ours", "reference"))
    ap.add_argument("--workload", default=workloads.HEADLINE, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    w = workloads.WORKLOADS[args.workload]
    if args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
