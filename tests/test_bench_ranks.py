"""The bench's multi-rank logic on CPU: two gloo ranks on 127.0.0.1.

Under torchrun every rank times its own replica; the step time reported is
the slowest rank's, every rank must agree on it, and the value is the units
all ranks processed over that time.  The reference arm (the CPU oracle) runs
on rank 0 alone: other ranks leave at once, printing nothing.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_env() == (rank, world, rank)
    local_ms = 1.5 + rank  # rank 1 is the slower replica
    ms = bench.max_over_ranks(local_ms, world)
    value = bench.job_throughput(1e9, world, ms)
    dist.barrier()
    with open(os.path.join(out, f"rank{rank}.json"), "w") as f:
        json.dump({"ms": ms, "value": value}, f)
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time(tmp_path):
    import multiprocessing as mp

    ctx = mp.get_context("spawn")
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, str(tmp_path))) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert res[0] == res[1]
    assert res[0]["ms"] == 2.5
    assert res[0]["value"] == pytest.approx(2 * 1e9 / 2.5e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.job_throughput(2.0, 1, 4.0) == pytest.approx(500.0)


def test_reference_arm_other_ranks_leave_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(_free_port()))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], env=env, capture_output=True,
                       text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_kernel_unit_finds_each_plans_definition():
    """bench.py ties the recorded DRAM traffic to the sources of the kernel's
    translation unit: the file that defines the plan, not one that only names
    it (host.cu names the packed plans in its table of tile-shape twins)."""
    sys.path.insert(0, ROOT)
    import bench
    import dense_fp32_gemm_07_gb300 as b2g
    from dense_fp32_gemm_07_gb300 import build

    build.build()
    for name in b2g.plans():
        unit = bench.kernel_unit(name)
        assert unit.startswith("csrc/") and unit != "csrc/host.cu", (name, unit)
        src = open(os.path.join(ROOT, "dense_fp32_gemm_07_gb300", unit)).read()
        assert f'"{name}"' in src and "PLAN" in src
