"""Compile the CUDA library in-tree: csrc/*.cu -> libb2g_sgemm.so (sm_103a only).

Each translation unit is compiled in parallel with nvcc, then linked into one
shared library with the CUDA runtime linked statically.  `-Xptxas -v` output
(registers, spills, shared memory per kernel) is kept in build/ptxas_<tu>.log,
and the build fails when ptxas reports a register spill in any kernel: the
packed FFMA kernels are capped at 128 registers to keep three CTAs per SM, and
a spill there would otherwise show up only as a quiet loss of speed.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import re
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "build")
LIB = os.path.join(PKG, "libb2g_sgemm.so")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                     "-Xptxas", "-v"]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [
        os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(d) <= t for d in _deps())


_SPILL = re.compile(r"(\d+) bytes spill stores, (\d+) bytes spill loads")
_ENTRY = re.compile(r"Function properties for (\S+)")


def spills(log_text: str):
    """[(function, spill store bytes, spill load bytes)] for every function
    whose ptxas report shows a spill."""
    out, fn = [], None
    for line in log_text.splitlines():
        m = _ENTRY.search(line)
        if m:
            fn = m.group(1)
            continue
        m = _SPILL.search(line)
        if m and (int(m.group(1)) or int(m.group(2))):
            out.append((fn, int(m.group(1)), int(m.group(2))))
    return out


def _compile(src: str) -> str:
    obj = os.path.join(BUILD, src[:-3] + ".o")
    log = os.path.join(BUILD, f"ptxas_{src[:-3]}.log")
    cmd = [nvcc(), *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    with open(log, "w") as f:
        f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr[-4000:]}")
    bad = spills(r.stdout + r.stderr)
    if bad:
        os.remove(obj)
        raise RuntimeError(f"ptxas reports register spills in {src}: " +
                           "; ".join(f"{f}: {st} B stored, {ld} B loaded" for f, st, ld in bad))
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Build the library if any source is newer than it; return its path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    srcs = sources()
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(_compile, srcs))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr[-4000:]}")
    os.replace(tmp, LIB)
    if verbose:
        for s in srcs:
            with open(os.path.join(BUILD, f"ptxas_{s[:-3]}.log")) as f:
                sys.stdout.write(f.read())
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
