"""The header as a plain C99 program sees it: compiled here (syntax only, no
GPU), and on a GPU built against the library and run (exact results through
b2g_sgemm and b2g_sgemm_host, an error code for a bad leading dimension)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c", "abi_example.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _gcc():
    gcc = shutil.which("gcc")
    if not gcc or not os.path.isdir(os.path.join(CUDA, "include")):
        pytest.skip("gcc or the CUDA headers are not available")
    return gcc


def test_header_compiles_as_c99():
    r = subprocess.run([_gcc(), "-std=c99", "-Wall", "-Wextra", "-Werror", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
                        SRC], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


@pytest.mark.gpu
def test_c_program_runs(tmp_path):
    from dense_fp32_gemm_07_gb300 import build

    build.build()
    pkg = os.path.join(ROOT, "dense_fp32_gemm_07_gb300")
    exe = str(tmp_path / "abi_example")
    lib64 = os.path.join(CUDA, "lib64")
    r = subprocess.run([_gcc(), "-std=c99", "-O2", "-o", exe, SRC,
                        "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
                        "-L", pkg, "-lb2g_sgemm", "-Wl,-rpath," + pkg,
                        "-L", lib64, "-lcudart", "-Wl,-rpath," + lib64],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.startswith("ok"), (r.stdout, r.stderr)
