"""The C ABI used from a plain C program (tests/c_abi_check.c).

The program includes include/swiglu_mlp.h as C, links libswiglu_mlp.so, takes
device memory from cudaMalloc and calls gemm, gemm_ex (forced split-K) and
swiglu_mlp with no Python or torch in the process; it checks the results
against host sums itself (exact for the integer GEMMs).  Compiling and
linking it needs no GPU; running it does.
"""
import os
import subprocess

import pytest

from swiglu_mlp_gb300 import build as swg_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi_check.c")
LIBDIR = os.path.join(ROOT, "swiglu_mlp_gb300")


def _compile(out):
    swg_build.build()
    nvcc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    cmd = [nvcc, "-O1", "-I", os.path.join(ROOT, "include"), SRC, "-o", out,
           "-L", LIBDIR, "-lswiglu_mlp", "-Xlinker", "-rpath=" + LIBDIR]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "warning" not in (r.stdout + r.stderr).lower(), r.stdout + r.stderr


def test_c_program_compiles_and_links(tmp_path):
    _compile(str(tmp_path / "c_abi_check"))


@pytest.mark.gpu
def test_c_program_runs(tmp_path):
    exe = str(tmp_path / "c_abi_check")
    _compile(exe)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "c_abi_check: ok" in r.stdout
