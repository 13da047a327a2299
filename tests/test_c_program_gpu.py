"""The C ABI used from C alone (tests/c/mhcpb_from_c.c): a C program, built
with nvcc against include/mhcpb.h and libmhcpb.so, runs the backward, the
split backward, the forward, the forward with fused gates and the gate
backward chain on exact integer inputs and checks the results exactly
(the cuDNN frontend page "DSv4.1 mHC projection/RMS backward", intro:
dX = P W + c X with c = 0 here, dW = P^T X).  Compiling needs no GPU;
running does."""
import os
import shutil
import subprocess

import pytest

from rms_backward_gb300 import abi
from rms_backward_gb300 import build as B

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "c", "mhcpb_from_c.c")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")


def _compile(out):
    if not os.path.exists(abi.LIB_PATH):
        B.build()
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    libdir = os.path.dirname(abi.LIB_PATH)
    subprocess.run([nvcc, "-O2", "-Xcompiler", "-Wall,-Wextra,-Werror", "-I", INCLUDE, SRC, "-L", libdir,
                    "-lmhcpb", "-Xlinker", f"-rpath,{libdir}", "-o", out],
                   check=True, capture_output=True, text=True)
    return out


def test_c_program_compiles(tmp_path):
    assert os.path.exists(_compile(str(tmp_path / "mhcpb_from_c")))


@pytest.mark.gpu
def test_c_program_runs_and_checks_exactly(tmp_path):
    exe = _compile(str(tmp_path / "mhcpb_from_c"))
    run = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "C ABI ok" in run.stdout
