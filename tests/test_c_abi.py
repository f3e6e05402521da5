"""The C ABI used from plain C (tests/c/abi_example.c): no Python binding and
no torch between the caller and libsmo_gemm.so.  The program is compiled
against include/smo_gemm.h on the host (CPU test) and run on a GPU, where it
checks exact integer products through gemm_bf16 and gemm_ex in both B
orientations against a triple loop."""
import os
import shutil
import subprocess

import pytest

import shared_memory_operand_gb300 as smo

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
SRC = os.path.join(ROOT, "tests", "c", "abi_example.c")


def _build() -> str:
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = smo.load_library(build=True)._name
    libdir = os.path.dirname(lib)
    exe = os.path.join(libdir, "abi_example")
    cmd = [cc, "-O2", "-std=c11", "-Wall", "-Wextra", "-Werror", SRC, "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA_HOME, "include"), "-L", libdir, "-l:" + os.path.basename(lib),
           "-L", os.path.join(CUDA_HOME, "lib64"), "-lcudart", "-Wl,-rpath," + libdir, "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_program_compiles_against_the_header():
    assert os.path.exists(_build())


@pytest.mark.gpu
def test_c_program_runs_exact():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    r = subprocess.run([_build()], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ABI OK")
