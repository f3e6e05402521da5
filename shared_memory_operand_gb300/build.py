"""Build ``libsmo_gemm.so`` in-tree (``shared_memory_operand_gb300/_build/``).

Two translation units compiled in parallel: the host planner (g++) and the
CUDA kernel + C ABI (nvcc, sm_103a only), linked with the shared CUDA runtime.
"""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libsmo_gemm.so")

CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
NVCC = os.path.join(CUDA_HOME, "bin", "nvcc")
GENCODE = "arch=compute_103a,code=sm_103a"

SOURCES_CU = ["capi.cu", "smem_probe.cu", "tc_probe.cu", "l2_probe.cu"]
SOURCES_CPP = ["planner.cpp"]
HEADERS = ["gemm_kernel.cuh", "gemm_kernel_pair.cuh", "gemm_common.cuh", "ptx.cuh", "gemm_params.h", "planner.h"]


def _inputs():
    files = [os.path.join(CSRC, f) for f in SOURCES_CU + SOURCES_CPP + HEADERS]
    files.extend(os.path.join(INCLUDE, h) for h in ("smo_gemm.h", "smo_probe.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB
    os.makedirs(OUT_DIR, exist_ok=True)
    inc = ["-I", CSRC, "-I", INCLUDE]
    objs, procs = [], []
    for src in SOURCES_CPP:
        obj = os.path.join(OUT_DIR, src + ".o")
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-c", os.path.join(CSRC, src), "-o", obj] + inc
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    for src in SOURCES_CU:
        obj = os.path.join(OUT_DIR, src + ".o")
        cmd = [NVCC, "-gencode", GENCODE, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
               "-Xptxas", "-v" if verbose else "-O3", "-c", os.path.join(CSRC, src), "-o", obj] + inc
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    for cmd, pr in procs:
        out, _ = pr.communicate()
        text = out.decode(errors="replace")
        if pr.returncode != 0:
            raise RuntimeError("build failed: " + " ".join(cmd) + "\n" + text)
        if verbose and text:
            print(text)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [NVCC, "-shared", "-gencode", GENCODE, "-cudart", "shared", "-o", tmp] + objs + [
        "-Xlinker", "-rpath," + os.path.join(CUDA_HOME, "lib64")]
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        raise RuntimeError("link failed: " + " ".join(cmd) + "\n" + r.stdout.decode(errors="replace"))
    os.replace(tmp, LIB)
    return LIB


def clean() -> None:
    if os.path.isdir(OUT_DIR):
        shutil.rmtree(OUT_DIR)


if __name__ == "__main__":
    import sys
    print(build(force=True, verbose="-v" in sys.argv))
