"""Compile the oracle's C GEMM into ``oracle/_build/libgemm_ref.so``.

TEST INFRASTRUCTURE ONLY: the library this builds is the parity oracle, loaded
by ``tests/``, the smoke check and the bench's CPU baseline leg, never by the
product path.  Plain gcc, no CUDA; ``-ffp-contract=off`` keeps every multiply
and add a separately rounded IEEE double operation on every host architecture.
"""
from __future__ import annotations

import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gemm_ref.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libgemm_ref.so")


def build(force: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", "-Wall", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
