"""Seeded random sweep of the CUDA path against the fp64 oracle (GPU).

Each case draws a shape (ragged M, N, K tails, batch 1-3, padded leading
dimensions), both operand orientations, the input type (bf16, f16, FP8 E4M3 /
E5M2), the output type, a tile mode (the planner's choice, or one forced:
128 / 256 one-CTA, 512 CTA pair, 1024 wide CTA pair) and stream-K (automatic or
forced on), and compares the whole output element by element.  A quarter of
the cases use integer inputs and must match bit for bit.
"""
import numpy as np
import pytest
import torch

import shared_memory_operand_gb300 as smo
from synthetic import make_problem
from tests.gemm_check import check, oracle_full, run_gpu

pytestmark = pytest.mark.gpu

N_CASES = 200


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    smo.load_library(build=True)
    yield


def _case(i):
    rng = np.random.default_rng(1000 + i)
    ind = ["bf16", "f16", "e4m3", "e5m2"][int(rng.integers(0, 4))]
    out = ["f32", "bf16", "f16"][int(rng.integers(0, 3))]
    if ind == "f16" and out == "bf16":
        out = "f16"
    dist = "int" if rng.random() < 0.25 else "uniform"
    if dist == "int":
        out = "f32"
    return dict(M=int(rng.integers(1, 700)), N=int(rng.integers(1, 700)), K=int(rng.integers(1, 1200)),
                batch=int(rng.integers(1, 4)), a_major=int(rng.integers(0, 2)), b_major=int(rng.integers(0, 2)),
                in_dtype=ind, out_dtype=out, dist=dist, ld_extra=int(rng.integers(0, 3)) * 16,
                mode=[None, 128, 256, 512, 1024][int(rng.integers(0, 5))],
                stream_k=bool(rng.random() < 0.3), seed=i)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case(i, monkeypatch):
    c = _case(i)
    if c["mode"]:
        monkeypatch.setenv("SMO_GEMM_FORCE_BN", str(c["mode"]))
    if c["stream_k"]:
        monkeypatch.setenv("SMO_GEMM_STREAM_K", "1")
    p = make_problem(c["M"], c["N"], c["K"], a_major=c["a_major"], b_major=c["b_major"],
                     in_dtype=c["in_dtype"], out_dtype=c["out_dtype"], dist=c["dist"], seed=c["seed"],
                     batch=c["batch"], ld_extra=c["ld_extra"])
    check(p, run_gpu(p), oracle_full(p), exact=c["dist"] == "int")
