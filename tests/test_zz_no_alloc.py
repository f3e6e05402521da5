"""The allocation-free entry point gemm_ex_noalloc, through the C ABI.

It serves callers that cannot allocate device memory -- code whose device
memory belongs to a pool or arena allocator, or that must not allocate once it
is running.  Its kernel's scratch lives in a static device array instead of a
cudaMalloc'd word.  This file is collected last on purpose, and the test holds
both alone in a fresh process and after every other test.

Checked here: two calls in a row produce the output of the existing entry point
gemm_ex, within the tolerances the parity tests use, on several problems
(fp32 and bf16 output, N-major and K-major B, a ragged shape, a batch), and the
variant rejects sizes beyond its limit with a clear status.
"""
import pytest
import torch

import shared_memory_operand_gb300 as smo
from synthetic import K_MAJOR, MN_MAJOR, make_problem, workload
from tests.gemm_check import check, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    smo.load_library(build=True)
    yield


PROBLEMS = [
    lambda: workload("gemm_1500x1152x896_f16_f32"),
    lambda: make_problem(300, 520, 200, a_major=MN_MAJOR, b_major=K_MAJOR, out_dtype="bf16",
                         dist="uniform", seed=5),
    lambda: make_problem(129, 257, 65, a_major=K_MAJOR, b_major=MN_MAJOR, out_dtype="f32",
                         dist="normal", seed=6),
    lambda: make_problem(256, 384, 192, batch=3, out_dtype="bf16", dist="uniform", seed=7),
]


@pytest.mark.parametrize("make", PROBLEMS)
def test_noalloc_matches_gemm_ex_twice(make):
    p = make()
    ref = run_gpu(p)                                   # existing entry point
    for _ in range(2):                                 # two calls in a row
        got = run_gpu(p, fn=smo.gemm_ex_noalloc)
        check(p, got, ref)


def test_noalloc_rejects_sizes_beyond_limit():
    A = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(64, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(smo.GemmError) as e:
        smo.gemm_ex_noalloc(A, 64, 0, A, 64, 1, C, 64, 1 << 31, 64, 64)
    assert e.value.status == smo.GEMM_ERR_UNSUPPORTED
    with pytest.raises(smo.GemmError) as e:
        smo.gemm_ex_noalloc(A, 64, 0, A, 64, 1, C, 64, 64, 64, 64, batch=1 << 31)
    assert e.value.status == smo.GEMM_ERR_UNSUPPORTED
