"""The allocation-free entry point gemm_ex_noalloc and its error report
gemm_check_noalloc, through the C ABI.

They serve callers that cannot allocate device memory: code whose device
memory belongs to a pool or arena allocator (a framework's caching allocator,
an inference runtime that hands a plugin a fixed workspace), or that must not
allocate once it is running (cudaMalloc may synchronise the device in the
middle of a latency-critical loop).  The kernel's scratch -- its error word --
lives in a static device array instead of a cudaMalloc'd word.  This file is
collected last on purpose, and it holds both alone in a fresh process and
after every other test; its own checks use gemm_check_noalloc, so nothing here
depends on the allocating entry points having run first.

Checked here:
  * two calls in a row give the output of the existing entry point gemm_ex,
    and the oracle's, within the parity tests' tolerances, on problems that
    run each kernel: one CTA (BN = 128), split K over a 2-CTA cluster, the
    CTA pair with 256 x 256 tiles and with 512 x 256 and 512 x 224 tiles, fp32
    and 16-bit output, both B orientations, a ragged shape and a batch;
  * a bounded-wait timeout of this variant is reported by gemm_check_noalloc,
    survives a later call until it is reported, is cleared by the report, and
    the next call is correct;
  * sizes beyond the limit are rejected with a clear status.
"""
import pytest
import torch

import shared_memory_operand_gb300 as smo
from synthetic import K_MAJOR, MN_MAJOR, make_problem, workload
from tests.gemm_check import check, oracle_full, run_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    smo.load_library(build=True)
    yield


# (problem, kernel the planner sends it to on a 152-SM GB300)
PROBLEMS = {
    "one_cta_bn128": lambda: workload("gemm_1500x1152x896_f16_f32"),
    "one_cta_ragged": lambda: make_problem(300, 520, 200, a_major=MN_MAJOR, b_major=K_MAJOR,
                                           out_dtype="bf16", dist="uniform", seed=5),
    "one_cta_f32": lambda: make_problem(129, 257, 65, a_major=K_MAJOR, b_major=MN_MAJOR, out_dtype="f32",
                                        dist="normal", seed=6),
    "one_cta_batch": lambda: make_problem(256, 384, 192, batch=3, out_dtype="bf16", dist="uniform", seed=7),
    "pair_256x256": lambda: make_problem(2048, 2048, 256, in_dtype="bf16", out_dtype="bf16",
                                         dist="uniform", seed=8),
    "pair_512x256": lambda: make_problem(3072, 3072, 3072, a_major=K_MAJOR, b_major=MN_MAJOR,
                                         in_dtype="bf16", out_dtype="bf16", dist="uniform", seed=9),
    "pair_512x224": lambda: make_problem(2048, 4096, 3072, a_major=K_MAJOR, b_major=MN_MAJOR,
                                         in_dtype="bf16", out_dtype="bf16", dist="uniform", seed=10),
    "split_k": lambda: make_problem(512, 512, 4096, a_major=K_MAJOR, b_major=MN_MAJOR,
                                    in_dtype="bf16", out_dtype="f32", dist="uniform", seed=11),
}
# tile width the planner picks (wide pairs) / whether it splits K
WIDTH = {"pair_512x256": 256, "pair_512x224": 224}


def _noalloc(p):
    return run_gpu(p, fn=smo.gemm_ex_noalloc, check_fn=smo.gemm_check_noalloc)


@pytest.mark.parametrize("name", list(PROBLEMS))
def test_noalloc_matches_gemm_ex_and_oracle_twice(name):
    p = PROBLEMS[name]()
    plan = smo.gemm_plan_describe(p.M, p.N, p.K, p.a_major, p.b_major, p.in_dtype, p.out_dtype,
                                  p.batch, torch.cuda.get_device_properties(0).multi_processor_count)
    if name.startswith("pair"):
        assert plan["pair"] == 1 and plan["wide"] == (1 if name in WIDTH else 0)
        if name in WIDTH:
            assert plan["BN"] == WIDTH[name]
    assert plan["split"] == (1 if name == "split_k" else 0)
    ref = oracle_full(p)
    existing = run_gpu(p)                              # the allocating entry point
    for _ in range(2):                                 # two calls in a row
        got = _noalloc(p)
        check(p, got, existing)                        # same product as gemm_ex
        check(p, got, ref)                             # and as the oracle


def test_noalloc_timeout_is_reported_then_cleared():
    """A stalled stage makes the kernel's bounded wait run out; the code lands
    in the static word, a later call does not erase it, gemm_check_noalloc
    reports it once and clears it, and the context stays usable."""
    assert smo.gemm_check_noalloc() == smo.GEMM_OK
    old = smo.gemm_set_timeout_ns(20_000_000)
    try:
        smo.gemm_debug_inject_stall(True)
        A = torch.zeros(512, 512, dtype=torch.bfloat16, device="cuda")
        C = torch.zeros(512, 512, dtype=torch.float32, device="cuda")
        smo.gemm_ex_noalloc(A, 512, 0, A, 512, 1, C, 512, 512, 512, 512, out_dtype="f32")
        smo.gemm_debug_inject_stall(False)
        smo.gemm_ex_noalloc(A, 512, 0, A, 512, 1, C, 512, 512, 512, 512, out_dtype="f32")   # healthy call
        assert smo.gemm_check_noalloc() == smo.GEMM_ERR_TIMEOUT
    finally:
        smo.gemm_debug_inject_stall(False)
        smo.gemm_set_timeout_ns(old)
    assert smo.gemm_check_noalloc() == smo.GEMM_OK     # cleared by the report
    p = PROBLEMS["pair_256x256"]()
    check(p, _noalloc(p), oracle_full(p))              # next call is correct


def test_noalloc_rejects_sizes_beyond_limit():
    A = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    C = torch.zeros(64, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(smo.GemmError) as e:
        smo.gemm_ex_noalloc(A, 64, 0, A, 64, 1, C, 64, 1 << 31, 64, 64)
    assert e.value.status == smo.GEMM_ERR_UNSUPPORTED
    with pytest.raises(smo.GemmError) as e:
        smo.gemm_ex_noalloc(A, 64, 0, A, 64, 1, C, 64, 64, 64, 64, batch=1 << 31)
    assert e.value.status == smo.GEMM_ERR_UNSUPPORTED
