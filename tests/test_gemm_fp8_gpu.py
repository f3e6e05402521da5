"""GPU parity of the 8-bit operand path (tcgen05.mma.kind::f8f6f4) against the
fp64 oracle, through the C ABI.

FP8 values multiply exactly and the tensor core accumulates in fp32, so the
tolerances are those of the 16-bit path (tests/gemm_check.py), and integer
inputs must match bit for bit.  The operands are E4M3 / E5M2 codes of the OCP
8-bit format ("An Educational GEMM Ladder for Helios GPUs": FP8 matrix units;
"A Deep Dive into LDS Optimizations on AMD Instinct MI450 GPUs", Part I: the
8-bit transposed load, whose GB300 counterpart is the MN-major descriptor).
"""
import numpy as np
import pytest
import torch

import shared_memory_operand_gb300 as smo
from synthetic import K_MAJOR, MN_MAJOR, make_problem, workload
from tests.gemm_check import check, oracle_full, run_gpu

pytestmark = pytest.mark.gpu

MAJORS = [(K_MAJOR, K_MAJOR), (K_MAJOR, MN_MAJOR), (MN_MAJOR, K_MAJOR), (MN_MAJOR, MN_MAJOR)]
FP8 = ["e4m3", "e5m2"]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    smo.load_library(build=True)
    yield


def _full(p, exact=False):
    return check(p, run_gpu(p), oracle_full(p), exact=exact)


@pytest.mark.parametrize("am,bm", MAJORS)
@pytest.mark.parametrize("dt", FP8)
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_small_ragged_all_orientations(am, bm, dt, out):
    # K = 65 / 200: one partial 128-deep stage; 129 x 257: ragged M and N
    for (M, N, K) in [(256, 256, 128), (300, 520, 200), (129, 257, 65), (1, 16, 32), (192, 384, 384)]:
        p = make_problem(M, N, K, a_major=am, b_major=bm, in_dtype=dt, out_dtype=out, dist="uniform",
                         seed=M + N + K)
        _full(p)


@pytest.mark.parametrize("mode", [128, 256, 512, 1024])
@pytest.mark.parametrize("am,bm", MAJORS)
def test_tile_modes_ragged(monkeypatch, mode, am, bm):
    monkeypatch.setenv("SMO_GEMM_FORCE_BN", str(mode))
    # (384, 640): MN extents multiples of 128 (one-instruction 4-D loads of
    # MN-major FP8 operands) but not of the tile
    for (M, N, K, out) in [(600, 700, 300, "bf16"), (257, 513, 129, "f32"), (384, 640, 256, "f32"),
                           (520, 1030, 1000, "f16")]:
        p = make_problem(M, N, K, a_major=am, b_major=bm, in_dtype="e4m3", out_dtype=out,
                         dist="uniform", seed=M + K + mode)
        _full(p)


@pytest.mark.parametrize("am,bm", MAJORS)
@pytest.mark.parametrize("dt", FP8)
def test_integer_inputs_bit_exact(am, bm, dt):
    """Integers in [-4, 4] are exact in both formats and every partial sum
    (|s| <= 16 K) is exact in fp32."""
    for (M, N, K) in [(200, 300, 1000), (256, 512, 4096)]:
        p = make_problem(M, N, K, a_major=am, b_major=bm, in_dtype=dt, out_dtype="f32", dist="int",
                         seed=3 + K)
        _full(p, exact=True)


@pytest.mark.parametrize("am,bm", MAJORS)
def test_permutation_operands_exact(am, bm):
    """A = permutation matrix: every output is one B element, moved; a wrong
    descriptor stride or major bit shows up as a moved row or column."""
    g = torch.Generator().manual_seed(21)
    K, N = 256, 384
    perm = torch.randperm(K, generator=g)
    p = make_problem(K, N, K, a_major=am, b_major=bm, in_dtype="e4m3", out_dtype="f32", dist="uniform",
                     seed=5)
    p.logical_A()[0].copy_(torch.eye(K)[perm].to(torch.float8_e4m3fn))
    gpu = run_gpu(p)
    want = p.logical_B()[0].to(torch.float64).numpy()[perm.numpy()]
    assert np.array_equal(gpu[0], want)


def test_batched_and_k_tails():
    for K in (1, 16, 127, 129, 383):
        p = make_problem(130, 260, K, in_dtype="e5m2", out_dtype="bf16", dist="uniform", seed=K, batch=3)
        _full(p)


def test_stream_k_full_compare(monkeypatch):
    """Stream-K on the CTA pair with FP8 stages (128 K per block)."""
    monkeypatch.setenv("SMO_GEMM_STREAM_K", "1")
    p = make_problem(1536, 2560, 4096, in_dtype="e4m3", out_dtype="f32", dist="uniform", seed=77)
    _full(p)
    q = make_problem(1536, 2560, 4096, in_dtype="e4m3", out_dtype="f32", dist="int", seed=78)
    _full(q, exact=True)


def test_alignment_rule_for_one_byte_elements():
    """FP8 leading dimensions must be multiples of 16 elements (16 bytes)."""
    A = torch.zeros(64 * 72, dtype=torch.uint8, device="cuda")
    B = torch.zeros(64 * 64, dtype=torch.uint8, device="cuda")
    C = torch.zeros(64 * 64, dtype=torch.float32, device="cuda")
    st = smo.gemm_ex_status(A, 72, 0, B, 64, 0, C, 64, 64, 64, 64, in_dtype="e4m3", out_dtype="f32")
    assert st == smo.GEMM_ERR_ALIGN
    st = smo.gemm_ex_status(A, 80, 0, B, 64, 0, C, 64, 64, 64, 64, in_dtype="e4m3", out_dtype="f32")
    assert st == smo.GEMM_OK
    assert smo.gemm_check(None) == smo.GEMM_OK


@pytest.mark.parametrize("name", ["gemm_8192_e4m3_bf16_AK_BN", "gemm_8192_e4m3_bf16_AK_BK"])
def test_config_8192_fp8(name):
    """Whole 8192^3 output against the oracle's whole product."""
    _full(workload(name))


def test_config_8192_fp8_integer_bit_exact():
    _full(workload("gemm_8192_e4m3_bf16_AK_BN", dist="int", out_dtype="f32"), exact=True)


@pytest.mark.parametrize("wbn", [224, 192, 160])
@pytest.mark.parametrize("am,bm", MAJORS)
def test_wide_tile_widths_fp8(wbn, am, bm, monkeypatch):
    """FP8 operands on 512 x wbn CTA-pair tiles (an N-major box is 128 values
    wide, so every half-width here is one box; each half starts on a 16-byte
    boundary, as TMA requires -- widths whose half does not are refused by the
    planner, tests/test_capi_host.py)."""
    monkeypatch.setenv("SMO_GEMM_FORCE_BN", "1024")
    monkeypatch.setenv("SMO_GEMM_WIDE_BN", str(wbn))
    for (M, N, K, out, dist) in [(600, 700, 384, "bf16", "uniform"), (1100, 1030, 520, "f32", "int")]:
        p = make_problem(M, N, K, a_major=am, b_major=bm, in_dtype="e4m3", out_dtype=out, dist=dist,
                         seed=M + wbn)
        _full(p, exact=(dist == "int"))


@pytest.mark.parametrize("am,bm", MAJORS)
def test_split_k_fp8(am, bm, monkeypatch):
    """Split-K over 2-CTA clusters with FP8 operands (fp32 output): 192-wide
    tiles, whose N-major B takes two 128-wide FP8 boxes per stage."""
    monkeypatch.setenv("SMO_GEMM_SPLIT_K", "1")
    for (M, N, K, dist) in [(1500, 1152, 896, "uniform"), (600, 700, 1000, "int")]:
        p = make_problem(M, N, K, a_major=am, b_major=bm, in_dtype="e4m3", out_dtype="f32", dist=dist,
                         seed=M + K)
        assert smo.gemm_plan_describe(M, N, K, am, bm, "e4m3", "f32")["split"] == 1
        _full(p, exact=(dist == "int"))


@pytest.mark.parametrize("bm,tail_bn", [(K_MAJOR, 176), (MN_MAJOR, 192)])
@pytest.mark.parametrize("out,dist", [("bf16", "uniform"), ("f32", "int")])
def test_batched_wide_tail_fp8(bm, tail_bn, out, dist):
    """FP8 operands in a batch whose last wave is re-tiled narrower across
    batch entries (an N-major FP8 B half-tile starts on a 16-byte boundary, so
    its tail width is a multiple of 32); integers bit-exact."""
    plan = smo.gemm_plan_describe(512, 1024, 4096, K_MAJOR, bm, "e4m3", out, 31)
    assert plan["wide"] and plan["tail"] and plan["tail_bn"] == tail_bn and plan["tail_b0"] == 19
    p = make_problem(512, 1024, 4096, a_major=K_MAJOR, b_major=bm, in_dtype="e4m3", out_dtype=out,
                     dist=dist, batch=31, seed=bm + 7)
    _full(p, exact=(dist == "int"))
