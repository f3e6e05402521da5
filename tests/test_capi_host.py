"""Host-side checks of the C-ABI library (no GPU): it builds, loads and exports
every symbol the header declares; arguments are validated before any device
work; and the layout planner's F2 model of every shared-memory layout agrees
with the oracle's independent restatement and bank simulator."""
import os
import re

import numpy as np
import pytest

import shared_memory_operand_gb300 as smo
from oracle import banksim

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    return smo.load_library(build=True)


def _header_functions():
    import glob
    text = "".join(open(f).read() for f in sorted(glob.glob(os.path.join(ROOT, "include", "*.h"))))
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z_][a-z0-9_]*)\s*\(", text)) - {"if", "defined"})


def test_exports_every_declared_symbol(lib):
    names = _header_functions()
    assert set(names) == set(smo.EXPORTS)
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings(lib):
    for st in range(0, -8, -1):
        s = smo.gemm_status_string(st)
        assert s and s != "unknown status"
    assert smo.gemm_status_string(-99) == "unknown status"


def _ex(A=0x1000, lda=64, am=0, B=0x2000, ldb=64, bm=1, C=0x3000, ldc=64, M=64, N=64, K=64,
        i=0, o=2, batch=1, sa=0, sb=0, sc=0):
    return smo.gemm_ex_status(A, lda, am, B, ldb, bm, C, ldc, M, N, K, i, o, batch, sa, sb, sc,
                              stream=0)


def test_argument_validation_without_device(lib):
    assert _ex(am=2) == smo.GEMM_ERR_ARG
    assert _ex(bm=-1) == smo.GEMM_ERR_ARG
    assert _ex(M=-1) == smo.GEMM_ERR_ARG
    assert _ex(batch=0) == smo.GEMM_ERR_ARG
    assert _ex(i=2) == smo.GEMM_ERR_UNSUPPORTED        # f32 operands
    assert _ex(o=7) == smo.GEMM_ERR_UNSUPPORTED
    assert _ex(M=0) == smo.GEMM_OK                       # empty product: no-op
    assert _ex(N=0, C=0) == smo.GEMM_OK
    assert _ex(C=0) == smo.GEMM_ERR_ARG
    assert _ex(A=0) == smo.GEMM_ERR_ARG
    assert _ex(ldc=63) == smo.GEMM_ERR_ARG
    assert _ex(lda=63) == smo.GEMM_ERR_ARG
    assert _ex(am=1, lda=64, M=65) == smo.GEMM_ERR_ARG  # M-major A needs lda >= M
    assert _ex(A=0x1008) == smo.GEMM_ERR_ALIGN
    assert _ex(C=0x3004) == smo.GEMM_ERR_ALIGN
    assert _ex(lda=68, K=66) == smo.GEMM_ERR_ALIGN      # 136-byte pitch
    assert _ex(o=0, ldc=68, N=66) == smo.GEMM_ERR_ALIGN
    assert _ex(batch=2, sa=64 * 64, sb=64 * 64, sc=64) == smo.GEMM_ERR_ARG   # C batches overlap
    assert _ex(batch=2, sa=4100, sb=4096, sc=4096) == smo.GEMM_ERR_ALIGN
    assert _ex(M=1 << 31) == smo.GEMM_ERR_UNSUPPORTED
    assert _ex(ldc=1 << 32) == smo.GEMM_ERR_UNSUPPORTED         # leading dimensions below 2^32
    assert _ex(lda=1 << 32) == smo.GEMM_ERR_UNSUPPORTED
    assert _ex(ldb=(1 << 32) + 64) == smo.GEMM_ERR_UNSUPPORTED
    assert _ex(batch=2, sa=1 << 39, sb=4096, sc=4096) == smo.GEMM_ERR_UNSUPPORTED   # 2^40 bytes
    assert _ex(batch=2, sa=4096, sb=4096, sc=1 << 38) == smo.GEMM_ERR_UNSUPPORTED   # fp32 C: 2^40 bytes
    assert _ex(i=5) == smo.GEMM_ERR_UNSUPPORTED        # no such input type
    # FP8 operands: one byte per element, so pitches need 16 elements
    assert _ex(i=3, lda=72, K=66) == smo.GEMM_ERR_ALIGN
    assert _ex(i=4, lda=80, bm=0, ldb=72, K=66) == smo.GEMM_ERR_ALIGN
    # well-formed arguments reach the device query: no GPU here
    if not _have_gpu():
        assert _ex() == smo.GEMM_ERR_NO_DEVICE
        assert _ex(K=0, lda=1 << 40) == smo.GEMM_ERR_NO_DEVICE   # K = 0: A and B unused
        assert _ex(i=3, lda=80, K=66) == smo.GEMM_ERR_NO_DEVICE
        assert smo.gemm_check(0) == smo.GEMM_ERR_NO_DEVICE


def _have_gpu():
    import torch
    return torch.cuda.is_available()


def test_timeout_knob(lib):
    old = smo.gemm_set_timeout_ns(12345)
    assert smo.gemm_set_timeout_ns(0) == 12345
    assert smo.gemm_set_timeout_ns(old) == 2_000_000_000


SHAPES = [(256, 256, 256), (1500, 1152, 896), (4096, 4096, 4096), (8192, 8192, 8192),
          (16384, 8192, 1024), (1, 1, 1), (129, 257, 65)]


@pytest.mark.parametrize("am", [0, 1])
@pytest.mark.parametrize("bm", [0, 1])
@pytest.mark.parametrize("out", ["f32", "bf16", "f16"])
def test_planner_layouts_match_oracle(lib, am, bm, out):
    for (M, N, K) in SHAPES:
        d = smo.gemm_plan_describe(M, N, K, am, bm, "bf16", out)
        assert d["ok"], d["why"]
        assert d["smem_bytes"] <= 232448
        # two accumulators, allocated as a power of two of columns
        tc = d["tmem_cols"]
        assert 2 * d["BN"] <= tc <= 512 and tc & (tc - 1) == 0 and tc < 4 * d["BN"]
        for name, major in (("A", am), ("B", bm)):
            op = d[name]
            tile = op["tile_mn"]          # per-CTA operand tile (half of BN in a pair)
            mn_major = bool(major)
            # planner's F2 basis images == oracle's 128B-swizzle TMA box layout
            # (one basis per bit of the largest row index: 8 for 192 rows)
            want_mn = [banksim.operand_tile_offset(1 << i, 0, mn_major, tile)
                       for i in range((tile - 1).bit_length())]
            want_k = [banksim.operand_tile_offset(0, 1 << i, mn_major, tile) for i in range(6)]
            assert op["basis_mn"] == want_mn
            assert op["basis_k"] == want_k
            # descriptor strides: the oracle's canonical layout with the
            # planner's LBO / SBO / K step reproduces the TMA layout exactly
            for mn in range(0, tile, 3):
                for k in range(64):
                    assert banksim.umma_canonical_offset(mn, k, mn_major, op["lbo"], op["sbo"],
                                                         op["kstep_bytes"]) == \
                        banksim.operand_tile_offset(mn, k, mn_major, tile)
            assert op["linear"] and op["bijective"] and op["tma_equals_umma"]
            assert op["core_matrix_divides"]
            # K-major: tile rows of 128 bytes; MN-major: whole 64-wide boxes
            # (a tile of 112 columns loads two, the MMA reads the first 112)
            loaded = -(-tile // 64) * 64 if mn_major else tile
            assert op["stage_bytes"] == loaded * 64 * 2


@pytest.mark.parametrize("am", [0, 1])
@pytest.mark.parametrize("bm", [0, 1])
@pytest.mark.parametrize("ind", ["e4m3", "e5m2"])
def test_planner_fp8_layouts_match_oracle(lib, am, bm, ind):
    """One-byte operands: a stage is 128 K values (one 128-byte swizzle row), an
    MMA takes 32, and an MN-major box is 128 MN values wide; the planner's F2
    bases and descriptor strides reproduce the oracle's layouts exactly."""
    for (M, N, K) in SHAPES:
        d = smo.gemm_plan_describe(M, N, K, am, bm, ind, "bf16")
        assert d["ok"], d["why"]
        assert d["BK"] == 128 and d["mma_k"] == 32 and d["kind"] == 1 and d["in_es"] == 1
        assert d["smem_bytes"] <= 232448
        for name, major in (("A", am), ("B", bm)):
            op = d[name]
            tile = op["tile_mn"]
            mn_major = bool(major)
            loaded = -(-tile // 128) * 128 if mn_major else tile
            want_mn = [banksim.operand_tile_offset(1 << i, 0, mn_major, tile, elem_bytes=1, box_k=128)
                       for i in range((loaded - 1).bit_length())]
            want_k = [banksim.operand_tile_offset(0, 1 << i, mn_major, tile, elem_bytes=1, box_k=128)
                      for i in range(7)]
            assert op["basis_mn"] == want_mn
            assert op["basis_k"] == want_k
            for mn in range(0, tile, 5):
                for k in range(128):
                    assert banksim.umma_canonical_offset(mn, k, mn_major, op["lbo"], op["sbo"],
                                                         op["kstep_bytes"], elem_bytes=1, mma_k=32) == \
                        banksim.operand_tile_offset(mn, k, mn_major, tile, elem_bytes=1, box_k=128)
            assert op["linear"] and op["bijective"] and op["tma_equals_umma"]
            assert op["core_matrix_divides"]
            assert op["stage_bytes"] == loaded * 128
            assert op["box"] == ([128, tile] if not mn_major else [128, 128])


@pytest.mark.parametrize("am", [0, 1])
@pytest.mark.parametrize("bm", [0, 1])
@pytest.mark.parametrize("ind", ["bf16", "e4m3"])
def test_wide_pair_plans(lib, monkeypatch, am, bm, ind):
    """Wide CTA pair (512 x 256 tiles): each CTA stages 256 rows of A, whose
    second 128-row half starts 16 KiB into the stage in every layout (the
    offset the issue loop adds); 4 stages of 48 KiB, one per barrier pair."""
    monkeypatch.setenv("SMO_GEMM_FORCE_BN", "1024")
    monkeypatch.setenv("SMO_GEMM_WIDE_BN", "256")
    es = 1 if ind == "e4m3" else 2
    bk = 128 // es
    for (M, N, K) in [(8192, 8192, 8192), (1500, 1152, 896), (129, 257, 65)]:
        d = smo.gemm_plan_describe(M, N, K, am, bm, ind, "bf16")
        assert d["ok"], d["why"]
        assert d["pair"] and d["wide"] and d["BM"] == 512 and d["BN"] == 256
        assert d["stages"] == 4 and d["kgroup"] == 1 and d["tmem_cols"] == 512
        assert d["smem_bytes"] <= 232448
        assert ((d["idesc"] >> 24) & 31) * 16 == 256 and ((d["idesc"] >> 17) & 63) * 8 == 256
        A = d["A"]
        assert A["tile_mn"] == 256 and A["stage_bytes"] == 256 * 128
        assert A["linear"] and A["bijective"] and A["tma_equals_umma"] and A["core_matrix_divides"]
        for mn in range(0, 256, 7):
            for k in range(0, bk, 3):
                off = banksim.operand_tile_offset(mn, k, bool(am), 256, elem_bytes=es, box_k=bk)
                assert banksim.umma_canonical_offset(mn, k, bool(am), A["lbo"], A["sbo"], A["kstep_bytes"],
                                                     elem_bytes=es, mma_k=32 // es) == off
                if mn >= 128:       # the second half, read by descriptors 16 KiB further on
                    assert off - banksim.operand_tile_offset(mn - 128, k, bool(am), 256, elem_bytes=es,
                                                             box_k=bk) == 16384
        assert d["B"]["tile_mn"] == 128 and d["stage_stride"] == 256 * 128 + 128 * 128


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_epilogue_stores_conflict_free(lib, out):
    d = smo.gemm_plan_describe(1024, 1024, 1024, 0, 1, "bf16", out)
    c = d["C"]
    assert c["chunk_cols"] * (4 if out == "f32" else 2) == 128
    seen = set()
    for addrs in c["store_addrs"]:
        rep = banksim.simulate(addrs, 16)
        assert rep.degree == 1, addrs
        assert rep.wavefronts == 4
        for a in addrs:
            assert a % 16 == 0
            assert d["off_epi"] <= a < d["off_bar"]
            seen.update(range(a, a + 16))
    # 4 warps x 2 buffers x 4 KiB, every byte written by exactly one (lane, store)
    assert len(seen) == 4 * 2 * 4096
    # the same chunk without the swizzle: the 8-way control
    rows = [c["store_addrs"][0][0] + 128 * l for l in range(32)]
    assert banksim.simulate(rows, 16).degree == 8


def test_instruction_descriptor_fields(lib):
    """Field layout of the tcgen05 kind::f16 instruction descriptor (PTX ISA):
    D fmt bits 4-5, A fmt 7-9, B fmt 10-12, A/B major 15/16, N>>3 17-22,
    M>>4 24-28."""
    for am in (0, 1):
        for bm in (0, 1):
            for ind, fmt in (("bf16", 1), ("f16", 0)):
                d = smo.gemm_plan_describe(2048, 2048, 2048, am, bm, ind, "f32")
                x = d["idesc"]
                assert (x >> 4) & 3 == 1
                assert (x >> 7) & 7 == fmt and (x >> 10) & 7 == fmt
                assert (x >> 15) & 1 == am and (x >> 16) & 1 == bm
                assert ((x >> 17) & 63) * 8 == d["BN"]
                assert ((x >> 24) & 31) * 16 == min(d["BM"], 256)
                assert x & 0b1111 == 0 and (x >> 13) & 3 == 0 and (x >> 23) & 1 == 0


def test_instruction_descriptor_fp8_fields(lib):
    """kind::f8f6f4 instruction descriptor: A / B format E4M3 = 0, E5M2 = 1 in
    bits 7-9 / 10-12, the other fields as for kind::f16."""
    for am in (0, 1):
        for bm in (0, 1):
            for ind, fmt in (("e4m3", 0), ("e5m2", 1)):
                d = smo.gemm_plan_describe(4096, 4096, 4096, am, bm, ind, "bf16")
                x = d["idesc"]
                assert (x >> 4) & 3 == 1
                assert (x >> 7) & 7 == fmt and (x >> 10) & 7 == fmt
                assert (x >> 15) & 1 == am and (x >> 16) & 1 == bm
                # a wide 512-row tile issues two MMAs of M = 256 (one per 128-row half per CTA)
                assert ((x >> 17) & 63) * 8 == d["BN"] and ((x >> 24) & 31) * 16 == min(d["BM"], 256)
                assert d["num_k"] == 4096 // 128


def test_tile_choice_and_grid(lib):
    # tile-starved: 128 x 128 one-CTA tiles on 108 SMs; splitting K (72 tiles of
    # 128 x 192 on 144 SMs) is modelled, and measured, slower at K = 896
    for out in ("f32", "f16"):
        d = smo.gemm_plan_describe(1500, 1152, 896, 0, 1, "f16", out)
        assert not d["pair"] and not d["split"] and d["BN"] == 128 and d["tiles"] == 12 * 9
        assert d["grid"] == 108
    # long K, few tiles, fp32 out: K split over 2-CTA clusters
    d = smo.gemm_plan_describe(1500, 1152, 2688, 0, 1, "f16", "f32")
    assert d["split"] and d["BN"] == 192 and d["tiles"] == 12 * 6 and d["grid"] == 144
    assert d["split_kh"] == 21 and d["stages"] == 4 and d["tmem_cols"] == 512
    x = d["idesc"]
    assert ((x >> 24) & 31) * 16 == 128 and ((x >> 17) & 63) * 8 == 192
    d = smo.gemm_plan_describe(512, 512, 4096, 0, 1, "bf16", "f32")
    assert d["split"] and d["BN"] == 128 and d["grid"] == 32 and d["split_kh"] == 32
    d = smo.gemm_plan_describe(512, 512, 4096, 0, 1, "bf16", "bf16")      # 16-bit out: never split
    assert not d["split"] and d["grid"] == 16
    # short K: no split
    d = smo.gemm_plan_describe(256, 256, 256, 0, 1, "bf16", "f32")
    assert not d["split"] and d["BN"] == 128 and d["grid"] == 4
    # long K: the wide pair (512 x 256 tiles); short K: 256 x 256
    d = smo.gemm_plan_describe(8192, 8192, 8192, 0, 1, "bf16", "bf16")
    assert d["pair"] and d["wide"] and d["BM"] == 512 and d["BN"] == 256
    assert d["tiles"] == 6 * 76 + 72 and d["tail"] and d["tail_bn"] == 208        # see test_wide_tail_*
    assert d["grid"] == 152 and d["stages"] == 4 and d["A"]["tile_mn"] == 256 and d["B"]["tile_mn"] == 128
    d = smo.gemm_plan_describe(16384, 8192, 1024, 0, 1, "bf16", "bf16")
    assert d["pair"] and not d["wide"] and d["BM"] == 256 and d["tiles"] == 64 * 32
    assert d["grid"] == 152 and d["stages"] == 6 and d["A"]["tile_mn"] == d["B"]["tile_mn"] == 128
    # 32 K blocks: wide 512 x 256 tiles (measured +1.8% over 256 x 256 here)
    d = smo.gemm_plan_describe(2048, 2048, 2048, 0, 1, "bf16", "bf16", batch=32)
    assert d["pair"] and d["wide"] and d["BN"] == 256 and d["tail_start"] == 13 * 76
    assert d["tail"] and d["tail_bn"] == 128 and d["tiles"] == 13 * 76 + 72      # the last wave re-tiled


def test_epilogue_warps_by_plan(lib, monkeypatch):
    """Eight epilogue warps (320 threads) for wide pairs and for one-CTA
    launches whose CTAs each hold one tile of at most four column chunks;
    four (192 threads) otherwise."""
    d = smo.gemm_plan_describe(1500, 1152, 896, 0, 1, "f16", "f32")        # 108 tiles, 4 fp32 chunks
    assert d["threads"] == 320 and d["tiles"] <= d["grid"] and d["C"]["chunks"] == 4
    d = smo.gemm_plan_describe(256, 256, 256, 0, 1, "bf16", "bf16")        # 4 tiles, 2 bf16 chunks
    assert d["threads"] == 320
    d = smo.gemm_plan_describe(512, 512, 4096, 0, 1, "bf16", "f32")        # split K: four warps
    assert d["split"] and d["threads"] == 192
    d = smo.gemm_plan_describe(8192, 8192, 8192, 0, 1, "bf16", "bf16")     # wide pair
    assert d["wide"] and d["threads"] == 320
    d = smo.gemm_plan_describe(16384, 8192, 1024, 0, 1, "bf16", "bf16")    # 256 x 256 pair
    assert d["pair"] and not d["wide"] and d["threads"] == 192
    monkeypatch.setenv("SMO_GEMM_FORCE_BN", "256")
    d = smo.gemm_plan_describe(2048, 2048, 1024, 0, 1, "bf16", "f32")      # one wave, 8 fp32 chunks
    assert d["tiles"] <= d["grid"] and d["C"]["chunks"] == 8 and d["threads"] == 192
    d = smo.gemm_plan_describe(2048, 2048, 1024, 0, 1, "bf16", "bf16")     # one wave, 4 bf16 chunks
    assert d["threads"] == 320
    monkeypatch.setenv("SMO_GEMM_FORCE_BN", "128")
    d = smo.gemm_plan_describe(4096, 4096, 1024, 0, 1, "bf16", "bf16")     # several tiles per CTA
    assert d["tiles"] > d["grid"] and d["threads"] == 192


def test_epilogue_pacing_by_plan(lib):
    """256 x 256 pair tiles with 16-bit output space their chunk stores (48 ns
    per K block for 16-bit operands, 24 for FP8, whose K blocks take half the
    time); fp32 output, wide and one-CTA tiles store back to back."""
    d = smo.gemm_plan_describe(16384, 8192, 1024, 0, 1, "bf16", "bf16")
    assert d["pair"] and not d["wide"] and d["epi_pace_ns_per_kb"] == 48
    d = smo.gemm_plan_describe(16384, 8192, 2048, 0, 1, "e4m3", "bf16")
    assert d["pair"] and not d["wide"] and d["epi_pace_ns_per_kb"] == 24
    d = smo.gemm_plan_describe(16384, 8192, 1024, 0, 1, "bf16", "f32")
    assert d["pair"] and not d["wide"] and d["epi_pace_ns_per_kb"] == 0
    d = smo.gemm_plan_describe(8192, 8192, 8192, 0, 1, "bf16", "bf16")
    assert d["wide"] and d["epi_pace_ns_per_kb"] == 0
    d = smo.gemm_plan_describe(1500, 1152, 896, 0, 1, "f16", "f16")
    assert not d["pair"] and d["epi_pace_ns_per_kb"] == 0


def test_split_k_policy(lib, monkeypatch):
    """Split-K is taken for fp32 output only, on one-CTA tiles; forced on it
    still keeps at least one K block per CTA; forced off the plan is the
    one-CTA 128 x 128 tiling."""
    monkeypatch.setenv("SMO_GEMM_SPLIT_K", "0")
    d = smo.gemm_plan_describe(512, 512, 4096, 0, 1, "bf16", "f32")
    assert not d["split"] and d["grid"] == 16
    monkeypatch.setenv("SMO_GEMM_SPLIT_K", "0")
    d = smo.gemm_plan_describe(1500, 1152, 896, 0, 1, "f16", "f32")
    assert not d["split"] and d["BN"] == 128 and d["grid"] == 108
    monkeypatch.setenv("SMO_GEMM_SPLIT_K", "1")
    d = smo.gemm_plan_describe(256, 256, 256, 0, 1, "bf16", "f32")
    assert d["split"] and d["split_kh"] == 2 and d["grid"] == 2 * d["tiles"]
    d = smo.gemm_plan_describe(256, 256, 64, 0, 1, "bf16", "f32")       # one K block: nothing to split
    assert not d["split"]
    d = smo.gemm_plan_describe(256, 256, 256, 0, 1, "bf16", "bf16")      # 16-bit output: never split
    assert not d["split"]
    d = smo.gemm_plan_describe(4096, 4096, 4096, 0, 1, "bf16", "f32")    # CTA-pair plans: never split
    assert d["pair"] and not d["split"]
    d = smo.gemm_plan_describe(1500, 1152, 896, 0, 1, "f16", "f32")      # forced on: narrowest one-wave width
    assert d["split"] and d["BN"] == 192 and d["grid"] == 2 * 12 * 6 and d["split_kh"] == 7
    monkeypatch.setenv("SMO_GEMM_FORCE_BN", "256")
    d = smo.gemm_plan_describe(1500, 1152, 896, 0, 1, "f16", "f32")
    assert d["split"] and d["BN"] == 256 and d["grid"] == 2 * 12 * 5 and d["split_kh"] == 7


def test_wide_tile_width_by_wave_quantisation(lib):
    """4096^2 on 76 clusters: 128 tiles of 512 x 256 run in 2 waves, the
    second 52/76 full; 152 tiles of 512 x 224 fill both waves exactly with 7/8
    of the work per tile.  8192^2: 512 x 256 tiles (7 waves), as 224 would
    need 8.  Each CTA then stages 112 B columns: one 112-row box (K-major) or
    two 64-wide boxes (N-major, the MMA reading the first 112); the bf16
    epilogue has 3 whole 64-column chunks and a 32-column one."""
    for am in (0, 1):
        for bm in (0, 1):
            d = smo.gemm_plan_describe(4096, 4096, 4096, am, bm, "bf16", "bf16")
            assert d["wide"] and d["BN"] == 224 and d["tiles"] == 8 * 19 and d["grid"] == 152
            B = d["B"]
            assert B["tile_mn"] == 112
            assert (B["nbox"], B["stage_bytes"]) == ((2, 16384) if bm else (1, 112 * 128))
            assert B["linear"] and B["bijective"] and B["tma_equals_umma"] and B["core_matrix_divides"]
            assert d["C"]["chunks"] == 4 and d["C"]["last_cols"] == 32
            x = d["idesc"]
            assert ((x >> 24) & 31) * 16 == 256 and ((x >> 17) & 63) * 8 == 224
            assert d["tmem_cols"] == 512
    d = smo.gemm_plan_describe(4096, 4096, 4096, 0, 1, "bf16", "f32")
    assert d["BN"] == 224 and d["C"]["chunks"] == 7 and d["C"]["last_cols"] == 32
    d = smo.gemm_plan_describe(8192, 8192, 8192, 0, 1, "bf16", "bf16")
    assert d["wide"] and d["BN"] == 256 and d["C"]["chunks"] == 4 and d["C"]["last_cols"] == 64


def test_tma_coordinate_rule_refuses_unaligned_widths(lib, monkeypatch):
    """A tiled TMA copy whose innermost coordinate times the element size is
    not a multiple of 16 bytes faults the GPU.  With one-byte operands and an
    N-major B, a pair tile of width w gives each CTA w / 2 columns: w / 2 must
    be a multiple of 16.  The planner refuses such a forced width (no launch)
    and its own choice never takes one."""
    monkeypatch.setenv("SMO_GEMM_FORCE_BN", "1024")
    for w in (208, 240, 112, 48):
        monkeypatch.setenv("SMO_GEMM_WIDE_BN", str(w))
        d = smo.gemm_plan_describe(600, 700, 384, 0, 1, "e4m3", "bf16")
        assert not d["ok"] and "TMA" in d["why"]
        assert smo.gemm_plan_describe(600, 700, 384, 0, 0, "e4m3", "bf16")["ok"]     # K-major B: fine
        assert smo.gemm_plan_describe(600, 700, 384, 0, 1, "bf16", "bf16")["ok"]     # 2-byte: fine
    monkeypatch.delenv("SMO_GEMM_WIDE_BN")
    for M, N in [(4096, 4096), (2048, 6144), (1536, 1000)]:
        d = smo.gemm_plan_describe(M, N, 8192, 0, 1, "e4m3", "bf16")
        assert d["ok"] and (d["BN"] // 2) % 16 == 0
    # every plan's MN-major coordinates are 16-byte aligned, whatever the width
    for w in range(16, 257, 16):
        monkeypatch.setenv("SMO_GEMM_WIDE_BN", str(w))
        for ind, es in (("bf16", 2), ("e4m3", 1)):
            d = smo.gemm_plan_describe(1000, 1000, 512, 1, 1, ind, "bf16")
            if d["ok"]:
                assert (d["BN"] * es) % 16 == 0 and (d["B"]["tile_mn"] * es) % 16 == 0
                assert (d["A"]["tile_mn"] * es) % 16 == 0


def _tiles_of(d):
    """The output rectangles (batch entry, first row, first column, width) of
    a plan's tiles, decoded as the wide CTA-pair kernel decodes them: tiles
    before tail_start problem by problem, in groups of group_m M blocks,
    column-major inside a group; the tail region in column blocks of
    tail_gsz tiles, tail_bn wide -- tail_k0 tiles of problem tail_b0 from
    column tail_n0, then tail_kfull per later problem from column 0."""
    BM, BN, gm = d["BM"], d["BN"], d["group_m"]
    num_m, num_n = d["num_m"], d["num_n"]
    per_batch = num_m * num_n
    out = []
    for t in range(d["tiles"]):
        if d["tail"] and t >= d["tail_start"]:
            r = t - d["tail_start"]
            b, base = d["tail_b0"], d["tail_n0"]
            if r >= d["tail_k0"]:
                r -= d["tail_k0"]
                j = r // d["tail_kfull"]
                b, r, base = b + 1 + j, r - j * d["tail_kfull"], 0
            mb = d["tail_m0"] + r % d["tail_gsz"]
            out.append((b, mb * BM, base + (r // d["tail_gsz"]) * d["tail_bn"], d["tail_bn"]))
            continue
        b, r = divmod(t, per_batch)
        span = gm * num_n
        g = r // span
        first = g * gm
        gsz = min(num_m - first, gm)
        rr = r - g * span
        out.append((b, (first + rr % gsz) * BM, (rr // gsz) * BN, BN))
    return out


def _assert_covers_once(d, M, N, batch=1):
    cover = np.zeros((batch, -(-M // 512) * 512, N + 256), dtype=np.int8)
    for (b, m0, n0, w) in _tiles_of(d):
        assert 0 <= b < batch
        cover[b, m0:m0 + 512, n0:n0 + w] += 1
    assert np.all(cover[:, :M, :N] == 1)


@pytest.mark.parametrize("M,N,K,bm,ind", [(8192, 8192, 8192, 1, "bf16"), (8192, 8192, 8192, 0, "bf16"),
                                          (8192, 8192, 8192, 1, "e4m3"), (4096, 6912, 3072, 1, "bf16"),
                                          (6144, 4608, 3072, 0, "bf16"), (6144, 6144, 3072, 1, "f16")])
def test_wide_tail_covers_the_output_once(lib, M, N, K, bm, ind):
    """The last, partial wave of a 256-wide wide tiling is re-tiled narrower:
    the tiles (main ones up to tail_start, then the tail's) cover every
    output element exactly once, the tail fits one wave of 76 clusters, the
    main tiles fill whole waves, and the tail width keeps the TMA rule."""
    d = smo.gemm_plan_describe(M, N, K, 0, bm, ind, "bf16")
    assert d["ok"] and d["wide"] and d["tail"], d
    assert d["tail_start"] % 76 == 0 and d["tail_tiles"] <= 76 and d["tail_bn"] < 256
    es = 1 if ind == "e4m3" else 2
    if bm:
        assert (d["tail_bn"] // 2 * es) % 16 == 0 and (d["tail_n0"] * es) % 16 == 0
    x = d["tail_idesc"]
    assert ((x >> 17) & 63) * 8 == d["tail_bn"] and ((x >> 24) & 31) * 16 == 256
    _assert_covers_once(d, M, N)


@pytest.mark.parametrize("M,N,batch,bm,later", [
    (2048, 2048, 32, 1, 1),      # the batched workload: last column of entry 30, all of entry 31
    (2048, 2048, 32, 0, 1),
    (1024, 2048, 31, 1, 2),      # the tail spans three entries
    (2048, 1280, 21, 1, 1),      # the first entry the tail touches is re-tiled whole
    (1500, 2048, 12, 1, 2),      # ragged M (three M blocks, the last one 476 rows)
    (2560, 2048, 20, 1, 0),      # five M blocks
    (1024, 4096, 31, 1, 0),      # 16-wide tail tiles
])
def test_batched_wide_tail_covers_every_entry_once(lib, M, N, batch, bm, later):
    """A batch of problems that are one M group each: the tiles left for a
    last, partial wave are whole columns at the end of the order, from the
    last columns of one problem and all of the problems after it; re-tiled
    narrower, they fit one wave and every output element of every problem
    is covered exactly once."""
    d = smo.gemm_plan_describe(M, N, 2048, 0, bm, "bf16", "bf16", batch, 152)
    assert d["ok"] and d["wide"] and d["tail"], d
    assert d["group_m"] == d["num_m"] and d["tail_start"] % 76 == 0 and d["tail_tiles"] <= 76
    assert (d["tail_tiles"] - d["tail_k0"]) // d["tail_kfull"] == later
    assert d["tail_b0"] == batch - 1 - later and d["tail_bn"] < 256
    if bm:
        assert (d["tail_bn"] // 2 * 2) % 16 == 0
    _assert_covers_once(d, M, N, batch)


def test_wide_tail_off_when_forced_or_full(lib, monkeypatch):
    d = smo.gemm_plan_describe(4096, 4096, 4096, 0, 1, "bf16", "bf16")     # two full waves of 224
    assert not d["tail"]
    monkeypatch.setenv("SMO_GEMM_WIDE_BN", "256")
    d = smo.gemm_plan_describe(8192, 8192, 8192, 0, 1, "bf16", "bf16")     # uniform 512 x 256
    assert not d["tail"] and d["tiles"] == 16 * 32


def test_pair_descriptors(lib, monkeypatch):
    """CTA pair: M = 256 and N = 256 in the instruction descriptor, each CTA
    stages 128 rows of A and 128 columns of B per 64-deep stage."""
    monkeypatch.setenv("SMO_GEMM_FORCE_BN", "512")
    for am in (0, 1):
        for bm in (0, 1):
            d = smo.gemm_plan_describe(8192, 8192, 8192, am, bm, "bf16", "bf16")
            x = d["idesc"]
            assert ((x >> 24) & 31) * 16 == 256 and ((x >> 17) & 63) * 8 == 256
            assert d["stage_stride"] == 2 * 128 * 64 * 2
            assert d["tmem_cols"] == 512


def test_wide_tail_random_shapes_cover_once(lib):
    """Seeded random shapes, batches, orientations and operand types: whenever
    the planner re-tiles a wide tiling's last wave, every output element of
    every batch entry is covered exactly once, the tail fits one wave of 76
    clusters and keeps the TMA coordinate rule."""
    rng = np.random.default_rng(12345)
    seen = 0
    for _ in range(1500):
        batch = int(rng.choice([1, 1, 1, 2, 3, 5, 8, 12, 17, 31, 32, 40]))
        M = int(rng.integers(256, 12000 if batch == 1 else 3000))
        N = int(rng.integers(256, 12000 if batch == 1 else 3000)) // 16 * 16 + 16
        if batch * M * N > 60_000_000:
            continue
        ind = str(rng.choice(["bf16", "f16", "e4m3"]))
        bm = int(rng.integers(0, 2))
        K = 8192 if ind == "e4m3" else 4096
        d = smo.gemm_plan_describe(M, N, K, 0, bm, ind, "bf16", batch, 152)
        if not (d["ok"] and d["wide"] and d["tail"]):
            continue
        seen += 1
        es = 1 if ind == "e4m3" else 2
        assert d["tail_start"] % 76 == 0 and 0 < d["tail_tiles"] <= 76 and 16 <= d["tail_bn"] < 256
        if bm:
            assert (d["tail_bn"] // 2 * es) % 16 == 0 and (d["tail_n0"] * es) % 16 == 0
        _assert_covers_once(d, M, N, batch)
    assert seen >= 30
