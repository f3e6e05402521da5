"""Pins for the oracle's 8-bit operand path (CPU only).

The FP8 formats are those of the OCP 8-bit floating point specification, the
plainest reading of the "FP8" the pages name ("An Educational GEMM Ladder for
Helios GPUs": matrix units for BF16, FP8, FP6 and FP4; "A Deep Dive into LDS
Optimizations on AMD Instinct MI450 GPUs", Part I: the 8-bit transposed load).
Each check ties the oracle to something other than itself: torch's float8
conversions over all 256 codes, values fixed by the format definition, exact
rational products, identity / permutation / closed-form products and numpy's
BLAS product.
"""
import itertools
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import gemm as og
from synthetic import K_MAJOR, MN_MAJOR, make_problem

MAJORS = [(K_MAJOR, K_MAJOR), (K_MAJOR, MN_MAJOR), (MN_MAJOR, K_MAJOR), (MN_MAJOR, MN_MAJOR)]
TORCH_FP8 = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


def _oracle(p):
    return og.gemm_f64(p.bits("A"), p.lda, p.a_major, p.bits("B"), p.ldb, p.b_major,
                       p.in_dtype, p.M, p.N, p.K, p.batch, p.strideA, p.strideB)


# ---------------------------------------------------------------- decoding
@pytest.mark.parametrize("dt", ["e4m3", "e5m2"])
def test_decode_matches_torch_all_codes(dt):
    codes = np.arange(256, dtype=np.uint8)
    ours = og.decode8(codes, dt)
    ref = torch.from_numpy(codes.copy()).view(TORCH_FP8[dt]).to(torch.float64).numpy()
    same = (ours == ref) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


@pytest.mark.parametrize("dt", ["e4m3", "e5m2"])
def test_exact_values_match_torch_all_finite_codes(dt):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(TORCH_FP8[dt]).to(torch.float64).numpy()
    for c in codes:
        if np.isfinite(ref[c]):
            assert og.exact_value8(int(c), dt) == Fraction(float(ref[c]))


def test_format_landmarks():
    d4 = lambda c: og.decode8(np.array([c], dtype=np.uint8), "e4m3")[0]
    d5 = lambda c: og.decode8(np.array([c], dtype=np.uint8), "e5m2")[0]
    # E4M3: bias 7, 3 fraction bits, no infinities, S.1111.111 is the only NaN
    assert d4(0x38) == 1.0 and d4(0xB8) == -1.0
    assert d4(0x7E) == 448.0 and d4(0xFE) == -448.0        # 1.110b x 2^8
    assert d4(0x78) == 256.0                               # all-ones exponent is a normal binade
    assert d4(0x08) == 2.0 ** -6                           # smallest normal
    assert d4(0x01) == 2.0 ** -9 and d4(0x07) == 7 * 2.0 ** -9
    assert np.isnan(d4(0x7F)) and np.isnan(d4(0xFF))
    assert d4(0x00) == 0.0 and np.signbit(d4(0x80))
    # E5M2: bias 15, 2 fraction bits, IEEE infinities and NaNs
    assert d5(0x3C) == 1.0 and d5(0x7B) == 57344.0          # 1.11b x 2^15
    assert d5(0x7C) == np.inf and d5(0xFC) == -np.inf
    assert np.isnan(d5(0x7D)) and np.isnan(d5(0x7F))
    assert d5(0x04) == 2.0 ** -14 and d5(0x01) == 2.0 ** -16


def test_small_integers_exact_in_both_formats():
    for dt in ("e4m3", "e5m2"):
        p = make_problem(9, 1, 1, in_dtype=dt, dist="int", seed=1)
        vals = p.logical_A().to(torch.float64).numpy().reshape(-1)
        assert np.array_equal(vals, np.round(vals)) and np.abs(vals).max() <= 4


# ---------------------------------------------------------------- the GEMM
@pytest.mark.parametrize("am,bm", MAJORS)
@pytest.mark.parametrize("dt", ["e4m3", "e5m2"])
def test_bruteforce_exact_tiny(am, bm, dt):
    """Products of FP8 values are exact in fp64 and these short sums stay
    exact, so the fp64 product must equal the rational one."""
    for (M, N, K) in [(1, 1, 1), (3, 5, 7), (8, 8, 8), (5, 2, 19)]:
        p = make_problem(M, N, K, a_major=am, b_major=bm, in_dtype=dt, dist="uniform",
                         seed=M * 100 + N * 10 + K, ld_extra=3)
        c = _oracle(p)
        exact = og.exact_gemm(p.bits("A"), p.lda, p.a_major, p.bits("B"), p.ldb, p.b_major,
                              p.in_dtype, M, N, K)
        for m, n in itertools.product(range(M), range(N)):
            assert Fraction(c[0, m, n]) == exact[0][m][n]


@pytest.mark.parametrize("am,bm", MAJORS)
def test_identity_and_permutation(am, bm):
    g = torch.Generator().manual_seed(17)
    K, N, M = 32, 48, 19
    for dt in ("e4m3", "e5m2"):
        B = (torch.rand(K, N, generator=g) * 2 - 1).to(TORCH_FP8[dt]).float()
        perm = torch.randperm(K, generator=g)
        for A, want in ((torch.eye(K), B), (torch.eye(K)[perm], B[perm])):
            p = make_problem(K, N, K, a_major=am, b_major=bm, in_dtype=dt, dist="ones", ld_extra=16)
            p.logical_A()[0].copy_(A.to(TORCH_FP8[dt]))
            p.logical_B()[0].copy_(B.to(TORCH_FP8[dt]))
            assert np.array_equal(_oracle(p)[0], want.double().numpy())
        A = (torch.rand(M, K, generator=g) * 2 - 1).to(TORCH_FP8[dt]).float()
        Q = torch.eye(K)[:, perm]
        p = make_problem(M, K, K, a_major=am, b_major=bm, in_dtype=dt, dist="ones", ld_extra=16)
        p.logical_A()[0].copy_(A.to(TORCH_FP8[dt]))
        p.logical_B()[0].copy_(Q.to(TORCH_FP8[dt]))
        assert np.array_equal(_oracle(p)[0], A[:, perm].double().numpy())


@pytest.mark.parametrize("am,bm", MAJORS)
def test_closed_forms(am, bm):
    M, N, K = 9, 11, 37
    p = make_problem(M, N, K, a_major=am, b_major=bm, in_dtype="e4m3", dist="ones")
    assert np.all(_oracle(p) == K)
    p = make_problem(M, N, K, a_major=am, b_major=bm, in_dtype="e5m2", dist="int", seed=8)
    A = p.logical_A().to(torch.float64).numpy()[0]
    B = p.logical_B().to(torch.float64).numpy()[0]
    assert np.array_equal(_oracle(p)[0], A @ B)         # integer sums: exact in any order


def test_against_numpy_blas_mid():
    for am, bm in MAJORS:
        for dt in ("e4m3", "e5m2"):
            p = make_problem(70, 45, 160, a_major=am, b_major=bm, in_dtype=dt, dist="normal",
                             seed=13, batch=2)
            c = _oracle(p)
            A = p.logical_A().to(torch.float64).numpy()
            B = p.logical_B().to(torch.float64).numpy()
            ref = A @ B
            scale = np.abs(A) @ np.abs(B)
            assert np.all(np.abs(c - ref) <= 1e-12 * scale + 1e-300)


def test_sampled_equals_full_and_padding_unread():
    p = make_problem(40, 36, 77, a_major=MN_MAJOR, b_major=K_MAJOR, in_dtype="e4m3", batch=2,
                     dist="normal", seed=9, ld_extra=16)
    c = _oracle(p)
    rng = np.random.default_rng(0)
    bi, mi, ni = rng.integers(0, 2, 200), rng.integers(0, 40, 200), rng.integers(0, 36, 200)
    s = og.gemm_f64_sampled(p.bits("A"), p.lda, p.a_major, p.bits("B"), p.ldb, p.b_major,
                            p.in_dtype, p.K, bi, mi, ni, p.strideA, p.strideB)
    assert np.array_equal(s, c[bi, mi, ni])
    q = make_problem(40, 36, 77, a_major=MN_MAJOR, b_major=K_MAJOR, in_dtype="e4m3", batch=2,
                     dist="normal", seed=9, ld_extra=48)
    assert np.array_equal(c, _oracle(q))
