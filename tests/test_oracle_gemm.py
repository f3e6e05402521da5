"""Pins for the oracle's fp64 GEMM and its IEEE rounding helpers (CPU only).

Each check ties the oracle to something other than itself: exact rational
arithmetic, the identity / permutation / closed-form products, numpy's and
torch's conversions and numpy's BLAS product, and exhaustive bit patterns.
"""
import itertools
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import gemm as og
from synthetic import K_MAJOR, MN_MAJOR, make_problem

MAJORS = [(K_MAJOR, K_MAJOR), (K_MAJOR, MN_MAJOR), (MN_MAJOR, K_MAJOR), (MN_MAJOR, MN_MAJOR)]


def _bits(p, which):
    return p.bits(which)


def _oracle(p, out=None):
    c = og.gemm_f64(_bits(p, "A"), p.lda, p.a_major, _bits(p, "B"), p.ldb, p.b_major,
                    p.in_dtype, p.M, p.N, p.K, p.batch, p.strideA, p.strideB)
    return c if out is None else og.round_to(c, out)


# ---------------------------------------------------------------- decoding
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_decode_encode_roundtrip_exhaustive(dt):
    bits = np.arange(65536, dtype=np.uint16)
    vals = og.decode16(bits, dt)
    finite = np.isfinite(vals)
    back = og.encode16(vals[finite], dt)
    assert np.array_equal(back, bits[finite])


def test_decode_matches_library_formats():
    bits = np.arange(65536, dtype=np.uint16)
    f16 = bits.view(np.float16).astype(np.float64)
    ours = og.decode16(bits, "f16")
    same = (ours == f16) | (np.isnan(ours) & np.isnan(f16))
    assert same.all()
    bf = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    ours = og.decode16(bits, "bf16")
    same = (ours == bf) | (np.isnan(ours) & np.isnan(bf))
    assert same.all()


# ---------------------------------------------------------------- rounding
def _random_doubles(n, seed):
    rng = np.random.default_rng(seed)
    mant = rng.uniform(-1, 1, n)
    exps = rng.integers(-140, 140, n)
    return np.ldexp(mant, exps)


pytestmark = pytest.mark.filterwarnings("ignore:overflow encountered in cast:RuntimeWarning")


def test_round_f16_matches_numpy():
    x = _random_doubles(200000, 1)
    x = x[np.abs(x) < 1e6]
    ours = og.round_to(x, "f16")
    ref = x.astype(np.float16).astype(np.float64)
    assert np.array_equal(ours, ref)


def test_round_f32_matches_numpy():
    x = _random_doubles(200000, 2)
    ours = og.round_to(x, "f32")
    ref = x.astype(np.float32).astype(np.float64)
    assert np.array_equal(ours, ref)


def test_round_bf16_matches_torch_on_f32_values():
    x = _random_doubles(200000, 3).astype(np.float32)
    ours = og.round_to(x.astype(np.float64), "bf16")
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, ref)


def test_round_ties_to_even():
    ulp = 2.0 ** -7                     # bf16 spacing in [1, 2)
    assert og.round_to(np.array([1 + ulp / 2]), "bf16")[0] == 1.0
    assert og.round_to(np.array([1 + 3 * ulp / 2]), "bf16")[0] == 1 + 2 * ulp
    assert og.round_to(np.array([1 + ulp / 2 + 2.0 ** -40]), "bf16")[0] == 1 + ulp
    u32 = 2.0 ** -23
    assert og.round_to(np.array([1 + u32 / 2]), "f32")[0] == 1.0
    assert og.round_to(np.array([1 + 3 * u32 / 2]), "f32")[0] == 1 + 2 * u32
    u16 = 2.0 ** -10
    assert og.round_to(np.array([-(1 + u16 / 2)]), "f16")[0] == -1.0
    # overflow: at or above max + ulp/2 goes to inf
    assert og.round_to(np.array([65520.0]), "f16")[0] == math.inf
    assert og.round_to(np.array([65519.99]), "f16")[0] == 65504.0


# ---------------------------------------------------------------- the GEMM
def _exact_bound_ok(p, c64):
    """|fp64 - exact| within the recursive-summation bound gamma_K * sum|terms|."""
    exact = og.exact_gemm(_bits(p, "A"), p.lda, p.a_major, _bits(p, "B"), p.ldb, p.b_major,
                          p.in_dtype, p.M, p.N, p.K, p.batch, p.strideA, p.strideB)
    A = p.logical_A().to(torch.float64).numpy()
    B = p.logical_B().to(torch.float64).numpy()
    absum = np.abs(A) @ np.abs(B)
    u = 2.0 ** -53
    gamma = p.K * u / (1 - p.K * u)
    for b in range(p.batch):
        for m in range(p.M):
            for n in range(p.N):
                err = abs(Fraction(c64[b, m, n]) - exact[b][m][n])
                if err > Fraction(gamma * absum[b, m, n]) + Fraction(0):
                    return False
    return True


@pytest.mark.parametrize("am,bm", MAJORS)
@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_bruteforce_exact_tiny(am, bm, dt):
    for (M, N, K) in [(1, 1, 1), (3, 5, 7), (8, 8, 8), (5, 2, 9)]:
        p = make_problem(M, N, K, a_major=am, b_major=bm, in_dtype=dt, dist="uniform",
                         seed=M * 100 + N * 10 + K, ld_extra=3)
        c = _oracle(p)
        assert _exact_bound_ok(p, c)


@pytest.mark.parametrize("am,bm", MAJORS)
def test_bruteforce_exact_integers_bitexact(am, bm):
    p = make_problem(6, 7, 9, a_major=am, b_major=bm, in_dtype="bf16", dist="int", seed=5, batch=2)
    c = _oracle(p)
    exact = og.exact_gemm(_bits(p, "A"), p.lda, p.a_major, _bits(p, "B"), p.ldb, p.b_major,
                          p.in_dtype, p.M, p.N, p.K, p.batch, p.strideA, p.strideB)
    for b, m, n in itertools.product(range(2), range(6), range(7)):
        assert Fraction(c[b, m, n]) == exact[b][m][n]


def _problem_from_logical(A, B, am, bm, dt="bf16"):
    """Store given logical fp32 matrices (values exact in dt) with the majors."""
    M, K = A.shape
    N = B.shape[1]
    p = make_problem(M, N, K, a_major=am, b_major=bm, in_dtype=dt, dist="ones", ld_extra=1)
    tdt = torch.bfloat16 if dt == "bf16" else torch.float16
    la = p.logical_A()
    lb = p.logical_B()
    la[0].copy_(A.to(tdt))
    lb[0].copy_(B.to(tdt))
    return p


@pytest.mark.parametrize("am,bm", MAJORS)
def test_identity_and_permutation(am, bm):
    g = torch.Generator().manual_seed(7)
    K, N = 24, 40
    B = (torch.rand(K, N, generator=g) * 2 - 1).to(torch.bfloat16).float()
    I = torch.eye(K)
    p = _problem_from_logical(I, B, am, bm)
    c = _oracle(p)[0]
    assert np.array_equal(c, B.double().numpy())
    perm = torch.randperm(K, generator=g)
    P = torch.eye(K)[perm]                      # (P B)[m] = B[perm[m]]
    p = _problem_from_logical(P, B, am, bm)
    c = _oracle(p)[0]
    assert np.array_equal(c, B[perm].double().numpy())
    # right identity / permutation: A Q with Q a column permutation
    M = 17
    A = (torch.rand(M, K, generator=g) * 2 - 1).to(torch.bfloat16).float()
    Q = torch.eye(K)[:, perm]                   # (A Q)[:, n] = A[:, perm[n]]
    p = _problem_from_logical(A, Q, am, bm)
    c = _oracle(p)[0]
    assert np.array_equal(c, A[:, perm].double().numpy())


@pytest.mark.parametrize("am,bm", MAJORS)
def test_closed_forms(am, bm):
    M, N, K = 9, 11, 37
    p = make_problem(M, N, K, a_major=am, b_major=bm, dist="ones")
    assert np.all(_oracle(p) == K)
    g = torch.Generator().manual_seed(3)
    u = torch.randint(-3, 4, (M,), generator=g).float()
    v = torch.randint(-3, 4, (N,), generator=g).float()
    x = torch.randint(-3, 4, (K,), generator=g).float()
    y = torch.randint(-3, 4, (K,), generator=g).float()
    A = u[:, None] * x[None, :]
    B = y[:, None] * v[None, :]
    p = _problem_from_logical(A, B, am, bm)
    want = (u[:, None] * v[None, :] * float(x @ y)).double().numpy()
    assert np.array_equal(_oracle(p)[0], want)


def test_against_numpy_blas_mid():
    for am, bm in MAJORS:
        p = make_problem(70, 45, 129, a_major=am, b_major=bm, in_dtype="f16", dist="normal",
                         seed=11, batch=3)
        c = _oracle(p)
        A = p.logical_A().to(torch.float64).numpy()
        B = p.logical_B().to(torch.float64).numpy()
        ref = A @ B
        scale = np.abs(A) @ np.abs(B)
        assert np.all(np.abs(c - ref) <= 1e-12 * scale + 1e-300)


def test_batched_equals_separate():
    p = make_problem(33, 21, 50, batch=4, dist="uniform", seed=2)
    c = _oracle(p)
    A = p.logical_A()
    B = p.logical_B()
    for b in range(4):
        q = _problem_from_logical(A[b].float(), B[b].float(), K_MAJOR, MN_MAJOR)
        assert np.array_equal(_oracle(q)[0], c[b])


def test_sampled_equals_full():
    p = make_problem(40, 36, 77, a_major=MN_MAJOR, b_major=K_MAJOR, batch=2, dist="normal", seed=9)
    c = _oracle(p)
    rng = np.random.default_rng(0)
    bi = rng.integers(0, 2, 200)
    mi = rng.integers(0, 40, 200)
    ni = rng.integers(0, 36, 200)
    s = og.gemm_f64_sampled(_bits(p, "A"), p.lda, p.a_major, _bits(p, "B"), p.ldb, p.b_major,
                            p.in_dtype, p.K, bi, mi, ni, p.strideA, p.strideB)
    assert np.array_equal(s, c[bi, mi, ni])


def test_poison_padding_never_read():
    """Leading-dimension padding holds a poison value; the product must not
    change when the padding changes (the oracle reads only in-range cells)."""
    p = make_problem(12, 10, 20, a_major=MN_MAJOR, b_major=MN_MAJOR, ld_extra=5, seed=4)
    c1 = _oracle(p)
    q = make_problem(12, 10, 20, a_major=MN_MAJOR, b_major=MN_MAJOR, ld_extra=13, seed=4)
    assert np.array_equal(c1, _oracle(q))
