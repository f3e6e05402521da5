"""Oracle GEMM: fp64 CPU product over the same 16-bit or 8-bit operands the GPU reads.

TEST INFRASTRUCTURE ONLY -- imported by ``tests/``, the smoke check and the
bench's CPU-baseline leg, never by the product path.  Shares no code with the
CUDA library: it wraps ``gemm_ref.c`` (plain C, fp64) through ctypes and adds a
pure-Python exact brute force over ``fractions.Fraction``.

What it computes: C = A B ("An Educational GEMM Ladder for Helios GPUs",
section "Educational GEMM Ladder": every rung computes C = AB, BF16 operands,
on matrix units that also take FP8; rocMLIR pull 2196, description: the f16
GEMM -m 1500 -n 1152 -k 896), each
element summed in IEEE double with k ascending, then rounded once to the output
format by round-to-nearest-even.

Operand addressing (majors, leading dimensions, batch strides) follows the
library's convention:
  A K-major: A[b,m,k] = a[b*sa + m*lda + k];   A M-major: a[b*sa + k*lda + m]
  B K-major: B[b,k,n] = b[b*sb + n*ldb + k];   B N-major: b[b*sb + k*ldb + n]
"""
from __future__ import annotations

import ctypes
import os
from fractions import Fraction

import numpy as np

from . import build as _build

DTYPES = {"bf16": 0, "f16": 1, "f32": 2, "e4m3": 3, "e5m2": 4}
FP8 = ("e4m3", "e5m2")
K_MAJOR, MN_MAJOR = 0, 1

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i64, i32 = ctypes.c_int64, ctypes.c_int
        p16 = ctypes.POINTER(ctypes.c_uint16)
        pd = ctypes.POINTER(ctypes.c_double)
        p64 = ctypes.POINTER(ctypes.c_int64)
        L.orc_decode16.restype = ctypes.c_double
        L.orc_decode16.argtypes = [ctypes.c_uint16, i32]
        L.orc_decode16_array.restype = None
        L.orc_decode16_array.argtypes = [p16, i64, i32, pd]
        L.orc_encode16.restype = ctypes.c_uint16
        L.orc_encode16.argtypes = [ctypes.c_double, i32]
        for name in ("orc_round_f32", "orc_round_bf16", "orc_round_f16"):
            getattr(L, name).restype = ctypes.c_double
            getattr(L, name).argtypes = [ctypes.c_double]
        L.orc_round_array.restype = None
        L.orc_round_array.argtypes = [pd, i64, i32, pd]
        p8 = ctypes.POINTER(ctypes.c_uint8)
        vp = ctypes.c_void_p
        L.orc_decode8.restype = ctypes.c_double
        L.orc_decode8.argtypes = [ctypes.c_uint8, i32]
        L.orc_decode8_array.restype = None
        L.orc_decode8_array.argtypes = [p8, i64, i32, pd]
        L.orc_elem_bytes.restype = i32
        L.orc_elem_bytes.argtypes = [i32]
        L.orc_gemm_f64.restype = i32
        L.orc_gemm_f64.argtypes = [vp, i64, i32, vp, i64, i32, i32, i64, i64, i64, i64, i64, i64, pd]
        L.orc_gemm_f64_sampled.restype = None
        L.orc_gemm_f64_sampled.argtypes = [vp, i64, i32, vp, i64, i32, i32, i64, i64, i64,
                                           p64, p64, p64, i64, pd]
        L.orc_num_threads.restype = i32
        L.orc_num_threads.argtypes = []
        _lib = L
    return _lib


def _u16(x) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(x)).reshape(-1)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError(f"operand bits must be uint16/int16, got {a.dtype}")
    return a


def _u8(x) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(x)).reshape(-1)
    if a.dtype == np.int8:
        a = a.view(np.uint8)
    if a.dtype != np.uint8:
        raise TypeError(f"8-bit operand bits must be uint8/int8, got {a.dtype}")
    return a


def _operand(x, dtype: str) -> np.ndarray:
    """Operand bit patterns as a contiguous uint8 (FP8) or uint16 array."""
    return _u8(x) if dtype in FP8 else _u16(x)


def _pv(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _p16(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16))


def _pd(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def num_threads() -> int:
    return int(lib().orc_num_threads())


def decode16(bits, dtype: str) -> np.ndarray:
    a = _u16(bits)
    out = np.empty(a.size, dtype=np.float64)
    lib().orc_decode16_array(_p16(a), a.size, DTYPES[dtype], _pd(out))
    return out


def decode8(bits, dtype: str) -> np.ndarray:
    """FP8 (E4M3 / E5M2) bit patterns -> float64 values."""
    a = _u8(bits)
    out = np.empty(a.size, dtype=np.float64)
    lib().orc_decode8_array(a.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)), a.size, DTYPES[dtype], _pd(out))
    return out


def decode(bits, dtype: str) -> np.ndarray:
    return decode8(bits, dtype) if dtype in FP8 else decode16(bits, dtype)


def encode16(x, dtype: str) -> np.ndarray:
    """fp64 -> 16-bit bit patterns, round-to-nearest-even."""
    xs = np.asarray(x, dtype=np.float64).reshape(-1)
    L = lib()
    return np.array([L.orc_encode16(float(v), DTYPES[dtype]) for v in xs], dtype=np.uint16)


def round_to(x, out_dtype: str) -> np.ndarray:
    """Round fp64 values once to f32 / bf16 / f16 (RNE); returned as float64."""
    xs = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    flat = xs.reshape(-1)
    out = np.empty_like(flat)
    lib().orc_round_array(_pd(flat), flat.size, DTYPES[out_dtype], _pd(out))
    return out.reshape(xs.shape)


def gemm_f64(A, lda, a_major, B, ldb, b_major, in_dtype, M, N, K,
             batch=1, strideA=0, strideB=0) -> np.ndarray:
    """Exact-definition fp64 product; returns float64 array (batch, M, N)."""
    a, b = _operand(A, in_dtype), _operand(B, in_dtype)
    c = np.empty((batch, M, N), dtype=np.float64)
    rc = lib().orc_gemm_f64(_pv(a), lda, int(a_major), _pv(b), ldb, int(b_major),
                            DTYPES[in_dtype], M, N, K, batch, strideA, strideB, _pd(c))
    if rc != 0:
        raise MemoryError("oracle gemm: scratch allocation failed")
    return c


def gemm_ref(A, lda, a_major, B, ldb, b_major, in_dtype, out_dtype, M, N, K,
             batch=1, strideA=0, strideB=0) -> np.ndarray:
    """fp64 product rounded once to ``out_dtype`` (values held as float64)."""
    return round_to(gemm_f64(A, lda, a_major, B, ldb, b_major, in_dtype, M, N, K,
                             batch, strideA, strideB), out_dtype)


def gemm_f64_sampled(A, lda, a_major, B, ldb, b_major, in_dtype, K, bi, mi, ni,
                     strideA=0, strideB=0) -> np.ndarray:
    """fp64 dot products for the listed (batch, m, n) positions only."""
    a, b = _operand(A, in_dtype), _operand(B, in_dtype)
    bi = np.ascontiguousarray(bi, dtype=np.int64)
    mi = np.ascontiguousarray(mi, dtype=np.int64)
    ni = np.ascontiguousarray(ni, dtype=np.int64)
    out = np.empty(bi.size, dtype=np.float64)
    p64 = ctypes.POINTER(ctypes.c_int64)
    lib().orc_gemm_f64_sampled(_pv(a), lda, int(a_major), _pv(b), ldb, int(b_major),
                               DTYPES[in_dtype], K, strideA, strideB,
                               bi.ctypes.data_as(p64), mi.ctypes.data_as(p64),
                               ni.ctypes.data_as(p64), bi.size, _pd(out))
    return out


# --------------------------------------------------------------------------
# Exact brute force (tiny shapes): rational arithmetic, no rounding anywhere.
# Bit decoding is re-derived here in Python, independently of gemm_ref.c.
# --------------------------------------------------------------------------

def exact_value16(h: int, dtype: str) -> Fraction:
    h = int(h) & 0xFFFF
    sign = -1 if (h >> 15) & 1 else 1
    if dtype == "bf16":
        ebits, fbits, bias = 8, 7, 127
    else:
        ebits, fbits, bias = 5, 10, 15
    e = (h >> fbits) & ((1 << ebits) - 1)
    f = h & ((1 << fbits) - 1)
    if e == (1 << ebits) - 1:
        raise ValueError("inf/nan has no exact value")
    if e == 0:
        mag = Fraction(f, 1 << fbits) * Fraction(2) ** (1 - bias)
    else:
        mag = (1 + Fraction(f, 1 << fbits)) * Fraction(2) ** (e - bias)
    return sign * mag


def exact_value8(h: int, dtype: str) -> Fraction:
    """Exact value of an FP8 code (OCP 8-bit floating point: E4M3 bias 7, whose
    only NaN is S.1111.111 and which has no infinities; E5M2 bias 15 with IEEE
    infinities and NaNs)."""
    h = int(h) & 0xFF
    sign = -1 if (h >> 7) & 1 else 1
    if dtype == "e4m3":
        ebits, fbits, bias = 4, 3, 7
        if (h & 0x7F) == 0x7F:
            raise ValueError("nan has no exact value")
    else:
        ebits, fbits, bias = 5, 2, 15
        if (h >> fbits) & 0x1F == 0x1F:
            raise ValueError("inf/nan has no exact value")
    e = (h >> fbits) & ((1 << ebits) - 1)
    f = h & ((1 << fbits) - 1)
    if e == 0:
        mag = Fraction(f, 1 << fbits) * Fraction(2) ** (1 - bias)
    else:
        mag = (1 + Fraction(f, 1 << fbits)) * Fraction(2) ** (e - bias)
    return sign * mag


def exact_value(h: int, dtype: str) -> Fraction:
    return exact_value8(h, dtype) if dtype in FP8 else exact_value16(h, dtype)


def exact_gemm(A, lda, a_major, B, ldb, b_major, in_dtype, M, N, K,
               batch=1, strideA=0, strideB=0):
    """Nested lists C[b][m][n] of Fractions: sum_k A[b,m,k] * B[b,k,n] exactly."""
    a, b = _operand(A, in_dtype), _operand(B, in_dtype)
    out = []
    for bb in range(batch):
        rows = []
        for m in range(M):
            row = []
            for n in range(N):
                s = Fraction(0)
                for k in range(K):
                    ia = bb * strideA + (k * lda + m if a_major == MN_MAJOR else m * lda + k)
                    ib = bb * strideB + (k * ldb + n if b_major == MN_MAJOR else n * ldb + k)
                    s += exact_value(a[ia], in_dtype) * exact_value(b[ib], in_dtype)
                row.append(s)
            rows.append(row)
        out.append(rows)
    return out
