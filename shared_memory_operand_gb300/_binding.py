"""ctypes binding of libsmo_gemm.so: the C ABI of include/smo_gemm.h, same
names, argument marshalling only.  Arguments that are torch tensors are passed
by their data pointer; ``stream=None`` means torch's current CUDA stream.

There is no fallback: if the shared library is missing or cannot be loaded,
every call raises.
"""
from __future__ import annotations

import ctypes
import json
import os
from typing import Any, Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libsmo_gemm.so")

GEMM_K_MAJOR, GEMM_MN_MAJOR = 0, 1
GEMM_BF16, GEMM_F16, GEMM_F32, GEMM_E4M3, GEMM_E5M2 = 0, 1, 2, 3, 4
GEMM_OK = 0
GEMM_ERR_ARG, GEMM_ERR_ALIGN, GEMM_ERR_UNSUPPORTED = -1, -2, -3
GEMM_ERR_LAUNCH, GEMM_ERR_TIMEOUT, GEMM_ERR_CUDA, GEMM_ERR_NO_DEVICE = -4, -5, -6, -7

DTYPE_CODES = {"bf16": GEMM_BF16, "f16": GEMM_F16, "f32": GEMM_F32, "e4m3": GEMM_E4M3, "e5m2": GEMM_E5M2}

# Every symbol include/smo_gemm.h declares.
EXPORTS = ("gemm_bf16", "gemm_ex", "gemm_check", "gemm_status_string", "gemm_set_timeout_ns",
           "gemm_plan_describe", "gemm_debug_inject_stall", "gemm_ex_noalloc", "gemm_check_noalloc",
           "smem_bank_probe", "tc_peak_probe",
           "l2_read_probe")


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        msg = status_text(status) if _lib is not None else str(status)
        super().__init__(f"{where}: {msg}" if where else msg)


_lib: Optional[ctypes.CDLL] = None


def load_library(path: str = LIB_PATH, build: bool = False) -> ctypes.CDLL:
    """Load (optionally build first) the CUDA library; raises if unavailable."""
    global _lib
    if _lib is not None:
        return _lib
    if build:
        from . import build as _b
        path = _b.build()
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built: {path} (run __graft_entry__.build())")
    L = ctypes.CDLL(path)
    i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    L.gemm_bf16.restype = i32
    L.gemm_bf16.argtypes = [vp, i64, i32, vp, i64, i32, vp, i64, i64, i64, i64, vp]
    L.gemm_ex.restype = i32
    L.gemm_ex.argtypes = [vp, i64, i32, vp, i64, i32, vp, i64, i64, i64, i64, i32, i32, i64, i64, i64,
                          i64, vp]
    L.gemm_ex_noalloc.restype = i32
    L.gemm_ex_noalloc.argtypes = [vp, i64, i32, vp, i64, i32, vp, i64, i64, i64, i64, i32, i32, i64,
                                  i64, i64, i64, vp]
    L.smem_bank_probe.restype = i32
    L.smem_bank_probe.argtypes = [vp, i32, i32, i32, vp, vp]
    L.tc_peak_probe.restype = i32
    L.tc_peak_probe.argtypes = [i32, vp, i32, vp]
    L.l2_read_probe.restype = i32
    L.l2_read_probe.argtypes = [vp, ctypes.c_size_t, i32, i32, vp, i32, vp]
    L.gemm_check.restype = i32
    L.gemm_check.argtypes = [vp]
    L.gemm_check_noalloc.restype = i32
    L.gemm_check_noalloc.argtypes = [vp]
    L.gemm_status_string.restype = ctypes.c_char_p
    L.gemm_status_string.argtypes = [i32]
    L.gemm_set_timeout_ns.restype = i64
    L.gemm_set_timeout_ns.argtypes = [i64]
    L.gemm_plan_describe.restype = i64
    L.gemm_plan_describe.argtypes = [i64, i64, i64, i32, i32, i32, i32, i64, i32, ctypes.c_char_p,
                                     ctypes.c_size_t]
    L.gemm_debug_inject_stall.restype = i32
    L.gemm_debug_inject_stall.argtypes = [i32]
    _lib = L
    return L


def _ptr(x: Any) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError(f"expected a tensor or an int address, got {type(x)}")


def _stream(stream: Any) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dt(x) -> int:
    return DTYPE_CODES[x] if isinstance(x, str) else int(x)


def status_text(status: int) -> str:
    return load_library().gemm_status_string(int(status)).decode()


def gemm_status_string(status: int) -> str:
    return status_text(status)


def _raise(st: int, where: str) -> None:
    if st != GEMM_OK:
        raise GemmError(st, where)


def gemm_bf16(A, lda, a_major, B, ldb, b_major, C, ldc, M, N, K, stream=None) -> None:
    st = load_library().gemm_bf16(_ptr(A), lda, a_major, _ptr(B), ldb, b_major, _ptr(C), ldc,
                                  M, N, K, _stream(stream))
    _raise(st, "gemm_bf16")


def gemm_ex(A, lda, a_major, B, ldb, b_major, C, ldc, M, N, K, in_dtype="bf16", out_dtype="f32",
            batch=1, strideA=0, strideB=0, strideC=0, stream=None) -> None:
    st = load_library().gemm_ex(_ptr(A), lda, a_major, _ptr(B), ldb, b_major, _ptr(C), ldc, M, N, K,
                                _dt(in_dtype), _dt(out_dtype), batch, strideA, strideB, strideC,
                                _stream(stream))
    _raise(st, "gemm_ex")


def gemm_ex_noalloc(A, lda, a_major, B, ldb, b_major, C, ldc, M, N, K, in_dtype="bf16",
                    out_dtype="f32", batch=1, strideA=0, strideB=0, strideC=0, stream=None) -> None:
    """gemm_ex without any device allocation (scratch in a static device array)."""
    st = load_library().gemm_ex_noalloc(_ptr(A), lda, a_major, _ptr(B), ldb, b_major, _ptr(C), ldc,
                                        M, N, K, _dt(in_dtype), _dt(out_dtype), batch, strideA,
                                        strideB, strideC, _stream(stream))
    _raise(st, "gemm_ex_noalloc")


def gemm_ex_status(*args, **kw) -> int:
    """Like gemm_ex but returns the raw status instead of raising."""
    try:
        gemm_ex(*args, **kw)
        return GEMM_OK
    except GemmError as e:
        return e.status


def gemm_check(stream=None) -> int:
    return int(load_library().gemm_check(_stream(stream)))


def gemm_check_noalloc(stream=None) -> int:
    """Error report of gemm_ex_noalloc (synchronises; allocates nothing)."""
    return int(load_library().gemm_check_noalloc(_stream(stream)))


def gemm_set_timeout_ns(ns: int) -> int:
    return int(load_library().gemm_set_timeout_ns(int(ns)))


def gemm_debug_inject_stall(on: bool) -> int:
    return int(load_library().gemm_debug_inject_stall(1 if on else 0))


def gemm_plan_describe(M, N, K, a_major, b_major, in_dtype="bf16", out_dtype="f32", batch=1,
                       num_sms=152) -> dict:
    L = load_library()
    n = L.gemm_plan_describe(M, N, K, a_major, b_major, _dt(in_dtype), _dt(out_dtype), batch,
                             num_sms, None, 0)
    if n < 0:
        raise GemmError(int(n), "gemm_plan_describe")
    buf = ctypes.create_string_buffer(int(n) + 1)
    L.gemm_plan_describe(M, N, K, a_major, b_major, _dt(in_dtype), _dt(out_dtype), batch, num_sms,
                         buf, n + 1)
    return json.loads(buf.value.decode())


def smem_bank_probe(offsets, access_bytes: int, is_store: bool, iters: int, cycles_out, stream=None) -> None:
    """Times one shared-memory access pattern (see include/smo_probe.h)."""
    st = load_library().smem_bank_probe(_ptr(offsets), int(access_bytes), 1 if is_store else 0, int(iters),
                                        _ptr(cycles_out), _stream(stream))
    if st != 0:
        raise RuntimeError(f"smem_bank_probe failed: {st}")


def l2_read_probe(src, nbytes: int, iters: int, out, max_ctas: int = 1 << 20, stages: int = 6,
                  stream=None) -> int:
    """Global-to-shared bandwidth probe (see include/smo_probe.h); returns CTAs."""
    n = load_library().l2_read_probe(_ptr(src), int(nbytes), int(iters), int(stages), _ptr(out),
                                     int(max_ctas), _stream(stream))
    if n < 1:
        raise RuntimeError(f"l2_read_probe failed: {n}")
    return int(n)


def tc_peak_probe(iters: int, out, max_clusters: int = 1 << 20, stream=None) -> int:
    """Tensor-core issue-rate probe (see include/smo_probe.h); returns clusters."""
    n = load_library().tc_peak_probe(int(iters), _ptr(out), int(max_clusters), _stream(stream))
    if n < 1:
        raise RuntimeError(f"tc_peak_probe failed: {n}")
    return int(n)
