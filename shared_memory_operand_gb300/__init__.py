"""GB300-native shared-memory-operand GEMM: C = A * B on sm_103a tensor cores.

The compute path is the CUDA library ``_build/libsmo_gemm.so`` (built from
``csrc/`` by ``build.py``); this package is its ctypes binding (same names as
the C ABI in ``include/smo_gemm.h``).  There is no CPU fallback.
"""
from ._binding import (  # noqa: F401
    DTYPE_CODES, EXPORTS, GEMM_BF16, GEMM_ERR_ALIGN, GEMM_ERR_ARG, GEMM_ERR_CUDA, GEMM_ERR_LAUNCH,
    GEMM_ERR_NO_DEVICE, GEMM_ERR_TIMEOUT, GEMM_ERR_UNSUPPORTED, GEMM_E4M3, GEMM_E5M2, GEMM_F16, GEMM_F32,
    GEMM_K_MAJOR,
    GEMM_MN_MAJOR, GEMM_OK, LIB_PATH, GemmError, gemm_bf16, gemm_check, gemm_check_noalloc,
    gemm_debug_inject_stall,
    gemm_ex, gemm_ex_noalloc, gemm_ex_status, gemm_plan_describe, gemm_set_timeout_ns, gemm_status_string, smem_bank_probe, tc_peak_probe, l2_read_probe,
    load_library, status_text,
)
