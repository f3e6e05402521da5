"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on a
synthetic problem and compare it with the oracle.

Tolerances (per element, in fp64; s = max|A| * max|B| over the operands):
  fp32 out : |gpu - ref| <= s * (1e-3 * sqrt(K) / 16 + 1e-5),
             ||gpu - ref||_F <= 1e-5 * ||ref||_F
  16-bit out: |gpu - ref| <= 2^-p * |ref| + s * (1e-3 * sqrt(K) / 16 + 1e-5)
             with p = 8 (bf16) or 11 (f16), ||.||_F relative <= 4e-3 (bf16) / 5e-4 (f16)
  integer-valued inputs (every partial sum exact in fp32): bit-exact.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import shared_memory_operand_gb300 as smo
from oracle import gemm as og

GUARD = 4096          # elements of canary on each side of C
_TORCH_OUT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


def canary(dt: torch.dtype) -> torch.Tensor:
    # a NaN bit pattern the kernel never produces from finite inputs
    if dt == torch.float32:
        return torch.tensor([0x7FC0DEAD], dtype=torch.int32).view(torch.float32)
    return torch.tensor([0x7E5A], dtype=torch.int16).view(dt)


def run_gpu(p, stream=None, device="cuda", fn=None, check_fn=None):
    """Copies the operands to the device, runs gemm_ex (or `fn`) on a
    NaN-poisoned C with canary guard bands, asks gemm_check (or `check_fn`)
    for the kernel's status, checks the guards, returns C (batch, M, N) as
    float64."""
    A = p.A.to(device)
    B = p.B.to(device)
    odt = _TORCH_OUT[p.out_dtype]
    n = p.c_numel()
    buf = torch.empty(n + 2 * GUARD, dtype=odt, device=device)
    buf.copy_(canary(odt).to(device).expand_as(buf))
    C = buf[GUARD:GUARD + n]
    call = fn or smo.gemm_ex
    call(A, p.lda, p.a_major, B, p.ldb, p.b_major, C, p.ldc, p.M, p.N, p.K,
         in_dtype=p.in_dtype, out_dtype=p.out_dtype, batch=p.batch, strideA=p.strideA,
         strideB=p.strideB, strideC=p.strideC, stream=stream)
    st = (check_fn or smo.gemm_check)(stream)
    assert st == smo.GEMM_OK, smo.gemm_status_string(st)
    raw = buf.view(torch.int32 if odt == torch.float32 else torch.int16).cpu()
    can = canary(odt).view(torch.int32 if odt == torch.float32 else torch.int16)
    assert torch.all(raw[:GUARD] == can), "write below C"
    assert torch.all(raw[GUARD + n:] == can), "write above C"
    c = C.cpu()
    ld_stride = p.strideC if p.batch > 1 else p.M * p.ldc
    full = torch.as_strided(c, (p.batch, p.M, p.ldc), (ld_stride, p.ldc, 1))
    if p.ldc > p.N:   # columns past N must stay untouched
        pad = full[:, :, p.N:].contiguous().view(torch.int32 if odt == torch.float32 else torch.int16)
        assert torch.all(pad == can), "write past N"
    return full[:, :, :p.N].to(torch.float64).numpy()


def oracle_full(p):
    return og.gemm_f64(p.bits("A"), p.lda, p.a_major, p.bits("B"), p.ldb, p.b_major, p.in_dtype,
                       p.M, p.N, p.K, p.batch, p.strideA, p.strideB)


def scale(p) -> float:
    a = p.logical_A().to(torch.float32).abs().max().item() if p.M * p.K else 0.0
    b = p.logical_B().to(torch.float32).abs().max().item() if p.K * p.N else 0.0
    return max(a * b, 1e-30)


def abs_tol(p) -> float:
    return scale(p) * (1e-3 * math.sqrt(max(p.K, 1)) / 16 + 1e-5)


def check(p, gpu: np.ndarray, ref64: np.ndarray, exact: bool = False) -> dict:
    """Element-wise comparison; ref64 is the unrounded fp64 oracle result
    (same shape as gpu).  Returns error statistics, raises AssertionError."""
    assert gpu.shape == ref64.shape
    assert np.all(np.isfinite(gpu)), "non-finite output (unwritten element?)"
    ref = og.round_to(ref64, p.out_dtype)
    if exact:
        bad = np.argwhere(gpu != ref)
        assert bad.size == 0, f"{len(bad)} mismatches, first at {bad[0].tolist()}: " \
                              f"gpu={gpu[tuple(bad[0])]} ref={ref[tuple(bad[0])]}"
        return {"max_abs": 0.0, "rel_fro": 0.0}
    err = np.abs(gpu - ref64)
    rel = {"f32": 0.0, "bf16": 2.0 ** -8, "f16": 2.0 ** -11}[p.out_dtype]
    tol = rel * np.abs(ref64) + abs_tol(p)
    worst = np.unravel_index(np.argmax(err - tol), err.shape) if err.size else None
    assert err.size == 0 or np.all(err <= tol), \
        f"max excess at {worst}: gpu={gpu[worst]} ref={ref64[worst]} tol={tol[worst]}"
    fro_ref = np.linalg.norm(ref64)
    rel_fro = float(np.linalg.norm(gpu - ref64) / fro_ref) if fro_ref > 0 else 0.0
    fro_tol = {"f32": 1e-5, "bf16": 4e-3, "f16": 5e-4}[p.out_dtype]
    assert rel_fro <= fro_tol, f"relative Frobenius error {rel_fro} > {fro_tol}"
    return {"max_abs": float(err.max()) if err.size else 0.0, "rel_fro": rel_fro}
