"""Seeded operand generation (CPU, torch.Generator) for the GEMM workloads.

Recipe (one generator per problem, seeded, draws A then B):
  uniform : torch.rand * 2 - 1 in fp32, rounded to the input type
            (bf16 / f16, or FP8 E4M3 / E5M2, by torch's round-to-nearest-even)
  normal  : torch.randn * sigma in fp32, rounded likewise
  int     : torch.randint(-4, 5) (integers in [-4, 4]), exact in every input type
Logical A is batch x M x K and logical B is batch x K x N; each is then stored
in the requested orientation:
  A K-major: rows of K (lda >= K)      A M-major: rows of M (lda >= M)
  B K-major: rows of K, one per n      B N-major: rows of N, one per k
Leading dimensions are padded up to ``ld_align`` elements (TMA needs 16-byte
row pitches: 8 elements of 16 bits, 16 of 8 bits); padding cells hold a poison
value the product must never read (4096, or 448 = the largest E4M3 value).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, Optional

import torch

K_MAJOR, MN_MAJOR = 0, 1
_TORCH_DT = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32,
             "e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}
FP8 = ("e4m3", "e5m2")
POISON = 4096.0
_POISON = {"e4m3": 448.0}


def elem_bytes(dtype: str) -> int:
    return {"bf16": 2, "f16": 2, "f32": 4, "e4m3": 1, "e5m2": 1}[dtype]


@dataclass
class Problem:
    M: int
    N: int
    K: int
    batch: int
    a_major: int
    b_major: int
    in_dtype: str
    out_dtype: str
    A: torch.Tensor            # CPU storage, 1-D, 16-bit or 8-bit
    B: torch.Tensor
    lda: int
    ldb: int
    ldc: int
    strideA: int
    strideB: int
    strideC: int
    dist: str = "uniform"
    seed: int = 0
    meta: Dict = field(default_factory=dict)

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K * self.batch

    def c_numel(self) -> int:
        return self.batch * self.strideC if self.batch > 1 else self.M * self.ldc

    def bits(self, which: str):
        """Operand storage as a numpy uint16 (16-bit types) or uint8 (FP8)
        array: the oracle's input."""
        t = self.A if which == "A" else self.B
        if self.in_dtype in FP8:
            return t.view(torch.uint8).numpy()
        return t.view(torch.int16).numpy().view("uint16")

    def logical_A(self) -> torch.Tensor:
        """batch x M x K view of A (values, not a copy of the arithmetic)."""
        return self._logical(self.A, self.M, self.K, self.lda, self.strideA, self.a_major)

    def logical_B(self) -> torch.Tensor:
        """batch x K x N view of B."""
        v = self._logical(self.B, self.N, self.K, self.ldb, self.strideB, self.b_major)
        return v.transpose(1, 2)

    def _logical(self, t, rows, kdim, ld, stride, major):
        # returns batch x rows x kdim
        if major == K_MAJOR:
            return torch.as_strided(t, (self.batch, rows, kdim), (stride, ld, 1))
        return torch.as_strided(t, (self.batch, rows, kdim), (stride, 1, ld))


def _round_up(x: int, a: int) -> int:
    return (x + a - 1) // a * a


def _draw(gen: torch.Generator, shape, dist: str, sigma: float) -> torch.Tensor:
    if dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2 - 1
    if dist == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32) * sigma
    if dist == "int":
        return torch.randint(-4, 5, shape, generator=gen).to(torch.float32)
    if dist == "ones":
        return torch.ones(shape, dtype=torch.float32)
    raise ValueError(dist)


def _store(logical: torch.Tensor, mn_major: bool, ld: int, dt: torch.dtype,
           poison: float = POISON) -> (torch.Tensor, int):
    """logical: batch x R x Kd (R = M for A, N for B).  Returns 1-D storage and
    the batch stride."""
    batch, R, Kd = logical.shape
    if not mn_major:
        rows, cols = R, Kd
        src = logical
    else:
        rows, cols = Kd, R
        src = logical.transpose(1, 2)
    stride = rows * ld
    if dt.itemsize == 2:
        # 16-bit: filled and written in the storage type directly (the logical
        # values are already rounded to it, so the conversion is exact)
        buf = torch.full((batch, rows, ld), poison, dtype=dt)
        buf[:, :, :cols] = src.to(dt)
        return buf.reshape(-1), stride
    buf = torch.full((batch, rows, ld), poison, dtype=torch.float32)
    buf[:, :, :cols] = src
    return buf.to(dt).reshape(-1).contiguous(), stride


def make_problem(M: int, N: int, K: int, *, a_major: int = K_MAJOR, b_major: int = MN_MAJOR,
                 in_dtype: str = "bf16", out_dtype: str = "bf16", dist: str = "uniform",
                 sigma: float = 1.0, seed: int = 0, batch: int = 1, ld_align: Optional[int] = None,
                 ld_extra: int = 0) -> Problem:
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    dt = _TORCH_DT[in_dtype]
    if ld_align is None:
        ld_align = 16 // elem_bytes(in_dtype)
    poison = _POISON.get(in_dtype, POISON)
    a_log = _draw(gen, (batch, M, K), dist, sigma).to(dt).to(torch.float32)
    b_log = _draw(gen, (batch, K, N), dist, sigma).to(dt).to(torch.float32)
    lda = _round_up((M if a_major == MN_MAJOR else K) + ld_extra, ld_align)
    ldb = _round_up((N if b_major == MN_MAJOR else K) + ld_extra, ld_align)
    A, sA = _store(a_log, a_major == MN_MAJOR, lda, dt, poison)
    # B logical batch x K x N; stored per n (K-major) or per k (N-major)
    B, sB = _store(b_log.transpose(1, 2), b_major == MN_MAJOR, ldb, dt, poison)
    out_align = 4 if out_dtype == "f32" else 8
    ldc = _round_up(N, out_align)
    return Problem(M, N, K, batch, a_major, b_major, in_dtype, out_dtype, A, B, lda, ldb, ldc,
                   sA, sB, M * ldc, dist=dist, seed=seed)


# Named workloads (shapes, orientations, distributions of the configurations
# the library is measured and checked on).
WORKLOADS: Dict[str, Dict] = {
    "gemm_256_bf16_f32": dict(M=256, N=256, K=256, a_major=K_MAJOR, b_major=MN_MAJOR,
                              in_dtype="bf16", out_dtype="f32", dist="uniform"),
    "gemm_1500x1152x896_f16_f32": dict(M=1500, N=1152, K=896, a_major=K_MAJOR, b_major=MN_MAJOR,
                                       in_dtype="f16", out_dtype="f32", dist="uniform"),
    "gemm_1500x1152x896_f16_f32_int": dict(M=1500, N=1152, K=896, a_major=K_MAJOR,
                                           b_major=MN_MAJOR, in_dtype="f16", out_dtype="f32",
                                           dist="int"),
    "gemm_4096_bf16_bf16_AK_BK": dict(M=4096, N=4096, K=4096, a_major=K_MAJOR, b_major=K_MAJOR,
                                      in_dtype="bf16", out_dtype="bf16", dist="normal"),
    "gemm_4096_bf16_bf16_AK_BN": dict(M=4096, N=4096, K=4096, a_major=K_MAJOR, b_major=MN_MAJOR,
                                      in_dtype="bf16", out_dtype="bf16", dist="normal"),
    "gemm_4096_bf16_bf16_AM_BK": dict(M=4096, N=4096, K=4096, a_major=MN_MAJOR, b_major=K_MAJOR,
                                      in_dtype="bf16", out_dtype="bf16", dist="normal"),
    "gemm_4096_bf16_bf16_AM_BN": dict(M=4096, N=4096, K=4096, a_major=MN_MAJOR, b_major=MN_MAJOR,
                                      in_dtype="bf16", out_dtype="bf16", dist="normal"),
    "gemm_8192_bf16_bf16_AK_BN": dict(M=8192, N=8192, K=8192, a_major=K_MAJOR, b_major=MN_MAJOR,
                                      in_dtype="bf16", out_dtype="bf16", dist="uniform"),
    "gemm_8192_bf16_bf16_AK_BK": dict(M=8192, N=8192, K=8192, a_major=K_MAJOR, b_major=K_MAJOR,
                                      in_dtype="bf16", out_dtype="bf16", dist="uniform"),
    "skinny_16384x8192x1024_bf16": dict(M=16384, N=8192, K=1024, a_major=K_MAJOR,
                                        b_major=MN_MAJOR, in_dtype="bf16", out_dtype="bf16",
                                        dist="normal", sigma=0.02),
    "batched_32x2048_bf16": dict(M=2048, N=2048, K=2048, batch=32, a_major=K_MAJOR,
                                 b_major=MN_MAJOR, in_dtype="bf16", out_dtype="bf16",
                                 dist="normal", sigma=0.02),
    # a tile-starved long-K shape with fp32 output: 16 tiles of 128 x 128, K
    # split over 2-CTA clusters
    "gemm_512x512x4096_bf16_f32": dict(M=512, N=512, K=4096, a_major=K_MAJOR, b_major=MN_MAJOR,
                                       in_dtype="bf16", out_dtype="f32", dist="uniform"),
    # 8-bit operands (E4M3), fp32 accumulate, bf16 out: the 8192^3 shape in the
    # transposed-B orientation and K-major B
    "gemm_8192_e4m3_bf16_AK_BN": dict(M=8192, N=8192, K=8192, a_major=K_MAJOR, b_major=MN_MAJOR,
                                      in_dtype="e4m3", out_dtype="bf16", dist="uniform"),
    "gemm_8192_e4m3_bf16_AK_BK": dict(M=8192, N=8192, K=8192, a_major=K_MAJOR, b_major=K_MAJOR,
                                      in_dtype="e4m3", out_dtype="bf16", dist="uniform"),
}


def workload(name: str, seed: int = 0, **overrides) -> Problem:
    kw = dict(WORKLOADS[name])
    kw.update(overrides)
    M, N, K = kw.pop("M"), kw.pop("N"), kw.pop("K")
    p = make_problem(M, N, K, seed=seed, **kw)
    p.meta["workload"] = name
    return p
