"""Per-lane shared-memory byte offsets of the access patterns the bank
microbenchmark times (32 lanes).  Test inputs only: no arithmetic of the
method.  Sources of the patterns:
  * the GEMM epilogue's 16-byte stores into a 128-byte-swizzled 32-row slab and
    the same stores without the swizzle;
  * "LDS Optimization" skill page, "Optimization Method 1: Swizzle Layout / The
    Problem" (a stride that is a multiple of the bank span) and "Optimization
    Method 2: Padding" / "Padding Amount" (one lane per row of a [64][64+PAD]
    fp16 tile reading one column, PAD 0, 1, 2, 4, 32);
  * rocMLIR pull 2196, description (the [kPackPerBlock, dPerBlock = 96,
    kPack = 4] f16 layout whose first 32 threads write an 8-way pattern).
"""


def epilogue(swizzled: bool, chunk: int = 0):
    return [l * 128 + (((chunk ^ (l & 7)) if swizzled else chunk) << 4) for l in range(32)]


def strided(stride_bytes: int):
    return [l * stride_bytes for l in range(32)]


def padded_column(pad: int):
    return strided((64 + pad) * 2)


def kpack_rows():
    def addr(m, k):
        return ((k // 4) * 96 + m) * 4 * 2 + (k % 4) * 2
    return [addr(0, 2 * t) for t in range(16)] + [addr(3, 2 * (t - 16)) for t in range(16, 32)]


# name -> (offsets, access bytes)
PATTERNS = {
    "st16_epilogue_swizzled": (epilogue(True), 16),
    "st16_epilogue_unswizzled": (epilogue(False), 16),
    "st16_linear": (strided(16), 16),
    "st8_linear": (strided(8), 8),
    "st8_stride128": (strided(128), 8),
    "st4_linear": (strided(4), 4),
    "st4_stride128": (strided(128), 4),
    "st4_stride132": (strided(132), 4),
    "st4_stride136": (strided(136), 4),
    "st4_kpack": (kpack_rows(), 4),
    "ld2_pad0": (padded_column(0), 2),
    "ld2_pad1": (padded_column(1), 2),
    "ld2_pad2": (padded_column(2), 2),
    "ld2_pad4": (padded_column(4), 2),
    "ld2_pad32": (padded_column(32), 2),
}
