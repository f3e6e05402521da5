"""Shared-memory bank-conflict simulator and the shared-memory layouts the GPU
path is expected to use -- the oracle's own restatement.

TEST INFRASTRUCTURE ONLY (tests/ and the smoke check import it; the product
path never does).  Independent of the C++ layout planner.

Bank model ("LDS Optimization" skill page, sections "LDS Architecture on CDNA3
(gfx942) / Hardware Facts" and "... CDNA4 (gfx950) / Hardware Facts"):
memory is split into NB banks of 4 bytes, bank = (byte_address / 4) % NB; two
or more lanes touching *different* 4-byte words of one bank in the same cycle
serialise (a conflict); lanes touching the same word are served by broadcast.
Conflicts are judged on the shared-memory addresses the lanes issue, not on
where the data lands in registers ("A Deep Dive into LDS Optimizations on AMD
Instinct MI450 GPUs", end of "What Does ds_load_tr Do?").

A request is served in phases, each phase holding a fixed group of lanes
(the rocMLIR pull 2196 description: ds_write2_b32 runs in two phases of 32
threads; the MI450 post, "Measuring It": ds_load_b128 serves 16 lanes per
group).  Per phase the degree is the largest number of distinct words any bank
must deliver; the request costs the sum of its phase degrees ("wavefronts").
On GB300 (an NVIDIA fact, not from the pages) the model is 32 banks x 4 B with
128 bytes served per phase: 32 lanes for 4-byte, 16 for 8-byte and 8 for
16-byte accesses -- the default below.
"""
from __future__ import annotations

from dataclasses import dataclass
from math import gcd
from typing import Dict, List, Optional, Sequence, Set


@dataclass
class Report:
    degree: int                 # worst phase: max distinct words on one bank
    wavefronts: int             # sum over phases of their degrees
    phases: int
    distinct_banks: List[int]   # per phase, number of banks touched

    @property
    def extra_wavefronts(self) -> int:
        return self.wavefronts - self.phases


def simulate(addresses: Sequence[Optional[int]], access_bytes: int, n_banks: int = 32,
             bank_bytes: int = 4, lanes_per_phase: Optional[int] = None) -> Report:
    """One access instruction: ``addresses[lane]`` is the byte address lane
    issues (None = inactive lane); each lane touches ``access_bytes`` bytes."""
    if lanes_per_phase is None:
        lanes_per_phase = max(1, (n_banks * bank_bytes) // access_bytes)
    n = len(addresses)
    degree, wavefronts, phases, banks_touched = 0, 0, 0, []
    for start in range(0, n, lanes_per_phase):
        words_by_bank: Dict[int, Set[int]] = {}
        any_active = False
        for lane in range(start, min(n, start + lanes_per_phase)):
            a = addresses[lane]
            if a is None:
                continue
            any_active = True
            first = a // bank_bytes
            last = (a + access_bytes - 1) // bank_bytes
            for w in range(first, last + 1):
                words_by_bank.setdefault(w % n_banks, set()).add(w)
        if not any_active:
            continue
        d = max(len(s) for s in words_by_bank.values())
        phases += 1
        wavefronts += d
        degree = max(degree, d)
        banks_touched.append(len(words_by_bank))
    return Report(degree, wavefronts, phases, banks_touched)


def padding_rule_degree(row_stride_dwords: int, n_banks: int) -> int:
    """Closed form for one lane per row, n_banks lanes, integer dword stride:
    lanes land on n_banks / gcd(stride, n_banks) distinct banks, so each bank
    serves gcd(stride, n_banks) distinct words ("LDS Optimization",
    "Optimization Method 2: Padding / The Solution")."""
    return gcd(row_stride_dwords, n_banks)


def xor_mask_rule(n_banks: int, vec_elems: int, elem_bytes: int) -> int:
    """The page's XOR-mask width rule ("Choosing Swizzle Parameters"):
    NB / (vec * element_size / 4) - 1."""
    return n_banks // (vec_elems * elem_bytes // 4) - 1


# ---------------------------------------------------------------------------
# GB300 shared-memory tile layouts (NVIDIA facts restated from the public PTX
# ISA / CUDA documentation, independently of the planner):
#   128-byte swizzle (TMA SWIZZLE_128B, tcgen05 SWIZZLE_128B): inside each
#   1024-byte block of eight 128-byte rows, the 16-byte chunk index (address
#   bits 4..6) is XORed with the row index within the block (bits 7..9).
# ---------------------------------------------------------------------------

def sw128(byte_offset: int) -> int:
    return byte_offset ^ (((byte_offset >> 7) & 7) << 4)


def sw128_row_major(row: int, byte_in_row: int) -> int:
    """Rows of 128 bytes, row r at r*128, chunk swizzled by r % 8."""
    assert 0 <= byte_in_row < 128
    return sw128(row * 128 + byte_in_row)


def operand_tile_offset(mn: int, k: int, mn_major: bool, tile_mn: int, elem_bytes: int = 2,
                        box_k: int = 64) -> int:
    """Byte offset of element (mn, k) of one pipeline-stage operand tile
    (tile_mn x box_k, 16-bit elements) as 128-byte-swizzled TMA boxes place it.

    K-major: one box, row = mn (128 bytes = 64 k-values per row).
    MN-major: boxes of 64 mn-values x box_k k-rows, box j = mn // 64 at
    j * (box_k * 128); inside a box row = k, byte = 2 * (mn % 64)."""
    per_row = 128 // elem_bytes
    if not mn_major:
        assert k < per_row
        return sw128_row_major(mn, k * elem_bytes)
    box = mn // per_row
    return box * box_k * 128 + sw128_row_major(k, (mn % per_row) * elem_bytes)


def umma_canonical_offset(mn: int, k: int, mn_major: bool, lbo: int, sbo: int,
                          kstep_bytes: int, elem_bytes: int = 2, mma_k: int = 16) -> int:
    """Byte offset the tensor core reads element (mn, k) from, for the
    SWIZZLE_128B canonical layouts of the tcgen05 shared-memory descriptor
    (PTX ISA, tcgen05 "Shared memory descriptor" / canonical layouts), with the
    descriptor's start address advanced by kstep_bytes per 16-wide K step.

    K-major  ((8,m),(T,2)) : ((8T,SBO),(1,T))  in 16-byte units T
    MN-major ((T,8,m),(8,2)) : ((1,T,LBO),(8T,SBO))
    The swizzle is a function of the absolute address (1024-byte aligned base)."""
    step, kk = divmod(k, mma_k)
    start = step * kstep_bytes
    if not mn_major:
        pre = start + (mn % 8) * 128 + (mn // 8) * sbo + kk * elem_bytes
    else:
        per_atom = 128 // elem_bytes
        pre = (start + (mn % per_atom) * elem_bytes + (mn // per_atom) * lbo
               + (kk % 8) * 128 + (kk // 8) * sbo)
    return sw128(pre)


def epilogue_store_addresses(slab_base: int, chunk: int, swizzled: bool = True,
                             lanes: int = 32) -> List[int]:
    """One 16-byte st.shared per lane: lane l writes 16-byte chunk ``chunk`` of
    row l of its warp's 32-row staging slab (rows of 128 bytes)."""
    out = []
    for l in range(lanes):
        off = l * 128 + chunk * 16
        out.append(slab_base + (sw128(off) if swizzled else off))
    return out
