"""Pins for the oracle's F2 layout algebra and bank-conflict simulator against
the worked examples the pages print (tests/golden/*.txt, each line cited
there) and against closed forms brute-forced over many cases."""
import os
from math import gcd

import pytest

from oracle import banksim
from oracle.f2 import LinearLayout, divide_left, enumerate_map, identity_1d


def _parse_layouts(path):
    layouts, evals = {}, {}
    for line in open(path):
        line = line.split("#")[0].strip()
        if not line:
            continue
        parts = line.split()
        if parts[0].endswith("_eval"):
            args = dict(kv.split("=") for kv in parts[1].split(","))
            evals[parts[0][:-5]] = ({k: int(v) for k, v in args.items()},
                                    tuple(int(v) for v in parts[2].split(",")))
            continue
        name, dim, idx, img = parts
        layouts.setdefault(name, {}).setdefault(dim, []).append(
            (int(idx), tuple(int(v) for v in img.split(","))))
    return layouts, evals


def _mk(spec, order, outs):
    ins = []
    for d in order:
        items = sorted(spec[d])
        assert [i for i, _ in items] == [1 << j for j in range(len(items))]
        ins.append((d, [img for _, img in items]))
    return LinearLayout(ins, outs)


@pytest.fixture(scope="module")
def mi450(golden_dir):
    return _parse_layouts(os.path.join(golden_dir, "mi450_linear_layouts.txt"))


def test_invert_and_compose_worked_table(mi450):
    L, _ = mi450
    dst = _mk(L["dst"], ["register", "lane"], [("M", 32), ("K", 8)])
    shared = _mk(L["shared"], ["offset"], [("M", 32), ("K", 8)])
    cvt = dst.invert_and_compose(shared)
    want = _mk(L["cvt"], ["register", "lane"], [("offset", 256)])
    assert cvt.bases("register") == want.bases("register")
    assert cvt.bases("lane") == want.bases("lane")
    # brute force: every (register, lane) lands on the offset holding its [M,K]
    for r in range(8):
        for ln in range(32):
            off = cvt.apply(register=r, lane=ln)[0]
            assert shared.apply(offset=off) == dst.apply(register=r, lane=ln)


def test_invert_and_compose_needs_surjective(mi450):
    L, _ = mi450
    dst = _mk(L["dst"], ["register", "lane"], [("M", 32), ("K", 8)])
    bad = LinearLayout([("offset", [(1, 0), (2, 0), (4, 0), (8, 0), (16, 0), (0, 1), (0, 2), (0, 2)])],
                       [("M", 32), ("K", 8)])
    with pytest.raises(ValueError):
        dst.invert_and_compose(bad)


def test_divide_left_eligibility(mi450):
    """Figure 5 caption: the first 3 lane bases of cvt must be [1],[2],[4] and
    every other basis a multiple of 8; rearranging repetition bases keeps it
    divisible; swapping two required lane bases makes it fail."""
    L, _ = mi450
    cvt = _mk(L["cvt"], ["register", "lane"], [("offset", 256)])
    tile = identity_1d(8, "lane", "offset")
    q = divide_left(cvt, tile)
    assert q is not None
    assert q.bases("lane") == [(1,), (2,)]
    assert q.bases("register") == [(4,), (8,), (16,)]
    assert dict(q.outs)["offset"] == 32
    scrambled = LinearLayout([("register", [(64,), (128,), (32,)]),
                              ("lane", [(1,), (2,), (4,), (16,), (8,)])], [("offset", 256)])
    assert divide_left(scrambled, tile) is not None
    swapped = LinearLayout([("register", [(32,), (64,), (128,)]),
                            ("lane", [(2,), (1,), (4,), (8,), (16,)])], [("offset", 256)])
    assert divide_left(swapped, tile) is None
    not_mult = LinearLayout([("register", [(33,), (64,), (128,)]),
                             ("lane", [(1,), (2,), (4,), (8,), (16,)])], [("offset", 256)])
    assert divide_left(not_mult, tile) is None


def test_cta_layouts(mi450):
    L, ev = mi450
    std = _mk(L["cta_standard"], ["warp"], [("M", 2), ("N", 2)])
    swz = _mk(L["cta_swizzled"], ["reg", "warp"], [("M", 4), ("N", 2)])
    args, img = ev["cta_standard"]
    assert std.apply(**args) == img
    args, img = ev["cta_swizzled"]
    assert swz.apply(**args) == img
    assert swz.is_bijective()                 # covers the 4 x 2 warp-tile grid
    # Pairs: even warps (SIMD pair A) and odd warps (pair B).  Standard layout:
    # w0 and w1 share M-row 0.  Swizzled: per instruction (fixed reg) the pairs
    # read disjoint M-rows.
    assert std.apply(warp=0)[0] == std.apply(warp=1)[0]
    for r in range(2):
        rows_a = {swz.apply(reg=r, warp=w)[0] for w in (0, 2)}
        rows_b = {swz.apply(reg=r, warp=w)[0] for w in (1, 3)}
        assert not rows_a & rows_b


def test_microbenchmark_layouts(mi450):
    L, _ = mi450
    dist = _mk(L["mb_dist"], ["reg", "lane", "warp"], [("d0", 4), ("d1", 256)])
    plain = _mk(L["mb_plain"], ["offset"], [("d0", 4), ("d1", 256)])
    part = _mk(L["mb_part"], ["offset", "partition"], [("d0", 4), ("d1", 256)])
    assert plain.is_bijective() and part.is_bijective()
    cvt_p = dist.invert_and_compose(plain)
    cvt_q = dist.invert_and_compose(part)
    for w in range(4):
        offs = set()
        for ln in range(32):
            for r in range(8):
                offs.add(cvt_p.apply(reg=r, lane=ln, warp=w)[0] * 2)     # fp16 bytes
                o, pidx = cvt_q.apply(reg=r, lane=ln, warp=w)
                assert pidx == w % 2                  # warp w on partition w % 2
        # one warp, one ds_load_b128: a single contiguous 512-byte window
        assert offs == set(range(512 * w, 512 * w + 512, 2))
    # 16 lanes per group, 16 bytes per lane, 64 banks: each bank exactly once
    addrs = [cvt_p.apply(reg=0, lane=ln, warp=0)[0] * 2 for ln in range(32)]
    rep = banksim.simulate(addrs, 16, n_banks=64, lanes_per_phase=16)
    assert rep.degree == 1 and rep.distinct_banks == [64, 64]


# ------------------------------------------------------------- bank model
def _parse_bank(golden_dir):
    rows = {}
    for line in open(os.path.join(golden_dir, "lds_bank_tables.txt")):
        line = line.split("#")[0].strip()
        if line:
            p = line.split()
            rows.setdefault(p[0], []).append([int(v) for v in p[1:]])
    return rows


def test_stride_examples(golden_dir):
    for nb, stride, lanes, banks in _parse_bank(golden_dir)["stride"]:
        rep = banksim.simulate([t * stride for t in range(lanes)], 4, n_banks=nb,
                               lanes_per_phase=lanes)
        assert rep.distinct_banks == [banks]
        assert rep.degree == lanes // banks


def _column_read(stride_bytes, lanes, nb):
    return banksim.simulate([t * stride_bytes for t in range(lanes)], 2, n_banks=nb,
                            lanes_per_phase=lanes)


def test_padding_tables(golden_dir):
    rows = _parse_bank(golden_dir)
    for pad, stride, deg in rows["pad64"]:
        assert stride == (64 + pad) * 2
        assert _column_read(stride, 64, 64).degree == deg
    for pad, stride, deg in rows["pad128"]:
        assert stride == (128 + pad) * 2
        got = _column_read(stride, 64, 64).degree
        if pad == 1:
            # printed 1-way; the page's own rule (bank = (t*258/4) % 64) puts
            # lanes 2i and 2i+1 on bank i at different words: 2-way.
            assert deg == 1 and got == 2
        else:
            assert got == deg


def test_padding_closed_form_bruteforce():
    for nb in (32, 64):
        for s in range(1, 257):
            rep = banksim.simulate([t * s * 4 for t in range(nb)], 4, n_banks=nb,
                                   lanes_per_phase=nb)
            assert rep.degree == banksim.padding_rule_degree(s, nb) == gcd(s, nb)
            assert rep.distinct_banks == [nb // gcd(s, nb)]


def test_broadcast_is_not_a_conflict():
    rep = banksim.simulate([0] * 32, 4)
    assert rep.degree == 1
    rep = banksim.simulate([0, 128] * 16, 4)
    assert rep.degree == 2


def test_xor_mask_rule_is_minimal_conflict_free(golden_dir):
    """The rule's mask is the smallest XOR mask on the 16-byte chunk index that
    makes a column of 16-byte vectors (rows one bank-span apart) conflict-free;
    brute force over masks."""
    for nb, vec, es, mask in _parse_bank(golden_dir)["mask"]:
        assert banksim.xor_mask_rule(nb, vec, es) == mask
        vbytes = vec * es
        lanes = nb * 4 // vbytes            # one phase
        span = nb * 4                       # row stride = all banks once
        best = None
        for m in range(0, span // vbytes):
            addrs = [r * span + (((0 ^ (r & m)) * vbytes) % span) for r in range(lanes)]
            if banksim.simulate(addrs, vbytes, n_banks=nb, lanes_per_phase=lanes).degree == 1:
                best = m
                break
        assert best == mask


def test_rocmlir_kpack_table(golden_dir):
    rows, degree = {}, None
    for line in open(os.path.join(golden_dir, "rocmlir_kpack_table.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        p = line.split()
        if p[0] == "row":
            rows[int(p[1])] = [tuple(int(x[1:]) for x in cell.split(":")) for cell in p[2:]]
        elif p[0] == "degree":
            degree = int(p[1])

    def addr(m, k):       # [kPackPerBlock, dPerBlock=96, kPack=4] f16
        return ((k // 4) * 96 + m) * 4 * 2 + (k % 4) * 2

    for m, cells in rows.items():
        for j, (t, bank) in enumerate(cells):
            k = 2 * j
            assert t == (m // 3) * 16 + j
            assert (addr(m, k) // 4) % 32 == bank
    # the phase that writes row m = 0 (threads 0..15) and m = 3 (16..31)
    addrs = [addr(0, 2 * t) for t in range(16)] + [addr(3, 2 * (t - 16)) for t in range(16, 32)]
    rep = banksim.simulate(addrs, 4, n_banks=32, lanes_per_phase=32)
    assert rep.degree == degree


# --------------------------------------------------- GB300 tile layouts
def test_sw128_is_bijective_and_matches_xor_rule():
    seen = set()
    for r in range(64):
        for b in range(0, 128, 2):
            o = banksim.sw128_row_major(r, b)
            assert (o >> 7) == r and (o & 15) == (b & 15)
            assert ((o >> 4) & 7) == ((b >> 4) ^ (r & 7))
            seen.add(o)
    assert seen == set(range(0, 64 * 128, 2))


def test_epilogue_store_pattern_conflict_free_and_control():
    for chunk in range(8):
        swz = banksim.simulate(banksim.epilogue_store_addresses(0, chunk, True), 16)
        assert swz.degree == 1 and swz.wavefronts == 4
        plain = banksim.simulate(banksim.epilogue_store_addresses(0, chunk, False), 16)
        assert plain.degree == 8 and plain.extra_wavefronts == 4 * 7


@pytest.mark.parametrize("mn_major", [False, True])
def test_tma_box_layout_equals_canonical_umma_layout(mn_major):
    """The 128B-swizzled TMA boxes and the tcgen05 SWIZZLE_128B canonical
    layout agree element by element when SBO = 1024 B (eight 128-byte rows)
    and, for MN-major tiles, LBO = one box (64 k-rows x 128 B); the K step
    advances the start address by 32 B (K-major) or 2 x SBO (MN-major)."""
    tile_mn = 256
    lbo = 64 * 128 if mn_major else 16
    sbo = 1024
    kstep = 2 * sbo if mn_major else 32
    offs = set()
    for mn in range(tile_mn):
        for k in range(64):
            a = banksim.operand_tile_offset(mn, k, mn_major, tile_mn)
            b = banksim.umma_canonical_offset(mn, k, mn_major, lbo, sbo, kstep)
            assert a == b
            offs.add(a)
    assert offs == set(range(0, tile_mn * 128, 2))


# ------------------------------------------------------------- invert
def test_invert_against_worked_cvt_table(mi450):
    """MI450 post, "Lowering local_load to ds_load_tr in Triton": the address
    step inverts the shared layout (offset -> [M, K]) and composes the result
    with the destination layout.  shared^-1 applied to each basis image of
    dstLL must give the printed cvt table, and shared^-1 must undo shared on
    every offset (brute force over the whole tile)."""
    L, _ = mi450
    dst = _mk(L["dst"], ["register", "lane"], [("M", 32), ("K", 8)])
    shared = _mk(L["shared"], ["offset"], [("M", 32), ("K", 8)])
    want = _mk(L["cvt"], ["register", "lane"], [("offset", 256)])
    inv = shared.invert()
    assert inv.in_names() == ["M", "K"] and inv.outs == [("offset", 256)]
    for dim in ("register", "lane"):
        got = [inv.apply(M=m, K=k) for (m, k) in dst.bases(dim)]
        assert got == want.bases(dim)
    seen = 0
    for ins, img in enumerate_map(shared):
        assert inv.apply(M=img[0], K=img[1]) == (ins["offset"],)
        seen += 1
    assert seen == 256


def test_invert_round_trip_on_swizzled_and_microbenchmark_layouts(mi450):
    """A 128-byte XOR swizzle in 16-byte units (offset chunk bits -> column,
    row bits -> row and column): its matrix is not a permutation, so a
    transpose in place of the inverse, or a dropped XOR term, fails the round
    trip.  Also the microbenchmark's plain [4, 256] layout."""
    L, _ = mi450
    sw = LinearLayout([("offset", [(0, 1), (0, 2), (0, 4), (1, 1), (2, 2), (4, 4)])],
                      [("row", 8), ("col", 8)])
    plain = _mk(L["mb_plain"], ["offset"], [("d0", 4), ("d1", 256)])
    for lay, names in ((sw, ("row", "col")), (plain, ("d0", "d1"))):
        inv = lay.invert()
        n = 0
        for ins, img in enumerate_map(lay):
            assert inv.apply(**dict(zip(names, img))) == (ins["offset"],)
            n += 1
        assert n == lay.in_size("offset")
        # and the other way round: lay(inv(x)) == x on every output coordinate
        for a in range(lay.out_size(names[0])):
            for b in range(lay.out_size(names[1])):
                (off,) = inv.apply(**{names[0]: a, names[1]: b})
                assert lay.apply(offset=off) == (a, b)
    # by hand: row bit i alone is offset bits (3 + i) and i (the XOR cancels
    # the column term); column bit i is offset bit i
    inv = sw.invert()
    assert inv.bases("row") == [(9,), (18,), (36,)]
    assert inv.bases("col") == [(1,), (2,), (4,)]


def test_invert_rejects_non_bijective_and_multi_input(mi450):
    L, _ = mi450
    part = _mk(L["mb_part"], ["offset", "partition"], [("d0", 4), ("d1", 256)])
    with pytest.raises(ValueError):
        part.invert()                         # two input dimensions
    collapsed = LinearLayout([("offset", [(1, 0), (2, 0), (0, 1), (0, 1)])], [("M", 4), ("K", 4)])
    with pytest.raises(ValueError):
        collapsed.invert()                    # rank 3 of 4
    short = LinearLayout([("offset", [(1, 0), (2, 0), (0, 1)])], [("M", 4), ("K", 4)])
    with pytest.raises(ValueError):
        short.invert()                        # injective, not surjective
