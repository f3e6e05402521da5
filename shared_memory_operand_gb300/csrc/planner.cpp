// Layout planner (host C++): see planner.h.
#include "planner.h"

#include <algorithm>
#include <cstdio>
#include <set>
#include <sstream>
#include <vector>

namespace smo {
namespace {

constexpr uint32_t kSwizzleSpan = 128;        // bytes per swizzled row
constexpr uint32_t kSwizzleAtom = 1024;       // 8 rows x 128 B

// 128-byte swizzle of a byte offset inside a 1024-byte aligned region: the
// 16-byte chunk index (bits 4..6) is XORed with the row-in-atom (bits 7..9).
inline uint32_t sw128(uint32_t off) { return off ^ (((off >> 7) & 7u) << 4); }

int log2i(uint32_t v) {
    int r = 0;
    while ((1u << r) < v) ++r;
    return r;
}

// Where TMA (SWIZZLE_128B, box inner extent 128 bytes) puts element (mn, k) of
// a stage tile.
uint32_t tma_offset(const OperandPlan& op, uint32_t mn, uint32_t k) {
    if (!op.mn_major) {
        // one box: outer = mn rows of 128 bytes (bk k values)
        return sw128(mn * kSwizzleSpan + k * op.es);
    }
    // boxes of T = 128 / es mn values x bk k rows: box j = mn / T, row = k
    const uint32_t T = kSwizzleSpan / op.es;
    uint32_t j = mn / T;
    return j * op.box_bytes + sw128(k * kSwizzleSpan + (mn % T) * op.es);
}

// Where the tensor core reads element (mn, k) given the descriptor fields
// (canonical SWIZZLE_128B layouts of the tcgen05 shared-memory descriptor),
// the start address advanced by kstep per MMA-wide K step.
uint32_t umma_offset(const OperandPlan& op, uint32_t mn, uint32_t k) {
    uint32_t step = k / op.mma_k, kk = k % op.mma_k;
    uint32_t start = step * op.kstep;
    uint32_t pre;
    if (!op.mn_major) {
        // ((8,m),(T,2)) : ((8T,SBO),(1,T)), T = 16 bytes
        pre = start + (mn % 8) * 128 + (mn / 8) * op.sbo + kk * op.es;
    } else {
        // ((T,8,m),(8,k)) : ((1,T,LBO),(8T,SBO)), T = 128 bytes of mn
        const uint32_t T = kSwizzleSpan / op.es;
        pre = start + (mn % T) * op.es + (mn / T) * op.lbo + (kk % 8) * 128 + (kk / 8) * op.sbo;
    }
    return sw128(pre);
}

uint64_t desc_hi(uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;     // leading dimension byte offset
    d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;     // stride dimension byte offset
    d |= (uint64_t)1 << 46;                          // fixed 0b001 (tcgen05 descriptor version)
    d |= (uint64_t)2 << 61;                          // layout: SWIZZLE_128B
    return d;                                        // base offset 0 (1024-aligned stages)
}

// es: bytes per element.  A stage holds one 128-byte swizzle row of K per
// K-major row (bk = 128 / es) and one MMA consumes 32 bytes of K.
void plan_operand(OperandPlan& op, int mn_major, int tile_mn, int es) {
    op.mn_major = mn_major;
    op.tile_mn = tile_mn;
    op.es = es;
    op.bk = (int)(kSwizzleSpan / es);
    op.mma_k = 32 / es;
    const uint32_t T = kSwizzleSpan / es;             // elements per 128-byte row
    if (!mn_major) {
        op.box_inner = op.bk;            // K, 128 bytes
        op.box_outer = tile_mn;          // MN rows
        op.nbox = 1;
        op.box_bytes = tile_mn * kSwizzleSpan;
        op.lbo = 16;                     // unused by swizzled K-major layouts
        op.sbo = kSwizzleAtom;           // next group of 8 rows
        op.kstep = op.mma_k * es;        // 32 bytes along the swizzled row
    } else {
        op.box_inner = T;                // MN, 128 bytes
        op.box_outer = op.bk;            // K rows
        op.nbox = (tile_mn + (int)T - 1) / (int)T;   // the last box may reach past the tile
        op.box_bytes = op.bk * kSwizzleSpan;
        op.lbo = op.box_bytes;           // next 128-byte-wide MN atom = next box
        op.sbo = kSwizzleAtom;           // next group of 8 k rows
        op.kstep = op.mma_k * kSwizzleSpan;   // mma_k k rows of 128 bytes
    }
    op.stage_bytes = op.box_bytes * op.nbox;
    op.desc_hi = desc_hi(op.lbo, op.sbo);

    // ---- F2 model and checks ------------------------------------------------
    // The stage holds what TMA writes: tile_mn rows of a K-major operand, or
    // nbox whole 128-byte-wide boxes of an MN-major one (loaded_mn >= tile_mn
    // when the tile is not a whole number of boxes; the MMA reads the first
    // tile_mn).  Linearity and bijectivity are checked over what is loaded,
    // TMA == tensor core over what the MMA reads.
    const uint32_t loaded_mn = op.mn_major ? (uint32_t)op.nbox * T : (uint32_t)tile_mn;
    op.bits_mn = log2i(loaded_mn);
    op.bits_k = log2i(op.bk);
    for (int i = 0; i < op.bits_mn; ++i) op.basis_mn[i] = tma_offset(op, 1u << i, 0);
    for (int i = 0; i < op.bits_k; ++i) op.basis_k[i] = tma_offset(op, 0, 1u << i);
    bool linear = true, same = true;
    std::vector<uint8_t> hit(op.nbox > 0 ? op.stage_bytes / es : 0, 0);
    bool inj = op.nbox > 0;
    for (uint32_t mn = 0; mn < loaded_mn; ++mn) {
        for (uint32_t k = 0; k < (uint32_t)op.bk; ++k) {
            uint32_t t = tma_offset(op, mn, k);
            uint32_t x = 0;
            for (int i = 0; i < op.bits_mn; ++i) if ((mn >> i) & 1) x ^= op.basis_mn[i];
            for (int i = 0; i < op.bits_k; ++i) if ((k >> i) & 1) x ^= op.basis_k[i];
            linear &= (x == t);
            if (mn < (uint32_t)tile_mn) same &= (umma_offset(op, mn, k) == t);
            if (t / es >= hit.size() || hit[t / es]) inj = false; else hit[t / es] = 1;
        }
    }
    op.linear = linear;
    op.tma_equals_umma = same;
    op.bijective = inj && std::all_of(hit.begin(), hit.end(), [](uint8_t h) { return h != 0; });
    // Left division by the 16-byte contiguous row of a core matrix: the bases
    // of the contiguous dimension must be es, 2 es, ..., 8 bytes and every
    // other basis a multiple of 16 bytes.
    const uint32_t* cont = op.mn_major ? op.basis_mn : op.basis_k;
    int ncont = op.mn_major ? op.bits_mn : op.bits_k;
    const int inner = log2i(16u / (uint32_t)es);      // bases inside one 16-byte row
    bool div = ncont >= inner;
    for (int i = 0; i < inner && i < ncont; ++i) div &= cont[i] == ((uint32_t)es << i);
    for (int i = inner; i < ncont; ++i) div &= (cont[i] % 16) == 0;
    const uint32_t* other = op.mn_major ? op.basis_k : op.basis_mn;
    int nother = op.mn_major ? op.bits_k : op.bits_mn;
    for (int i = 0; i < nother; ++i) div &= (other[i] % 16) == 0;
    op.core_matrix_divides = div;
}

// Epilogue staging: warp-private slabs of 32 rows x 128 bytes, 128-byte
// swizzled; lane l stores 16-byte chunk j of row l.
uint32_t epi_offset(uint32_t row, uint32_t chunk) { return sw128(row * 128 + chunk * 16); }

int bank_degree_16B(const uint32_t* addr, int lanes) {
    // 32 banks x 4 bytes; 16-byte accesses served 8 lanes per phase.
    int worst = 0;
    for (int p = 0; p < lanes; p += 8) {
        std::set<uint32_t> words[32];
        for (int l = p; l < p + 8 && l < lanes; ++l)
            for (uint32_t w = addr[l] / 4; w < (addr[l] + 16) / 4; ++w) words[w % 32].insert(w);
        for (auto& s : words) worst = std::max<int>(worst, (int)s.size());
    }
    return worst;
}

}  // namespace

uint32_t make_idesc(int in_dtype, int a_mn_major, int b_mn_major, int M, int N) {
    // A / B format field: kind::f16 F16 = 0, BF16 = 1; kind::f8f6f4 E4M3 = 0, E5M2 = 1
    uint32_t fmt = (in_dtype == 0 || in_dtype == 4) ? 1u : 0u;
    uint32_t d = 0;
    d |= 1u << 4;                                  // D format: F32
    d |= fmt << 7;                                 // A format
    d |= fmt << 10;                                // B format
    d |= (uint32_t)(a_mn_major & 1) << 15;         // A major: 0 K, 1 MN
    d |= (uint32_t)(b_mn_major & 1) << 16;         // B major
    d |= (uint32_t)((N >> 3) & 0x3F) << 17;        // N >> 3
    d |= (uint32_t)((M >> 4) & 0x1F) << 24;        // M >> 4
    return d;
}

Plan make_plan(int64_t M, int64_t N, int64_t K, int a_major, int b_major, int in_dtype,
               int out_dtype, int64_t batch, int num_sms, int force, int split, int wide_bn) {
    Plan p;
    p.M = M; p.N = N; p.K = K; p.batch = batch;
    p.in_dtype = in_dtype; p.out_dtype = out_dtype;
    p.num_sms = num_sms > 0 ? num_sms : 1;
    if (M >= (1ll << 31) || N >= (1ll << 31) || K >= (1ll << 31) || batch >= (1ll << 31)) {
        p.why = "dimension beyond 2^31-1";
        return p;
    }
    if (in_dtype != 0 && in_dtype != 1 && in_dtype != 3 && in_dtype != 4) {
        p.why = "input type";
        return p;
    }
    p.in_es = (in_dtype == 3 || in_dtype == 4) ? 1 : 2;
    p.kind = p.in_es == 1 ? 1 : 0;
    p.bk = (int)(kSwizzleSpan / p.in_es);
    p.mma_k = 32 / p.in_es;
    p.num_k = (int)((K + p.bk - 1) / p.bk);
    auto tiles_for = [&](int tm, int bn) { return ((M + tm - 1) / tm) * ((N + bn - 1) / bn) * batch; };
    // Wave quantisation, in units of one 128 x 256 tile on one SM: a 128-wide
    // tile costs a bit over half of that; a CTA pair computes a 256 x 256 tile
    // on two SMs in about 0.85 of it (half the B bytes per SM, deeper pipeline).
    const int64_t clusters = std::max(1, p.num_sms / 2);
    const int64_t t256 = tiles_for(kBM, 256), t128 = tiles_for(kBM, 128), tpair = tiles_for(2 * kBM, 256);
    const int64_t twide = tiles_for(4 * kBM, 256);
    const double c256 = (double)((t256 + p.num_sms - 1) / p.num_sms) * 1.0;
    const double c128 = (double)((t128 + p.num_sms - 1) / p.num_sms) * 0.55;
    const double cpair = (double)((tpair + clusters - 1) / clusters) * 0.85;
    // A wide pair tile is two pair tiles' work on three quarters of the
    // operand bytes (measured about 5% cheaper per flop at 8192^3), but its
    // single accumulator is held once per tile while the epilogue warps read
    // it out: it wins when every tile runs a long enough K loop.  Measured
    // with the 8-warp epilogue that hands the accumulator back from
    // registers: 16 K blocks (skinny) -7%, 32 (batched) +1.8%.
    const double cwide = (double)((twide + clusters - 1) / clusters) * 1.62;
    const bool long_k = p.num_k >= 32;
    int choice;
    if (force == 128 || force == 192 || force == 256 || force == 384 || force == 512 || force == 1024) choice = force;
    else if (cpair <= c256 && cpair <= c128) choice = (long_k && cwide < cpair) ? 1024 : 512;
    else choice = (c128 < c256) ? 128 : 256;
    // Split-K over a 2-CTA cluster (fp32 output): for a tile-starved problem
    // -- one wave of one-CTA tiles on fewer SMs than the GPU has -- the two
    // CTAs of each tile's cluster read half of its K panel each, on twice the
    // SMs, and their partials meet in global memory.  Main-loop model,
    // measured on GB300 with one-CTA tiles: an SM takes operands in at about
    // 135 GB/s, and all SMs together at about 16 TB/s; the main loop lasts
    // max(bytes per SM / 135 GB/s, total bytes / 16 TB/s).  The split's
    // second pass over C (plain stores, their completion, then TMA
    // reduce-adds) costs about 1.8 us more than one epilogue.  The split is
    // taken for the tile width (128 / 192 / 256) whose two CTAs per tile fit
    // one wave and whose modelled time beats the unsplit plan by more than
    // that (measured: 512^2 x 4096 22.5 -> 15.4 us, 1024^2 x 1536 12.1 ->
    // 10.9 us; 1500 x 1152 x 896 would lose 0.9 us and is not split).
    const bool one_cta = choice == 128 || choice == 192 || choice == 256;
    if (one_cta && out_dtype == 2 && p.num_k >= 2 && split != 0) {
        auto main_us = [&](int64_t ctas, int bn, int64_t kblocks) {
            const double per_cta = (double)(kBM + bn) * kSwizzleSpan * (double)kblocks;   // operand bytes
            const int64_t waves = (ctas + p.num_sms - 1) / p.num_sms;
            const int64_t active = std::min<int64_t>(ctas, p.num_sms);
            const double per_sm_us = per_cta / 135e3;                                     // 135 GB/s
            const double agg_us = per_cta * (double)active / 16e6;                          // 16 TB/s
            return (double)waves * std::max(per_sm_us, agg_us);
        };
        const double base_us = main_us(tiles_for(kBM, choice), choice, p.num_k);
        int sbn = 0;
        double best = 0.0;
        for (int bn : {128, 192, 256}) {
            if (force == 128 || force == 192 || force == 256) {
                if (bn != force) continue;
            } else if (2 * tiles_for(kBM, bn) > p.num_sms) {
                continue;
            }
            const double t = main_us(2 * tiles_for(kBM, bn), bn, (p.num_k + 1) / 2) + 1.8;
            if (sbn == 0 || t < best) {
                sbn = bn;
                best = t;
            }
        }
        const bool starved = tiles_for(kBM, choice) <= p.num_sms && sbn != 0 && best < base_us;
        if (split == 1 || starved) {
            p.split = 1;
            choice = sbn != 0 ? sbn : 256;
        }
    }
    p.pair = choice == 384 || choice == 512 || choice == 1024;
    p.wide = choice == 1024;
    p.tile_m = p.wide ? 4 * kBM : p.pair ? 2 * kBM : kBM;
    int bn = choice == 384 ? 128 : p.pair ? 256 : choice;
    if (p.wide) {
        // Wave quantisation of wide tiles: a narrower tile (still a multiple
        // of 16 columns, so that each CTA's half is a whole number of 8-column
        // core matrices) takes fewer tensor cycles, so a width whose tile
        // count fills the last wave better can win: 4096^2 has 128 tiles of
        // 512 x 256 on 76 clusters (1.68 waves, run as 2), but 152 of 512 x
        // 224 (exactly 2 waves).  A tile's time is modelled as 0.35 + 0.65 x
        // width / 256 of a 256-wide one: its A panel, fill and epilogue do not
        // shrink with the width (measured: 4096^3 +5% at 224, 8192^3's tail
        // wave +1.4% at 208, 32 x 2048^3 -8% at 208).  Ties keep 256.
        if (wide_bn >= 16 && wide_bn <= 256 && wide_bn % 16 == 0) {
            bn = wide_bn;
        } else {
            double best = 0.0;
            for (int w : {256, 240, 224, 208, 192}) {
                // an N-major B half-tile must start on a 16-byte boundary (TMA)
                if (b_major && ((w / 2) * p.in_es) % 16 != 0) continue;
                const int64_t t = tiles_for(4 * kBM, w);
                const double cost = (double)((t + clusters - 1) / clusters) * (0.35 + 0.65 * (double)w / 256.0);
                if (w == 256 || cost < best - 1e-9) {
                    best = cost;
                    bn = w;
                }
            }
        }
    }
    p.BN = bn;
    p.num_m = (int)((M + p.tile_m - 1) / p.tile_m);
    p.num_n = (int)((N + bn - 1) / bn);
    p.tiles = tiles_for(p.tile_m, bn);
    p.group_m = std::min(p.pair ? 8 : 16, p.num_m);
    // Tail of a wide tiling (256 wide): when the tiles leave a last wave only
    // partly full and those tiles, in the grouped order, are whole columns of
    // the last M group -- the last q N blocks of one problem, or, in a batch
    // whose problems are one M group each, the last columns of one problem and
    // the problems after it -- they are re-tiled with the narrowest width (a
    // multiple of 16 that keeps the TMA coordinate rule) whose tiles still fit
    // one wave: 8192^2 has 6 full waves of 76 tiles and 56 left over (8 M
    // blocks x 7 N blocks); as 72 tiles of 512 x 208 the last wave takes
    // 13/16 of a full one.  32 x 2048^2 leaves 36 tiles (the last column of
    // one problem and the whole next one), re-tiled as 72 of 512 x 128.
    const bool one_group = p.group_m == p.num_m;
    if (p.wide && bn == 256 && (batch == 1 || one_group) && force != 1024 && wide_bn == 0) {
        const int64_t C = clusters;
        const int64_t T = p.tiles;
        const int64_t R = T % C;
        const int gstart = batch == 1 ? ((p.num_m - 1) / p.group_m) * p.group_m : 0;
        const int gsz = p.num_m - gstart;
        if (T / C >= 1 && R > 0 && R % gsz == 0) {
            const int64_t q = R / gsz;                         // tail columns, in the grouped order
            // problems after the first one the tail touches, and the first one's columns
            const int64_t later = batch == 1 ? 0 : (q - 1) / p.num_n;
            const int64_t q_first = q - later * p.num_n;
            if (batch > 1 || q < p.num_n) {       // one problem: not its whole last group
                const int64_t n0 = (int64_t)(p.num_n - q_first) * bn;
                for (int w = 16; w < bn; w += 16) {
                    if (b_major && ((w / 2) * p.in_es) % 16 != 0) continue;
                    const int64_t k0 = gsz * ((N - n0 + w - 1) / w);
                    const int64_t kfull = gsz * ((N + w - 1) / w);
                    if (k0 + later * kfull > C) continue;
                    p.tail = 1;
                    p.tail_bn = w;
                    p.tail_m0 = gstart;
                    p.tail_gsz = gsz;
                    p.tail_n0 = (int)n0;
                    p.tail_b0 = (int)(batch - 1 - later);
                    p.tail_k0 = (int)k0;
                    p.tail_kfull = (int)kfull;
                    p.tail_start = T - R;
                    p.tail_tiles = (int)(k0 + later * kfull);
                    break;
                }
            }
        }
        if (p.tail) p.tiles = p.tail_start + p.tail_tiles;
    }
    if (p.split) {
        // one tile per cluster (the epilogue stages in the idle operand ring)
        if (2 * p.tiles >= (1ll << 31)) {
            p.why = "too many tiles for a split-K grid";
            return p;
        }
        p.grid = (int)(2 * p.tiles);
        p.split_kh = (p.num_k + 1) / 2;
    } else {
        p.grid = p.pair ? (int)(2 * std::min<int64_t>(p.tiles, clusters)) : (int)std::min<int64_t>(p.tiles, p.num_sms);
    }
    p.idesc = make_idesc(in_dtype, a_major, b_major, p.pair ? 2 * kBM : kBM, bn);
    if (p.tail) p.tail_idesc = make_idesc(in_dtype, a_major, b_major, 2 * kBM, p.tail_bn);

    // Per-CTA operand tiles: A 128 rows (256 in a wide pair); B all BN columns,
    // or half of them in a pair.
    plan_operand(p.a, a_major, p.wide ? 2 * kBM : kBM, p.in_es);
    plan_operand(p.b, b_major, p.pair ? bn / 2 : bn, p.in_es);

    // TMA rule: a tiled copy's innermost coordinate times the element size
    // must be a multiple of 16 bytes, or the copy faults.  For an MN-major
    // operand that coordinate is the tile's MN origin (a multiple of the tile
    // step) plus the CTA's offset inside a pair tile (a multiple of its own
    // tile) plus whole 128-byte boxes; for a K-major operand it is a multiple
    // of the 128-byte stage.  The C map's innermost coordinate is a tile's
    // column origin plus whole 128-byte chunks.  A plan that breaks this is
    // never launched.
    auto x_aligned = [](int64_t elems, int es) { return (elems * es) % 16 == 0; };
    const bool a_ok = !a_major || (x_aligned(p.tile_m, p.in_es) && x_aligned(p.a.tile_mn, p.in_es));
    const bool b_ok = !b_major || (x_aligned(bn, p.in_es) && x_aligned(p.b.tile_mn, p.in_es));
    const bool c_ok = x_aligned(bn, out_dtype == 2 ? 4 : 2) &&
                      (!p.tail || (x_aligned(p.tail_bn, out_dtype == 2 ? 4 : 2) && x_aligned(p.tail_n0, out_dtype == 2 ? 4 : 2) &&
                                   (!b_major || (x_aligned(p.tail_bn / 2, p.in_es) && x_aligned(p.tail_n0, p.in_es)))));
    if (!a_ok || !b_ok || !c_ok) {
        p.why = "tile width breaks the 16-byte TMA coordinate rule";
        return p;
    }

    p.c.out_es = (out_dtype == 2) ? 4 : 2;
    p.c.chunk_cols = 128 / p.c.out_es;
    p.c.chunks = (bn + p.c.chunk_cols - 1) / p.c.chunk_cols;
    p.c.last_cols = bn - (p.c.chunks - 1) * p.c.chunk_cols;
    // 256 x 256 pair tiles with 16-bit output: each epilogue warp reads its
    // four chunks into registers, hands the accumulator back and spaces the
    // four stores over about half of the next tile's main loop instead of
    // issuing them in one burst, which competed with that loop's operand
    // loads for the SM's path to L2 (measured on 16384 x 8192 x 1024: +1.5%
    // for the early hand-back, +2.9% with 40-56 ns per K block, -9% at 85,
    // where the stores run into the next epilogue).  A K block takes about
    // 265 ns at the 16-bit MMA rate and half that with FP8.
    if (p.pair && !p.wide && out_dtype != 2 && p.c.chunks == 4 && p.c.last_cols == p.c.chunk_cols)
        p.epi_pace_ns_per_kb = p.in_es == 1 ? 24 : 48;
    if (p.tail) {
        p.tail_chunks = (p.tail_bn + p.c.chunk_cols - 1) / p.c.chunk_cols;
        p.tail_last_cols = p.tail_bn - (p.tail_chunks - 1) * p.c.chunk_cols;
    }
    for (int i = 0; i < 5; ++i) p.c.basis_row[i] = epi_offset(1u << i, 0);
    for (int i = 0; i < 3; ++i) p.c.basis_chunk[i] = epi_offset(0, 1u << i);
    {
        std::set<uint32_t> offs;
        bool lin = true;
        for (uint32_t r = 0; r < 32; ++r)
            for (uint32_t c = 0; c < 8; ++c) {
                uint32_t o = epi_offset(r, c);
                uint32_t x = 0;
                for (int i = 0; i < 5; ++i) if ((r >> i) & 1) x ^= p.c.basis_row[i];
                for (int i = 0; i < 3; ++i) if ((c >> i) & 1) x ^= p.c.basis_chunk[i];
                lin &= (x == o);
                offs.insert(o);
            }
        p.c.bijective = lin && offs.size() == 256 && *offs.rbegin() == kEpiSlabBytes - 16;
        int worst = 0;
        for (uint32_t j = 0; j < 8; ++j) {
            uint32_t addr[32];
            for (uint32_t l = 0; l < 32; ++l) addr[l] = epi_offset(l, j);
            worst = std::max(worst, bank_degree_16B(addr, 32));
        }
        p.c.planner_degree = worst;
    }

    // Shared-memory carve-up (offsets from a 1024-byte aligned base).
    p.stage_stride = p.a.stage_bytes + p.b.stage_bytes;
    uint32_t epi_bytes = kEpiWarps * kEpiBufs * kEpiSlabBytes;
    uint32_t fixed = 1024 /* alignment slack */ + epi_bytes + kBarrierBytes;
    int stages = (int)((kSmemLimit - fixed) / p.stage_stride);
    stages = std::min(stages, kMaxStages);
    if (stages < 2) {
        p.why = "shared memory too small for two stages";
        return p;
    }
    p.stages = stages;
    // Two stages per barrier pair halve the waits and commits the single
    // MMA-issuing thread executes per MMA.  With fewer than six stages the
    // one-CTA ring would have too few groups in flight to hide the load
    // latency; the CTA-pair kernel (32 KiB stages, six of them) always
    // groups two.
    if (p.pair && !p.wide && stages < 4) {
        p.why = "shared memory too small for two groups of two stages";
        return p;
    }
    if (p.wide && stages < 3) {
        p.why = "shared memory too small for three wide stages";
        return p;
    }
    // A wide pair's stage already holds 8 MMAs (two 128-row halves of A).
    p.kgroup = p.wide ? 1 : (p.pair || stages >= 6) ? 2 : 1;
    p.off_epi = stages * p.stage_stride;
    p.off_bar = p.off_epi + epi_bytes;
    p.smem_bytes = p.off_bar + kBarrierBytes + 1024;
    p.tmem_cols = 32;                              // two accumulators, allocated as a power of two >= 32
    while (p.tmem_cols < (uint32_t)(2 * bn)) p.tmem_cols <<= 1;
    // a split CTA stages its partial of the peer's half of the tile (4 warps x
    // up to 4 chunks of 4 KiB) in the idle operand ring
    if (p.split && (uint32_t)p.stages * p.stage_stride < kEpiWarps * 4 * kEpiSlabBytes) {
        p.why = "operand ring too small to stage a split tile";
        return p;
    }

    bool layouts_ok = p.a.linear && p.a.bijective && p.a.tma_equals_umma && p.a.core_matrix_divides &&
                      p.b.linear && p.b.bijective && p.b.tma_equals_umma && p.b.core_matrix_divides &&
                      p.c.bijective && p.c.planner_degree == 1;
    if (!layouts_ok) {
        p.why = "layout check failed";
        return p;
    }
    p.ok = true;
    return p;
}

void fill_params(const Plan& p, KParams* kp) {
    kp->M = (int32_t)p.M; kp->N = (int32_t)p.N; kp->K = (int32_t)p.K; kp->batch = (int32_t)p.batch;
    kp->num_m = p.num_m; kp->num_n = p.num_n; kp->num_k = p.num_k;
    kp->group_m = p.group_m;
    kp->tiles_per_batch = (int64_t)p.num_m * p.num_n;
    kp->total_tiles = p.tiles;
    kp->BN = p.BN; kp->stages = p.stages;
    kp->kgroup = p.kgroup;
    kp->bk = p.bk;
    kp->m_sub = p.wide ? 2 : 1;
    kp->idesc = p.idesc;
    kp->a_mn_major = p.a.mn_major; kp->b_mn_major = p.b.mn_major;
    kp->a_nbox = p.a.nbox; kp->b_nbox = p.b.nbox;
    kp->a_box_bytes = p.a.box_bytes; kp->b_box_bytes = p.b.box_bytes;
    kp->a_box_mn = p.a.mn_major ? p.a.box_inner : p.a.box_outer;
    kp->b_box_mn = p.b.mn_major ? p.b.box_inner : p.b.box_outer;
    kp->a_kstep = p.a.kstep; kp->b_kstep = p.b.kstep;
    kp->a_desc_hi = p.a.desc_hi; kp->b_desc_hi = p.b.desc_hi;
    kp->stage_stride = p.stage_stride;
    kp->b_off = p.a.stage_bytes;
    kp->off_epi = p.off_epi; kp->off_bar = p.off_bar;
    kp->tmem_cols = p.tmem_cols;
    kp->tx_bytes = p.pair ? 2 * p.stage_stride : p.stage_stride;   // a pair's even CTA arms both CTAs' bytes
    kp->epi_chunk_cols = p.c.chunk_cols;
    kp->epi_chunks = p.c.chunks;
    kp->epi_last_cols = p.c.last_cols;
    kp->split_kh = p.split ? p.split_kh : 0;
    kp->tail_start = p.tail ? p.tail_start : p.tiles;
    kp->tail_m0 = p.tail_m0;
    kp->tail_gsz = p.tail_gsz;
    kp->tail_n0 = p.tail_n0;
    kp->tail_bn = p.tail_bn;
    kp->epi_pace_ns_per_kb = p.epi_pace_ns_per_kb;
    kp->tail_b0 = p.tail_b0;
    kp->tail_k0 = p.tail_tiles == 0 ? 0 : p.tail_k0;
    kp->tail_kfull = p.tail_kfull > 0 ? p.tail_kfull : 1;
    kp->tail_idesc = p.tail_idesc;
    kp->tail_epi_chunks = p.tail_chunks;
    kp->tail_epi_last_cols = p.tail_last_cols;
}

std::string describe_json(const Plan& p) {
    std::ostringstream o;
    auto op_json = [&](const OperandPlan& a) {
        o << "{\"mn_major\":" << a.mn_major << ",\"tile_mn\":" << a.tile_mn
          << ",\"box\":[" << a.box_inner << "," << a.box_outer << "],\"nbox\":" << a.nbox
          << ",\"box_bytes\":" << a.box_bytes << ",\"stage_bytes\":" << a.stage_bytes
          << ",\"lbo\":" << a.lbo << ",\"sbo\":" << a.sbo << ",\"kstep_bytes\":" << a.kstep
          << ",\"desc_hi\":" << a.desc_hi << ",\"swizzle\":\"128B\"";
        o << ",\"basis_mn\":[";
        for (int i = 0; i < a.bits_mn; ++i) o << (i ? "," : "") << a.basis_mn[i];
        o << "],\"basis_k\":[";
        for (int i = 0; i < a.bits_k; ++i) o << (i ? "," : "") << a.basis_k[i];
        o << "],\"linear\":" << (a.linear ? "true" : "false")
          << ",\"bijective\":" << (a.bijective ? "true" : "false")
          << ",\"tma_equals_umma\":" << (a.tma_equals_umma ? "true" : "false")
          << ",\"core_matrix_divides\":" << (a.core_matrix_divides ? "true" : "false") << "}";
    };
    o << "{\"ok\":" << (p.ok ? "true" : "false") << ",\"why\":\"" << p.why << "\""
      << ",\"M\":" << p.M << ",\"N\":" << p.N << ",\"K\":" << p.K << ",\"batch\":" << p.batch
      << ",\"pair\":" << p.pair << ",\"wide\":" << p.wide << ",\"split\":" << p.split
      << ",\"split_kh\":" << p.split_kh << ",\"tail\":" << p.tail << ",\"tail_start\":" << p.tail_start
      << ",\"tail_m0\":" << p.tail_m0 << ",\"tail_gsz\":" << p.tail_gsz << ",\"tail_n0\":" << p.tail_n0
      << ",\"tail_bn\":" << p.tail_bn << ",\"tail_tiles\":" << p.tail_tiles << ",\"tail_b0\":" << p.tail_b0
      << ",\"tail_k0\":" << p.tail_k0 << ",\"tail_kfull\":" << p.tail_kfull
      << ",\"epi_pace_ns_per_kb\":" << p.epi_pace_ns_per_kb << ",\"tail_idesc\":" << p.tail_idesc
      << ",\"tail_chunks\":" << p.tail_chunks << ",\"tail_last_cols\":" << p.tail_last_cols << ",\"BM\":" << p.tile_m << ",\"BN\":" << p.BN << ",\"BK\":" << p.bk << ",\"mma_k\":" << p.mma_k << ",\"kind\":" << p.kind << ",\"in_es\":" << p.in_es
      << ",\"stages\":" << p.stages << ",\"kgroup\":" << p.kgroup << ",\"num_m\":" << p.num_m << ",\"num_n\":" << p.num_n
      << ",\"num_k\":" << p.num_k << ",\"tiles\":" << p.tiles << ",\"grid\":" << p.grid
      << ",\"group_m\":" << p.group_m << ",\"threads\":" << (p.wide || (!p.pair && !p.split && p.tiles <= p.grid && p.c.chunks <= 4) ? kWideThreads : kThreads)
      << ",\"idesc\":" << p.idesc << ",\"smem_bytes\":" << p.smem_bytes
      << ",\"stage_stride\":" << p.stage_stride << ",\"off_epi\":" << p.off_epi
      << ",\"off_bar\":" << p.off_bar << ",\"tmem_cols\":" << p.tmem_cols;
    o << ",\"A\":";
    op_json(p.a);
    o << ",\"B\":";
    op_json(p.b);
    o << ",\"C\":{\"out_es\":" << p.c.out_es << ",\"chunk_cols\":" << p.c.chunk_cols
      << ",\"chunks\":" << p.c.chunks << ",\"last_cols\":" << p.c.last_cols << ",\"slab_bytes\":" << kEpiSlabBytes
      << ",\"bufs\":" << kEpiBufs << ",\"basis_row\":[";
    for (int i = 0; i < 5; ++i) o << (i ? "," : "") << p.c.basis_row[i];
    o << "],\"basis_chunk\":[";
    for (int i = 0; i < 3; ++i) o << (i ? "," : "") << p.c.basis_chunk[i];
    o << "],\"bijective\":" << (p.c.bijective ? "true" : "false")
      << ",\"planner_degree\":" << p.c.planner_degree;
    // Addresses (from the aligned smem base) of the 8 st.shared.v4 of one chunk
    // for every epilogue warp slot and staging buffer.
    o << ",\"store_addrs\":[";
    bool first = true;
    for (uint32_t w = 0; w < (uint32_t)kEpiWarps; ++w)
        for (uint32_t sb = 0; sb < (uint32_t)kEpiBufs; ++sb)
            for (uint32_t j = 0; j < 8; ++j) {
                o << (first ? "" : ",") << "[";
                first = false;
                uint32_t base = p.off_epi + (w * kEpiBufs + sb) * kEpiSlabBytes;
                for (uint32_t l = 0; l < 32; ++l) o << (l ? "," : "") << base + epi_offset(l, j);
                o << "]";
            }
    o << "]}}";
    return o.str();
}

}  // namespace smo
