// Device pieces shared by the one-CTA and CTA-pair GEMM kernels: error
// reporting, tile decoding, the producer's per-lane TMA load slots, the
// stream-K work split (whole tiles, then K ranges of the last wave's tiles),
// its fp32 partials and their fix-up, and the epilogue (tensor memory ->
// registers -> 128-byte-swizzled shared-memory slab -> TMA store, ragged row
// tails stored directly).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "gemm_params.h"
#include "ptx.cuh"

namespace smo {

__device__ __forceinline__ void report_error(int32_t* err, int32_t code) {
    if (err) atomicCAS(err, 0, code);
}

// Tile id -> (batch, m block, n block), grouped along M for L2 reuse.
__device__ __forceinline__ void decode_tile(const KParams& p, int64_t t, int& b, int& mb, int& nb) {
    b = (int)(t / p.tiles_per_batch);
    const int64_t r = t - (int64_t)b * p.tiles_per_batch;
    const int64_t span = (int64_t)p.group_m * p.num_n;
    const int g = (int)(r / span);
    const int first_m = g * p.group_m;
    const int gsz = min(p.num_m - first_m, p.group_m);
    const int rr = (int)(r - (int64_t)g * span);
    mb = first_m + rr % gsz;
    nb = rr / gsz;
}

// Tile id -> (batch, m block, first column, width), with the tail region of a
// wide tiling: tiles [tail_start, total_tiles) are tail_bn wide and cover M
// blocks [tail_m0, tail_m0 + tail_gsz) in column blocks of tail_gsz tiles --
// the first tail_k0 of them columns [tail_n0, N) of problem tail_b0, then
// tail_kfull per later problem, columns [0, N).  Tiles before tail_start
// decode as decode_tile does (the tail region is the end of the grouped
// order).
__device__ __forceinline__ void decode_tile_w(const KParams& p, int64_t t, int& b, int& mb, int32_t& n0,
                                              int32_t& bn) {
    if (t >= p.tail_start) {
        int32_t r = (int32_t)(t - p.tail_start);
        int32_t base = p.tail_n0;
        b = p.tail_b0;
        if (r >= p.tail_k0) {
            r -= p.tail_k0;
            const int32_t j = r / p.tail_kfull;
            b += 1 + j;
            r -= j * p.tail_kfull;
            base = 0;
        }
        mb = p.tail_m0 + r % p.tail_gsz;
        n0 = base + (r / p.tail_gsz) * p.tail_bn;
        bn = p.tail_bn;
        return;
    }
    int nb;
    decode_tile(p, t, b, mb, nb);
    n0 = nb * p.BN;
    bn = p.BN;
}

// One TMA load of a pipeline stage, owned by one lane of the producer warp.
// All of a stage's loads (A boxes, then B boxes) are issued by consecutive
// lanes in a single instruction: the producer's issue cost is then one
// instruction per stage instead of one per box.  Every operand map is 4-D;
// T = 128 bytes of MN elements (64 of 16 bits, 128 of 8 bits):
//   fused MN-major (extent % T == 0): {T, K, MN / T, batch}, one load
//   K-major box:                      {K, MN, 1, batch}
//   MN-major T-wide box:              {MN, K, 1, batch}
struct LoadSlot {
    const CUtensorMap* tm;
    uint32_t dst_off;      // from the stage base
    uint32_t mode;         // 0 fused, 1 K-major box, 2 MN-major box
    int32_t mn_off;        // offset of this box along MN
    int32_t box_mn_log2;   // log2 of the MN extent of one box (64 or 128 elements, or a tile's rows)
    bool is_a;
};

__device__ __forceinline__ uint32_t stage_loads(const KParams& p) {
    return (p.a_fused ? 1u : p.a_nbox) + (p.b_fused ? 1u : p.b_nbox);
}

__device__ __forceinline__ LoadSlot load_slot(const KParams& p, const CUtensorMap* tmA, const CUtensorMap* tmB,
                                              uint32_t lane) {
    const uint32_t na = p.a_fused ? 1u : p.a_nbox;
    LoadSlot s;
    s.is_a = lane < na;
    const uint32_t j = s.is_a ? lane : lane - na;
    const uint32_t fused = s.is_a ? p.a_fused : p.b_fused;
    const uint32_t mn_major = s.is_a ? p.a_mn_major : p.b_mn_major;
    s.tm = s.is_a ? tmA : tmB;
    s.dst_off = (s.is_a ? 0u : p.b_off) + j * (s.is_a ? p.a_box_bytes : p.b_box_bytes);
    s.mode = fused ? 0u : (mn_major ? 2u : 1u);
    const uint32_t box_mn = s.is_a ? p.a_box_mn : p.b_box_mn;   // a power of two
    s.box_mn_log2 = 31 - __clz((int)box_mn);
    s.mn_off = (int32_t)(j * box_mn);
    return s;
}

// Coordinates of a slot's load for K block k0 of the tile whose operand rows
// (A) / columns (B) start at mn0.
__device__ __forceinline__ void slot_coords(const LoadSlot& s, int32_t mn0, int32_t k0, int32_t& c0, int32_t& c1,
                                            int32_t& c2) {
    if (s.mode == 0) {
        c0 = 0; c1 = k0; c2 = mn0 >> s.box_mn_log2;
    } else if (s.mode == 1) {
        c0 = k0; c1 = mn0 + s.mn_off; c2 = 0;
    } else {
        c0 = mn0 + s.mn_off; c1 = k0; c2 = 0;
    }
}

// ---------------------------------------------------------------- work items
// One unit of a CTA's (or CTA pair's) work: K blocks [kb0, kb1) of one tile.
enum WorkRole : int32_t {
    ROLE_WHOLE = 0,     // every K block: normal epilogue
    ROLE_OWNER = 1,     // the tile's first K blocks: adds the later pieces' partials, then the epilogue
    ROLE_PARTIAL = 2,   // later K blocks of a tile: publishes an fp32 partial into this cluster's slot
};

struct WorkItem {
    int64_t tile;
    int32_t kb0, kb1;
    int32_t role;
    int32_t sk_tile;    // index among the stream-K tiles (ROLE_OWNER / ROLE_PARTIAL)
    int32_t last_slot;  // ROLE_OWNER: partials come from clusters (self, last_slot]
};

struct WorkIter {
    int64_t dp, dp_stride;      // next whole tile, stride = clusters
    int64_t u, u1;              // stream-K unit cursor and end
    int64_t self;               // this cluster
};

// First stream-K unit of cluster c.
__device__ __forceinline__ int64_t sk_bound(const KParams& p, int64_t c) {
    return c * p.sk_units / p.sk_clusters;
}

// Cluster whose unit range holds unit u: the largest c with sk_bound(c) <= u.
__device__ __forceinline__ int64_t sk_cluster_of(const KParams& p, int64_t u) {
    return ((u + 1) * p.sk_clusters + p.sk_units - 1) / p.sk_units - 1;
}

__device__ __forceinline__ void work_begin(const KParams& p, int64_t cluster, int64_t nclusters, WorkIter& it) {
    it.dp = cluster;
    it.dp_stride = nclusters;
    it.self = cluster;
    if (p.sk_clusters > 0) {
        it.u = sk_bound(p, cluster);
        it.u1 = sk_bound(p, cluster + 1);
    } else {
        it.u = it.u1 = 0;
    }
}

__device__ __forceinline__ bool work_next(const KParams& p, WorkIter& it, WorkItem& w) {
    if (it.dp < p.dp_tiles) {
        w.tile = it.dp;
        w.kb0 = 0;
        w.kb1 = p.num_k;
        w.role = ROLE_WHOLE;
        w.sk_tile = -1;
        w.last_slot = -1;
        it.dp += it.dp_stride;
        return true;
    }
    if (it.u < it.u1) {
        const int64_t j = it.u / p.num_k;
        const int32_t kb0 = (int32_t)(it.u - j * p.num_k);
        const int32_t kb1 = (int32_t)min((int64_t)p.num_k, kb0 + (it.u1 - it.u));
        w.tile = p.dp_tiles + j;
        w.kb0 = kb0;
        w.kb1 = kb1;
        w.sk_tile = (int32_t)j;
        w.last_slot = -1;
        if (kb0 != 0) {
            w.role = ROLE_PARTIAL;
        } else if (kb1 == p.num_k) {
            w.role = ROLE_WHOLE;
        } else {
            w.role = ROLE_OWNER;
            w.last_slot = (int32_t)sk_cluster_of(p, (j + 1) * p.num_k - 1);
        }
        it.u += kb1 - kb0;
        return true;
    }
    return false;
}

__device__ __forceinline__ int32_t ld_acquire_gpu(const int32_t* ptr) {
    int32_t v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

template <int OUT>
__device__ __forceinline__ uint32_t pack2(uint32_t lo, uint32_t hi) {
    const float a = __uint_as_float(lo), b = __uint_as_float(hi);
    if (OUT == OUT_BF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);   // .x (low half) = a
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}

// Stream-K partials.  A warp's partial of one accumulator region (its 32
// rows, BN fp32 columns) is BN / 32 blocks of 4 KiB, one per 32-column chunk,
// each laid out like an fp32 epilogue slab: row r (the warp's lane r) is 128
// bytes and its 16-byte piece j sits at piece j ^ (r % 8).  Written from and
// read into shared memory with 16-byte accesses, every 8 lanes of an access
// phase hit 8 different bank groups; between shared and global memory the
// blocks move as plain bulk copies.

// Writes the warp's partial of one region (tensor memory `tmem_acc`) to `dst`
// through its staging slabs; `release` is called once the region has been
// read.  With `announce` the warp then waits for its copies to land and adds
// 1 to `flag`.
template <typename Release>
__device__ __forceinline__ void epilogue_partial(const KParams& p, uint32_t tmem_acc, uint32_t lane_field, int lane,
                                                 uint32_t slabs, uint32_t& sbuf, float* dst, int32_t* flag,
                                                 bool announce, Release release) {
    const uint32_t row = (uint32_t)lane * 128u;
    for (int c = 0; c < p.BN / 32; ++c) {
        const uint32_t slab = slabs + sbuf * kEpiSlabBytes;
        if (lane == 0) bulk_wait_read<1>();        // this slab's previous copy has read it
        __syncwarp();
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_acc + lane_field + (uint32_t)(c * 32), v);
        tmem_ld_wait();
        if (c == p.BN / 32 - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release();
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
            st_shared_v4(slab + row + ((uint32_t)(j ^ (lane & 7)) << 4), v[4 * j], v[4 * j + 1], v[4 * j + 2],
                         v[4 * j + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            bulk_store(dst + (int64_t)c * 32 * 32, slab, kEpiSlabBytes);
            bulk_commit();
        }
        sbuf ^= 1u;
    }
    if (!announce) return;
    if (lane == 0) {
        bulk_wait<0>();             // every copy of this warp has landed
        fence_proxy_async_all();    // ... and comes before the generic release below
        __threadfence();
        atomicAdd(flag, 1);
    }
    __syncwarp();
}

// Stream-K fix-up of one epilogue warp: adds the partials of the slots set in
// `mask` to its 32 accumulator rows of regions 0 .. nreg-1 (256 tensor memory
// columns apart), slot by slot in increasing order -- a fixed order, so the
// sum does not depend on timing.  The partials arrive in blocks of kFixChunks
// chunks, copied by bulk loads into the warp's kFixBufs buffers kFixBufs
// blocks ahead of the additions; every warp streams only its own rows.
//   parts        : the warp's partial of region 0 in slot 0
//   slot_stride  : floats from one slot to the next; region_stride likewise
//   bufs, bars   : the warp's first buffer and first mbarrier (count 1)
// The buffers lie in the operand ring: the owner's piece is the last piece of
// its cluster's range, so once its accumulator is full no load or MMA touches
// the ring again.  Returns false if a copy did not land within the budget
// (the copies still in flight are then waited for, again with the budget).
__device__ __forceinline__ bool sk_fixup(uint32_t tmem_acc, uint32_t lane_field, int lane, int BN, int nreg,
                                        const float* parts, int64_t slot_stride, int64_t region_stride,
                                        uint32_t mask, uint32_t bufs, uint32_t bars, int64_t budget) {
    const int nh = BN / (32 * kFixChunks);          // blocks per region and slot
    const int ns = __popc(mask);
    const int nb = nreg * ns * nh;
    // block b: part h, k-th slot of the mask, region i (region-major order)
    auto src_of = [&](int b) {
        const int h = b % nh, t = b / nh, k = t % ns, i = t / ns;
        uint32_t m = mask;
        for (int j = 0; j < k; ++j) m &= m - 1;
        return parts + (int64_t)(__ffs(m) - 1) * slot_stride + (int64_t)i * region_stride +
               (int64_t)h * (kFixChunks * 32 * 32);
    };
    if (lane == 0) {
        fence_proxy_async_all();    // the partials were acquired through the generic proxy
        for (int b = 0; b < nb && b < kFixBufs; ++b) {
            mbar_arrive_expect_tx(bars + 8u * b, kFixBlockBytes);
            bulk_load(bufs + b * kFixBlockBytes, src_of(b), kFixBlockBytes, bars + 8u * b);
        }
    }
    const uint32_t row = (uint32_t)lane * 128u;
    for (int b = 0; b < nb; ++b) {
        const int j = b % kFixBufs;
        const uint32_t buf = bufs + j * kFixBlockBytes;
        if (!__all_sync(0xffffffffu, mbar_wait(bars + 8u * j, (uint32_t)(b / kFixBufs) & 1u, budget))) {
            if (lane == 0)
                for (int r = b + 1; r < nb && r < b + kFixBufs; ++r)
                    (void)mbar_wait(bars + 8u * (r % kFixBufs), (uint32_t)(r / kFixBufs) & 1u, budget);
            return false;
        }
        const int h = b % nh, i = (b / nh) / ns;
        const uint32_t col0 = (uint32_t)(i * 256 + h * kFixChunks * 32);
#pragma unroll 1
        for (int cc = 0; cc < kFixChunks; cc += 2) {
            const uint32_t taddr = tmem_acc + lane_field + col0 + (uint32_t)(cc * 32);
            uint32_t v0[32], v1[32];
            tmem_ld_32x32b_x32(taddr, v0);
            tmem_ld_32x32b_x32(taddr + 32, v1);
            tmem_ld_wait();
            const uint32_t s0 = buf + (uint32_t)cc * kEpiSlabBytes + row, s1 = s0 + kEpiSlabBytes;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const uint32_t piece = (uint32_t)(q ^ (lane & 7)) << 4;
                const uint4 a = ld_shared_v4(s0 + piece), c = ld_shared_v4(s1 + piece);
                v0[4 * q] = __float_as_uint(__uint_as_float(v0[4 * q]) + __uint_as_float(a.x));
                v0[4 * q + 1] = __float_as_uint(__uint_as_float(v0[4 * q + 1]) + __uint_as_float(a.y));
                v0[4 * q + 2] = __float_as_uint(__uint_as_float(v0[4 * q + 2]) + __uint_as_float(a.z));
                v0[4 * q + 3] = __float_as_uint(__uint_as_float(v0[4 * q + 3]) + __uint_as_float(a.w));
                v1[4 * q] = __float_as_uint(__uint_as_float(v1[4 * q]) + __uint_as_float(c.x));
                v1[4 * q + 1] = __float_as_uint(__uint_as_float(v1[4 * q + 1]) + __uint_as_float(c.y));
                v1[4 * q + 2] = __float_as_uint(__uint_as_float(v1[4 * q + 2]) + __uint_as_float(c.z));
                v1[4 * q + 3] = __float_as_uint(__uint_as_float(v1[4 * q + 3]) + __uint_as_float(c.w));
            }
            tmem_st_32x32b_x32(taddr, v0);
            tmem_st_32x32b_x32(taddr + 32, v1);
        }
        tmem_st_wait();
        __syncwarp();
        if (lane == 0 && b + kFixBufs < nb) {
            fence_proxy_async_smem();   // the lanes' reads of this buffer come before the next copy
            mbar_arrive_expect_tx(bars + 8u * j, kFixBlockBytes);
            bulk_load(buf, src_of(b + kFixBufs), kFixBlockBytes, bars + 8u * j);
        }
    }
    return true;
}

// One 128-byte column chunk of the epilogue, step 1: read the warp's 32 rows
// of it from tensor memory (fp32 output: 32 columns; 16-bit output: 64
// columns, packed in pairs).
template <int OUT>
__device__ __forceinline__ void epi_load_chunk(uint32_t tmem_acc, uint32_t lane_field, int c, uint32_t (&v)[32]) {
    constexpr int kChunkCols = (OUT == OUT_F32) ? 32 : 64;
    const uint32_t col = (uint32_t)(c * kChunkCols);
    if (OUT == OUT_F32) {
        tmem_ld_32x32b_x32(tmem_acc + lane_field + col, v);
        tmem_ld_wait();
    } else {
        uint32_t r0[32], r1[32];
        tmem_ld_32x32b_x32(tmem_acc + lane_field + col, r0);
        tmem_ld_32x32b_x32(tmem_acc + lane_field + col + 32, r1);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            v[i] = pack2<OUT>(r0[2 * i], r0[2 * i + 1]);
            v[16 + i] = pack2<OUT>(r1[2 * i], r1[2 * i + 1]);
        }
    }
}

// Step 1 for 16-bit output with fewer registers: the chunk's two 32-column
// halves are read and packed one after the other (32 raw values live at a
// time instead of 64), for a warp that holds a whole accumulator in
// registers.
template <int OUT>
__device__ __forceinline__ void epi_load_chunk_halves(uint32_t tmem_acc, uint32_t lane_field, int c,
                                                      uint32_t (&v)[32]) {
    static_assert(OUT != OUT_F32, "16-bit output");
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem_acc + lane_field + (uint32_t)(c * 64 + h * 32), r);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i) v[16 * h + i] = pack2<OUT>(r[2 * i], r[2 * i + 1]);
    }
}

// Step 2: stage the chunk in this warp's swizzled slab and store it with TMA
// (the ragged < 16-byte end of a row is copied from the slab directly).  The
// caller has made sure the slab's previous store has finished reading it.
template <int OUT>
__device__ __forceinline__ void epi_store_chunk(const KParams& p, const CUtensorMap* tmC, uint32_t slab, int lane,
                                                int32_t m0, int32_t nc, int b, const uint32_t (&v)[32]) {
    constexpr int kOutBytes = (OUT == OUT_F32) ? 4 : 2;
    constexpr int kChunkCols = 128 / kOutBytes;
    // Row `lane` of the slab; 16-byte chunk j goes to j ^ (row % 8): the 8
    // lanes of each store phase hit 8 different bank groups.
    const uint32_t row = slab + (uint32_t)lane * 128u;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        st_shared_v4(row + ((uint32_t)(j ^ (lane & 7)) << 4), v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
        if (m0 < p.M && nc < p.n_tma) tma_store_3d(tmC, slab, nc, m0, b);
        bulk_commit();
    }
    if (nc + kChunkCols > p.n_tma && nc < p.N) {
        // TMA stores write whole 16-byte pieces at the row end; the last
        // < 16 bytes of a ragged row are copied from this lane's own row of
        // the swizzled slab (its own st.shared above are visible to it).
        const int32_t m = m0 + lane;
        if (m < p.M) {
            char* rowp = static_cast<char*>(p.C) + ((int64_t)b * p.strideC + (int64_t)m * p.ldc) * kOutBytes;
            const int32_t n_lo = max(p.n_tma, nc), n_hi = min(p.N, nc + kChunkCols);
#pragma unroll 1
            for (int32_t n = n_lo; n < n_hi; ++n) {
                const uint32_t byte = (uint32_t)(n - nc) * kOutBytes;
                const uint32_t src = row + ((((byte >> 4) ^ (uint32_t)(lane & 7)) << 4) | (byte & 15u));
                if (OUT == OUT_F32)
                    *reinterpret_cast<uint32_t*>(rowp + (int64_t)n * 4) = ld_shared_u32(src);
                else
                    *reinterpret_cast<uint16_t*>(rowp + (int64_t)n * 2) = ld_shared_u16(src);
            }
        }
    }
}

// A chunk of which only the first `cols` columns belong to the tile (the last
// chunk of a tile whose width is not a whole number of 128-byte chunks): a
// TMA store of the whole chunk would write into the next tile, so each lane
// stores its own row's columns from registers, 16 bytes at a time (the
// chunk starts 16-byte aligned: tile widths are multiples of 16 columns),
// element by element past the matrix's last column N.
template <int OUT>
__device__ __forceinline__ void epi_store_partial(const KParams& p, int lane, int32_t m0, int32_t nc, int cols,
                                                  int b, const uint32_t (&v)[32]) {
    constexpr int kOutBytes = (OUT == OUT_F32) ? 4 : 2;
    constexpr int kPer16 = 16 / kOutBytes;
    const int32_t m = m0 + lane;
    if (m >= p.M) return;
    char* rowp = static_cast<char*>(p.C) + ((int64_t)b * p.strideC + (int64_t)m * p.ldc) * kOutBytes;
    const int32_t n_hi = min(p.N, nc + cols);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
        const int32_t n = nc + q * kPer16;
        if (n + kPer16 <= n_hi) {
            asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(rowp + (int64_t)n * kOutBytes),
                         "r"(v[4 * q]), "r"(v[4 * q + 1]), "r"(v[4 * q + 2]), "r"(v[4 * q + 3])
                         : "memory");
        } else if (n < n_hi) {
            // static register indices only (a runtime index would move v to local memory)
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                const uint32_t word = v[4 * q + w];
                if (OUT == OUT_F32) {
                    const int32_t e = n + w;
                    if (e < n_hi) *reinterpret_cast<uint32_t*>(rowp + (int64_t)e * 4) = word;
                } else {
                    const int32_t e = n + 2 * w;
                    if (e < n_hi) *reinterpret_cast<uint16_t*>(rowp + (int64_t)e * 2) = (uint16_t)(word & 0xFFFFu);
                    if (e + 1 < n_hi) *reinterpret_cast<uint16_t*>(rowp + (int64_t)(e + 1) * 2) = (uint16_t)(word >> 16);
                }
            }
        }
    }
}

// Epilogue of one accumulator tile for one warp: its 32 rows (TMEM lanes
// 32*(warp % 4) ...), all p.epi_chunks column chunks of 128 bytes (the last
// one partial when the tile width is not a whole number of chunks).
//   tmem_acc : tensor-memory address of the accumulator (lane field 0)
//   slabs    : this warp's first staging slab (kEpiBufs slabs of kEpiSlabBytes)
//   m0, n0   : first output row of the warp and first column of the tile
// `release` is called once every accumulator column has been read, so the MMA
// issuer may overwrite the accumulator while the stores drain.
template <int OUT, typename Release>
__device__ __forceinline__ void epilogue_tile(const KParams& p, const CUtensorMap* tmC, uint32_t tmem_acc,
                                              uint32_t lane_field, uint32_t slabs, uint32_t& sbuf, int lane,
                                              int32_t m0, int32_t n0, int b, Release release,
                                              int chunks, int last_cols) {
    constexpr int kChunkCols = (OUT == OUT_F32) ? 32 : 64;
    for (int c = 0; c < chunks; ++c) {
        const bool last = c == chunks - 1;
        const bool partial = last && last_cols < kChunkCols;
        const uint32_t slab = slabs + sbuf * kEpiSlabBytes;
        if (!partial) {
            if (lane == 0) bulk_wait_read<1>();    // this slab's previous store has read it
            __syncwarp();
        }
        uint32_t v[32];
        epi_load_chunk<OUT>(tmem_acc, lane_field, c, v);
        if (last) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release();
        }
        if (partial) {
            epi_store_partial<OUT>(p, lane, m0, n0 + c * kChunkCols, last_cols, b, v);
        } else {
            epi_store_chunk<OUT>(p, tmC, slab, lane, m0, n0 + c * kChunkCols, b, v);
            sbuf ^= 1u;
        }
    }
}

// The tile of the launch's main width (p.epi_chunks chunks, the last one
// holding p.epi_last_cols columns).
template <int OUT, typename Release>
__device__ __forceinline__ void epilogue_tile(const KParams& p, const CUtensorMap* tmC, uint32_t tmem_acc,
                                              uint32_t lane_field, uint32_t slabs, uint32_t& sbuf, int lane,
                                              int32_t m0, int32_t n0, int b, Release release) {
    epilogue_tile<OUT>(p, tmC, tmem_acc, lane_field, slabs, sbuf, lane, m0, n0, b, release, p.epi_chunks,
                       p.epi_last_cols);
}

// Epilogue of one warp of a 256 x 256 CTA-pair tile with 16-bit output (four
// whole 64-column chunks): the warp reads all four chunks into registers
// (128 per thread, packed), hands the accumulator back -- the MMA issuer
// starts the tile after next at once -- and then stores chunk j no earlier
// than j x pace_ns after the hand-back, so that the tile's C leaves the SM
// spread over the next tile's main loop instead of in one burst against its
// operand loads (pace_ns = 0: back to back).  The waits are bounded by
// 3 x pace_ns.
template <int OUT, typename Release>
__device__ __forceinline__ void epilogue_tile_paced(const KParams& p, const CUtensorMap* tmC, uint32_t acc,
                                                    uint32_t lane_field, uint32_t slabs, uint32_t& sbuf, int lane,
                                                    int32_t m0, int32_t n0, int b, int64_t pace_ns,
                                                    Release release) {
    static_assert(OUT != OUT_F32, "16-bit output");
    uint32_t v[4][32];
#pragma unroll
    for (int j = 0; j < 4; ++j) epi_load_chunk_halves<OUT>(acc, lane_field, j, v[j]);
    tc_fence_before();
    __syncwarp();
    if (lane == 0) release();
    const uint64_t t0 = globaltimer();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        if (j > 0 && pace_ns > 0 && lane == 0) {
            const uint64_t until = t0 + (uint64_t)j * (uint64_t)pace_ns;
            while (globaltimer() < until) __nanosleep(128);
        }
        if (lane == 0) bulk_wait_read<1>();         // the slab's previous store has read it
        __syncwarp();
        epi_store_chunk<OUT>(p, tmC, slabs + sbuf * kEpiSlabBytes, lane, m0, n0 + j * 64, b, v[j]);
        sbuf ^= 1u;
    }
}

// One of eight epilogue warps of a one-CTA tile: tensor-memory lane quarter
// `lane_field`, chunks [c0, c0 + nc) of the tile's `chunks` (the last one
// holding `last_cols` columns), staged through the warp's one slab.  With at
// most two chunks the warp reads both into registers and hands the
// accumulator back before it stores them; with more it goes chunk by chunk
// and hands back after its last tensor-memory read.
template <int OUT, typename Release>
__device__ __forceinline__ void epilogue_tile_part(const KParams& p, const CUtensorMap* tmC, uint32_t tmem_acc,
                                                   uint32_t lane_field, uint32_t slab, int lane, int32_t m0,
                                                   int32_t n0, int b, int c0, int nc, int chunks, int last_cols,
                                                   Release release) {
    constexpr int kChunkCols = (OUT == OUT_F32) ? 32 : 64;
    if (nc <= 0) {                                  // a narrow tile may leave this warp nothing
        __syncwarp();
        if (lane == 0) release();
        return;
    }
    if (nc <= 2) {
        uint32_t v[2][32];
#pragma unroll
        for (int j = 0; j < 2; ++j)
            if (j < nc) epi_load_chunk<OUT>(tmem_acc, lane_field, c0 + j, v[j]);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) release();
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            if (j < nc) {
                const int c = c0 + j;
                if (c == chunks - 1 && last_cols < kChunkCols) {
                    epi_store_partial<OUT>(p, lane, m0, n0 + c * kChunkCols, last_cols, b, v[j]);
                } else {
                    if (lane == 0) bulk_wait_read<0>();   // the slab's previous store has read it
                    __syncwarp();
                    epi_store_chunk<OUT>(p, tmC, slab, lane, m0, n0 + c * kChunkCols, b, v[j]);
                }
            }
        }
        return;
    }
    for (int j = 0; j < nc; ++j) {
        const int c = c0 + j;
        const bool partial = c == chunks - 1 && last_cols < kChunkCols;
        if (!partial) {
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
        }
        uint32_t v[32];
        epi_load_chunk<OUT>(tmem_acc, lane_field, c, v);
        if (j == nc - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release();
        }
        if (partial)
            epi_store_partial<OUT>(p, lane, m0, n0 + c * kChunkCols, last_cols, b, v);
        else
            epi_store_chunk<OUT>(p, tmC, slab, lane, m0, n0 + c * kChunkCols, b, v);
    }
}

// Split-K epilogue of one warp (fp32 output; one tile per 2-CTA cluster, the
// two CTAs holding the partial sums of the two halves of K).  The tile's
// column chunks are shared out: CTA rank 0 owns chunks [0, h), rank 1 chunks
// [h, epi_chunks), h = epi_chunks / 2.  Each CTA
//   1. stores its own chunks' partial plainly (slab + TMA store);
//   2. stages its partial of the peer's chunks in the idle operand ring;
//   3. once its plain stores are complete, arrives (release, cluster scope)
//      on the peer's `peer_bar`, every lane for its own direct stores;
//   4. waits (acquire, cluster scope) until the peer's plain stores of those
//      chunks are complete and adds its staged partial to them with TMA
//      reduce-adds (fp32, rounded to nearest; ragged row tails by atomic
//      adds).
// Every output is then fl(p0 + p1) of the two partials: one rounding of two
// addends, independent of which add came first, so the result is
// deterministic.  `stage`: this warp's staging slots (up to 4 chunks of
// kEpiSlabBytes).  Returns false if the wait for the peer ran out.
template <typename Release>
__device__ __forceinline__ bool epilogue_split_tile(const KParams& p, const CUtensorMap* tmC, uint32_t tmem_acc,
                                                    uint32_t lane_field, uint32_t slabs, uint32_t& sbuf, int lane,
                                                    int32_t m0, int32_t n0, int b, uint32_t rank, uint32_t stage,
                                                    uint32_t peer_bar, uint32_t own_bar, int64_t budget,
                                                    Release release) {
    constexpr int kChunkCols = 32;                  // fp32: 32 columns per 128-byte chunk
    const int h = p.epi_chunks / 2;
    const int own0 = rank ? h : 0, own1 = rank ? p.epi_chunks : h;
    const int oth0 = rank ? 0 : h, oth1 = rank ? h : p.epi_chunks;
    for (int c = own0; c < own1; ++c) {
        const uint32_t slab = slabs + sbuf * kEpiSlabBytes;
        if (lane == 0) bulk_wait_read<1>();         // this slab's previous store has read it
        __syncwarp();
        uint32_t v[32];
        epi_load_chunk<OUT_F32>(tmem_acc, lane_field, c, v);
        epi_store_chunk<OUT_F32>(p, tmC, slab, lane, m0, n0 + c * kChunkCols, b, v);
        sbuf ^= 1u;
    }
    const uint32_t row = (uint32_t)lane * 128u;
    for (int c = oth0; c < oth1; ++c) {
        uint32_t v[32];
        epi_load_chunk<OUT_F32>(tmem_acc, lane_field, c, v);
        const uint32_t slot = stage + (uint32_t)(c - oth0) * kEpiSlabBytes + row;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            st_shared_v4(slot + ((uint32_t)(j ^ (lane & 7)) << 4), v[4 * j], v[4 * j + 1], v[4 * j + 2],
                         v[4 * j + 3]);
    }
    tc_fence_before();
    fence_proxy_async_smem();                       // staged partials visible to the TMA reduce
    __syncwarp();
    if (lane == 0) {
        release();                                  // every accumulator column has been read
        bulk_wait<0>();                             // own TMA stores complete
        fence_proxy_async_all();
    }
    __syncwarp();
    mbar_arrive_cluster(peer_bar);
    const bool ok = __all_sync(0xffffffffu, mbar_wait_cluster(own_bar, 0, budget));
    if (!ok) return false;
    fence_proxy_async_all();                        // the peer's stores, acquired, before our reduces
    if (lane == 0) {
        for (int c = oth0; c < oth1; ++c) {
            const int32_t nc = n0 + c * kChunkCols;
            if (m0 < p.M && nc < p.n_tma)
                tma_reduce_add_3d(tmC, stage + (uint32_t)(c - oth0) * kEpiSlabBytes, nc, m0, b);
        }
        bulk_commit();
    }
    const int32_t m = m0 + lane;
    for (int c = oth0; c < oth1; ++c) {
        const int32_t nc = n0 + c * kChunkCols;
        if (nc + kChunkCols > p.n_tma && nc < p.N && m < p.M) {
            // the ragged < 16-byte end of a row: not covered by the tensor map
            float* rowp = static_cast<float*>(p.C) + (int64_t)b * p.strideC + (int64_t)m * p.ldc;
            const uint32_t slot = stage + (uint32_t)(c - oth0) * kEpiSlabBytes + row;
            const int32_t n_lo = max(p.n_tma, nc), n_hi = min(p.N, nc + kChunkCols);
#pragma unroll 1
            for (int32_t n = n_lo; n < n_hi; ++n) {
                const uint32_t byte = (uint32_t)(n - nc) * 4u;
                atomicAdd(rowp + n,
                          __uint_as_float(ld_shared_u32(slot + ((((byte >> 4) ^ (uint32_t)(lane & 7)) << 4) |
                                                                (byte & 15u)))));
            }
        }
    }
    return true;
}

// Epilogue of a wide tile (two 128-row accumulator regions per CTA) for one
// of its 8 warps: TMEM lane quarter `lane_field`, chunks [c0, c0 + nc) of
// each region (its half of the tile's columns).
//   16-bit output: the warp reads its (at most 2 + 2) chunks of both regions
//     from tensor memory into registers (128 per thread, packed), hands the
//     accumulator back -- the MMA issuer starts the next tile at once -- and
//     then stores the chunks through its slab while the next tile's MMAs run.
//   fp32 output (twice the registers): chunk by chunk, the accumulator handed
//     back after the warp's last tensor-memory read.
// A partial last chunk (tile width not a multiple of the chunk) is stored
// directly.  mrow: the warp's first row in region 0 (region 1 is 128 below).
template <int OUT, typename Release>
__device__ __forceinline__ void epilogue_wide_warp(const KParams& p, const CUtensorMap* tmC, uint32_t acc,
                                                   uint32_t lane_field, uint32_t slab, int lane, int32_t mrow,
                                                   int32_t n0, int b, int c0, int nc, int chunks, int last_cols,
                                                   Release release) {
    constexpr int kChunkCols = (OUT == OUT_F32) ? 32 : 64;
    if (nc <= 0) {                                  // a narrow tile may leave this warp nothing
        __syncwarp();
        if (lane == 0) release();
        return;
    }
    if constexpr (OUT != OUT_F32) {
        if (last_cols == kChunkCols) {
            // whole chunks: everything into registers, hand back, then store
            uint32_t v[2][2][32];
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int j = 0; j < 2; ++j)
                    if (j < nc) epi_load_chunk_halves<OUT>(acc + (uint32_t)(r * 256), lane_field, c0 + j, v[r][j]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) release();
#pragma unroll
            for (int r = 0; r < 2; ++r) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    if (j < nc) {
                        if (lane == 0) bulk_wait_read<0>();   // the slab's previous store has read it
                        __syncwarp();
                        epi_store_chunk<OUT>(p, tmC, slab, lane, mrow + r * kBM, n0 + (c0 + j) * kChunkCols, b,
                                             v[r][j]);
                    }
                }
            }
            return;
        }
    }
    // fp32 output (twice the registers), or a partial last chunk (the tail
    // of a wide tiling): chunk by chunk, the accumulator handed back after the
    // warp's last tensor-memory read.
    for (int r = 0; r < 2; ++r) {
        for (int j = 0; j < nc; ++j) {
            const int c = c0 + j;
            const int32_t m0 = mrow + r * kBM;
            const bool partial = c == chunks - 1 && last_cols < kChunkCols;
            if (!partial) {
                if (lane == 0) bulk_wait_read<0>();
                __syncwarp();
            }
            uint32_t v[32];
            epi_load_chunk<OUT>(acc + (uint32_t)(r * 256), lane_field, c, v);
            if (r == 1 && j == nc - 1) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) release();
            }
            if (partial)
                epi_store_partial<OUT>(p, lane, m0, n0 + c * kChunkCols, last_cols, b, v);
            else
                epi_store_chunk<OUT>(p, tmC, slab, lane, m0, n0 + c * kChunkCols, b, v);
        }
    }
}

}  // namespace smo
