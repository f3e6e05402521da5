// CTA-pair variant of the persistent GEMM for sm_103a: output tiles computed
// by two CTAs of a cluster with tcgen05.mma.cta_group::2 (256 x 256 x K_mma
// per instruction).
//
// Each CTA of the pair holds its own rows of A and its own 128 columns of B
// per pipeline stage; the even CTA's single MMA thread issues MMAs that read
// both CTAs' shared memory and accumulate the even CTA's rows in its tensor
// memory and the odd CTA's rows in the odd CTA's.  Compared with one CTA per
// 128 x 256 tile this halves the B bytes each SM stages per flop and doubles
// the pipeline depth for the same shared memory ("An Educational GEMM Ladder
// for Helios GPUs", Level 4: larger output tiles raise arithmetic intensity;
// Level 9: a cluster of workgroups shares operand panels instead of
// re-requesting them).  Two tile shapes (template parameter WIDE):
//   256 x 256: 128 A rows per CTA, 6 stages of 32 KiB handed over two at a
//              time (one full/empty barrier pair, one wait and one commit per
//              8 MMAs: the single issuing thread, not the tensor pipe, set the
//              pace with a wait and a commit per 4), two accumulators;
//   512 x 256: 256 A rows per CTA in two 128-row halves with their own MMAs,
//              4 stages of 48 KiB, one accumulator of 512 columns, 8
//              epilogue warps (320 threads) that read the whole accumulator
//              into registers and hand it back before storing.
//
// Synchronisation across the pair:
//   full[g]    (even CTA only) -- both CTAs' TMA loads of the group complete
//                                 on it (cp.async.bulk.tensor ... .cta_group::2);
//                                 the even producer arms it for both CTAs' bytes
//   empty[g]   (both)          -- the MMA thread's commit multicasts to both
//   acc_full   (both)          -- likewise, after the last K block of a tile
//   acc_empty  (even CTA only) -- the epilogue warps of each CTA arrive (4, or 8
//                                 for wide tiles)
// Every wait is bounded; cluster barriers at start (barriers initialised,
// tensor memory allocated) and end (no CTA leaves while its peer may still
// signal it).
#pragma once
#include <cuda.h>
#include <stdint.h>

#include "gemm_common.cuh"

namespace smo {

static_assert(kStageKBytes / kMmaKBytes == 4, "the issue loop unrolls four MMAs per K block");
constexpr int kPairGroup = 2;       // stages per full/empty barrier pair (the ring holds 6)
constexpr uint32_t kHalfABytes = kBM * kStageKBytes;   // 128 A rows of one stage, every layout

// KIND: MmaKind (kind::f16 for 16-bit operands, kind::f8f6f4 for FP8).
// WIDE: 0 -- 256 x 256 tiles, 128 A rows per CTA, two accumulators, stages
//            handed over in groups of two (6 x 32 KiB);
//       1 -- 512 x BN tiles (BN <= 256), 256 A rows per CTA (two 128-row
//            halves, each with its own 256 x BN MMAs into TMEM columns
//            0..BN-1 / 256..256+BN-1), one accumulator, one stage per barrier
//            pair (4 x 48 KiB).  The B half-panel of a stage then feeds twice
//            the MMAs: 47 instead of 64 operand bytes per tensor cycle, so the
//            same ring keeps more MMA work in flight.  8 epilogue warps hand
//            the single accumulator back as soon as it sits in registers
//            (16-bit output); no stream-K.
template <int OUT, int KIND, int WIDE>
__global__ void __launch_bounds__(WIDE ? kWideThreads : kThreads, 1)
    smo_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                         const __grid_constant__ CUtensorMap tmC, const __grid_constant__ KParams p) {
    constexpr int KG = WIDE ? 1 : kPairGroup;      // stages per full/empty barrier pair
    constexpr int EPIW = WIDE ? kWideEpiWarps : kEpiWarps;   // epilogue warps per CTA
    constexpr int MSUB = WIDE ? 2 : 1;             // 128-row A halves (and accumulator regions) per CTA
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank() & 1u;      // 0: even CTA of the pair, issues the MMAs
    const uint32_t lead = cluster_ctarank() & ~1u;     // cluster rank of the even CTA

    const uint32_t bars = base + p.off_bar;
    auto full_bar = [&](uint32_t s) { return bars + 8u * s; };
    auto empty_bar = [&](uint32_t s) { return bars + 8u * (kMaxStages + s); };
    auto accf_bar = [&](uint32_t b) { return bars + 8u * (2 * kMaxStages + b); };
    auto acce_bar = [&](uint32_t b) { return bars + 8u * (2 * kMaxStages + 2 + b); };
    const uint32_t drain_bar = bars + 8u * (2 * kMaxStages + 4);
    const uint32_t tmem_slot = bars + 8u * (2 * kMaxStages + 5);
    auto fix_bar = [&](uint32_t j) { return bars + 8u * (2 * kMaxStages + 6 + j); };   // kEpiWarps x kFixBufs

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), 2 * EPIW);
        }
        mbar_init(drain_bar, 1);
        for (int j = 0; j < kEpiWarps * kFixBufs; ++j) mbar_init(fix_bar(j), 1);
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, p.tmem_cols);       // one warp of each CTA, same columns in both
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    // The prologue above touches only shared memory, tensor memory and the
    // kernel parameters, so it may overlap the previous kernel in the stream
    // (launched with programmatic stream serialization); every global memory
    // access comes after this wait.
    griddep_wait();
    griddep_launch_dependents();
    const uint32_t tmem_base = ld_shared_u32(tmem_slot);
    const int64_t budget = p.timeout_ns;
    const int64_t cluster_id = blockIdx.x >> 1;
    const int64_t nclusters = gridDim.x >> 1;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        // Lanes 0 .. nloads-1 each own one load of every stage and issue them
        // together; lane 0 waits for the free slot and (even CTA) arms the
        // stage for both CTAs' bytes.
        const uint32_t nloads = stage_loads(p);
        if ((uint32_t)lane < nloads) {
            const uint32_t lmask = (1u << nloads) - 1u;
            const LoadSlot slot = load_slot(p, &tmA, &tmB, (uint32_t)lane);
            const uint32_t ngroups = (uint32_t)(p.stages / KG);
            const uint32_t group_bytes = KG * p.stage_stride;
            uint32_t g = 0, ph = 0, gst = base;           // group index, ring parity, group's smem
            uint32_t issued_mask = 0, issued_ph = 0;
            bool skip_one = p.stall != 0;
            bool ok = true;
            WorkIter wi;
            WorkItem w;
            work_begin(p, cluster_id, nclusters, wi);
            for (uint32_t tix = 0; ok && work_next(p, wi, w); ++tix) {
                int b, mb;
                int32_t n0, tbn;
                decode_tile_w(p, w.tile, b, mb, n0, tbn);
                // this CTA's A rows / B columns
                const int32_t mn0 = slot.is_a ? mb * (2 * MSUB * kBM) + (int32_t)rank * (MSUB * kBM)
                                              : n0 + (int32_t)rank * (tbn / 2);
                // Wide tiles (one stage per barrier pair): every other tile of
                // this cluster loads its K blocks last to first.  A wave then
                // begins on the K slices of A the previous wave read last,
                // which are the ones still in L2.  The MMAs consume the
                // stages in ring order either way (only the summation order
                // changes).
                const bool rev = KG == 1 && p.serp && (tix & 1u);
                for (int kb = w.kb0; kb < w.kb1; kb += KG) {
                    const int kload = rev ? w.kb0 + w.kb1 - 1 - kb : kb;
                    const bool two = KG == 2 && kb + 1 < w.kb1;   // a range's last group may hold one block
                    int good = 1;
                    if (lane == 0) good = mbar_wait(empty_bar(g), ph ^ 1u, budget) ? 1 : 0;
                    good = __shfl_sync(lmask, good, 0);
                    if (!good) {
                        if (lane == 0) report_error(p.err, DEV_TIMEOUT_PRODUCER);
                        ok = false;
                        break;
                    }
                    if (skip_one) {
                        skip_one = false;          // test hook: this group never fills
                    } else {
                        const uint32_t fb = mapa_shared(full_bar(g), lead);
                        if (rank == 0 && lane == 0) {
                            mbar_arrive_expect_tx(full_bar(g), two ? 2 * p.tx_bytes : p.tx_bytes);   // both CTAs
                            issued_mask |= 1u << g;
                            issued_ph = (issued_ph & ~(1u << g)) | (ph << g);
                        }
                        __syncwarp(lmask);
                        int32_t c0, c1, c2;
                        slot_coords(slot, mn0, kload * p.bk, c0, c1, c2);
                        tma_load_4d_pair(gst + slot.dst_off, slot.tm, fb, c0, c1, c2, b);
                        if (two) {
                            slot_coords(slot, mn0, (kb + 1) * p.bk, c0, c1, c2);
                            tma_load_4d_pair(gst + p.stage_stride + slot.dst_off, slot.tm, fb, c0, c1, c2, b);
                        }
                    }
                    if (++g == ngroups) {
                        g = 0;
                        ph ^= 1u;
                        gst = base;
                    } else {
                        gst += group_bytes;
                    }
                }
            }
            if (lane == 0 && rank == 0) {
                // Every armed group has received both CTAs' bytes (immediate when
                // the MMA thread already consumed it).
                for (uint32_t q = 0; q < (uint32_t)(p.stages / KG); ++q) {
                    if ((issued_mask >> q) & 1u) {
                        if (!mbar_wait(full_bar(q), (issued_ph >> q) & 1u, budget))
                            report_error(p.err, DEV_TIMEOUT_TEARDOWN);
                    }
                }
            } else if (lane == 0 && !ok) {
                // The odd CTA cannot observe the even CTA's barrier: after a
                // timeout give its own loads in flight a bounded time to land.
                const uint64_t t0 = globaltimer();
                while (globaltimer() - t0 < 2000000ull) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer (even CTA)
        if (lane == 0 && rank == 0) {
            // Everything the issue loop needs sits in registers: the single
            // issuing thread, not the tensor pipe, is the limit when each K
            // block's MMAs wait behind parameter loads and address arithmetic.
            const uint32_t ngroups = (uint32_t)(p.stages / KG);
            const uint64_t stage_desc = p.stage_stride >> 4;                // descriptor units per stage
            const uint64_t group_desc = KG * stage_desc;
            const uint64_t a_desc0 = p.a_desc_hi | (uint64_t)((base >> 4) & 0x3FFFu);
            const uint64_t b_desc0 = p.b_desc_hi | (uint64_t)(((base + p.b_off) >> 4) & 0x3FFFu);
            const uint64_t ak = p.a_kstep >> 4, bk = p.b_kstep >> 4;
            const uint32_t idesc_main = p.idesc;
            uint32_t g = 0, ph = 0;
            uint64_t so = 0;                                                 // group's descriptor offset
            uint32_t it = 0;
            bool ok = true;
            WorkIter wi;
            WorkItem w;
            work_begin(p, cluster_id, nclusters, wi);
            for (; ok && work_next(p, wi, w); ++it) {
                // two accumulators alternate; a wide tile fills all 512 columns
                const uint32_t buf = WIDE ? 0u : (it & 1u), aph = WIDE ? (it & 1u) : ((it >> 1) & 1u);
                if (!mbar_wait(acce_bar(buf), aph ^ 1u, budget)) {
                    report_error(p.err, DEV_TIMEOUT_MMA);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * (uint32_t)p.BN;
                const uint32_t idesc = w.tile >= p.tail_start ? p.tail_idesc : idesc_main;   // tile width
                for (int kb = w.kb0; kb < w.kb1; kb += KG) {
                    if (!mbar_wait(full_bar(g), ph, budget)) {
                        report_error(p.err, DEV_TIMEOUT_MMA);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint64_t ad = a_desc0 + so, bd = b_desc0 + so;
                    const uint32_t acc0 = (uint32_t)(kb != w.kb0);
                    umma_pair<KIND>(d_tmem, ad, bd, idesc, acc0);
                    umma_pair<KIND>(d_tmem, ad + ak, bd + bk, idesc, 1u);
                    umma_pair<KIND>(d_tmem, ad + 2 * ak, bd + 2 * bk, idesc, 1u);
                    umma_pair<KIND>(d_tmem, ad + 3 * ak, bd + 3 * bk, idesc, 1u);
                    if (WIDE) {
                        // second 128-row half of A (16 KiB further in every layout)
                        // into accumulator columns 256..511
                        const uint64_t ah = ad + (kHalfABytes >> 4);
                        const uint32_t d1 = d_tmem + 256u;
                        umma_pair<KIND>(d1, ah, bd, idesc, acc0);
                        umma_pair<KIND>(d1, ah + ak, bd + bk, idesc, 1u);
                        umma_pair<KIND>(d1, ah + 2 * ak, bd + 2 * bk, idesc, 1u);
                        umma_pair<KIND>(d1, ah + 3 * ak, bd + 3 * bk, idesc, 1u);
                    } else if (kb + 1 < w.kb1) {
                        ad += stage_desc;
                        bd += stage_desc;
                        umma_pair<KIND>(d_tmem, ad, bd, idesc, 1u);
                        umma_pair<KIND>(d_tmem, ad + ak, bd + bk, idesc, 1u);
                        umma_pair<KIND>(d_tmem, ad + 2 * ak, bd + 2 * bk, idesc, 1u);
                        umma_pair<KIND>(d_tmem, ad + 3 * ak, bd + 3 * bk, idesc, 1u);
                    }
                    umma_commit_pair_mc(empty_bar(g), (uint16_t)(3u << lead));   // both CTAs' group g free
                    if (++g == ngroups) {
                        g = 0;
                        ph ^= 1u;
                        so = 0;
                    } else {
                        so += group_desc;
                    }
                }
                if (!ok) break;
                umma_commit_pair_mc(accf_bar(buf), (uint16_t)(3u << lead));       // both accumulators ready
            }
            umma_commit_pair_mc(drain_bar, (uint16_t)(1u << lead));
            if (!mbar_wait(drain_bar, 0, budget)) report_error(p.err, DEV_TIMEOUT_TEARDOWN);
        }
        __syncwarp();
    } else if constexpr (WIDE != 0) {
        // ------------------------------------------------ epilogue, wide tiles (both CTAs, 8 warps)
        // warp 2 + e: tensor-memory lane quarter warp % 4 (the warps a CTA
        // may read a quarter with), column half e / 4; one staging slab each
        const uint32_t e = (uint32_t)warp - 2u;
        const uint32_t q = (uint32_t)warp & 3u;
        const uint32_t h = e >> 2;
        const uint32_t lane_field = (q * 32u) << 16;
        const uint32_t slab = base + p.off_epi + e * kEpiSlabBytes;
        uint32_t it = 0;
        WorkIter wi;
        WorkItem w;
        work_begin(p, cluster_id, nclusters, wi);
        for (; work_next(p, wi, w); ++it) {
            int b, mb;
            int32_t n0, tbn;
            decode_tile_w(p, w.tile, b, mb, n0, tbn);
            const bool tail = w.tile >= p.tail_start;
            const int chunks = tail ? p.tail_epi_chunks : p.epi_chunks;
            const int last_cols = tail ? p.tail_epi_last_cols : p.epi_last_cols;
            int good = 1;
            if (lane == 0) good = mbar_wait(accf_bar(0), it & 1u, budget) ? 1 : 0;
            good = __shfl_sync(0xffffffffu, good, 0);
            if (!good) {
                if (lane == 0) report_error(p.err, DEV_TIMEOUT_EPILOGUE);
                break;
            }
            tc_fence_after();
            const uint32_t acce = mapa_shared(acce_bar(0), lead);
            const int half = (chunks + 1) / 2;
            const int c0 = (int)h * half;
            const int nc = min(chunks - c0, half);
            // CTA `rank` holds tile rows rank * 256 .. (region 0) and + 128 (region 1)
            const int32_t mrow = mb * (4 * kBM) + (int32_t)rank * (2 * kBM) + (int32_t)q * kEpiRowsPerWarp;
            epilogue_wide_warp<OUT>(p, &tmC, tmem_base, lane_field, slab, lane, mrow, n0, b, c0, nc, chunks,
                                    last_cols, [&] { mbar_arrive_cluster(acce); });
        }
        if (lane == 0) bulk_wait<0>();
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (both CTAs)
        const uint32_t q = (uint32_t)warp & 3u;
        const uint32_t lane_field = (q * 32u) << 16;
        uint32_t it = 0, sbuf = 0;
        WorkIter wi;
        WorkItem w;
        work_begin(p, cluster_id, nclusters, wi);
        const int64_t slot_floats = 2 * MSUB * kBM * (int64_t)p.BN;   // one cluster's partial slot
        // this warp's share of accumulator region i in a slot: 32 rows x BN fp32
        auto warp_rows = [&](int i) {
            return (((int64_t)rank * MSUB + i) * kEpiWarps + (int64_t)q) * kEpiRowsPerWarp * p.BN;
        };
        for (; work_next(p, wi, w); ++it) {
            int b, mb;
            int32_t n0, tbn;
            decode_tile_w(p, w.tile, b, mb, n0, tbn);
            const bool tail = w.tile >= p.tail_start;
            const int chunks = tail ? p.tail_epi_chunks : p.epi_chunks;
            const int last_cols = tail ? p.tail_epi_last_cols : p.epi_last_cols;
            const uint32_t buf = WIDE ? 0u : (it & 1u), aph = WIDE ? (it & 1u) : ((it >> 1) & 1u);
            int good = 1;
            if (lane == 0) good = mbar_wait(accf_bar(buf), aph, budget) ? 1 : 0;
            good = __shfl_sync(0xffffffffu, good, 0);
            if (!good) {
                if (lane == 0) report_error(p.err, DEV_TIMEOUT_EPILOGUE);
                break;
            }
            tc_fence_after();
            const uint32_t acce = mapa_shared(acce_bar(buf), lead);
            const uint32_t acc = tmem_base + buf * (uint32_t)p.BN;
            const uint32_t slabs = base + p.off_epi + q * kEpiBufs * kEpiSlabBytes;
            if (w.role == ROLE_PARTIAL) {
                // later K blocks of a stream-K tile: publish the fp32 partial
                // (the warp announces it once, after its last region)
                for (int i = 0; i < MSUB; ++i) {
                    epilogue_partial(p, acc + (uint32_t)(i * 256), lane_field, lane, slabs, sbuf,
                                     p.sk_work + cluster_id * slot_floats + warp_rows(i), p.sk_flags + w.sk_tile,
                                     i == MSUB - 1, [&] {
                                         if (i == MSUB - 1) mbar_arrive_cluster(acce);
                                     });
                }
                continue;
            }
            uint32_t mask = 0;
            if (w.role == ROLE_OWNER) {
                // partials of clusters (self, last_slot] with a non-empty range,
                // 8 epilogue warps each (4 per CTA of the pair)
                int32_t want = 0;
                for (int64_t c = cluster_id + 1; c <= w.last_slot; ++c) {
                    if (sk_bound(p, c) < sk_bound(p, c + 1)) {
                        mask |= 1u << (uint32_t)(c - cluster_id - 1);
                        want += 2 * kEpiWarps;
                    }
                }
                int ready = 1;
                if (lane == 0) {
                    const uint64_t t0 = globaltimer();
                    while (ld_acquire_gpu(p.sk_flags + w.sk_tile) < want) {
                        if ((int64_t)(globaltimer() - t0) > budget) {
                            ready = 0;
                            break;
                        }
                    }
                }
                ready = __shfl_sync(0xffffffffu, ready, 0);
                if (!ready) {
                    if (lane == 0) report_error(p.err, DEV_TIMEOUT_FIXUP);
                } else if (mask != 0 &&
                           !sk_fixup(acc, lane_field, lane, p.BN, MSUB,
                                     p.sk_work + (cluster_id + 1) * slot_floats + warp_rows(0), slot_floats,
                                     (int64_t)kEpiWarps * kEpiRowsPerWarp * p.BN, mask,
                                     base + q * (kFixBufs * kFixBlockBytes), fix_bar(q * kFixBufs), budget)) {
                    if (lane == 0) report_error(p.err, DEV_TIMEOUT_FIXUP);
                }
            }
            if constexpr (WIDE == 0 && OUT != OUT_F32) {
                if (p.epi_pace_ns_per_kb > 0 && w.role == ROLE_WHOLE && chunks == 4 && last_cols == 64) {
                    const int32_t m0 = mb * (2 * kBM) + (int32_t)rank * kBM + (int32_t)q * kEpiRowsPerWarp;
                    // spaced only while this cluster has a next main loop to
                    // hide the stores behind (the last tile stores at once)
                    const bool more = wi.dp < p.dp_tiles || wi.u < wi.u1;
                    epilogue_tile_paced<OUT>(p, &tmC, acc, lane_field, slabs, sbuf, lane, m0, n0, b,
                                             more ? (int64_t)p.epi_pace_ns_per_kb * (w.kb1 - w.kb0) : 0,
                                             [&] { mbar_arrive_cluster(acce); });
                    continue;
                }
            }
            for (int i = 0; i < MSUB; ++i) {
                // CTA `rank`'s accumulator region i holds tile rows rank * 128 * MSUB + i * 128 ...
                const int32_t m0 = mb * (2 * MSUB * kBM) + (int32_t)rank * (MSUB * kBM) + i * kBM +
                                   (int32_t)q * kEpiRowsPerWarp;
                epilogue_tile<OUT>(p, &tmC, acc + (uint32_t)(i * 256), lane_field, slabs, sbuf, lane, m0, n0, b,
                                   [&] {
                                       if (i == MSUB - 1) mbar_arrive_cluster(acce);
                                   },
                                   chunks, last_cols);
            }
        }
        if (lane == 0) bulk_wait<0>();
        __syncwarp();
    }

    tc_fence_before();
    cluster_sync_all();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, p.tmem_cols);
}

}  // namespace smo
