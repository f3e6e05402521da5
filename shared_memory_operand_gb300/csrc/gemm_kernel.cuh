// Persistent, warp-specialised GEMM for sm_103a (GB300), one CTA per
// 128 x BN output tile: bf16 / f16 operands (tcgen05.mma kind::f16) or FP8
// E4M3 / E5M2 operands (kind::f8f6f4), fp32 accumulation.
//
//   warp 0               TMA producer: lane 0 waits for a free group of
//                        stages and arms its barrier; lanes 0 .. n-1 then
//                        issue the group's loads of 128-byte-swizzled A and B
//                        tiles together (cp.async.bulk.tensor, mbarrier
//                        complete_tx), `kgroup` stages per barrier pair.
//   warp 1 (one thread)  MMA issuer: 4 x tcgen05.mma (128 x BN x 32 bytes of
//                        K: K = 16 for 16-bit, 32 for FP8) per stage,
//                        accumulating in tensor memory; tcgen05.commit frees
//                        the group (split barrier) and, after the last K block,
//                        publishes the accumulator.
//   warps 2..5 (or 2..9) epilogue: tcgen05.ld -> fp32/bf16/f16 ->
//                        conflict-free swizzled st.shared -> TMA store (clips
//                        ragged edges).  A launch in which every CTA has one
//                        tile (its epilogue is not overlapped by a next main
//                        loop) of at most four column chunks has 8 epilogue
//                        warps, two per tensor-memory lane quarter, each
//                        taking half of the tile's chunks; with several tiles
//                        per CTA 4 warps measured as fast or faster.
// Two tensor-memory accumulators let the epilogue of tile i overlap the main
// loop of tile i + 1.
//
// Design lineage (prior art, re-made for tcgen05/TMA): "An Educational GEMM
// Ladder for Helios GPUs" -- Level 1 (multi-buffered operand stages), Level 2
// (direct global-to-shared copies), Level 3/4 (large output tiles, arithmetic
// intensity 2MNK/(MK+KN+MN)), Level 5 (deep K per stage), Level 7 (descriptor
// DMA issued by a single producer, zero fill at the K tail), Level 8 (split
// barrier: release a stage as soon as its last MMA retires), Level 10
// (epilogue staged through shared memory for wide coalesced stores), Level 12
// (overlap of epilogue and main loop).  Operand orientation: an N-contiguous B
// (or M-contiguous A) is consumed directly through the MN-major canonical
// layout and the instruction descriptor's major bit -- the job the transposed
// shared-memory load does in "A Deep Dive into LDS Optimizations on AMD
// Instinct MI450 GPUs", Part I.
//
// Split-K (SPLIT = 1; fp32 output): the grid is one 2-CTA cluster per tile.
// The CTA of cluster rank 0 computes the tile's first split_kh K blocks,
// rank 1 the rest, each into its own tensor memory; the two partial sums
// meet in global memory (see epilogue_split_tile): each CTA stores half of
// the tile's columns plainly and adds its partial of the other half with TMA
// reduce-adds once the peer's plain stores are complete.  A tile-starved
// problem (fewer tiles than SMs) then runs on twice the SMs, each reading
// half of the tile's K panel ("An Educational GEMM Ladder for Helios GPUs",
// Level 3: large tiles leave a small problem with too few workgroups).
//
// Every mbarrier wait is bounded by p.timeout_ns of the global timer; on
// timeout the thread records an error code, stops, and the CTA still drains
// its in-flight copies and MMAs and frees tensor memory before returning.
#pragma once
#include <cuda.h>
#include <stdint.h>

#include "gemm_common.cuh"

namespace smo {

static_assert(kStageKBytes / kMmaKBytes == 4, "the issue loops unroll four MMAs per K block");

// KG: stages per full/empty barrier pair (1 or 2).  KIND: MmaKind.  SPLIT:
// 1 = split-K over a 2-CTA cluster, one tile per cluster (fp32 output only).
// EPI8: 1 = eight epilogue warps (320 threads), for launches in which every
// CTA has one tile of at most four column chunks.
template <int OUT, int KG, int KIND, int SPLIT, int EPI8>
__global__ void __launch_bounds__(EPI8 ? kWideThreads : kThreads, 1)
    smo_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const __grid_constant__ KParams p) {
    static_assert(!SPLIT || OUT == OUT_F32, "split-K partials meet in fp32");
    static_assert(!(SPLIT && EPI8), "the split-K epilogue has four warps");
    constexpr uint32_t epiw = EPI8 ? 8u : 4u;      // epilogue warps
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // tiles and K range of this CTA
    const uint32_t crank = SPLIT ? (cluster_ctarank() & 1u) : 0u;
    const int64_t tile0 = SPLIT ? (int64_t)(blockIdx.x >> 1) : (int64_t)blockIdx.x;
    const int64_t tstride = SPLIT ? (int64_t)(gridDim.x >> 1) : (int64_t)gridDim.x;
    const int kb_begin = SPLIT && crank ? p.split_kh : 0;
    const int kb_end = SPLIT && !crank ? p.split_kh : p.num_k;

    const uint32_t bars = base + p.off_bar;
    auto full_bar = [&](uint32_t s) { return bars + 8u * s; };
    auto empty_bar = [&](uint32_t s) { return bars + 8u * (kMaxStages + s); };
    auto accf_bar = [&](uint32_t b) { return bars + 8u * (2 * kMaxStages + b); };
    auto acce_bar = [&](uint32_t b) { return bars + 8u * (2 * kMaxStages + 2 + b); };
    const uint32_t drain_bar = bars + 8u * (2 * kMaxStages + 4);
    const uint32_t tmem_slot = bars + 8u * (2 * kMaxStages + 5);
    // SPLIT: every epilogue thread of the peer CTA arrives once its plain
    // stores of the tile are complete
    const uint32_t plain_bar = bars + 8u * (2 * kMaxStages + 6);

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), epiw);
        }
        mbar_init(drain_bar, 1);
        if (SPLIT) mbar_init(plain_bar, kEpiWarps * 32);
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmC);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    if (SPLIT) cluster_sync_all();      // the peer's barriers are initialised before any remote arrive
    else __syncthreads();
    tc_fence_after();
    // The prologue above touches only shared memory, tensor memory and the
    // kernel parameters, so it may overlap the previous kernel in the stream
    // (launched with programmatic stream serialization); every global memory
    // access comes after this wait.
    griddep_wait();
    griddep_launch_dependents();
    const uint32_t tmem_base = ld_shared_u32(tmem_slot);
    const int64_t budget = p.timeout_ns;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        // Lanes 0 .. nloads-1 each own one load of every stage and issue them
        // together; lane 0 waits for the free slot and arms the stage.
        const uint32_t nloads = stage_loads(p);
        if ((uint32_t)lane < nloads) {
            const uint32_t lmask = (1u << nloads) - 1u;
            const LoadSlot slot = load_slot(p, &tmA, &tmB, (uint32_t)lane);
            const uint32_t ngroups = (uint32_t)(p.stages / KG);
            const uint32_t group_bytes = KG * p.stage_stride;
            uint32_t g = 0, ph = 0, gst = base;        // group index, ring parity, group's smem
            uint32_t issued_mask = 0, issued_ph = 0;   // last issued phase per group (lane 0)
            bool skip_one = p.stall != 0;
            bool ok = true;
            for (int64_t t = tile0; t < p.total_tiles && ok; t += tstride) {
                int b, mb, nb;
                decode_tile(p, t, b, mb, nb);
                const int32_t mn0 = slot.is_a ? mb * kBM : nb * p.BN;
                for (int kb = kb_begin; kb < kb_end; kb += KG) {
                    const bool two = KG == 2 && kb + 1 < kb_end;    // the last group may hold one block
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
                        if (lane == 0) {
                            mbar_arrive_expect_tx(full_bar(g), two ? 2 * p.tx_bytes : p.tx_bytes);
                            issued_mask |= 1u << g;
                            issued_ph = (issued_ph & ~(1u << g)) | (ph << g);
                        }
                        __syncwarp(lmask);
                        int32_t c0, c1, c2;
                        slot_coords(slot, mn0, kb * p.bk, c0, c1, c2);
                        tma_load_4d(gst + slot.dst_off, slot.tm, full_bar(g), c0, c1, c2, b);
                        if (two) {
                            slot_coords(slot, mn0, (kb + 1) * p.bk, c0, c1, c2);
                            tma_load_4d(gst + p.stage_stride + slot.dst_off, slot.tm, full_bar(g), c0, c1, c2, b);
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
            // Every load issued has landed before the CTA may exit (immediate
            // when the consumer already waited for it).
            if (lane == 0) {
                for (uint32_t q = 0; q < (uint32_t)(p.stages / KG); ++q) {
                    if ((issued_mask >> q) & 1u) {
                        if (!mbar_wait(full_bar(q), (issued_ph >> q) & 1u, budget))
                            report_error(p.err, DEV_TIMEOUT_TEARDOWN);
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            // Descriptors, steps and ring bounds sit in registers: one thread
            // issues every MMA, and its per-K-block instruction latency must
            // stay below the tensor pipe's time for that block.
            const uint32_t ngroups = (uint32_t)(p.stages / KG);
            const uint64_t stage_desc = p.stage_stride >> 4;
            const uint64_t group_desc = KG * stage_desc;
            const uint64_t a_desc0 = p.a_desc_hi | (uint64_t)((base >> 4) & 0x3FFFu);
            const uint64_t b_desc0 = p.b_desc_hi | (uint64_t)(((base + p.b_off) >> 4) & 0x3FFFu);
            const uint64_t ak = p.a_kstep >> 4, bk = p.b_kstep >> 4;
            const uint32_t idesc = p.idesc;
            uint32_t g = 0, ph = 0;
            uint64_t so = 0;                           // group's descriptor offset
            uint32_t it = 0;
            bool ok = true;
            for (int64_t t = tile0; t < p.total_tiles && ok; t += tstride, ++it) {
                const uint32_t buf = it & 1u, aph = (it >> 1) & 1u;
                if (!mbar_wait(acce_bar(buf), aph ^ 1u, budget)) {
                    report_error(p.err, DEV_TIMEOUT_MMA);
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + buf * (uint32_t)p.BN;
                for (int kb = kb_begin; kb < kb_end; kb += KG) {
                    if (!mbar_wait(full_bar(g), ph, budget)) {
                        report_error(p.err, DEV_TIMEOUT_MMA);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint64_t ad = a_desc0 + so, bd = b_desc0 + so;
                    umma<KIND>(d_tmem, ad, bd, idesc, (uint32_t)(kb != kb_begin));
                    umma<KIND>(d_tmem, ad + ak, bd + bk, idesc, 1u);
                    umma<KIND>(d_tmem, ad + 2 * ak, bd + 2 * bk, idesc, 1u);
                    umma<KIND>(d_tmem, ad + 3 * ak, bd + 3 * bk, idesc, 1u);
                    if (KG == 2 && kb + 1 < kb_end) {
                        ad += stage_desc;
                        bd += stage_desc;
                        umma<KIND>(d_tmem, ad, bd, idesc, 1u);
                        umma<KIND>(d_tmem, ad + ak, bd + bk, idesc, 1u);
                        umma<KIND>(d_tmem, ad + 2 * ak, bd + 2 * bk, idesc, 1u);
                        umma<KIND>(d_tmem, ad + 3 * ak, bd + 3 * bk, idesc, 1u);
                    }
                    umma_commit(empty_bar(g));     // group free once these MMAs retire
                    if (++g == ngroups) {
                        g = 0;
                        ph ^= 1u;
                        so = 0;
                    } else {
                        so += group_desc;
                    }
                }
                if (!ok) break;
                umma_commit(accf_bar(buf));        // accumulator ready for the epilogue
            }
            // All MMAs issued by this thread have completed before teardown.
            umma_commit(drain_bar);
            if (!mbar_wait(drain_bar, 0, budget)) report_error(p.err, DEV_TIMEOUT_TEARDOWN);
        }
        __syncwarp();
    } else if constexpr (SPLIT) {
        // ------------------------------------------------ epilogue (split-K, warps 2..5)
        const uint32_t q = (uint32_t)warp & 3u;           // TMEM lane quarter of this warp
        const uint32_t lane_field = (q * 32u) << 16;
        uint32_t it = 0, sbuf = 0;
        for (int64_t t = tile0; t < p.total_tiles; t += tstride, ++it) {
            int b, mb, nb;
            decode_tile(p, t, b, mb, nb);
            const uint32_t buf = it & 1u, aph = (it >> 1) & 1u;
            int good = 1;
            if (lane == 0) good = mbar_wait(accf_bar(buf), aph, budget) ? 1 : 0;
            good = __shfl_sync(0xffffffffu, good, 0);
            if (!good) {
                if (lane == 0) report_error(p.err, DEV_TIMEOUT_EPILOGUE);
                break;
            }
            tc_fence_after();
            const int32_t m0 = mb * kBM + (int32_t)q * kEpiRowsPerWarp;
            const uint32_t slabs = base + p.off_epi + q * kEpiBufs * kEpiSlabBytes;
            const uint32_t acce = acce_bar(buf);
            // one tile per cluster: the operand ring is idle once the
            // accumulator is full; each warp stages the peer's chunks in its
            // own 16 KiB of it
            if (!epilogue_split_tile(p, &tmC, tmem_base + buf * (uint32_t)p.BN, lane_field, slabs, sbuf, lane, m0,
                                     nb * p.BN, b, crank, base + q * 4u * kEpiSlabBytes,
                                     mapa_shared(plain_bar, crank ^ 1u), plain_bar, budget,
                                     [&] { mbar_arrive(acce); })) {
                if (lane == 0) report_error(p.err, DEV_TIMEOUT_SPLIT);
                break;
            }
        }
        if (lane == 0) bulk_wait<0>();
        __syncwarp();
    } else {
        // ------------------------------------------------ epilogue (warps 2..5, or 2..9 with EPI8)
        // warp 2 + e: tensor-memory lane quarter warp % 4 (the warps a CTA may
        // read a quarter with); with 8 warps, chunk half e / 4 and one
        // staging slab each, with 4 warps all chunks and two slabs each
        const uint32_t e = (uint32_t)warp - 2u;
        const uint32_t q = (uint32_t)warp & 3u;
        const uint32_t lane_field = (q * 32u) << 16;
        const int half = (p.epi_chunks + 1) / 2;
        const int c0 = (int)(e >> 2) * half;
        const int nc = min(p.epi_chunks - c0, half);
        uint32_t it = 0, sbuf = 0;
        for (int64_t t = tile0; t < p.total_tiles; t += tstride, ++it) {
            int b, mb, nb;
            decode_tile(p, t, b, mb, nb);
            const uint32_t buf = it & 1u, aph = (it >> 1) & 1u;
            int good = 1;
            if (lane == 0) good = mbar_wait(accf_bar(buf), aph, budget) ? 1 : 0;
            good = __shfl_sync(0xffffffffu, good, 0);
            if (!good) {
                if (lane == 0) report_error(p.err, DEV_TIMEOUT_EPILOGUE);
                break;
            }
            tc_fence_after();
            const int32_t m0 = mb * kBM + (int32_t)q * kEpiRowsPerWarp;
            const uint32_t acce = acce_bar(buf);
            const uint32_t acc = tmem_base + buf * (uint32_t)p.BN;
            if constexpr (EPI8)
                epilogue_tile_part<OUT>(p, &tmC, acc, lane_field, base + p.off_epi + e * kEpiSlabBytes, lane, m0,
                                        nb * p.BN, b, c0, nc, p.epi_chunks, p.epi_last_cols,
                                        [&] { mbar_arrive(acce); });
            else
                epilogue_tile<OUT>(p, &tmC, acc, lane_field, base + p.off_epi + q * kEpiBufs * kEpiSlabBytes, sbuf,
                                   lane, m0, nb * p.BN, b, [&] { mbar_arrive(acce); });
        }
        if (lane == 0) bulk_wait<0>();
        __syncwarp();
    }

    tc_fence_before();
    if (SPLIT) cluster_sync_all();      // no CTA leaves while its peer may still arrive on its barrier
    else __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, p.tmem_cols);
}

}  // namespace smo
