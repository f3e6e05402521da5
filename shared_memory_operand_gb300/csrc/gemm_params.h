// Kernel parameter block shared by the host planner and the sm_103a kernel.
// Plain C++ (no CUDA headers) so the planner compiles with the host compiler.
#pragma once
#include <stdint.h>

namespace smo {

constexpr int kBM = 128;            // output rows per tile (tcgen05 M, cta_group::1)
constexpr int kStageKBytes = 128;   // K bytes per pipeline stage: one 128-byte swizzle row
                                    // (64 bf16 / f16 values, 128 FP8 values)
constexpr int kMmaKBytes = 32;      // K bytes per tcgen05.mma (kind::f16 K = 16, kind::f8f6f4 K = 32)
constexpr int kThreads = 192;       // warp 0 TMA producer, warp 1 MMA issuer, warps 2..5 epilogue
constexpr int kEpiWarps = 4;
// Wide CTA-pair tiles, and one-CTA launches with one tile per CTA: 8
// epilogue warps (two per tensor-memory lane quarter, one per half of the
// tile's columns), 320 threads.
constexpr int kWideEpiWarps = 8;
constexpr int kWideThreads = 64 + 32 * kWideEpiWarps;
constexpr int kEpiRowsPerWarp = 32;
constexpr int kEpiBufs = 2;         // staging buffers per epilogue warp
constexpr uint32_t kEpiSlabBytes = kEpiRowsPerWarp * 128;   // 32 rows x 128 B
constexpr int kMaxStages = 8;
constexpr uint32_t kSmemLimit = 232448;                      // 227 KiB opt-in per block
constexpr uint32_t kBarrierBytes = 512;
// Stream-K fix-up: each epilogue warp streams the fp32 partials it adds in
// blocks of 4 accumulator column chunks (32 rows x 128 columns x 4 B) through
// kFixBufs buffers of its own in the operand ring, idle by then.
constexpr int kFixBufs = 3;
constexpr int kFixChunks = 4;
constexpr uint32_t kFixBlockBytes = kEpiRowsPerWarp * 32 * 4 * kFixChunks;    // 16 KiB
constexpr uint32_t kFixRingBytes = kEpiWarps * kFixBufs * kFixBlockBytes;   // 192 KiB

// Out element types.
enum OutKind { OUT_F32 = 0, OUT_BF16 = 1, OUT_F16 = 2 };

// tcgen05.mma instruction kinds: 16-bit operands, or 8-bit floating point.
enum MmaKind { KIND_F16 = 0, KIND_F8F6F4 = 1 };

// Error codes written to the device error word (first writer wins).
enum DevErr : int32_t {
    DEV_OK = 0,
    DEV_TIMEOUT_PRODUCER = 1,
    DEV_TIMEOUT_MMA = 2,
    DEV_TIMEOUT_EPILOGUE = 3,
    DEV_TIMEOUT_TEARDOWN = 4,
    DEV_TIMEOUT_FIXUP = 5,
    DEV_TIMEOUT_SPLIT = 6,
};

struct KParams {
    int32_t M, N, K, batch;
    int32_t num_m, num_n, num_k;
    int32_t group_m;
    int64_t tiles_per_batch, total_tiles;
    int32_t BN, stages;
    int32_t kgroup;                 // K blocks (stages) per full/empty barrier pair: 1 or 2
    int32_t bk;                     // K elements per stage (128 / input element bytes)
    int32_t m_sub;                  // 128-row accumulator regions per CTA (2 in a wide CTA pair)
    uint32_t idesc;                 // tcgen05 instruction descriptor
    uint32_t a_mn_major, b_mn_major;
    uint32_t a_nbox, b_nbox;        // TMA boxes per stage and operand
    uint32_t a_fused, b_fused;      // 1: an MN-major operand's boxes come from one 4-D TMA load
    uint32_t a_box_bytes, b_box_bytes;
    uint32_t a_box_mn, b_box_mn;    // MN extent of one box
    uint32_t a_kstep, b_kstep;      // descriptor start-address advance per MMA K step (bytes)
    uint64_t a_desc_hi, b_desc_hi;  // smem descriptor fields other than the start address
    uint32_t stage_stride;          // bytes per pipeline stage (A then B)
    uint32_t b_off;                 // offset of B inside a stage
    uint32_t off_epi, off_bar;      // from the 1024-aligned smem base
    uint32_t tmem_cols;
    uint32_t tx_bytes;              // bytes TMA delivers per stage
    int32_t epi_chunk_cols;         // output columns per 128-byte chunk
    int32_t epi_chunks;             // chunks per tile row (ceil(BN / epi_chunk_cols))
    int32_t epi_last_cols;          // tile columns in the last chunk (epi_chunk_cols unless BN is not a multiple)
    // 256 x 256 pair tiles with 16-bit output: spacing of a warp's four chunk
    // stores, in ns per K block of the tile (0: stored back to back)
    int32_t epi_pace_ns_per_kb;
    void* C;                        // output base (ragged 16-byte row tails are stored directly)
    int64_t ldc, strideC;           // elements
    int32_t n_tma;                  // columns [0, n_tma) are written by TMA (n_tma * es % 16 == 0)
    // Stream-K (CTA-pair kernel): tiles [0, dp_tiles) are computed whole,
    // round-robin over the clusters; the K blocks of the remaining tiles
    // (sk_units in all) are shared out evenly, cluster c taking units
    // [c * sk_units / sk_clusters, (c + 1) * sk_units / sk_clusters).
    int32_t sk_clusters;            // clusters of the launch; 0 = no stream-K
    int64_t dp_tiles;
    int64_t sk_units;
    float* sk_work;                 // one fp32 partial-accumulator slot per cluster
    int32_t* sk_flags;              // per stream-K tile: epilogue warps that published
    // Narrower tiles for the last, partial wave (CTA-pair wide kernel): tiles
    // [tail_start, total_tiles) cover M blocks [tail_m0, tail_m0 + tail_gsz)
    // x columns [tail_n0, N) with tiles tail_bn wide, so that they fit one
    // wave; tail_start >= total_tiles: every tile is BN wide.
    // Wide tiles: a cluster's odd-numbered tiles run their K loop from the
    // last K block down (1 = on), so that a wave starts on the K slices the
    // previous wave used last, still in L2.
    int32_t serp;
    int64_t tail_start;
    int32_t tail_m0, tail_gsz, tail_n0, tail_bn;
    // batches: tail tiles [0, tail_k0) lie in problem tail_b0 from column
    // tail_n0; then tail_kfull tiles per later problem, from column 0
    int32_t tail_b0, tail_k0, tail_kfull;
    uint32_t tail_idesc;
    int32_t tail_epi_chunks, tail_epi_last_cols;
    // Split-K over a 2-CTA cluster (one-CTA kernel, fp32 output): the CTA of
    // cluster rank 0 takes K blocks [0, split_kh), rank 1 [split_kh, num_k);
    // 0 = no split.
    int32_t split_kh;
    int32_t* err;                   // device error word
    int64_t timeout_ns;             // budget of each bounded wait
    int32_t stall;                  // test hook: skip the first TMA load
};

}  // namespace smo
