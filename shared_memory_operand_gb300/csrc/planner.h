// Layout planner: chooses the tile, the pipeline depth, the TMA boxes and the
// tcgen05 descriptors, and proves on the host -- by modelling every
// shared-memory layout as an F2-linear map from element coordinates to byte
// offsets -- that the layout TMA writes is the layout the tensor core reads.
//
// Linear-layout view: "A Deep Dive into LDS Optimizations on AMD Instinct MI450
// GPUs", "A Linear Layout Refresher" (a layout is a binary matrix on index
// bits; images XOR) and "Dividing Layouts" (left division = block-diagonal
// factor; here the factor is the 16-byte contiguous core-matrix row).
// XOR swizzle: "LDS Optimization" skill page, "Optimization Method 1: Swizzle
// Layout" (col ^= f(row)); mask width rule from "Choosing Swizzle Parameters"
// (32 banks, 16-byte vectors -> a 3-bit mask, i.e. the 128-byte swizzle).
#pragma once
#include <stdint.h>
#include <string>

#include "gemm_params.h"

namespace smo {

struct OperandPlan {
    int mn_major = 0;
    int tile_mn = 0;                // rows of the operand tile in its MN dimension
    int es = 2;                     // bytes per element (2: bf16 / f16, 1: FP8)
    int bk = 64;                    // K per stage: one 128-byte swizzle row of K-major elements
    int mma_k = 16;                 // K per tcgen05.mma: 32 bytes of K
    uint32_t box_inner = 0, box_outer = 0;   // TMA box (elements)
    int nbox = 0;
    uint32_t box_bytes = 0, stage_bytes = 0;
    uint32_t lbo = 0, sbo = 0, kstep = 0;
    uint64_t desc_hi = 0;
    // F2 model of the stage tile: byte offset of unit coordinates
    int bits_mn = 0, bits_k = 0;
    uint32_t basis_mn[16] = {0}, basis_k[16] = {0};
    bool linear = false, bijective = false, tma_equals_umma = false, core_matrix_divides = false;
};

struct EpiPlan {
    int out_es = 4;
    int chunk_cols = 32;
    int chunks = 0;                 // ceil(BN / chunk_cols)
    int last_cols = 32;             // tile columns in the last chunk
    uint32_t basis_row[5] = {0}, basis_chunk[3] = {0};
    bool bijective = false;
    int planner_degree = 0;         // planner's own bank-degree estimate of one store
};

struct Plan {
    int64_t M = 0, N = 0, K = 0, batch = 1;
    int in_dtype = 0, out_dtype = 0;
    int in_es = 2;                  // input element bytes
    int bk = 64, mma_k = 16;        // K per stage / per MMA (128 / in_es, 32 / in_es)
    int kind = 0;                   // tcgen05.mma kind: 0 kind::f16, 1 kind::f8f6f4
    int pair = 0;                   // 1: CTA pair (cta_group::2), 256 x BN tiles over two SMs
    int wide = 0;                   // 1 (pair only): 512 x 256 tiles, 256 A rows per CTA, one accumulator
    int split = 0;                  // 1 (one CTA, fp32 out): split-K over a 2-CTA cluster, one tile per cluster
    // Tail (wide CTA pair, BN = 256): the last partial wave's tiles re-tiled
    // tail_bn wide: M blocks [tail_m0, tail_m0 + tail_gsz) x columns [tail_n0, N)
    int tail = 0;
    int64_t tail_start = 0;
    int tail_m0 = 0, tail_gsz = 0, tail_n0 = 0, tail_bn = 0, tail_tiles = 0;
    // batches: the tail starts in problem tail_b0 at column tail_n0 (its first
    // tail_k0 tiles); each later problem is re-tiled whole (tail_kfull tiles)
    int tail_b0 = 0, tail_k0 = 0, tail_kfull = 0;
    // 256 x 256 pair tiles, 16-bit output (four whole chunks per warp): the
    // epilogue spaces its chunk stores by this many ns per K block of a tile
    int epi_pace_ns_per_kb = 0;
    uint32_t tail_idesc = 0;
    int tail_chunks = 0, tail_last_cols = 0;
    int split_kh = 0;               // K blocks of the cluster's rank-0 CTA
    int tile_m = 128;               // output rows per tile (128; 256 for a pair; 512 for a wide pair)
    int BN = 256, stages = 4;
    int kgroup = 1;                 // stages per full/empty barrier pair
    int num_m = 0, num_n = 0, num_k = 0, group_m = 16;
    int64_t tiles = 0;
    int grid = 0, num_sms = 0;
    uint32_t idesc = 0;
    OperandPlan a, b;
    EpiPlan c;
    uint32_t stage_stride = 0, off_epi = 0, off_bar = 0, smem_bytes = 0, tmem_cols = 0;
    bool ok = false;
    std::string why;                // reason when !ok
};

// in_dtype: 0 bf16, 1 f16, 3 FP8 E4M3, 4 FP8 E5M2.  out_dtype: 0 bf16, 1 f16,
// 2 f32 (gemm_dtype_t).
// force: 0 = choose; 128, 192 or 256 = one CTA with that BN; 384 = CTA pair
// with 256 x 128 tiles; 512 = CTA pair (256 x 256); 1024 = wide CTA pair
// (512 x 256).
// split: -1 = choose, 0 = never, 1 = split K over a 2-CTA cluster whenever the
// plan allows it (one-CTA tiles, fp32 output, at least two K blocks).
// wide_bn: tile width of a wide CTA pair (0 = choose among 256, 240, 224, 208,
// 192 by wave quantisation; otherwise that width, a multiple of 16 <= 256).
Plan make_plan(int64_t M, int64_t N, int64_t K, int a_major, int b_major, int in_dtype,
               int out_dtype, int64_t batch, int num_sms, int force, int split = -1, int wide_bn = 0);

// Fills the kernel parameter block from a plan (pointers and runtime knobs are
// set by the caller).
void fill_params(const Plan& p, KParams* kp);

std::string describe_json(const Plan& p);

// tcgen05 instruction descriptor for kind::f16 with fp32 accumulation.
uint32_t make_idesc(int in_dtype, int a_mn_major, int b_mn_major, int M, int N);

}  // namespace smo
