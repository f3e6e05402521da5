// Tensor-core issue-rate probe (sm_103a): every 2-CTA cluster fills one
// 128 x 64 A tile and one 128 x 64 B tile per CTA in shared memory (128-byte
// swizzled, K-major, pseudo-random bf16 values), then the even CTA issues
// back-to-back tcgen05.mma.cta_group::2 (256 x 256 x 16) on that resident data
// and waits for the last one.  No global-memory traffic: the launch's duration
// bounds the dense BF16 rate the GEMM's main loop could reach on this GPU.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cstring>

#include "gemm_params.h"
#include "planner.h"
#include "ptx.cuh"
#include "smo_probe.h"

namespace {

constexpr uint32_t kTileBytes = 128 * 64 * 2;          // one operand tile per CTA
// Asks for far more shared memory than it uses, so that no SM holds two CTAs.
constexpr uint32_t kProbeSmemBytes = 160 * 1024;

__global__ void __launch_bounds__(128, 1)
    tc_peak_kernel(uint32_t idesc, uint64_t adesc_hi, uint64_t bdesc_hi, int iters, long long* out,
                   int64_t budget_ns) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t base = (smo::smem_u32(smem_raw) + 1023u) & ~1023u;
    uint8_t* gbase = smem_raw + (base - smo::smem_u32(smem_raw));
    const uint32_t bar = base + 2 * kTileBytes;
    const uint32_t slot = bar + 8;
    const uint32_t rank = smo::cluster_ctarank() & 1u;
    const uint32_t lead = smo::cluster_ctarank() & ~1u;

    // bf16 values from an integer hash of the element index (exponent kept in
    // range so the products stay finite)
    uint32_t* words = reinterpret_cast<uint32_t*>(gbase);
    for (uint32_t i = threadIdx.x; i < 2 * kTileBytes / 4; i += blockDim.x) {
        uint32_t h = (i + 1u + 977u * blockIdx.x) * 2654435761u;
        h ^= h >> 15;
        words[i] = (h & 0x807F807Fu) | 0x3F003F00u;
    }
    smo::fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        smo::mbar_init(bar, 1);
        smo::fence_barrier_init();
    }
    if (threadIdx.x < 32) {
        smo::tmem_alloc_pair(slot, 256);
        smo::tmem_relinquish_pair();
    }
    smo::tc_fence_before();
    smo::cluster_sync_all();
    smo::tc_fence_after();
    const uint32_t tmem = smo::ld_shared_u32(slot);

    if (rank == 0 && threadIdx.x == 0) {
        const uint64_t a_desc = adesc_hi | (uint64_t)((base >> 4) & 0x3FFFu);
        const uint64_t b_desc = bdesc_hi | (uint64_t)(((base + kTileBytes) >> 4) & 0x3FFFu);
        const long long c0 = clock64();
        const uint64_t g0 = smo::globaltimer();
        for (int i = 0; i < iters; ++i) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                smo::umma_pair<smo::KIND_F16>(tmem, a_desc + (uint64_t)(k * 2), b_desc + (uint64_t)(k * 2), idesc, (i | k) != 0);
        }
        smo::umma_commit_pair_mc(bar, (uint16_t)(1u << lead));
        const bool ok = smo::mbar_wait(bar, 0, budget_ns);
        const long long c1 = clock64();
        const uint64_t g1 = smo::globaltimer();
        const int cl = blockIdx.x >> 1;
        out[2 * cl] = ok ? c1 - c0 : -1;
        out[2 * cl + 1] = ok ? (long long)(g1 - g0) : -1;
    }
    smo::tc_fence_before();
    smo::cluster_sync_all();
    smo::tc_fence_after();
    if (threadIdx.x < 32) smo::tmem_dealloc_pair(tmem, 256);
}

}  // namespace

extern "C" int tc_peak_probe(int iters, void* out, int max_clusters, void* stream) {
    if (iters < 1 || !out || max_clusters < 1) return -1;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return -4;
    }
    // K-major, 128-byte swizzle, 8-row groups 1 KiB apart; bf16 x bf16 -> f32, M = N = 256
    const uint32_t idesc = smo::make_idesc(0, 0, 0, 256, 256);
    const uint64_t desc_hi = ((uint64_t)(16 >> 4) << 16) | ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) |
                             ((uint64_t)2 << 61);
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.blockDim = dim3(128, 1, 1);
    cfg.dynamicSmemBytes = kProbeSmemBytes;
    cfg.stream = reinterpret_cast<cudaStream_t>(stream);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaFuncSetAttribute(tc_peak_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kProbeSmemBytes) !=
        cudaSuccess) {
        cudaGetLastError();
        return -4;
    }
    // at most one cluster per SM pair, and no more than can be co-resident
    cfg.gridDim = dim3(2 * (unsigned)std::max(1, sms / 2), 1, 1);
    int resident = 0;
    if (cudaOccupancyMaxActiveClusters(&resident, tc_peak_kernel, &cfg) != cudaSuccess || resident < 1) {
        cudaGetLastError();
        return -4;
    }
    const int clusters = std::min(std::min(max_clusters, std::max(1, sms / 2)), resident);
    cfg.gridDim = dim3(2 * clusters, 1, 1);
    if (cudaLaunchKernelEx(&cfg, tc_peak_kernel, idesc, desc_hi, desc_hi, iters, static_cast<long long*>(out),
                           (int64_t)2000000000) != cudaSuccess) {
        cudaGetLastError();
        return -4;
    }
    return clusters;
}
