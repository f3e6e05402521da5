// Global-to-shared bandwidth probe (sm_103a): every CTA (one per SM) streams
// 32 KiB blocks of a caller's device buffer into a ring of shared-memory
// stages with untiled bulk copies (cp.async.bulk, mbarrier complete_tx),
// keeping every stage in flight (1 to 6 stages), and does nothing else.  With a buffer that
// fits in L2 the launch measures how fast L2 feeds the SMs -- the path the
// GEMM's TMA operand loads take; with a buffer several times larger than L2,
// the rate from HBM through L2.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <cstring>

#include "ptx.cuh"
#include "smo_probe.h"

namespace {

constexpr int kStages = 6;
constexpr uint32_t kChunk = 32 * 1024;
constexpr uint32_t kSmemBytes = kStages * kChunk + 1024 /* alignment */ + 8 * kStages;

// CTA c copies blocks c, c + grid, c + 2 grid, ... (modulo the buffer's
// `nchunks` blocks), `iters` of them, so that the SMs sweep the buffer
// together as a GEMM's wave sweeps its operand panels.
__global__ void __launch_bounds__(32, 1)
    l2_read_kernel(const uint8_t* src, uint64_t nchunks, int iters, int stages, long long* out,
                   int64_t budget_ns) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    if (threadIdx.x != 0) return;
    const uint32_t base = (smo::smem_u32(smem_raw) + 1023u) & ~1023u;
    const uint32_t bars = base + kStages * kChunk;
    for (int s = 0; s < stages; ++s) smo::mbar_init(bars + 8u * s, 1);
    smo::fence_barrier_init();
    smo::fence_proxy_async_smem();
    const long long c0 = clock64();
    const uint64_t t0 = smo::globaltimer();
    uint64_t blk = blockIdx.x % nchunks;
    const uint64_t step = gridDim.x % nchunks;
    bool ok = true;
    int issued = 0;
    for (; issued < iters; ++issued) {
        const int s = issued % stages;
        // the copy `stages` earlier into the same stage must have landed
        if (issued >= stages &&
            !smo::mbar_wait(bars + 8u * s, (uint32_t)(issued / stages - 1) & 1u, budget_ns)) {
            ok = false;
            break;
        }
        smo::mbar_arrive_expect_tx(bars + 8u * s, kChunk);
        smo::bulk_load(base + (uint32_t)s * kChunk, src + blk * kChunk, kChunk, bars + 8u * s);
        blk += step;
        if (blk >= nchunks) blk -= nchunks;
    }
    // wait (bounded) for every copy still in flight
    for (int i = issued > stages ? issued - stages : 0; i < issued; ++i)
        if (!smo::mbar_wait(bars + 8u * (i % stages), (uint32_t)(i / stages) & 1u, budget_ns)) ok = false;
    out[2 * blockIdx.x] = ok ? (long long)(clock64() - c0) : -1;
    out[2 * blockIdx.x + 1] = ok ? (long long)(smo::globaltimer() - t0) : -1;
}

}  // namespace

extern "C" int l2_read_probe(const void* src, size_t bytes, int iters, int stages, void* out, int max_ctas,
                             void* stream) {
    if (!src || !out || iters < 1 || max_ctas < 1 || bytes < kChunk || stages < 1 || stages > kStages) return -1;
    if ((reinterpret_cast<uintptr_t>(src) & 15u) != 0) return -2;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return -4;
    }
    if (cudaFuncSetAttribute(l2_read_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) !=
        cudaSuccess) {
        cudaGetLastError();
        return -4;
    }
    const int ctas = std::min(max_ctas, sms);       // the shared memory request allows one CTA per SM
    l2_read_kernel<<<ctas, 32, kSmemBytes, reinterpret_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t*>(src), (uint64_t)(bytes / kChunk), iters, stages, static_cast<long long*>(out),
        (int64_t)2000000000);
    if (cudaGetLastError() != cudaSuccess) return -4;
    return ctas;
}
