// Shared-memory bank microbenchmark (sm_103a): one warp repeats one shared
// memory access whose per-lane byte offsets the caller supplies, and records
// the clock cycles per access instruction.  With the address pattern alone on
// the SM, the cycles per instruction track the number of wavefronts the
// request needs (phases x worst bank degree), which is what a bank-conflict
// simulator predicts for the same offsets.
//
// Method: "A Deep Dive into LDS Optimizations on AMD Instinct MI450 GPUs",
// "Measuring It: An LDS Bandwidth Microbenchmark" (a kernel that only accesses
// shared memory, bracketed by clock reads; cycles = fixed + bytes / rate, the
// rate recovered as the slope over burst lengths) and the padding
// microbenchmark of the "LDS Optimization" skill page ("Padding Amount"): the
// same access pattern timed under several row strides.
#include <cuda_runtime.h>
#include <stdint.h>

#include "smo_probe.h"

namespace {

constexpr int kProbeSmem = 64 * 1024;

template <int BYTES, bool STORE>
__device__ __forceinline__ void access(uint32_t addr, uint32_t& acc) {
    if (STORE) {
        if (BYTES == 16)
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(acc) : "memory");
        else if (BYTES == 8)
            asm volatile("st.shared.v2.b32 [%0], {%1, %1};" ::"r"(addr), "r"(acc) : "memory");
        else if (BYTES == 4)
            asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(acc) : "memory");
        else
            asm volatile("st.shared.b16 [%0], %1;" ::"r"(addr), "h"((uint16_t)acc) : "memory");
    } else {
        uint32_t a, b, c, d;
        if (BYTES == 16) {
            asm volatile("ld.volatile.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(a), "=r"(b), "=r"(c), "=r"(d) : "r"(addr)
                         : "memory");
            acc += a ^ b ^ c ^ d;
        } else if (BYTES == 8) {
            asm volatile("ld.volatile.shared.v2.b32 {%0, %1}, [%2];" : "=r"(a), "=r"(b) : "r"(addr) : "memory");
            acc += a ^ b;
        } else if (BYTES == 4) {
            asm volatile("ld.volatile.shared.b32 %0, [%1];" : "=r"(a) : "r"(addr) : "memory");
            acc += a;
        } else {
            uint16_t h;
            asm volatile("ld.volatile.shared.b16 %0, [%1];" : "=h"(h) : "r"(addr) : "memory");
            acc += h;
        }
    }
}

template <int BYTES, bool STORE>
__global__ void __launch_bounds__(32, 1) smem_probe_kernel(const uint32_t* offsets, int iters, long long* out) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int lane = threadIdx.x & 31;
    const uint32_t base = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    // in range and aligned to the access width whatever the caller passed
    const uint32_t addr = base + ((offsets[lane] % (uint32_t)(kProbeSmem - 4096)) & ~(uint32_t)(BYTES - 1));
    uint32_t acc = (uint32_t)lane;
    // Warm the path once, then time `iters` rounds of 8 back-to-back accesses.
    // Access n is shifted by (n % 32) * 128 bytes: the whole pattern moves by a
    // multiple of the 32-bank span, so every lane keeps its bank, while no two
    // consecutive accesses repeat an address (the compiler may not merge them).
    access<BYTES, STORE>(addr, acc);
    __syncwarp();
    const long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int u = 0; u < 8; ++u) access<BYTES, STORE>(addr + (((uint32_t)(i * 8 + u) & 31u) << 7), acc);
    }
    __syncwarp();
    const long long t1 = clock64();
    if (lane == 0) out[0] = t1 - t0;
    if (acc == 0xFFFFFFFFu) out[1] = acc;   // keeps loads live
}

template <int BYTES>
cudaError_t launch_bytes(bool store, const uint32_t* offsets, int iters, long long* out, cudaStream_t s) {
    if (store) {
        auto k = smem_probe_kernel<BYTES, true>;
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem);
        k<<<1, 32, kProbeSmem, s>>>(offsets, iters, out);
    } else {
        auto k = smem_probe_kernel<BYTES, false>;
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kProbeSmem);
        k<<<1, 32, kProbeSmem, s>>>(offsets, iters, out);
    }
    return cudaGetLastError();
}

}  // namespace

extern "C" int smem_bank_probe(const void* offsets, int access_bytes, int is_store, int iters, void* cycles_out,
                               void* stream) {
    if (!offsets || !cycles_out || iters < 1) return -1;
    if (reinterpret_cast<uintptr_t>(offsets) & 3 || reinterpret_cast<uintptr_t>(cycles_out) & 7) return -2;
    const uint32_t* off = static_cast<const uint32_t*>(offsets);
    long long* out = static_cast<long long*>(cycles_out);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (access_bytes) {
        case 2: e = launch_bytes<2>(is_store != 0, off, iters, out, s); break;
        case 4: e = launch_bytes<4>(is_store != 0, off, iters, out, s); break;
        case 8: e = launch_bytes<8>(is_store != 0, off, iters, out, s); break;
        case 16: e = launch_bytes<16>(is_store != 0, off, iters, out, s); break;
        default: return -1;
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return -4;
    }
    return 0;
}
