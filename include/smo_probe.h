/*
 * smo_probe.h -- shared-memory bank microbenchmark exported by libsmo_gemm.so
 *
 * A measurement tool beside the GEMM, not part of it.  It times one shared
 * memory access pattern in isolation so that the bank-conflict degree a
 * simulator predicts for that pattern can be checked on the hardware (method:
 * "A Deep Dive into LDS Optimizations on AMD Instinct MI450 GPUs", "Measuring
 * It: An LDS Bandwidth Microbenchmark", and the padding measurement of the
 * "LDS Optimization" skill page, "Padding Amount").
 */
#ifndef SMO_PROBE_H
#define SMO_PROBE_H

#ifdef __cplusplus
extern "C" {
#endif

/*
 * smem_bank_probe: launches one warp on `stream` that performs, `iters` x 8
 * times back to back, the shared-memory access in which lane l uses byte
 * offset offsets[l] of a 64 KiB dynamic shared buffer.
 *   offsets      device pointer to 32 uint32 byte offsets (caller-owned; each is
 *                reduced modulo 60 KiB and rounded down to the access width,
 *                so every access stays in bounds and aligned).  Access n of the
 *                loop adds (n % 32) * 128 bytes to every lane's offset: the
 *                banks stay the same, the addresses do not repeat.
 *   access_bytes 2, 4, 8 or 16 (b16, b32, v2.b32, v4.b32)
 *   is_store     0 = ld.shared, 1 = st.shared
 *   cycles_out   device pointer to 2 int64; [0] receives the clock64 cycles
 *                of the timed loop (divide by iters * 8 for cycles/access)
 * Returns 0, -1 for a bad argument, -2 for a misaligned pointer, -4 if the
 * launch failed.  Asynchronous; synchronise `stream` before reading cycles_out.
 */
int smem_bank_probe(const void* offsets, int access_bytes, int is_store, int iters, void* cycles_out,
                    void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SMO_PROBE_H */
