/*
 * smo_probe.h -- measurement probes exported by libsmo_gemm.so: the
 * shared-memory bank microbenchmark, the tensor-core issue-rate probe and the
 * global-to-shared bandwidth probe.
 *
 * Measurement tools beside the GEMM, not part of it.  The bank microbenchmark
 * times one shared-memory access pattern in isolation so that the
 * bank-conflict degree a simulator predicts for that pattern can be checked
 * on the hardware (method:
 * "A Deep Dive into LDS Optimizations on AMD Instinct MI450 GPUs", "Measuring
 * It: An LDS Bandwidth Microbenchmark", and the padding measurement of the
 * "LDS Optimization" skill page, "Padding Amount").
 */
#ifndef SMO_PROBE_H
#define SMO_PROBE_H

#include <stddef.h>

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

/*
 * tc_peak_probe: tensor-core issue-rate probe.  Launches up to max_clusters
 * 2-CTA clusters (at most one per SM pair) on `stream`; in each, the even CTA
 * issues iters x 4 back-to-back tcgen05.mma.cta_group::2.kind::f16 of
 * 256 x 256 x 16 (bf16 in, fp32 accumulate in tensor memory) on operand tiles
 * resident in shared memory -- no global-memory traffic -- and waits (bounded)
 * for the last one.  out: device pointer to 2 * max_clusters int64, per
 * cluster [clock64 cycles, global-timer ns] of its issue loop (-1 on timeout).
 * Each cluster performs iters * 4 * 2 * 256 * 256 * 16 flops.  Returns the
 * number of clusters launched, or a negative value on error.  Asynchronous.
 */
int tc_peak_probe(int iters, void* out, int max_clusters, void* stream);

/*
 * l2_read_probe: global-to-shared-memory bandwidth probe.  Launches up to
 * max_ctas CTAs (at most one per SM) on `stream`; each streams `iters` blocks
 * of 32 KiB of the device buffer `src` (`bytes` long, 16-byte aligned,
 * caller-owned, only read) into a ring of `stages` (1..6) shared-memory
 * stages with untiled bulk copies (cp.async.bulk, mbarrier completion), all
 * of them in flight, and nothing else.  CTA c reads blocks c, c + ctas, c + 2 ctas, ... modulo
 * bytes / 32 KiB.  A buffer that fits in L2 (after one warm-up launch)
 * measures the rate at which L2 feeds the SMs -- the path of the GEMM's
 * operand loads; a buffer several times the L2 size measures the HBM-fed rate.
 * out: device pointer to 2 * max_ctas int64, per CTA [clock64 cycles,
 * global-timer ns] of its copy loop (-1 if a bounded wait ran out).
 * Bytes moved: ctas * iters * 32768.  Returns the number of CTAs launched, or
 * -1 (bad argument), -2 (misaligned src), -4 (launch failed).  Asynchronous.
 */
int l2_read_probe(const void* src, size_t bytes, int iters, int stages, void* out, int max_ctas,
                  void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SMO_PROBE_H */
