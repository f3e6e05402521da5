/*
 * smo_gemm.h -- C ABI of the shared-memory-operand GEMM library (libsmo_gemm.so)
 *
 * One operation: the dense matrix product C = A * B with 16-bit operands
 * (bfloat16 or float16) or 8-bit floating-point operands (FP8 E4M3 or E5M2 of
 * the OCP 8-bit format), fp32 accumulation in tensor memory, and fp32 / bf16 /
 * f16 output.  Source of the operation: "An Educational GEMM Ladder for Helios
 * GPUs", section "Educational GEMM Ladder" (every rung computes C = AB with
 * A in R^{MxK}, B in R^{KxN}, BF16 inputs, on matrix units that also take
 * FP8); the f16 variant is the GEMM of rocMLIR pull 2196's description
 * (-m 1500 -n 1152 -k 896, f16); the 8-bit operands are those of the 8-bit
 * transposed load of the MI450 post, Part I (ds_load_tr8_b64).  Operands are
 * staged through shared memory in 128-byte-swizzled layouts, and an
 * N-contiguous ("transposed") B is consumed directly -- the role that
 * "A Deep Dive into LDS Optimizations on AMD Instinct MI450 GPUs", Part I
 * ("Why Is It Important?") gives to the transposed shared-memory load.
 *
 * Conventions shared by every entry point
 *   Logical shapes: A is M x K, B is K x N, C is M x N (per batch entry).
 *   Orientation ("major" = the contiguous dimension):
 *     A, GEMM_K_MAJOR : A[m][k] at A[m*lda + k]      (row-major M x K)
 *     A, GEMM_MN_MAJOR: A[m][k] at A[k*lda + m]      (M contiguous)
 *     B, GEMM_K_MAJOR : B[k][n] at B[n*ldb + k]      (K contiguous per column)
 *     B, GEMM_MN_MAJOR: B[k][n] at B[k*ldb + n]      (row-major K x N, N contiguous)
 *     C               : C[m][n] at C[m*ldc + n]      (always row-major)
 *   Batch entry b adds b*strideA / b*strideB / b*strideC elements.
 *   Leading dimensions and strides are in elements.
 *   Pointers: caller-owned DEVICE memory of the current CUDA device.  The
 *   library keeps no reference after the call returns (the kernel reads and
 *   writes them asynchronously on `stream`; keep them alive until it is done).
 *   C is fully overwritten (alpha = 1, beta = 0).  C must not alias A or B.
 *   Alignment (tensor-memory-accelerator rule): A, B, C 16-byte aligned; lda,
 *   ldb and (batch > 1) strideA, strideB times the element size multiples of
 *   16 bytes; the same for ldc and strideC with the output element size.
 *   Streams: `stream` is a cudaStream_t (NULL = legacy default stream).  No
 *   entry point except gemm_check synchronises.
 *   Allocation: the library allocates one 4-byte error word per device on its
 *   first launch there.  A launch that splits tiles along K (stream-K: chosen
 *   automatically only for CTA-pair tiles whose last wave leaves every
 *   cluster a long share of K, or forced with SMO_GEMM_STREAM_K=1) also uses
 *   one workspace per (device, stream): an fp32 partial slot per cluster
 *   (clusters x tile rows x tile columns x 4 bytes; 76 x 256 x 256 x 4 =
 *   19.9 MB on a 152-SM GPU) and a counter per cluster.  It is allocated on
 *   the first split launch on that stream, grown when a larger one is needed,
 *   and kept until the process exits; while the stream is being captured into
 *   a CUDA graph nothing is allocated and a launch without a large enough
 *   workspace does not split.  A tile-starved fp32-output GEMM whose K loop is
 *   long may instead split K over the two CTAs of a cluster (chosen by the
 *   planner, or forced with SMO_GEMM_SPLIT_K=0/1); that allocates nothing:
 *   one CTA stores its partial of each output plainly and the other adds its
 *   own with a TMA reduce-add, so C receives exactly one rounding of the two
 *   partials.  Nothing else is allocated per call (gemm_ex_noalloc allocates
 *   nothing at all).
 *   Errors: every entry point returns GEMM_OK (0) or a negative gemm_status_t;
 *   argument errors launch nothing and leave C untouched.
 */
#ifndef SMO_GEMM_H
#define SMO_GEMM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { GEMM_K_MAJOR = 0, GEMM_MN_MAJOR = 1 } gemm_major_t;
typedef enum { GEMM_BF16 = 0, GEMM_F16 = 1, GEMM_F32 = 2, GEMM_E4M3 = 3, GEMM_E5M2 = 4 } gemm_dtype_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_ARG = -1,          /* null pointer, negative size, ld below the row length, bad enum */
    GEMM_ERR_ALIGN = -2,        /* base address / ld / stride breaks the 16-byte rules above */
    GEMM_ERR_UNSUPPORTED = -3,  /* dtype combination, or a size beyond the library's limits */
    GEMM_ERR_LAUNCH = -4,       /* the CUDA launch (or tensor-map encoding) failed */
    GEMM_ERR_TIMEOUT = -5,      /* a bounded wait inside a kernel ran out (reported by gemm_check) */
    GEMM_ERR_CUDA = -6,         /* another CUDA runtime error (see gemm_check) */
    GEMM_ERR_NO_DEVICE = -7     /* no usable sm_103 device / driver entry point */
} gemm_status_t;

/*
 * gemm_bf16: bf16 A and B, fp32 C, one problem.
 * Equivalent to gemm_ex(..., GEMM_BF16, GEMM_F32, 1, 0, 0, 0, stream).
 * a_major, b_major: gemm_major_t.  M, N, K >= 0; M == 0 or N == 0 is a no-op;
 * K == 0 writes C = 0.
 */
int gemm_bf16(const void* A, int64_t lda, int a_major,
              const void* B, int64_t ldb, int b_major,
              void* C, int64_t ldc,
              int64_t M, int64_t N, int64_t K, void* stream);

/*
 * gemm_ex: general entry point.
 * in_dtype : GEMM_BF16, GEMM_F16, GEMM_E4M3 or GEMM_E5M2 (A and B share it;
 *            FP8 operands are one byte per element, so lda / ldb / strides
 *            must be multiples of 16 elements).
 * out_dtype: GEMM_F32, GEMM_BF16 or GEMM_F16 (fp32 accumulator rounded to
 *            nearest-even on output).
 * batch >= 1 independent problems; strideA/B/C are ignored when batch == 1.
 * Limits (else GEMM_ERR_UNSUPPORTED): M, N, K and batch below 2^31; lda, ldb
 * and ldc below 2^32 elements; each batch stride below 2^40 bytes (the
 * tensor-memory-access unit's stride limit).
 */
int gemm_ex(const void* A, int64_t lda, int a_major,
            const void* B, int64_t ldb, int b_major,
            void* C, int64_t ldc,
            int64_t M, int64_t N, int64_t K,
            int in_dtype, int out_dtype,
            int64_t batch, int64_t strideA, int64_t strideB, int64_t strideC,
            void* stream);

/*
 * gemm_check: synchronises `stream`, then reports the first error since the
 * previous gemm_check on this device: GEMM_ERR_TIMEOUT if a kernel's bounded
 * wait ran out (the kernel then returned early and C is incomplete),
 * GEMM_ERR_CUDA for a CUDA error, else GEMM_OK.  Clears the device error word.
 */
int gemm_check(void* stream);

/* Human-readable name of a gemm_status_t value (static string, never NULL). */
const char* gemm_status_string(int status);

/*
 * gemm_set_timeout_ns: budget of every bounded wait inside the kernels, in
 * nanoseconds of the GPU's global timer (default 2e9).  Values <= 0 restore the
 * default.  Applies to launches made after the call.  Returns the old value.
 */
int64_t gemm_set_timeout_ns(int64_t ns);

/*
 * gemm_plan_describe: host-only.  Writes into buf (NUL-terminated, at most
 * buflen bytes) a JSON description of the plan gemm_ex would use for these
 * arguments on a GPU with num_sms multiprocessors: tile shape, pipeline depth,
 * tensor-map boxes, tcgen05 instruction and shared-memory descriptors, the
 * planner's F2 matrices of every shared-memory layout, its own layout checks
 * and the shared-memory addresses the epilogue stores issue.  No GPU needed.
 * Returns the length the full text needs (excluding the NUL), or a negative
 * gemm_status_t if the arguments are invalid.
 */
int64_t gemm_plan_describe(int64_t M, int64_t N, int64_t K, int a_major, int b_major,
                           int in_dtype, int out_dtype, int64_t batch, int num_sms,
                           char* buf, size_t buflen);

/*
 * gemm_debug_inject_stall: test hook.  When on != 0, the next launches skip the
 * producer's first tensor-memory-accelerator load, so the consumer's bounded
 * wait on that stage can never complete: the kernel times out (after the
 * gemm_set_timeout_ns budget), sets GEMM_ERR_TIMEOUT and returns cleanly.
 * Returns the previous setting.
 */
int gemm_debug_inject_stall(int on);

/*
 * gemm_ex_noalloc: gemm_ex for callers that cannot allocate device memory.
 * None of the source pages describes such an entry point; it exists for
 * users of this library, not for the method.
 *
 * Who needs it: callers whose device memory is owned entirely by a pool or
 * arena allocator (framework caching allocators, inference runtimes that hand
 * a plugin a fixed workspace and forbid other allocations), and callers that
 * must not allocate once they are running (latency-critical serving loops,
 * where cudaMalloc may synchronise the device).  gemm_ex allocates one 4-byte
 * error word per device on its first launch there; this entry point allocates
 * nothing: its kernel's scratch (the same error word) lives in a file-scope
 * device array of 256 bytes (64 words, word 0 used), which every GPU that
 * loads the library holds until the process exits.
 *
 * Arguments, layouts, ownership and return codes are those of gemm_ex.  Sizes:
 * the scratch needed is one word for every problem size the library accepts;
 * dimensions or batch >= 2^31 are rejected with GEMM_ERR_UNSUPPORTED.
 * Set-up: the first call on a device (made with that device current) resolves
 * the array's device address once (cudaGetSymbolAddress); make that first call
 * before any stream capture.
 * Calls no cudaMalloc, cudaFree or other allocating routine.
 * Every call shares the array.  Its error word starts at zero on each device
 * and is written only when a kernel's bounded wait runs out (first writer
 * wins); it keeps that code, across later calls, until gemm_check_noalloc
 * reads and clears it.  gemm_check does not read it.  Calls that overlap on
 * the GPU race on the shared word: a reported timeout cannot be attributed to
 * one of them, and C of each of them may be incomplete.
 */
int gemm_ex_noalloc(const void* A, int64_t lda, int a_major,
                    const void* B, int64_t ldb, int b_major,
                    void* C, int64_t ldc,
                    int64_t M, int64_t N, int64_t K,
                    int in_dtype, int out_dtype,
                    int64_t batch, int64_t strideA, int64_t strideB, int64_t strideC,
                    void* stream);

/*
 * gemm_check_noalloc: the error report of gemm_ex_noalloc, itself allocating
 * nothing.  None of the source pages describes it; it belongs to the
 * allocation-free entry point above.  Synchronises `stream`, then reads the
 * static error word: GEMM_ERR_TIMEOUT if a gemm_ex_noalloc kernel's bounded
 * wait ran out since the previous gemm_check_noalloc on this device (that
 * kernel returned early and its C is incomplete; the word is cleared),
 * GEMM_ERR_CUDA for a CUDA error, else GEMM_OK.  Reads and clears with
 * synchronous cudaMemcpy / cudaMemset of the 4-byte word: call it outside
 * stream capture.  Like gemm_ex_noalloc, its first call on a device resolves
 * the array's address.
 */
int gemm_check_noalloc(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SMO_GEMM_H */
