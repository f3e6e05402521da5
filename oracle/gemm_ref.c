/*
 * Oracle: plain fp64 CPU GEMM and IEEE-754 round-to-nearest-even helpers.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, the smoke check and the bench's CPU
 * baseline leg may load this library.  It shares no code, header, table or
 * constant with the CUDA path: it re-derives everything from the definitions.
 *
 * What it computes (the plain definition of the product the GPU path reaches):
 *   "An Educational GEMM Ladder for Helios GPUs", section "Educational GEMM
 *   Ladder": every rung computes C = A B with A in R^{M x K}, B in R^{K x N},
 *   BF16 inputs.  "Fix LDS vectorization logic ..." (rocMLIR pull 2196),
 *   description: the same product on f16 operands (1500 x 1152 x 896).
 *
 *   C_ref[b][m][n] = sum_{k = 0 .. K-1} A[b][m][k] * B[b][k][n]
 *
 * evaluated in IEEE double with k ascending for every element, no fused
 * multiply-add (build with -ffp-contract=off), from the operand bit patterns
 * the GPU reads (16-bit formats as uint16 arrays, 8-bit formats as uint8
 * arrays).  The loop nest walks n innermost so that each
 * element's partial sum still receives its terms in ascending k; the per-element
 * arithmetic is exactly the dot product above.
 *
 * Operand addressing (the library's convention, stated once):
 *   A K-major : A[b][m][k] at a[b*sa + m*lda + k]
 *   A M-major : A[b][m][k] at a[b*sa + k*lda + m]
 *   B K-major : B[b][k][n] at b[b*sb + n*ldb + k]
 *   B N-major : B[b][k][n] at b[b*sb + k*ldb + n]
 *   C         : C[b][m][n] at c[b*sc + m*ldc + n]
 *
 *   "An Educational GEMM Ladder for Helios GPUs", section "Educational GEMM
 *   Ladder": the matrix units take BF16, FP8, FP6 and FP4 operands; "A Deep
 *   Dive into LDS Optimizations on AMD Instinct MI450 GPUs", Part I: the 8-bit
 *   transposed operand load (ds_load_tr8_b64).  The 8-bit operand product is the
 *   same definition over FP8 inputs.
 *
 * 16-bit formats (IEEE 754-2008 binary16, and bfloat16 = the top half of
 * binary32) and the two 8-bit formats of the OCP 8-bit floating point
 * specification (E4M3: bias 7, no infinities, S.1111.111 is NaN; E5M2: bias 15,
 * IEEE-style infinities and NaNs) are decoded from their bit fields here, and
 * doubles are rounded to
 * binary32 / bfloat16 / binary16 by round-to-nearest, ties-to-even, written
 * from the standard's definition: scale by the quantum of the target binade,
 * round the (exact) quotient to an integer with nearbyint() under the default
 * rounding mode, scale back, overflow to infinity.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_BF16 = 0, ORC_F16 = 1, ORC_F32 = 2, ORC_E4M3 = 3, ORC_E5M2 = 4 };

/* ---- decoding ------------------------------------------------------------ */

/* bfloat16: sign 1 | exponent 8 (bias 127) | fraction 7; same fields as the
 * upper 16 bits of binary32. */
static double bf16_bits_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xFF;
    int f = h & 0x7F;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -126 - 7);                 /* subnormal / zero */
    } else if (e == 0xFF) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(128 + f), e - 127 - 7);      /* 1.f * 2^(e-127) */
    }
    return sign ? -v : v;
}

/* binary16: sign 1 | exponent 5 (bias 15) | fraction 10. */
static double f16_bits_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -14 - 10);
    } else if (e == 0x1F) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 15 - 10);
    }
    return sign ? -v : v;
}

double orc_decode16(uint16_t h, int dtype) {
    return dtype == ORC_BF16 ? bf16_bits_to_f64(h) : f16_bits_to_f64(h);
}

void orc_decode16_array(const uint16_t* h, int64_t n, int dtype, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_decode16(h[i], dtype);
}

/* E4M3: sign 1 | exponent 4 (bias 7) | fraction 3.  Exponent field 0 holds the
 * subnormals f * 2^(1-7-3); the all-ones exponent is an ordinary binade except
 * for fraction 111, the only NaN (no infinities), so the largest value is
 * 1.110b * 2^8 = 448. */
static double e4m3_bits_to_f64(uint8_t h) {
    int sign = (h >> 7) & 1;
    int e = (h >> 3) & 0xF;
    int f = h & 0x7;
    double v;
    if (e == 0xF && f == 0x7) {
        v = NAN;
    } else if (e == 0) {
        v = ldexp((double)f, 1 - 7 - 3);
    } else {
        v = ldexp((double)(8 + f), e - 7 - 3);          /* 1.f * 2^(e-7) */
    }
    return sign ? -v : v;
}

/* E5M2: sign 1 | exponent 5 (bias 15) | fraction 2, with IEEE 754 conventions:
 * exponent 0 is subnormal, all-ones exponent is infinity (fraction 0) or NaN. */
static double e5m2_bits_to_f64(uint8_t h) {
    int sign = (h >> 7) & 1;
    int e = (h >> 2) & 0x1F;
    int f = h & 0x3;
    double v;
    if (e == 0x1F) {
        v = f ? NAN : INFINITY;
    } else if (e == 0) {
        v = ldexp((double)f, 1 - 15 - 2);
    } else {
        v = ldexp((double)(4 + f), e - 15 - 2);         /* 1.f * 2^(e-15) */
    }
    return sign ? -v : v;
}

double orc_decode8(uint8_t h, int dtype) {
    return dtype == ORC_E4M3 ? e4m3_bits_to_f64(h) : e5m2_bits_to_f64(h);
}

void orc_decode8_array(const uint8_t* h, int64_t n, int dtype, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_decode8(h[i], dtype);
}

/* Bytes per operand element of an input format. */
int orc_elem_bytes(int dtype) { return (dtype == ORC_E4M3 || dtype == ORC_E5M2) ? 1 : 2; }

/* Element idx of an operand array of the given input format. */
static inline double operand_at(const void* p, int64_t idx, int dtype) {
    if (dtype == ORC_E4M3 || dtype == ORC_E5M2) return orc_decode8(((const uint8_t*)p)[idx], dtype);
    return orc_decode16(((const uint16_t*)p)[idx], dtype);
}

/* ---- rounding ------------------------------------------------------------ */

/* Round x to the nearest value with p significand bits (p = fraction bits + 1),
 * minimum normal exponent emin and maximum exponent emax (ties to even).
 * Returns +-inf on overflow.  NaN passes through. */
static double round_rne(double x, int p, int emin, int emax) {
    if (x != x || x == 0.0 || isinf(x)) return x;
    int e2;
    (void)frexp(x, &e2);            /* x = f * 2^e2, 0.5 <= |f| < 1 */
    int E = e2 - 1;                 /* x in [2^E, 2^(E+1)) */
    if (E < emin) E = emin;         /* subnormal range shares emin's quantum */
    int qexp = E - (p - 1);         /* quantum (ulp) of that binade */
    double scaled = ldexp(x, -qexp);        /* exact: a power-of-two scaling */
    double r = ldexp(nearbyint(scaled), qexp);
    if (fabs(r) >= ldexp(1.0, emax + 1)) return x > 0 ? INFINITY : -INFINITY;
    return r;
}

double orc_round_f32(double x) { return round_rne(x, 24, -126, 127); }
double orc_round_bf16(double x) { return round_rne(x, 8, -126, 127); }
double orc_round_f16(double x) { return round_rne(x, 11, -14, 15); }

/* Encode an already-representable value to bfloat16 bits. */
static uint16_t bf16_encode_exact(double v) {
    float f = (float)v;             /* exact: v is a bfloat16 value */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

/* Encode an already-representable value to binary16 bits. */
static uint16_t f16_encode_exact(double v) {
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (v != v) return 0x7E00;
    if (isinf(a)) return sign | 0x7C00;
    if (a == 0.0) return sign;
    if (a < ldexp(1.0, -14)) {                          /* subnormal */
        return sign | (uint16_t)(a * ldexp(1.0, 24));
    }
    int e2;
    double f = frexp(a, &e2);                           /* a = f * 2^e2 */
    int E = e2 - 1;
    uint16_t frac = (uint16_t)((f * 2.0 - 1.0) * 1024.0);
    return sign | (uint16_t)((E + 15) << 10) | frac;
}

uint16_t orc_encode16(double x, int dtype) {
    if (dtype == ORC_BF16) return bf16_encode_exact(orc_round_bf16(x));
    return f16_encode_exact(orc_round_f16(x));
}

void orc_round_array(const double* in, int64_t n, int out_dtype, double* out) {
    for (int64_t i = 0; i < n; ++i) {
        double x = in[i];
        out[i] = out_dtype == ORC_F32 ? orc_round_f32(x)
               : out_dtype == ORC_BF16 ? orc_round_bf16(x)
               : orc_round_f16(x);
    }
}

/* ---- the GEMM ------------------------------------------------------------ */

static inline double a_at(const void* a, int dt, int a_mn_major, int64_t lda,
                          int64_t sa, int64_t b, int64_t m, int64_t k) {
    int64_t idx = b * sa + (a_mn_major ? k * lda + m : m * lda + k);
    return operand_at(a, idx, dt);
}

static inline double b_at(const void* bm, int dt, int b_mn_major, int64_t ldb,
                          int64_t sb, int64_t b, int64_t k, int64_t n) {
    int64_t idx = b * sb + (b_mn_major ? k * ldb + n : n * ldb + k);
    return operand_at(bm, idx, dt);
}

/* Full product into a dense fp64 array c[b][m][n] (row-major, ld = N).
 * Returns 0, or -1 if scratch could not be allocated. */
int orc_gemm_f64(const void* a, int64_t lda, int a_mn_major,
                 const void* bmat, int64_t ldb, int b_mn_major,
                 int in_dtype, int64_t M, int64_t N, int64_t K,
                 int64_t batch, int64_t sa, int64_t sb, double* c) {
    int err = 0;
    for (int64_t b = 0; b < batch && !err; ++b) {
        /* Decode this batch entry's B once: bd[k][n]. */
        double* bd = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1) * (size_t)(N > 0 ? N : 1));
        if (!bd) return -1;
        for (int64_t k = 0; k < K; ++k)
            for (int64_t n = 0; n < N; ++n)
                bd[k * N + n] = b_at(bmat, in_dtype, b_mn_major, ldb, sb, b, k, n);
        #pragma omp parallel for schedule(static)
        for (int64_t m = 0; m < M; ++m) {
            double* crow = c + (b * M + m) * N;
            for (int64_t n = 0; n < N; ++n) crow[n] = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double av = a_at(a, in_dtype, a_mn_major, lda, sa, b, m, k);
                const double* brow = bd + k * N;
                for (int64_t n = 0; n < N; ++n) {
                    double t = av * brow[n];        /* rounded product */
                    crow[n] = crow[n] + t;          /* rounded sum, k ascending */
                }
            }
        }
        free(bd);
    }
    return err;
}

/* Selected elements only: out[i] = C_ref[bi[i]][mi[i]][ni[i]], each one a plain
 * dot product with k ascending (used to check full-size GPU results at sampled
 * positions). */
void orc_gemm_f64_sampled(const void* a, int64_t lda, int a_mn_major,
                          const void* bmat, int64_t ldb, int b_mn_major,
                          int in_dtype, int64_t K, int64_t sa, int64_t sb,
                          const int64_t* bi, const int64_t* mi, const int64_t* ni,
                          int64_t count, double* out) {
    #pragma omp parallel for schedule(dynamic, 16)
    for (int64_t i = 0; i < count; ++i) {
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double t = a_at(a, in_dtype, a_mn_major, lda, sa, bi[i], mi[i], k) *
                       b_at(bmat, in_dtype, b_mn_major, ldb, sb, bi[i], k, ni[i]);
            acc = acc + t;
        }
        out[i] = acc;
    }
}

/* Number of OpenMP threads a parallel region would use (reported beside
 * oracle timings). */
int orc_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
