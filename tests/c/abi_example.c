/*
 * A plain-C user of libsmo_gemm.so: no Python, no torch.  It multiplies small
 * integer matrices (exact in bf16 and in fp32 accumulation) through the C ABI
 * of smo_gemm.h, in both B orientations and through both entry points, and
 * compares every element with a triple loop.  Prints "ABI OK" and exits 0 on
 * success.  Test program; built and run by tests/test_c_abi.py.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "smo_gemm.h"

static uint16_t bf16_of_int(int v) {
    /* small integers are exact in bf16: the top 16 bits of the fp32 pattern */
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

#define CK(x)                                                                          \
    do {                                                                               \
        cudaError_t e_ = (x);                                                          \
        if (e_ != cudaSuccess) {                                                       \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));                   \
            return 2;                                                                  \
        }                                                                              \
    } while (0)

static int run(int M, int N, int K, int b_major, int use_ex) {
    /* leading dimensions padded to 16 bytes (the TMA rule of the header) */
    const int lda = (K + 7) / 8 * 8;                                   /* A K-major: M x K */
    const int ldb = ((b_major == GEMM_MN_MAJOR ? N : K) + 7) / 8 * 8;  /* B N-major: K x N; K-major: N x K */
    const int ldc = (N + 3) / 4 * 4;                                   /* fp32 C */
    uint16_t* hA = malloc(sizeof(uint16_t) * (size_t)M * lda);
    uint16_t* hB = malloc(sizeof(uint16_t) * (size_t)(b_major == GEMM_MN_MAJOR ? K : N) * ldb);
    float* hC = malloc(sizeof(float) * (size_t)M * ldc);
    int* a = malloc(sizeof(int) * (size_t)M * K);
    int* b = malloc(sizeof(int) * (size_t)K * N);
    if (!hA || !hB || !hC || !a || !b) return 2;
    unsigned s = 12345u + (unsigned)(M * 7 + N * 13 + K * 17 + b_major);
    for (int i = 0; i < M * K; ++i) { s = s * 1103515245u + 12345u; a[i] = (int)((s >> 16) % 9u) - 4; }
    for (int i = 0; i < K * N; ++i) { s = s * 1103515245u + 12345u; b[i] = (int)((s >> 16) % 9u) - 4; }
    for (int m = 0; m < M; ++m)
        for (int k = 0; k < K; ++k) hA[(size_t)m * lda + k] = bf16_of_int(a[m * K + k]);
    for (int k = 0; k < K; ++k)
        for (int n = 0; n < N; ++n) {
            size_t at = b_major == GEMM_MN_MAJOR ? (size_t)k * ldb + n : (size_t)n * ldb + k;
            hB[at] = bf16_of_int(b[k * N + n]);
        }
    void *dA, *dB, *dC;
    CK(cudaMalloc(&dA, sizeof(uint16_t) * (size_t)M * lda));
    CK(cudaMalloc(&dB, sizeof(uint16_t) * (size_t)(b_major == GEMM_MN_MAJOR ? K : N) * ldb));
    CK(cudaMalloc(&dC, sizeof(float) * (size_t)M * ldc));
    CK(cudaMemcpy(dA, hA, sizeof(uint16_t) * (size_t)M * lda, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(dB, hB, sizeof(uint16_t) * (size_t)(b_major == GEMM_MN_MAJOR ? K : N) * ldb,
                  cudaMemcpyHostToDevice));
    cudaStream_t st;
    CK(cudaStreamCreate(&st));
    int rc = use_ex ? gemm_ex(dA, lda, GEMM_K_MAJOR, dB, ldb, b_major, dC, ldc, M, N, K, GEMM_BF16, GEMM_F32, 1, 0,
                              0, 0, (void*)st)
                    : gemm_bf16(dA, lda, GEMM_K_MAJOR, dB, ldb, b_major, dC, ldc, M, N, K, (void*)st);
    if (rc != GEMM_OK) {
        fprintf(stderr, "launch: %s\n", gemm_status_string(rc));
        return 1;
    }
    rc = gemm_check((void*)st);
    if (rc != GEMM_OK) {
        fprintf(stderr, "check: %s\n", gemm_status_string(rc));
        return 1;
    }
    CK(cudaMemcpy(hC, dC, sizeof(float) * (size_t)M * ldc, cudaMemcpyDeviceToHost));
    long bad = 0;
    for (int m = 0; m < M; ++m)
        for (int n = 0; n < N; ++n) {
            long ref = 0;
            for (int k = 0; k < K; ++k) ref += (long)a[m * K + k] * b[k * N + n];
            if (hC[(size_t)m * ldc + n] != (float)ref) ++bad;
        }
    cudaStreamDestroy(st);
    cudaFree(dA); cudaFree(dB); cudaFree(dC);
    free(hA); free(hB); free(hC); free(a); free(b);
    if (bad) {
        fprintf(stderr, "%dx%dx%d b_major=%d ex=%d: %ld mismatches\n", M, N, K, b_major, use_ex, bad);
        return 1;
    }
    return 0;
}

int main(void) {
    /* an argument error is reported without a launch */
    if (gemm_bf16(NULL, 8, 0, NULL, 8, 1, NULL, 8, 8, 8, 8, NULL) != GEMM_ERR_ARG) {
        fprintf(stderr, "null pointers not rejected\n");
        return 1;
    }
    const int shapes[][3] = {{1, 1, 1}, {100, 72, 40}, {300, 520, 777}, {1024, 1024, 1024}};
    for (int i = 0; i < 4; ++i)
        for (int bm = 0; bm < 2; ++bm)
            for (int ex = 0; ex < 2; ++ex) {
                int r = run(shapes[i][0], shapes[i][1], shapes[i][2], bm, ex);
                if (r) return r;
            }
    printf("ABI OK\n");
    return 0;
}
