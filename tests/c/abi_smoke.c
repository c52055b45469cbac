/*
 * C-only check of the library's C ABI (include/tiled_gemm.h): no Python.
 *
 * Fills A (M x K) and B (K x N) with small integers in BF16, multiplies them
 * on the GPU through gemm (FP32 out), gemm_ex (BF16 out), gemm_general
 * (C = 2 A^T B + C with A stored K x M), gemm_ex_kernel with the single-tile
 * kernel and gemm_ex_host_ws (host buffers in and out), and compares every
 * element with a plain integer loop on the host: the products are exact, so
 * equality is required.  Exit status 0 on success; 1 on a mismatch; 2 on an API error;
 * 77 when no CUDA device is present.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "tiled_gemm.h"

static uint16_t bf16_of_int(int v)
{
    /* small integers are exact in BF16: the top 16 bits of the FP32 value */
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

#define CHECK(call)                                                                   \
    do {                                                                              \
        int rc_ = (int)(call);                                                        \
        if (rc_ != 0) {                                                               \
            fprintf(stderr, "%s failed: %d (%s)\n", #call, rc_, gemm_error_string(rc_)); \
            return 2;                                                                 \
        }                                                                             \
    } while (0)

#define CUDA_CHECK(call)                                                               \
    do {                                                                               \
        cudaError_t e_ = (call);                                                       \
        if (e_ != cudaSuccess) {                                                       \
            fprintf(stderr, "%s failed: %s\n", #call, cudaGetErrorString(e_));         \
            return 2;                                                                  \
        }                                                                              \
    } while (0)

int main(void)
{
    const int64_t M = 300, N = 264, K = 520; /* several tiles, ragged in every dimension */
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
        fprintf(stderr, "no CUDA device\n");
        return 77;
    }
    int *ai = malloc(sizeof(int) * M * K), *bi = malloc(sizeof(int) * K * N);
    uint16_t *a = malloc(2 * M * K), *at = malloc(2 * M * K), *b = malloc(2 * K * N);
    float *c32 = malloc(4 * M * N), *cin = malloc(4 * M * N);
    uint16_t *c16 = malloc(2 * M * N);
    int64_t *ref = malloc(sizeof(int64_t) * M * N);
    if (!ai || !bi || !a || !at || !b || !c32 || !cin || !c16 || !ref)
        return 2;
    uint32_t seed = 12345u;
    for (int64_t i = 0; i < M * K; ++i) {
        seed = seed * 1664525u + 1013904223u;
        ai[i] = (int)(seed >> 28) - 8;
    }
    for (int64_t i = 0; i < K * N; ++i) {
        seed = seed * 1664525u + 1013904223u;
        bi[i] = (int)(seed >> 28) - 8;
    }
    for (int64_t i = 0; i < M; ++i)
        for (int64_t k = 0; k < K; ++k) {
            a[i * K + k] = bf16_of_int(ai[i * K + k]);
            at[k * M + i] = a[i * K + k];
        }
    for (int64_t i = 0; i < K * N; ++i)
        b[i] = bf16_of_int(bi[i]);
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            int64_t s = 0;
            for (int64_t k = 0; k < K; ++k)
                s += (int64_t)ai[i * K + k] * bi[k * N + j];
            ref[i * N + j] = s;
            cin[i * N + j] = (float)((i + j) % 7 - 3);
        }

    void *dA, *dAt, *dB, *dC;
    CUDA_CHECK(cudaMalloc(&dA, 2 * M * K));
    CUDA_CHECK(cudaMalloc(&dAt, 2 * M * K));
    CUDA_CHECK(cudaMalloc(&dB, 2 * K * N));
    CUDA_CHECK(cudaMalloc(&dC, 4 * M * N));
    CUDA_CHECK(cudaMemcpy(dA, a, 2 * M * K, cudaMemcpyHostToDevice));
    CUDA_CHECK(cudaMemcpy(dAt, at, 2 * M * K, cudaMemcpyHostToDevice));
    CUDA_CHECK(cudaMemcpy(dB, b, 2 * K * N, cudaMemcpyHostToDevice));

    int bad = 0;
    /* gemm: FP32 accumulate, C written in the accumulator type */
    CHECK(gemm(dA, dB, dC, M, N, K, GEMM_BF16, GEMM_F32, NULL));
    CHECK(gemm_device_status(NULL));
    CUDA_CHECK(cudaMemcpy(c32, dC, 4 * M * N, cudaMemcpyDeviceToHost));
    for (int64_t i = 0; i < M * N; ++i)
        bad += c32[i] != (float)ref[i];
    /* gemm_ex: BF16 output; the exact sum rounded to nearest-even BF16 */
    CHECK(gemm_ex(dA, dB, dC, M, N, K, GEMM_BF16, GEMM_F32, GEMM_BF16, NULL));
    CHECK(gemm_device_status(NULL));
    CUDA_CHECK(cudaMemcpy(c16, dC, 2 * M * N, cudaMemcpyDeviceToHost));
    for (int64_t i = 0; i < M * N; ++i) {
        const float want = (float)ref[i];
        uint32_t u;
        memcpy(&u, &want, sizeof u);
        const uint32_t r = u + 0x7fffu + ((u >> 16) & 1u); /* nearest-even to BF16 (finite values) */
        bad += c16[i] != (uint16_t)(r >> 16);
    }
    /* gemm_general: C = 2 op(A) B + C_in, op(A) = the transpose of A stored
       K x M, i.e. the same M x K matrix as above */
    CUDA_CHECK(cudaMemcpy(dC, cin, 4 * M * N, cudaMemcpyHostToDevice));
    CHECK(gemm_general(dAt, dB, dC, M, N, K, GEMM_OP_T, GEMM_OP_N, 2.0f, 1.0f, GEMM_BF16, GEMM_F32,
                       GEMM_F32, GEMM_KERNEL_AUTO, NULL));
    CHECK(gemm_device_status(NULL));
    CUDA_CHECK(cudaMemcpy(c32, dC, 4 * M * N, cudaMemcpyDeviceToHost));
    for (int64_t i = 0; i < M * N; ++i)
        bad += c32[i] != (float)(2 * ref[i]) + cin[i];
    /* the single-tile kernel, forced */
    CHECK(gemm_ex_kernel(dA, dB, dC, M, N, K, GEMM_BF16, GEMM_F32, GEMM_F32, GEMM_KERNEL_TC_SMALL,
                         NULL));
    CHECK(gemm_device_status(NULL));
    CUDA_CHECK(cudaMemcpy(c32, dC, 4 * M * N, cudaMemcpyDeviceToHost));
    for (int64_t i = 0; i < M * N; ++i)
        bad += c32[i] != (float)ref[i];
    /* the latency-path SIMT kernel, forced */
    CHECK(gemm_ex_kernel(dA, dB, dC, M, N, K, GEMM_BF16, GEMM_F32, GEMM_F32,
                         GEMM_KERNEL_TILE16, NULL));
    CHECK(gemm_device_status(NULL));
    CUDA_CHECK(cudaMemcpy(c32, dC, 4 * M * N, cudaMemcpyDeviceToHost));
    for (int64_t i = 0; i < M * N; ++i)
        bad += c32[i] != (float)ref[i];
    /* host buffers in and out, through the workspace form of the host path */
    {
        const size_t ws_bytes = gemm_workspace_size(M, N, K);
        void* ws = NULL;
        CUDA_CHECK(cudaMalloc(&ws, ws_bytes > 0 ? ws_bytes : 16));
        memset(c32, 0, 4 * M * N);
        CHECK(gemm_ex_host_ws(a, b, c32, M, N, K, GEMM_BF16, GEMM_F32, GEMM_F32, dA, dB, dC, ws,
                              ws_bytes, NULL));
        CUDA_CHECK(cudaDeviceSynchronize());
        CHECK(gemm_device_status(NULL));
        for (int64_t i = 0; i < M * N; ++i)
            bad += c32[i] != (float)ref[i];
        cudaFree(ws);
    }
    if (gemm_host_panel_rows(M) != M || gemm_host_panel_rows(8192) != 1024)
        bad += 1;
    /* argument errors come back as codes */
    if (gemm(dA, dB, NULL, M, N, K, GEMM_BF16, GEMM_F32, NULL) != GEMM_ERR_INVALID_VALUE)
        bad += 1;
    if (gemm(dA, dB, dC, GEMM_MAX_DIM + 1, N, K, GEMM_BF16, GEMM_F32, NULL) != GEMM_ERR_INVALID_VALUE)
        bad += 1;

    cudaFree(dA);
    cudaFree(dAt);
    cudaFree(dB);
    cudaFree(dC);
    free(ai);
    free(bi);
    free(a);
    free(at);
    free(b);
    free(c32);
    free(cin);
    free(c16);
    free(ref);
    printf("%s: %d mismatches\n", bad ? "FAIL" : "ok", bad);
    return bad ? 1 : 0;
}
