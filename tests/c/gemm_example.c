/* A plain C99 program using the library through include/tcgemm.h and the
 * CUDA runtime's C API only (no Python, no torch): D = relu(A @ B + bias) for
 * a ragged 200 x 136 x 96 problem with small integer inputs, fp32 D, checked
 * element for element against a direct sum (exact: every partial sum is an
 * integer below 2^24).  Built and run by tests/test_c_example_gpu.py. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "tcgemm.h"

static uint16_t to_bf16(float x) {   /* exact for the small integers used here */
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    return (uint16_t)(u >> 16);
}

#define CUDA_OK(call)                                                                  \
    do {                                                                               \
        cudaError_t e_ = (call);                                                       \
        if (e_ != cudaSuccess) {                                                       \
            fprintf(stderr, "%s: %s\n", #call, cudaGetErrorString(e_));                \
            return 2;                                                                  \
        }                                                                              \
    } while (0)

int main(void) {
    enum { M = 200, N = 136, K = 96 };
    const int lda = K, ldb = K, ldd = N;                 /* A row-major, B column-major, D row-major */
    static float a[M * K], b[N * K], bias[N], ref[M * N], got[M * N];
    static uint16_t ha[M * K], hb[N * K], hbias[N];
    unsigned s = 12345u;
    for (int i = 0; i < M * K; ++i) { s = s * 1103515245u + 12345u; a[i] = (float)((int)((s >> 16) % 9) - 4); ha[i] = to_bf16(a[i]); }
    for (int i = 0; i < N * K; ++i) { s = s * 1103515245u + 12345u; b[i] = (float)((int)((s >> 16) % 9) - 4); hb[i] = to_bf16(b[i]); }
    for (int j = 0; j < N; ++j) { bias[j] = (float)(j % 7 - 3); hbias[j] = to_bf16(bias[j]); }
    for (int i = 0; i < M; ++i)
        for (int j = 0; j < N; ++j) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) acc += a[i * lda + k] * b[j * ldb + k];
            acc += bias[j];
            ref[i * N + j] = acc > 0.0f ? acc : 0.0f;
        }

    void *dA, *dB, *dBias, *dD, *ws;
    CUDA_OK(cudaMalloc(&dA, sizeof ha));
    CUDA_OK(cudaMalloc(&dB, sizeof hb));
    CUDA_OK(cudaMalloc(&dBias, sizeof hbias));
    CUDA_OK(cudaMalloc(&dD, sizeof got));
    CUDA_OK(cudaMemcpy(dA, ha, sizeof ha, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dB, hb, sizeof hb, cudaMemcpyHostToDevice));
    CUDA_OK(cudaMemcpy(dBias, hbias, sizeof hbias, cudaMemcpyHostToDevice));
    const size_t ws_bytes = tcg_workspace_size(M, N, K, TCG_BF16);
    CUDA_OK(cudaMalloc(&ws, ws_bytes));
    if (tcg_workspace_init(ws, ws_bytes, NULL) != TCG_OK) return 3;

    tcg_epilogue epi = {dBias, TCG_BF16, TCG_ACT_RELU};
    tcg_scales sc = {1.0f, 1.0f, NULL, NULL, NULL, NULL};
    tcg_status st = tcg_gemm(M, N, K, 1.0f, dA, lda, TCG_ROW, dB, ldb, TCG_COL, 0.0f, NULL, 0, TCG_BF16, dD, ldd,
                             TCG_F32, epi, TCG_BF16, sc, ws, ws_bytes, NULL);
    if (st != TCG_OK) { fprintf(stderr, "tcg_gemm: %d (%s)\n", (int)st, tcg_last_error()); return 4; }
    st = tcg_device_status(ws, NULL);
    if (st != TCG_OK) { fprintf(stderr, "device status %d\n", (int)st); return 5; }
    CUDA_OK(cudaMemcpy(got, dD, sizeof got, cudaMemcpyDeviceToHost));
    int bad = 0;
    for (int i = 0; i < M * N; ++i)
        if (got[i] != ref[i]) {
            if (bad < 5) fprintf(stderr, "D[%d][%d] = %g, expected %g\n", i / N, i % N, got[i], ref[i]);
            ++bad;
        }
    cudaFree(dA); cudaFree(dB); cudaFree(dBias); cudaFree(dD); cudaFree(ws);
    if (bad) { fprintf(stderr, "%d of %d elements differ\n", bad, M * N); return 6; }
    printf("gemm_example ok: %dx%dx%d relu(A@B + bias), every element exact\n", M, N, K);
    return 0;
}
