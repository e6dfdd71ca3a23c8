/* Uses the library through its C ABI alone (no Python): fp32 FFMA and bf16
 * tensor-core GEMM + bias + ReLU, and the staged copy, on device buffers the
 * program allocates itself.  Writes the results to the file named by argv[1]
 * (the test compares them with the oracle) and prints "ok" when every call
 * and the status check succeeded. */
#include <cuda_runtime.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "gbr.h"

#define CHECK_CUDA(x) do { cudaError_t e_ = (x); if (e_ != cudaSuccess) { \
    fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_)); return 1; } } while (0)
#define CHECK_GBR(x) do { int r_ = (x); if (r_ != GBR_OK) { \
    fprintf(stderr, "%s: %d %s\n", #x, r_, gbr_last_error()); return 1; } } while (0)

static unsigned short to_bf16(float f) {   /* round to nearest even */
    unsigned int u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (unsigned short)(u >> 16);
}

int main(int argc, char** argv) {
    if (argc < 2) return 2;
    const int M = 300, N = 264, K = 200;
    float *hA = malloc(sizeof(float) * M * K), *hB = malloc(sizeof(float) * K * N);
    float *hbias = malloc(sizeof(float) * N), *hC = malloc(sizeof(float) * M * N);
    unsigned short *hAb = malloc(2 * (size_t)M * K), *hBb = malloc(2 * (size_t)K * N);
    unsigned short *hCb = malloc(2 * (size_t)M * N);
    unsigned int seed = 12345u;
    for (int i = 0; i < M * K; ++i) {
        seed = seed * 1664525u + 1013904223u;
        hA[i] = (float)((seed >> 9) % 17) - 8.0f;
        hAb[i] = to_bf16(hA[i]);
    }
    for (int i = 0; i < K * N; ++i) {
        seed = seed * 1664525u + 1013904223u;
        hB[i] = ((float)((seed >> 9) % 13) - 6.0f) * 0.25f;
        hBb[i] = to_bf16(hB[i]);
    }
    for (int i = 0; i < N; ++i) hbias[i] = (float)(i % 7) - 3.0f;

    float *dA, *dB, *dbias, *dC, *dsrc, *ddst;
    void *dAb, *dBb, *dCb;
    CHECK_CUDA(cudaMalloc((void**)&dA, sizeof(float) * M * K));
    CHECK_CUDA(cudaMalloc((void**)&dB, sizeof(float) * K * N));
    CHECK_CUDA(cudaMalloc((void**)&dbias, sizeof(float) * N));
    CHECK_CUDA(cudaMalloc((void**)&dC, sizeof(float) * M * N));
    CHECK_CUDA(cudaMalloc(&dAb, 2 * (size_t)M * K));
    CHECK_CUDA(cudaMalloc(&dBb, 2 * (size_t)K * N));
    CHECK_CUDA(cudaMalloc(&dCb, 2 * (size_t)M * N));
    CHECK_CUDA(cudaMalloc((void**)&dsrc, sizeof(float) * M * K));
    CHECK_CUDA(cudaMalloc((void**)&ddst, sizeof(float) * M * K));
    CHECK_CUDA(cudaMemcpy(dA, hA, sizeof(float) * M * K, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dB, hB, sizeof(float) * K * N, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dbias, hbias, sizeof(float) * N, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dAb, hAb, 2 * (size_t)M * K, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dBb, hBb, 2 * (size_t)K * N, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dsrc, hA, sizeof(float) * M * K, cudaMemcpyHostToDevice));

    cudaStream_t st;
    CHECK_CUDA(cudaStreamCreate(&st));
    CHECK_GBR(gemm_bias_relu(dA, dB, dbias, dC, M, N, K, GBR_F32_FFMA, 3, st));
    CHECK_GBR(gemm_bias_relu(dAb, dBb, dbias, dCb, M, N, K, GBR_BF16, 3, st));
    CHECK_GBR(staged_copy(dsrc, ddst, M, K, 128, 64, 2, st));
    CHECK_GBR(gbr_device_status(st));
    CHECK_CUDA(cudaMemcpy(hC, dC, sizeof(float) * M * N, cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(hCb, dCb, 2 * (size_t)M * N, cudaMemcpyDeviceToHost));
    float* hcopy = malloc(sizeof(float) * M * K);
    CHECK_CUDA(cudaMemcpy(hcopy, ddst, sizeof(float) * M * K, cudaMemcpyDeviceToHost));

    FILE* f = fopen(argv[1], "wb");
    if (!f) return 3;
    fwrite(hA, sizeof(float), (size_t)M * K, f);
    fwrite(hB, sizeof(float), (size_t)K * N, f);
    fwrite(hbias, sizeof(float), N, f);
    fwrite(hC, sizeof(float), (size_t)M * N, f);
    fwrite(hCb, 2, (size_t)M * N, f);
    fwrite(hcopy, sizeof(float), (size_t)M * K, f);
    fclose(f);
    printf("ok\n");
    return 0;
}
