/*
 * A plain C99 user of the library's C ABI (include/fp8gemm.h), with no
 * Python and no C++: fp32 operands generated on the host, quantised on the
 * device to E4M3 with power-of-two 1x32 block scales (fp8g_quantize), one
 * block-scaled GEMM with a bf16 output (fp8_gemm_blockscaled), the device
 * status word read back (fp8_gemm_status).  It writes M, N, K, the fp32
 * operands and C (as fp32) to the file named on the command line, for the
 * test to compare with the oracle.
 *
 *   abi_gemm M N K out.bin        exit 0 on FP8G_OK everywhere
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "fp8gemm.h"

/* Numerical Recipes' LCG; the operands need only be deterministic. */
static float next_value(uint32_t *s) {
    *s = *s * 1664525u + 1013904223u;
    return ((float)(*s >> 8) / 16777216.0f * 2.0f - 1.0f) * 4.0f;
}

#define CHECK_CUDA(x)                                                               \
    do {                                                                            \
        cudaError_t e_ = (x);                                                       \
        if (e_ != cudaSuccess) {                                                    \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));               \
            return 3;                                                               \
        }                                                                           \
    } while (0)

#define CHECK_FP8G(x)                                                               \
    do {                                                                            \
        fp8g_status s_ = (x);                                                       \
        if (s_ != FP8G_OK) {                                                        \
            fprintf(stderr, "%s: %s\n", #x, fp8g_status_string(s_));               \
            return 4;                                                               \
        }                                                                           \
    } while (0)

int main(int argc, char **argv) {
    if (argc != 5) {
        fprintf(stderr, "usage: %s M N K out.bin\n", argv[0]);
        return 2;
    }
    const int64_t M = atoll(argv[1]), N = atoll(argv[2]), K = atoll(argv[3]);
    if (M < 1 || N < 1 || K < 32 || K % 32 != 0) return 2;
    float *a = (float *)malloc((size_t)(M * K) * sizeof(float));
    float *b = (float *)malloc((size_t)(N * K) * sizeof(float));
    float *c = (float *)malloc((size_t)(M * N) * sizeof(float));
    uint16_t *c16 = (uint16_t *)malloc((size_t)(M * N) * sizeof(uint16_t));
    if (!a || !b || !c || !c16) return 3;
    uint32_t seed = 20261203u;
    for (int64_t i = 0; i < M * K; ++i) a[i] = next_value(&seed);
    for (int64_t i = 0; i < N * K; ++i) b[i] = next_value(&seed) * 0.25f;

    float *da, *db, *dsa, *dsb;
    uint8_t *dqa, *dqb;
    void *dc;
    CHECK_CUDA(cudaMalloc((void **)&da, (size_t)(M * K) * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void **)&db, (size_t)(N * K) * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void **)&dqa, (size_t)(M * K)));
    CHECK_CUDA(cudaMalloc((void **)&dqb, (size_t)(N * K)));
    CHECK_CUDA(cudaMalloc((void **)&dsa, (size_t)(M * (K / 32)) * sizeof(float)));
    CHECK_CUDA(cudaMalloc((void **)&dsb, (size_t)(N * (K / 32)) * sizeof(float)));
    CHECK_CUDA(cudaMalloc(&dc, (size_t)(M * N) * sizeof(uint16_t)));
    CHECK_CUDA(cudaMemcpy(da, a, (size_t)(M * K) * sizeof(float), cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(db, b, (size_t)(N * K) * sizeof(float), cudaMemcpyHostToDevice));

    cudaStream_t stream;
    CHECK_CUDA(cudaStreamCreate(&stream));
    CHECK_FP8G(fp8g_quantize(da, M, K, 32, FP8G_E4M3, dqa, dsa, stream));
    CHECK_FP8G(fp8g_quantize(db, N, K, 32, FP8G_E4M3, dqb, dsb, stream));
    CHECK_FP8G(fp8_gemm_blockscaled(dqa, dqb, dsa, dsb, dc, FP8G_OUT_BF16, M, N, K, stream));
    int32_t detail = 0;
    CHECK_FP8G(fp8_gemm_status(stream, &detail));
    CHECK_CUDA(cudaMemcpy(c16, dc, (size_t)(M * N) * sizeof(uint16_t), cudaMemcpyDeviceToHost));
    for (int64_t i = 0; i < M * N; ++i) {
        const uint32_t bits = (uint32_t)c16[i] << 16;  /* bf16 -> fp32, exact */
        memcpy(&c[i], &bits, sizeof bits);
    }

    FILE *f = fopen(argv[4], "wb");
    if (!f) return 5;
    const int64_t dims[3] = {M, N, K};
    fwrite(dims, sizeof dims, 1, f);
    fwrite(a, sizeof(float), (size_t)(M * K), f);
    fwrite(b, sizeof(float), (size_t)(N * K), f);
    fwrite(c, sizeof(float), (size_t)(M * N), f);
    fclose(f);
    printf("library %d: %s\n", fp8g_version(), fp8g_status_string(FP8G_OK));

    cudaStreamDestroy(stream);
    cudaFree(da);
    cudaFree(db);
    cudaFree(dqa);
    cudaFree(dqb);
    cudaFree(dsa);
    cudaFree(dsb);
    cudaFree(dc);
    free(a);
    free(b);
    free(c);
    free(c16);
    fp8g_shutdown();
    return 0;
}
