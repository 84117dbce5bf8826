/*
 * A plain C11 caller of the library's C ABI (include/gemm_epi.h): what a program with no
 * Python or C++ in it does to run the fused GEMM.  It plans, executes and frees
 * RELU_AUX_BIAS plans on device buffers from the CUDA runtime, and checks the results with
 * exact integer arithmetic: every input is an integer in {-1, 0, 1} (bias in {-2, ..., 2}),
 * so every sum has |value| <= k + 2 < 256, exact in the fp32 accumulator and in bf16.  It
 * also checks the shape and alignment errors the header documents.
 *
 * Build: cc -std=c11 -I include -I <cuda>/include tests/c_caller.c
 *           -L <dir of libgemmepi.so> -lgemmepi -L <cuda>/lib64 -lcudart
 * Run:   c_caller          (prints "ok" and exits 0 when every check passes)
 */
#include <cuda_runtime_api.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "gemm_epi.h"

static uint64_t rng_state = 0x9E3779B97F4A7C15ull;

/* xorshift64*: a small deterministic generator for the test inputs */
static int draw(int lo, int hi)
{
    rng_state ^= rng_state >> 12;
    rng_state ^= rng_state << 25;
    rng_state ^= rng_state >> 27;
    const uint64_t r = (rng_state * 0x2545F4914F6CDD1Dull) >> 33;
    return lo + (int)(r % (uint64_t)(hi - lo + 1));
}

/* bf16 bits of a small integer (|v| <= 256 is exact: the low 16 bits of its float are 0) */
static uint16_t bf16_of_int(int v)
{
    const float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof(u));
    return (uint16_t)(u >> 16);
}

#define CHECK_CUDA(x)                                                                      \
    do {                                                                                   \
        cudaError_t e_ = (x);                                                              \
        if (e_ != cudaSuccess) {                                                           \
            fprintf(stderr, "%s:%d: %s\n", __FILE__, __LINE__, cudaGetErrorString(e_));     \
            return 1;                                                                      \
        }                                                                                  \
    } while (0)

#define EXPECT(cond, ...)                                                                  \
    do {                                                                                   \
        if (!(cond)) {                                                                     \
            fprintf(stderr, __VA_ARGS__);                                                  \
            fputc('\n', stderr);                                                           \
            return 1;                                                                      \
        }                                                                                  \
    } while (0)

/* One RELU_AUX_BIAS problem through plan / execute / sync_status / free. */
static int run_case(int64_t m, int64_t n, int64_t k, cudaStream_t stream)
{
    const int64_t words = gemm_epi_aux_words_per_row(n);
    int* a = malloc(sizeof(int) * (size_t)(m * k));
    int* b = malloc(sizeof(int) * (size_t)(k * n));
    int* bias = malloc(sizeof(int) * (size_t)n);
    uint16_t* hA = malloc(sizeof(uint16_t) * (size_t)(m * k));
    uint16_t* hB = malloc(sizeof(uint16_t) * (size_t)(k * n));
    uint16_t* hbias = malloc(sizeof(uint16_t) * (size_t)n);
    uint16_t* hD = malloc(sizeof(uint16_t) * (size_t)(m * n));
    uint32_t* haux = malloc(sizeof(uint32_t) * (size_t)(m * words));
    EXPECT(a && b && bias && hA && hB && hbias && hD && haux, "host allocation failed");
    for (int64_t i = 0; i < m * k; ++i) hA[i] = bf16_of_int(a[i] = draw(-1, 1));
    for (int64_t i = 0; i < k * n; ++i) hB[i] = bf16_of_int(b[i] = draw(-1, 1));
    for (int64_t j = 0; j < n; ++j) hbias[j] = bf16_of_int(bias[j] = draw(-2, 2));

    void *dA, *dB, *dbias, *dD, *daux;
    CHECK_CUDA(cudaMalloc(&dA, sizeof(uint16_t) * (size_t)(m * k)));
    CHECK_CUDA(cudaMalloc(&dB, sizeof(uint16_t) * (size_t)(k * n)));
    CHECK_CUDA(cudaMalloc(&dbias, sizeof(uint16_t) * (size_t)n));
    CHECK_CUDA(cudaMalloc(&dD, sizeof(uint16_t) * (size_t)(m * n)));
    CHECK_CUDA(cudaMalloc(&daux, sizeof(uint32_t) * (size_t)(m * words)));
    CHECK_CUDA(cudaMemcpy(dA, hA, sizeof(uint16_t) * (size_t)(m * k), cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dB, hB, sizeof(uint16_t) * (size_t)(k * n), cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dbias, hbias, sizeof(uint16_t) * (size_t)n, cudaMemcpyHostToDevice));
    /* poison the outputs: every value and bit must be written */
    CHECK_CUDA(cudaMemset(dD, 0xFF, sizeof(uint16_t) * (size_t)(m * n)));
    CHECK_CUDA(cudaMemset(daux, 0xFF, sizeof(uint32_t) * (size_t)(m * words)));

    gemm_epi_plan_t plan = NULL;
    gemm_epi_status st = gemm_epi_plan(&plan, m, n, k, GEMM_EPI_BF16, GEMM_EPI_RELU_AUX_BIAS,
                                       GEMM_EPI_BIAS_1N);
    EXPECT(st == GEMM_EPI_OK, "plan %lldx%lldx%lld: %s", (long long)m, (long long)n,
           (long long)k, gemm_epi_status_string(st));
    st = gemm_epi_execute(plan, dA, dB, dbias, dD, (uint32_t*)daux, stream);
    EXPECT(st == GEMM_EPI_OK, "execute: %s", gemm_epi_status_string(st));
    st = gemm_epi_sync_status(plan, stream);
    EXPECT(st == GEMM_EPI_OK, "device status: %s", gemm_epi_status_string(st));
    printf("%s\n", gemm_epi_plan_describe(plan));

    /* misaligned D (one element past a 16-byte boundary): refused before any launch */
    st = gemm_epi_execute(plan, dA, dB, dbias, (char*)dD + 2, (uint32_t*)daux, stream);
    EXPECT(st == GEMM_EPI_ERR_MISALIGNED, "misaligned D gave %s", gemm_epi_status_string(st));
    /* RELU_AUX_BIAS without its mask buffer */
    st = gemm_epi_execute(plan, dA, dB, dbias, dD, NULL, stream);
    EXPECT(st == GEMM_EPI_ERR_INVALID_ARG, "missing aux gave %s", gemm_epi_status_string(st));

    CHECK_CUDA(cudaMemcpy(hD, dD, sizeof(uint16_t) * (size_t)(m * n), cudaMemcpyDeviceToHost));
    CHECK_CUDA(cudaMemcpy(haux, daux, sizeof(uint32_t) * (size_t)(m * words),
                          cudaMemcpyDeviceToHost));
    for (int64_t i = 0; i < m; ++i) {
        for (int64_t w = 0; w < words; ++w) {
            uint32_t want = 0;
            for (int64_t j = 32 * w; j < 32 * w + 32 && j < n; ++j) {
                int pre = bias[j];
                for (int64_t t = 0; t < k; ++t) pre += a[i * k + t] * b[t * n + j];
                const int d = pre > 0 ? pre : 0;
                const uint16_t got = hD[i * n + j];
                EXPECT(got == bf16_of_int(d), "D[%lld][%lld] = 0x%04x, want %d", (long long)i,
                       (long long)j, got, d);
                if (pre > 0) want |= 1u << (j - 32 * w);
            }
            EXPECT(haux[i * words + w] == want, "aux[%lld][%lld] = 0x%08x, want 0x%08x",
                   (long long)i, (long long)w, haux[i * words + w], want);
        }
    }

    EXPECT(gemm_epi_free(plan) == GEMM_EPI_OK, "free");
    cudaFree(dA);
    cudaFree(dB);
    cudaFree(dbias);
    cudaFree(dD);
    cudaFree(daux);
    free(a);
    free(b);
    free(bias);
    free(hA);
    free(hB);
    free(hbias);
    free(hD);
    free(haux);
    return 0;
}

int main(void)
{
    /* shape errors are reported at plan time, before any device work */
    gemm_epi_plan_t bad = NULL;
    gemm_epi_status st = gemm_epi_plan(&bad, 64, 12, 64, GEMM_EPI_BF16, GEMM_EPI_BIAS,
                                       GEMM_EPI_BIAS_1N);
    EXPECT(st == GEMM_EPI_ERR_UNSUPPORTED_SHAPE && bad == NULL, "n = 12 gave %s",
           gemm_epi_status_string(st));
    EXPECT(gemm_epi_free(NULL) == GEMM_EPI_OK, "free(NULL)");

    cudaStream_t stream;
    CHECK_CUDA(cudaStreamCreate(&stream));
    /* small-m (K split over a cluster), swapped, single-CTA row tiles with ragged edges,
       CTA pairs */
    const int64_t shapes[][3] = {{16, 264, 72}, {100, 264, 72}, {300, 264, 136}, {2048, 2048, 200}};
    for (size_t s = 0; s < sizeof(shapes) / sizeof(shapes[0]); ++s)
        if (run_case(shapes[s][0], shapes[s][1], shapes[s][2], stream) != 0) return 1;
    CHECK_CUDA(cudaStreamDestroy(stream));
    printf("ok\n");
    return 0;
}
