/*
 * A plain C11 caller of the library's C ABI (include/gemm_epi.h): what a program with no
 * Python or C++ in it does to run the fused GEMM.  It plans, executes and frees
 * RELU_AUX_BIAS plans on device buffers from the CUDA runtime, and checks the results with
 * exact integer arithmetic: every input is an integer in {-1, 0, 1} (bias in {-2, ..., 2}),
 * so every sum has |value| <= k + 2 < 256, exact in the fp32 accumulator and in bf16.  It
 * also checks the shape and alignment errors the header documents.  The FFN block
 * (gemm_epi_ffn_*) runs in each of its modes and without allocation; its GELU makes the
 * hidden activation non-integer, so that check is in double against the stated bound
 * max |got - want| / (|want| + 1) <= 2e-2 (bf16).
 *
 * Build: cc -std=c11 -I include -I <cuda>/include tests/c_caller.c
 *           -L <dir of libgemmepi.so> -lgemmepi -L <cuda>/lib64 -lcudart
 * Run:   c_caller          (prints "ok" and exits 0 when every check passes)
 */
#include <cuda_runtime_api.h>
#include <math.h>
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

/* bf16 bits -> double, and double -> bf16 bits rounded to nearest even (finite values) */
static double double_of_bf16(uint16_t h)
{
    const uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof(f));
    return (double)f;
}

static uint16_t bf16_round(double x)
{
    const float f = (float)x;
    uint32_t u;
    memcpy(&u, &f, sizeof(u));
    u += 0x7FFFu + ((u >> 16) & 1u);
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

/* GELU(x) = x * Phi(x), Phi the standard normal distribution function */
static double gelu(double x) { return 0.5 * x * erfc(-x / sqrt(2.0)); }

/*
 * The FFN block Y = GELU(X.W1 + b1).W2 + b2 + R, t x d, hidden width f, bf16, run with
 * LAUNCHES = `launches` (-1: the call without allocation).  X, W1, W2 are in {-1, 0, 1},
 * b1 in {-2, ..., 2}, so X.W1 + b1 is an exact integer; the reference rounds GELU of it to
 * bf16 as the stored H is, then forms Y in double.
 */
static int run_ffn_case(int64_t t, int64_t d, int64_t f, int launches, cudaStream_t stream)
{
    uint16_t* hX = malloc(sizeof(uint16_t) * (size_t)(t * d));
    uint16_t* hW1 = malloc(sizeof(uint16_t) * (size_t)(d * f));
    uint16_t* hb1 = malloc(sizeof(uint16_t) * (size_t)f);
    uint16_t* hW2 = malloc(sizeof(uint16_t) * (size_t)(f * d));
    uint16_t* hb2 = malloc(sizeof(uint16_t) * (size_t)d);
    uint16_t* hR = malloc(sizeof(uint16_t) * (size_t)(t * d));
    uint16_t* hY = malloc(sizeof(uint16_t) * (size_t)(t * d));
    double* H = malloc(sizeof(double) * (size_t)f);
    EXPECT(hX && hW1 && hb1 && hW2 && hb2 && hR && hY && H, "host allocation failed");
    for (int64_t i = 0; i < t * d; ++i) hX[i] = bf16_of_int(draw(-1, 1));
    for (int64_t i = 0; i < d * f; ++i) hW1[i] = bf16_of_int(draw(-1, 1));
    for (int64_t j = 0; j < f; ++j) hb1[j] = bf16_of_int(draw(-2, 2));
    for (int64_t i = 0; i < f * d; ++i) hW2[i] = bf16_of_int(draw(-1, 1));
    for (int64_t j = 0; j < d; ++j) hb2[j] = bf16_of_int(draw(-2, 2));
    for (int64_t i = 0; i < t * d; ++i) hR[i] = bf16_of_int(draw(-3, 3));

    void *dX, *dW1, *db1, *dW2, *db2, *dR, *dY;
    CHECK_CUDA(cudaMalloc(&dX, sizeof(uint16_t) * (size_t)(t * d)));
    CHECK_CUDA(cudaMalloc(&dW1, sizeof(uint16_t) * (size_t)(d * f)));
    CHECK_CUDA(cudaMalloc(&db1, sizeof(uint16_t) * (size_t)f));
    CHECK_CUDA(cudaMalloc(&dW2, sizeof(uint16_t) * (size_t)(f * d)));
    CHECK_CUDA(cudaMalloc(&db2, sizeof(uint16_t) * (size_t)d));
    CHECK_CUDA(cudaMalloc(&dR, sizeof(uint16_t) * (size_t)(t * d)));
    CHECK_CUDA(cudaMalloc(&dY, sizeof(uint16_t) * (size_t)(t * d)));
    CHECK_CUDA(cudaMemcpy(dX, hX, sizeof(uint16_t) * (size_t)(t * d), cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dW1, hW1, sizeof(uint16_t) * (size_t)(d * f), cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(db1, hb1, sizeof(uint16_t) * (size_t)f, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dW2, hW2, sizeof(uint16_t) * (size_t)(f * d), cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(db2, hb2, sizeof(uint16_t) * (size_t)d, cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemcpy(dR, hR, sizeof(uint16_t) * (size_t)(t * d), cudaMemcpyHostToDevice));
    CHECK_CUDA(cudaMemset(dY, 0xFF, sizeof(uint16_t) * (size_t)(t * d)));

    gemm_epi_status st;
    if (launches < 0) {
        st = gemm_epi_ffn_execute_noalloc(t, d, f, GEMM_EPI_BF16, dX, dW1, db1, dW2, db2, dR, dY,
                                          stream);
        EXPECT(st == GEMM_EPI_OK, "ffn noalloc: %s", gemm_epi_status_string(st));
        CHECK_CUDA(cudaStreamSynchronize(stream));
        printf("ffn noalloc\n");
    } else {
        gemm_epi_ffn_plan_t plan = NULL;
        st = gemm_epi_ffn_plan(&plan, t, d, f, GEMM_EPI_BF16);
        EXPECT(st == GEMM_EPI_OK, "ffn plan: %s", gemm_epi_status_string(st));
        st = gemm_epi_ffn_set_option(plan, GEMM_EPI_FFN_OPT_LAUNCHES, launches);
        EXPECT(st == GEMM_EPI_OK, "ffn LAUNCHES=%d: %s", launches, gemm_epi_status_string(st));
        st = gemm_epi_ffn_execute(plan, dX, dW1, db1, dW2, db2, dR, dY, stream);
        EXPECT(st == GEMM_EPI_OK, "ffn execute: %s", gemm_epi_status_string(st));
        st = gemm_epi_ffn_sync_status(plan, stream);
        EXPECT(st == GEMM_EPI_OK, "ffn device status: %s", gemm_epi_status_string(st));
        printf("ffn %s\n", gemm_epi_ffn_plan_describe(plan));
        EXPECT(gemm_epi_ffn_free(plan) == GEMM_EPI_OK, "ffn free");
    }
    CHECK_CUDA(cudaMemcpy(hY, dY, sizeof(uint16_t) * (size_t)(t * d), cudaMemcpyDeviceToHost));
    double worst = 0.0;
    for (int64_t i = 0; i < t; ++i) {
        for (int64_t c = 0; c < f; ++c) {
            double pre = double_of_bf16(hb1[c]);
            for (int64_t kk = 0; kk < d; ++kk)
                pre += double_of_bf16(hX[i * d + kk]) * double_of_bf16(hW1[kk * f + c]);
            H[c] = double_of_bf16(bf16_round(gelu(pre)));
        }
        for (int64_t j = 0; j < d; ++j) {
            double y = double_of_bf16(hb2[j]) + double_of_bf16(hR[i * d + j]);
            for (int64_t c = 0; c < f; ++c) y += H[c] * double_of_bf16(hW2[c * d + j]);
            const double err = fabs(double_of_bf16(hY[i * d + j]) - y) / (fabs(y) + 1.0);
            if (!(err <= worst)) worst = err; /* a NaN from an unwritten element sticks */
        }
    }
    EXPECT(worst <= 2e-2, "ffn LAUNCHES=%d %lldx%lldx%lld: rel err %g", launches, (long long)t,
           (long long)d, (long long)f, worst);

    cudaFree(dX);
    cudaFree(dW1);
    cudaFree(db1);
    cudaFree(dW2);
    cudaFree(db2);
    cudaFree(dR);
    cudaFree(dY);
    free(hX);
    free(hW1);
    free(hb1);
    free(hW2);
    free(hb2);
    free(hR);
    free(hY);
    free(H);
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
    /* the FFN block: automatic, one launch, two launches, H on chip, no allocation */
    const int ffn_modes[] = {0, 1, 2, 3, -1};
    for (size_t s = 0; s < sizeof(ffn_modes) / sizeof(ffn_modes[0]); ++s)
        if (run_ffn_case(200, 256, 512, ffn_modes[s], stream) != 0) return 1;
    CHECK_CUDA(cudaStreamDestroy(stream));
    printf("ok\n");
    return 0;
}
