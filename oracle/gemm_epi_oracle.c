/*
 * CPU oracle for the fused GEMM + bias/activation epilogue.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library links, loads or calls this file:
 * only the tests, the smoke check and the benchmark's CPU-baseline leg do.  It shares
 * no code, header, table or constant with the CUDA path.
 *
 * What it computes, step by step, in the order the method is described:
 *
 *   "Fusing bias into cuBLASLt matmul with nvmath-python for PyTorch inference"
 *   (blog.hotdry.top, 2025-09-22), code example and the paragraph on shape constraints:
 *     D[m,n] = A[m,k] . B[k,n] + bias, with bias of shape (m,1) (added to every column)
 *     or (1,n) (added to every row); the BIAS / RELU_BIAS epilogs apply the bias and then
 *     the activation inside the matmul kernel; RELU_AUX_BIAS also emits a mask that the
 *     backward pass needs; the limitations paragraph lists Tanh among the predefined
 *     epilogs (TANH_BIAS: tanh(A.B + bias)).
 *   "Operator fusion in model inference, from LayerNorm to residual connections"
 *   (wmrh.cn/news/429806), section 1 and its flowchart: the FFN chain
 *     matmul -> bias -> GELU -> matmul -> bias, and (section 3) the residual added to the
 *     output of the op that precedes it; section 2: LayerNorm,
 *     y = (x - mu) / sqrt(sigma^2 + eps) * gamma + beta over each row, with the mean and
 *     the variance taken in two passes as the section's code does, optionally followed by
 *     a residual add (the section's LayerNorm-and-residual function).
 *
 * Readings where the pages are silent (each is listed with its reason in the design notes):
 *   - inputs are 16-bit (IEEE binary16 or bfloat16); every element is decoded exactly to
 *     double, and all arithmetic after that is double;
 *   - GELU is the erf form, x * Phi(x) = 0.5 * x * erfc(-x / sqrt(2)) (the same function as
 *     0.5 * x * (1 + erf(x / sqrt(2))), written with erfc so that it keeps its relative
 *     accuracy for negative x);
 *   - the aux mask bit for (i, j) is [pre(i, j) > 0] (strict), stored as bit (j mod 32) of
 *     32-bit word floor(j / 32) of row i, rows ceil(n / 32) words long, pad bits 0;
 *   - ReLU output is +0 whenever pre <= 0;
 *   - the FFN's hidden activation H is stored as bfloat16 rounded to nearest-even;
 *   - GELU_AUX_BIAS keeps the pre-activation for backward (the caller gets it as "pre");
 *   - the backward epilogues multiply A.B by the ReLU mask (DRELU) or by GELU'(pre) of the
 *     stored 16-bit pre-activation (DGELU), and reduce the product over the dimension the
 *     bias was broadcast along to give the bias gradient.
 *
 * Rounding to 16 bits (used only for the FFN's stored H) is written from the IEEE 754
 * definitions of the two formats, with round-to-nearest, ties-to-even.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -shared -fPIC (no fast-math), so the results
 * are the same on x86-64 and aarch64 hosts.
 */
#define _GNU_SOURCE
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F16 = 0, OR_BF16 = 1 };
enum {
    OR_EPI_BIAS = 0,
    OR_EPI_RELU_BIAS = 1,
    OR_EPI_GELU_BIAS = 2,
    OR_EPI_RELU_AUX_BIAS = 3,
    OR_EPI_BIAS_RESIDUAL = 4,
    OR_EPI_NONE = 5,
    OR_EPI_TANH_BIAS = 6,
    OR_EPI_GELU_AUX_BIAS = 7
};
enum { OR_BWD_DRELU = 0, OR_BWD_DGELU = 1 };
enum { OR_BIAS_M1 = 0, OR_BIAS_1N = 1 };

/* ---- 16-bit decode, from the format definitions ------------------------------------- */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_decode_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24);                 /* subnormal: frac * 2^(1-15-10) */
    else if (expo == 0x1f)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(frac + 1024), expo - 25);  /* (1 + frac/2^10) * 2^(expo-15) */
    return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_decode_bf16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 7) & 0xff;
    int frac = h & 0x7f;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -133);                /* subnormal: frac * 2^(1-127-7) */
    else if (expo == 0xff)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(frac + 128), expo - 134);  /* (1 + frac/2^7) * 2^(expo-127) */
    return sign ? -v : v;
}

static double decode(int dtype, uint16_t h)
{
    return dtype == OR_BF16 ? oracle_decode_bf16(h) : oracle_decode_f16(h);
}

/*
 * The 8-bit floating-point format E4M3 (the "FN" variant of the OCP 8-bit formats): 1 sign
 * bit, 4 exponent bits with bias 7, 3 fraction bits; no infinities; S.1111.111 is NaN, so the
 * largest finite magnitude is 1.75 * 2^8 = 448; exponent field 0 holds the subnormals
 * frac/8 * 2^-6.
 */
double oracle_decode_e4m3(uint8_t h)
{
    const int sign = (h >> 7) & 1;
    const int expo = (h >> 3) & 15;
    const int frac = h & 7;
    double v;
    if (expo == 15 && frac == 7)
        v = NAN;
    else if (expo == 0)
        v = ldexp((double)frac, -9);                  /* frac/8 * 2^(1-7) */
    else
        v = ldexp((double)(frac + 8), expo - 10);     /* (1 + frac/8) * 2^(expo-7) */
    return sign ? -v : v;
}

/* ---- 16-bit encode, round to nearest, ties to even ---------------------------------- */

/* A binary format with `fbits` fraction bits, `ebits` exponent bits and bias 2^(ebits-1)-1. */
static uint16_t encode_rne(double x, int fbits, int ebits)
{
    const int bias = (1 << (ebits - 1)) - 1;
    const int emin = 1 - bias;                       /* exponent of the smallest normal */
    const uint16_t sign = signbit(x) ? (uint16_t)(1u << (fbits + ebits)) : 0;
    const uint16_t inf_bits = (uint16_t)(((1u << ebits) - 1) << fbits);
    double a = fabs(x);
    if (isnan(x))
        return (uint16_t)(inf_bits | (1u << (fbits - 1)));   /* a quiet NaN */
    if (a == 0.0)
        return sign;
    if (isinf(x))
        return (uint16_t)(sign | inf_bits);

    int e2;
    frexp(a, &e2);                                   /* a = f * 2^e2 with f in [0.5, 1) */
    int lead = e2 - 1;                               /* exponent of the leading bit */
    if (lead < emin)
        lead = emin;                                 /* subnormal range: fixed quantum */
    /* Spacing of representable numbers at this exponent: 2^(lead - fbits). */
    double scaled = ldexp(a, fbits - lead);          /* exact: scaling by a power of two */
    double q = nearbyint(scaled);                    /* default mode: ties to even */
    double v = ldexp(q, lead - fbits);               /* the rounded magnitude */
    if (v >= ldexp(1.0, bias + 1))                   /* at or above 2^(emax+1): overflow */
        return (uint16_t)(sign | inf_bits);
    if (v < ldexp(1.0, emin)) {                      /* subnormal (or rounded up to min normal) */
        uint32_t f = (uint32_t)ldexp(v, fbits - emin);
        return (uint16_t)(sign | f);                 /* f == 2^fbits encodes the min normal */
    }
    int e3;
    frexp(v, &e3);
    int E = e3 - 1;
    uint32_t frac = (uint32_t)(ldexp(v, fbits - E) - ldexp(1.0, fbits));
    return (uint16_t)(sign | ((uint32_t)(E + bias) << fbits) | frac);
}

uint16_t oracle_encode_f16(double x) { return encode_rne(x, 10, 5); }
uint16_t oracle_encode_bf16(double x) { return encode_rne(x, 7, 8); }

void oracle_encode_array(int dtype, const double* x, int64_t count, uint16_t* out)
{
    for (int64_t i = 0; i < count; ++i)
        out[i] = dtype == OR_BF16 ? oracle_encode_bf16(x[i]) : oracle_encode_f16(x[i]);
}

void oracle_decode_array(int dtype, const uint16_t* h, int64_t count, double* out)
{
    for (int64_t i = 0; i < count; ++i)
        out[i] = decode(dtype, h[i]);
}

/* ---- the activation functions ------------------------------------------------------- */

/* GELU, erf form: x * Phi(x), Phi the standard normal CDF = 0.5 * erfc(-x / sqrt 2). */
double oracle_gelu(double x)
{
    return x * 0.5 * erfc(-x / sqrt(2.0));
}

static double activation(int epilog, double pre)
{
    switch (epilog) {
    case OR_EPI_RELU_BIAS:
    case OR_EPI_RELU_AUX_BIAS:
        return pre > 0.0 ? pre : 0.0;                /* +0 for every pre <= 0 */
    case OR_EPI_GELU_BIAS:
    case OR_EPI_GELU_AUX_BIAS:
        return oracle_gelu(pre);
    case OR_EPI_TANH_BIAS:
        return tanh(pre);
    default:
        return pre;                                  /* BIAS, BIAS_RESIDUAL, NONE */
    }
}

/* ---- the GEMM + epilogue ------------------------------------------------------------ */

/*
 * For every (rows[r], cols[c]) pair:
 *   pre[r][c] = sum over kk of A[rows[r]][kk] * B[kk][cols[c]]  +  beta(rows[r], cols[c])
 *   D[r][c]   = act(pre[r][c])            (+ residual[rows[r]][cols[c]] for BIAS_RESIDUAL)
 * with beta(i, j) = bias[i] for the (m,1) layout, bias[j] for (1,n), and no bias for NONE.
 * A is m x k, B is k x n, residual m x n, all row-major 16-bit of `dtype`.
 * pre (may be NULL) and D are nrows x ncols doubles.  The sum runs over kk = 0..k-1 in
 * order.  Returns 0, or -1 on an argument error or an allocation failure.
 */
int oracle_gemm_epi(int64_t m, int64_t n, int64_t k, int dtype, int epilog, int bias_layout,
                    const uint16_t* A, const uint16_t* B, const uint16_t* bias,
                    const uint16_t* residual,
                    const int64_t* rows, int64_t nrows, const int64_t* cols, int64_t ncols,
                    double* pre, double* D)
{
    if (m < 0 || n < 0 || k < 0 || nrows < 0 || ncols < 0 || !rows || !cols || !D)
        return -1;
    if (epilog < OR_EPI_BIAS || epilog > OR_EPI_GELU_AUX_BIAS)
        return -1;
    if (epilog != OR_EPI_NONE && !bias)
        return -1;
    if (epilog == OR_EPI_BIAS_RESIDUAL && !residual)
        return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= m) return -1;
    for (int64_t c = 0; c < ncols; ++c)
        if (cols[c] < 0 || cols[c] >= n) return -1;
    if (nrows == 0 || ncols == 0)
        return 0;

    /* The selected columns of B, decoded once: Bsel[kk][c] = B[kk][cols[c]]. */
    double* Bsel = (double*)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1) * (size_t)ncols);
    if (!Bsel)
        return -1;
    for (int64_t kk = 0; kk < k; ++kk)
        for (int64_t c = 0; c < ncols; ++c)
            Bsel[kk * ncols + c] = decode(dtype, B[kk * n + cols[c]]);

    int failed = 0;
#pragma omp parallel
    {
        double* acc = (double*)malloc(sizeof(double) * (size_t)ncols);
        if (!acc) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < nrows; ++r) {
            if (!acc) continue;
            const int64_t i = rows[r];
            for (int64_t c = 0; c < ncols; ++c)
                acc[c] = 0.0;
            for (int64_t kk = 0; kk < k; ++kk) {
                const double a = decode(dtype, A[i * k + kk]);
                const double* brow = Bsel + kk * ncols;
                for (int64_t c = 0; c < ncols; ++c)
                    acc[c] += a * brow[c];
            }
            for (int64_t c = 0; c < ncols; ++c) {
                const int64_t j = cols[c];
                double beta = 0.0;
                if (epilog != OR_EPI_NONE)
                    beta = decode(dtype, bias_layout == OR_BIAS_M1 ? bias[i] : bias[j]);
                const double p = acc[c] + beta;
                double d = activation(epilog, p);
                if (epilog == OR_EPI_BIAS_RESIDUAL)
                    d = p + decode(dtype, residual[i * n + j]);
                if (pre)
                    pre[r * ncols + c] = p;
                D[r * ncols + c] = d;
            }
        }
        free(acc);
    }
    free(Bsel);
    return failed ? -1 : 0;
}

/*
 * The aux ReLU mask of full rows: words is rows x ceil(n/32) uint32; bit (j mod 32) of word
 * floor(j/32) in row r is [pre[r][j] > 0]; bits for j >= n are 0.  pre is rows x n.
 */
void oracle_aux_pack(const double* pre, int64_t nrows, int64_t n, uint32_t* words)
{
    const int64_t ldw = (n + 31) / 32;
    for (int64_t r = 0; r < nrows; ++r) {
        for (int64_t w = 0; w < ldw; ++w)
            words[r * ldw + w] = 0u;
        for (int64_t j = 0; j < n; ++j)
            if (pre[r * n + j] > 0.0)
                words[r * ldw + j / 32] |= 1u << (j % 32);
    }
}

/*
 * The FFN block, all of it (full rows and columns):
 *   H = round_bf16(GELU(X . W1 + b1))       X: t x d, W1: d x f, b1: f        (stored 16-bit)
 *   Y = H . W2 + b2 + R                     W2: f x d, b2: d, R: t x d
 * H_bits receives the stored hidden activation (t x f, 16-bit of `dtype`), Hpre the
 * unrounded GELU output in double (may be NULL), Y the output in double (t x d).
 */
int oracle_ffn(int64_t t, int64_t d, int64_t f, int dtype,
               const uint16_t* X, const uint16_t* W1, const uint16_t* b1,
               const uint16_t* W2, const uint16_t* b2, const uint16_t* R,
               uint16_t* H_bits, double* H_exact, double* Y)
{
    int rc = -1;
    int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)(t > 0 ? t : 1));
    int64_t* cf = (int64_t*)malloc(sizeof(int64_t) * (size_t)(f > 0 ? f : 1));
    int64_t* cd = (int64_t*)malloc(sizeof(int64_t) * (size_t)(d > 0 ? d : 1));
    double* H = (double*)malloc(sizeof(double) * (size_t)(t * f > 0 ? t * f : 1));
    if (!rows || !cf || !cd || !H)
        goto out;
    for (int64_t i = 0; i < t; ++i) rows[i] = i;
    for (int64_t j = 0; j < f; ++j) cf[j] = j;
    for (int64_t j = 0; j < d; ++j) cd[j] = j;

    /* GEMM 1: bias (1,f), then GELU. */
    if (oracle_gemm_epi(t, f, d, dtype, OR_EPI_GELU_BIAS, OR_BIAS_1N, X, W1, b1, NULL,
                        rows, t, cf, f, NULL, H) != 0)
        goto out;
    if (H_exact)
        memcpy(H_exact, H, sizeof(double) * (size_t)(t * f));
    oracle_encode_array(dtype, H, t * f, H_bits);   /* H is stored in 16 bits */

    /* GEMM 2 on the stored H: bias (1,d), then the residual. */
    if (oracle_gemm_epi(t, d, f, dtype, OR_EPI_BIAS_RESIDUAL, OR_BIAS_1N, H_bits, W2, b2, R,
                        rows, t, cd, d, NULL, Y) != 0)
        goto out;
    rc = 0;
out:
    free(rows);
    free(cf);
    free(cd);
    free(H);
    return rc;
}

/*
 * LayerNorm of the rows of X (t x d): mu = sum(x) / d, var = sum((x - mu)^2) / d (the
 * biased variance, second pass over the centred row), y = (x - mu) / sqrt(var + eps) *
 * gamma + beta (+ residual when it is not NULL).  Y (t x d) in double; stats (may be NULL)
 * receives mu and 1 / sqrt(var + eps) per row.
 */
int oracle_layernorm(int64_t t, int64_t d, int dtype, const uint16_t* X, const uint16_t* residual,
                     const uint16_t* gamma, const uint16_t* beta, double eps, double* Y,
                     double* stats)
{
    if (t < 0 || d < 0 || !X || !gamma || !beta || !Y || !(eps >= 0.0)) return -1;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < t; ++i) {
        double sum = 0.0;
        for (int64_t j = 0; j < d; ++j)
            sum += decode(dtype, X[i * d + j]);
        const double mu = d > 0 ? sum / (double)d : 0.0;
        double ss = 0.0;
        for (int64_t j = 0; j < d; ++j) {
            const double c = decode(dtype, X[i * d + j]) - mu;
            ss += c * c;
        }
        const double var = d > 0 ? ss / (double)d : 0.0;
        const double rstd = 1.0 / sqrt(var + eps);
        if (stats) {
            stats[2 * i] = mu;
            stats[2 * i + 1] = rstd;
        }
        for (int64_t j = 0; j < d; ++j) {
            double y = (decode(dtype, X[i * d + j]) - mu) * rstd * decode(dtype, gamma[j]) +
                       decode(dtype, beta[j]);
            if (residual)
                y += decode(dtype, residual[i * d + j]);
            Y[i * d + j] = y;
        }
    }
    return 0;
}

/*
 * A GEMM on layer-normalised rows, the first GEMM of a pre-LayerNorm FFN block:
 *   D = GELU(LayerNorm(A) . W + b)      A: m x k, gamma, beta: k, W: k x n, b: n
 * LayerNorm(A) is kept in double (never rounded: it is an intermediate).
 */
int oracle_ln_gemm_gelu(int64_t m, int64_t n, int64_t k, int dtype, const uint16_t* A,
                        const uint16_t* gamma, const uint16_t* beta, double eps,
                        const uint16_t* W, const uint16_t* b, double* D)
{
    if (m < 0 || n < 0 || k < 0 || !A || !W || !b || !D) return -1;
    double* An = (double*)malloc(sizeof(double) * (size_t)(m * k > 0 ? m * k : 1));
    double* Wd = (double*)malloc(sizeof(double) * (size_t)(k * n > 0 ? k * n : 1));
    if (!An || !Wd) {
        free(An);
        free(Wd);
        return -1;
    }
    int rc = oracle_layernorm(m, k, dtype, A, NULL, gamma, beta, eps, An, NULL);
    if (rc == 0) {
        for (int64_t i = 0; i < k * n; ++i)
            Wd[i] = decode(dtype, W[i]);
#pragma omp parallel for schedule(dynamic, 1)
        for (int64_t i = 0; i < m; ++i) {
            for (int64_t j = 0; j < n; ++j)
                D[i * n + j] = 0.0;
            for (int64_t q = 0; q < k; ++q) {
                const double xq = An[i * k + q];
                for (int64_t j = 0; j < n; ++j)
                    D[i * n + j] += xq * Wd[q * n + j];
            }
            for (int64_t j = 0; j < n; ++j)
                D[i * n + j] = oracle_gelu(D[i * n + j] + decode(dtype, b[j]));
        }
    }
    free(An);
    free(Wd);
    return rc;
}

/*
 * The pre-LayerNorm FFN block: H = round(GELU(LayerNorm(X) . W1 + b1)) stored in 16 bits,
 * Y = H . W2 + b2 + R (the residual is usually X itself).  As oracle_ffn otherwise.
 */
int oracle_ln_ffn(int64_t t, int64_t d, int64_t f, int dtype, const uint16_t* X,
                  const uint16_t* gamma, const uint16_t* beta, double eps, const uint16_t* W1,
                  const uint16_t* b1, const uint16_t* W2, const uint16_t* b2, const uint16_t* R,
                  uint16_t* H_bits, double* H_exact, double* Y)
{
    int rc = -1;
    int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)(t > 0 ? t : 1));
    int64_t* cd = (int64_t*)malloc(sizeof(int64_t) * (size_t)(d > 0 ? d : 1));
    double* H = (double*)malloc(sizeof(double) * (size_t)(t * f > 0 ? t * f : 1));
    if (!rows || !cd || !H)
        goto out;
    for (int64_t i = 0; i < t; ++i) rows[i] = i;
    for (int64_t j = 0; j < d; ++j) cd[j] = j;
    if (oracle_ln_gemm_gelu(t, f, d, dtype, X, gamma, beta, eps, W1, b1, H) != 0)
        goto out;
    if (H_exact)
        memcpy(H_exact, H, sizeof(double) * (size_t)(t * f));
    oracle_encode_array(dtype, H, t * f, H_bits);
    if (oracle_gemm_epi(t, d, f, dtype, OR_EPI_BIAS_RESIDUAL, OR_BIAS_1N, H_bits, W2, b2, R,
                        rows, t, cd, d, NULL, Y) != 0)
        goto out;
    rc = 0;
out:
    free(rows);
    free(cd);
    free(H);
    return rc;
}

/*
 * FP8 inputs with per-tensor scales (the page names FP8 among the types the fused matmul
 * supports): D = epi(sa * sb * (A . B) + bias), A: m x k E4M3 row-major, Bt: n x k E4M3
 * row-major (B transposed: both operands contiguous along k), bias (m,1) or (1,n) and the
 * residual in bfloat16, sa and sb the dequantisation scales.  pre (may be NULL) receives
 * sa * sb * (A . B) + bias, D the output (both m x n, double).  Forward epilogs only.
 */
int oracle_gemm_epi_fp8(int64_t m, int64_t n, int64_t k, int epilog, int bias_layout,
                        const uint8_t* A, const uint8_t* Bt, double sa, double sb,
                        const uint16_t* bias, const uint16_t* residual, double* pre, double* D)
{
    if (m < 0 || n < 0 || k < 0 || !D) return -1;
    if (epilog < OR_EPI_BIAS || epilog > OR_EPI_GELU_AUX_BIAS) return -1;
    if (epilog != OR_EPI_NONE && !bias) return -1;
    if (epilog == OR_EPI_BIAS_RESIDUAL && !residual) return -1;
    double* Bd = (double*)malloc(sizeof(double) * (size_t)(n * k > 0 ? n * k : 1));
    if (!Bd) return -1;
    for (int64_t i = 0; i < n * k; ++i)
        Bd[i] = oracle_decode_e4m3(Bt[i]);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < m; ++i) {
        for (int64_t j = 0; j < n; ++j) {
            double acc = 0.0;
            for (int64_t q = 0; q < k; ++q)
                acc += oracle_decode_e4m3(A[i * k + q]) * Bd[j * k + q];
            const int64_t bi = bias_layout == OR_BIAS_M1 ? i : j;  /* the bias element */
            const double beta = epilog != OR_EPI_NONE ? decode(OR_BF16, bias[bi]) : 0.0;
            const double p = sa * sb * acc + beta;
            double d = activation(epilog, p);
            if (epilog == OR_EPI_BIAS_RESIDUAL)
                d = p + decode(OR_BF16, residual[i * n + j]);
            if (pre)
                pre[i * n + j] = p;
            D[i * n + j] = d;
        }
    }
    free(Bd);
    return 0;
}

/* GELU'(x) = Phi(x) + x phi(x): the derivative of x Phi(x), phi the standard normal density. */
double oracle_gelu_grad(double x)
{
    const double phi = exp(-0.5 * x * x) / sqrt(2.0 * M_PI);
    return 0.5 * erfc(-x / sqrt(2.0)) + x * phi;
}

/*
 * Backward epilogues.  With g(i, j) = bit (j mod 32) of word floor(j/32) of row i of `mask`
 * (kind DRELU) or g(i, j) = GELU'(pre[i][j]) of the stored 16-bit pre-activation (kind
 * DGELU):
 *   dpre[i][j] = (A.B)[i][j] * g(i, j)            (D, m x n doubles)
 *   dbias[j]   = sum over i of dpre[i][j]         (bias layout (1,n): n doubles)
 *   dbias[i]   = sum over j of dpre[i][j]         (bias layout (m,1): m doubles)
 * The products A.B come from oracle_gemm_epi with no epilog.  Returns 0, or -1.
 */
int oracle_gemm_bwd(int64_t m, int64_t n, int64_t k, int dtype, int kind, int bias_layout,
                    const uint16_t* A, const uint16_t* B, const uint32_t* mask,
                    const uint16_t* pre, double* D, double* dbias)
{
    if (m < 0 || n < 0 || k < 0 || !D || !dbias) return -1;
    if (kind == OR_BWD_DRELU ? !mask : (kind == OR_BWD_DGELU ? !pre : 1)) return -1;
    int rc = -1;
    int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)(m > 0 ? m : 1));
    int64_t* cols = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n > 0 ? n : 1));
    if (!rows || !cols) goto out;
    for (int64_t i = 0; i < m; ++i) rows[i] = i;
    for (int64_t j = 0; j < n; ++j) cols[j] = j;
    if (oracle_gemm_epi(m, n, k, dtype, OR_EPI_NONE, bias_layout, A, B, NULL, NULL, rows, m, cols,
                        n, NULL, D) != 0)
        goto out;
    const int64_t ldw = (n + 31) / 32;
    for (int64_t i = 0; i < m; ++i)
        for (int64_t j = 0; j < n; ++j) {
            double g;
            if (kind == OR_BWD_DRELU)
                g = (mask[i * ldw + j / 32] >> (j % 32)) & 1u ? 1.0 : 0.0;
            else
                g = oracle_gelu_grad(decode(dtype, pre[i * n + j]));
            D[i * n + j] *= g;
        }
    const int64_t nb = bias_layout == OR_BIAS_M1 ? m : n;
    for (int64_t b = 0; b < nb; ++b)
        dbias[b] = 0.0;
    for (int64_t i = 0; i < m; ++i)
        for (int64_t j = 0; j < n; ++j)
            dbias[bias_layout == OR_BIAS_M1 ? i : j] += D[i * n + j];
    rc = 0;
out:
    free(rows);
    free(cols);
    return rc;
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
