// LayerNorm calls of the C ABI ("Operator fusion in model inference, from LayerNorm to
// residual connections" (wmrh.cn/news/429806), section 2): the one-pass LayerNorm
// (+ residual), the per-row statistics and the weight fold of the form folded into a GEMM.
#include "plan.h"

using namespace gemm_epi;
using namespace gemm_epi_impl;

namespace {

bool ln_shape_ok(int64_t t, int64_t d)
{
    const int64_t kMax = (1ll << 31) - 1;
    return t >= 0 && d >= 8 && d % 8 == 0 && t <= kMax && d <= kMax && t * d <= (1ll << 40);
}

}  // namespace

extern "C" {

gemm_epi_status gemm_epi_layernorm(int64_t t, int64_t d, gemm_epi_dtype dtype, const void* X,
                                   const void* residual, const void* gamma, const void* beta,
                                   float eps, void* Y, cudaStream_t stream)
{
    if (dtype != GEMM_EPI_F16 && dtype != GEMM_EPI_BF16) return GEMM_EPI_ERR_INVALID_ARG;
    if (!ln_shape_ok(t, d)) return GEMM_EPI_ERR_UNSUPPORTED_SHAPE;
    if (!(eps >= 0.0f) || !(eps < 1e30f)) return GEMM_EPI_ERR_INVALID_ARG;
    if (t == 0) return GEMM_EPI_OK;
    if (!X || !gamma || !beta || !Y) return GEMM_EPI_ERR_INVALID_ARG;
    if (!aligned(X, 16) || !aligned(Y, 16) || (residual && !aligned(residual, 16)) ||
        !aligned(gamma, 2) || !aligned(beta, 2))
        return GEMM_EPI_ERR_MISALIGNED;
    int sms = 0;
    gemm_epi_status st = current_device(&sms);
    if (st != GEMM_EPI_OK) return st;
    return layernorm_launch(X, residual, gamma, beta, Y, static_cast<int>(t), static_cast<int>(d),
                            dtype == GEMM_EPI_BF16 ? 1 : 0, eps, sms, stream) == cudaSuccess
               ? GEMM_EPI_OK
               : GEMM_EPI_ERR_LAUNCH;
}

gemm_epi_status gemm_epi_layernorm_stats(int64_t t, int64_t d, gemm_epi_dtype dtype,
                                         const void* X, float eps, float* stats,
                                         cudaStream_t stream)
{
    if (dtype != GEMM_EPI_F16 && dtype != GEMM_EPI_BF16) return GEMM_EPI_ERR_INVALID_ARG;
    if (!ln_shape_ok(t, d)) return GEMM_EPI_ERR_UNSUPPORTED_SHAPE;
    if (!(eps >= 0.0f) || !(eps < 1e30f)) return GEMM_EPI_ERR_INVALID_ARG;
    if (t == 0) return GEMM_EPI_OK;
    if (!X || !stats) return GEMM_EPI_ERR_INVALID_ARG;
    if (!aligned(X, 16) || !aligned(stats, 8)) return GEMM_EPI_ERR_MISALIGNED;
    int sms = 0;
    gemm_epi_status st = current_device(&sms);
    if (st != GEMM_EPI_OK) return st;
    return layernorm_stats_launch(X, static_cast<int>(t), static_cast<int>(d),
                                  dtype == GEMM_EPI_BF16 ? 1 : 0, eps, stats, sms, stream) ==
                   cudaSuccess
               ? GEMM_EPI_OK
               : GEMM_EPI_ERR_LAUNCH;
}

gemm_epi_status gemm_epi_layernorm_fold(int64_t d, int64_t f, gemm_epi_dtype dtype,
                                        const void* gamma, const void* beta, const void* W,
                                        const void* b, void* W_folded, float* colsum,
                                        float* bias_folded, cudaStream_t stream)
{
    if (dtype != GEMM_EPI_F16 && dtype != GEMM_EPI_BF16) return GEMM_EPI_ERR_INVALID_ARG;
    if (!ln_shape_ok(f, d) || f % 8 != 0) return GEMM_EPI_ERR_UNSUPPORTED_SHAPE;
    if (f == 0) return GEMM_EPI_OK;
    if (!gamma || !beta || !W || !b || !W_folded || !colsum || !bias_folded)
        return GEMM_EPI_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(W_folded, 16) || !aligned(gamma, 2) || !aligned(beta, 2) ||
        !aligned(b, 2) || !aligned(colsum, 4) || !aligned(bias_folded, 4))
        return GEMM_EPI_ERR_MISALIGNED;
    int sms = 0;
    gemm_epi_status st = current_device(&sms);
    if (st != GEMM_EPI_OK) return st;
    return layernorm_fold_launch(gamma, beta, W, b, W_folded, colsum, bias_folded,
                                 static_cast<int>(d), static_cast<int>(f),
                                 dtype == GEMM_EPI_BF16 ? 1 : 0, sms, stream) == cudaSuccess
               ? GEMM_EPI_OK
               : GEMM_EPI_ERR_LAUNCH;
}

}  // extern "C"
