// LayerNorm next to the FFN GEMMs, after "Operator fusion in model inference, from LayerNorm to
// residual connections" (wmrh.cn/news/429806), section 2: y = (x - mu) / sqrt(var + eps) *
// gamma + beta over each row, optionally plus a residual, done in one kernel.
//
// Three kernels:
//   * layernorm_kernel: the section's fused LayerNorm (+ residual), one warp per row: the
//     mean, the variance of the centred row and the normalised output, from the row held
//     in registers (d <= 1024; longer rows are re-read from L1/L2 for each pass);
//     16-byte accesses.
//   * layernorm_stats_kernel: only the per-row mean and 1/sqrt(var + eps).  With them the
//     LayerNorm in front of a GEMM folds into the GEMM's epilogue:
//         LN(x) . W + b = rstd (x . W' - mu c) + b',
//     W' = diag(gamma) W, c_j = sum_k W'[k][j], b' = beta . W + b,
//     so the GEMM runs on the raw rows and the normalised rows never exist in memory.
//   * layernorm_fold_kernel: W' (rounded to the 16-bit type, as the GEMM reads it), c (the
//     column sums of that rounded W', so x . W' - mu c is exactly sum_k (x_k - mu) W'[k][j]
//     up to fp32 rounding) and b', once per weight update.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kernel_params.h"

namespace gemm_epi {

namespace {

__device__ __forceinline__ float dec(uint32_t h, int bf16)
{
    if (bf16) return __uint_as_float(h << 16);
    return __half2float(__ushort_as_half(static_cast<uint16_t>(h)));
}

__device__ __forceinline__ void load8(const uint16_t* p, float (&x)[8], int bf16)
{
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        x[2 * h] = dec(ww[h] & 0xFFFFu, bf16);
        x[2 * h + 1] = dec(ww[h] >> 16, bf16);
    }
}

__device__ __forceinline__ uint16_t enc(float a, int bf16)
{
    if (bf16) return __bfloat16_as_ushort(__float2bfloat16_rn(a));
    return __half_as_ushort(__float2half_rn(a));
}

__device__ __forceinline__ void store8(uint16_t* p, const float (&x)[8], int bf16)
{
    uint32_t w[4];
#pragma unroll
    for (int h = 0; h < 4; ++h)
        w[h] = static_cast<uint32_t>(enc(x[2 * h], bf16)) |
               (static_cast<uint32_t>(enc(x[2 * h + 1], bf16)) << 16);
    *reinterpret_cast<uint4*>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Mean and 1/sqrt(var + eps) of one row, two passes (the second over the centred values).
__device__ __forceinline__ void row_stats(const uint16_t* x, int d, int bf16, float eps,
                                          int lane, float& mu, float& rstd)
{
    float s = 0.0f;
    for (int c = lane * 8; c < d; c += 256) {
        float v[8];
        load8(x + c, v, bf16);
#pragma unroll
        for (int j = 0; j < 8; ++j) s += v[j];
    }
    const float inv_d = __fdividef(1.0f, static_cast<float>(d));
    mu = warp_sum(s) * inv_d;
    float q = 0.0f;
    for (int c = lane * 8; c < d; c += 256) {
        float v[8];
        load8(x + c, v, bf16);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float e = v[j] - mu;
            q = fmaf(e, e, q);
        }
    }
    const float var = warp_sum(q) * inv_d;
    rstd = rsqrtf(var + eps);  // hardware reciprocal square root (about 2 ulp)
}

// Rows of at most kRegVec * 256 elements are held in registers: every load of the row is
// issued before any is used (one memory round trip per row instead of one per 256
// columns), and the variance and the normalisation reuse the values.
constexpr int kRegVec = 4;  // d <= 1024: about 50 registers, four 256-thread blocks per SM

__device__ __forceinline__ void row_load_regs(const uint16_t* x, int d, int bf16, int lane,
                                              float (&v)[kRegVec][8])
{
#pragma unroll
    for (int i = 0; i < kRegVec; ++i) {
        const int c = i * 256 + lane * 8;
        if (c < d) {
            load8(x + c, v[i], bf16);
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) v[i][j] = 0.0f;
        }
    }
}

__device__ __forceinline__ void row_stats_regs(const float (&v)[kRegVec][8], int d, int lane,
                                               float eps, float& mu, float& rstd)
{
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < kRegVec; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) s += v[i][j];
    const float inv_d = __fdividef(1.0f, static_cast<float>(d));
    mu = warp_sum(s) * inv_d;
    float q = 0.0f;
#pragma unroll
    for (int i = 0; i < kRegVec; ++i) {
        if (i * 256 + lane * 8 < d) {  // (padding lanes hold 0, not mu)
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float e = v[i][j] - mu;
                q = fmaf(e, e, q);
            }
        }
    }
    rstd = rsqrtf(warp_sum(q) * inv_d + eps);
}

template <bool REGS>
__global__ void __launch_bounds__(256) layernorm_stats_kernel(const uint16_t* __restrict__ X,
                                                              int t, int d, int bf16, float eps,
                                                              float* __restrict__ stats)
{
    const int lane = threadIdx.x & 31;
    const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    for (long long r = warp; r < t; r += nwarps) {
        float mu, rstd;
        if constexpr (REGS) {
            float v[kRegVec][8];
            row_load_regs(X + r * d, d, bf16, lane, v);
            row_stats_regs(v, d, lane, eps, mu, rstd);
        } else {
            row_stats(X + r * d, d, bf16, eps, lane, mu, rstd);
        }
        if (lane == 0) {
            stats[2 * r] = mu;
            stats[2 * r + 1] = rstd;
        }
    }
}

__global__ void __launch_bounds__(256) layernorm_kernel(
    const uint16_t* __restrict__ X, const uint16_t* __restrict__ R,
    const uint16_t* __restrict__ gamma, const uint16_t* __restrict__ beta,
    uint16_t* __restrict__ Y, int t, int d, int bf16, float eps)
{
    const int lane = threadIdx.x & 31;
    const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    for (long long r = warp; r < t; r += nwarps) {
        const uint16_t* x = X + r * d;
        float mu, rstd;
        if (d <= kRegVec * 256) {
            float v[kRegVec][8];
            row_load_regs(x, d, bf16, lane, v);
            row_stats_regs(v, d, lane, eps, mu, rstd);
#pragma unroll
            for (int i = 0; i < kRegVec; ++i) {
                const int c = i * 256 + lane * 8;
                if (c >= d) continue;
                float rv[8];
                if (R) load8(R + r * d + c, rv, bf16);
                float y[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float o = (v[i][j] - mu) * rstd * dec(gamma[c + j], bf16) +
                                    dec(beta[c + j], bf16);
                    y[j] = R ? o + rv[j] : o;
                }
                store8(Y + r * d + c, y, bf16);
            }
            continue;
        }
        row_stats(x, d, bf16, eps, lane, mu, rstd);
        for (int c = lane * 8; c < d; c += 256) {
            float v[8];
            load8(x + c, v, bf16);
            float rv[8];
            if (R) load8(R + r * d + c, rv, bf16);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                // gamma and beta are only 2-byte aligned: element loads (they stay in L1)
                float y = (v[j] - mu) * rstd * dec(gamma[c + j], bf16) + dec(beta[c + j], bf16);
                v[j] = R ? y + rv[j] : y;
            }
            store8(Y + r * d + c, v, bf16);
        }
    }
}

// A warp folds 256 columns (8 per lane) over kFoldRows rows of W and adds its partial
// column sums to colsum and bias_f (zeroed before the launch); the warps of row chunk 0
// also add b.
constexpr int kFoldRows = 64;

__global__ void __launch_bounds__(256) layernorm_fold_kernel(
    const uint16_t* __restrict__ gamma, const uint16_t* __restrict__ beta,
    const uint16_t* __restrict__ W, const uint16_t* __restrict__ b, uint16_t* __restrict__ Wf,
    float* __restrict__ colsum, float* __restrict__ bias_f, int d, int f, int bf16)
{
    const int lane = threadIdx.x & 31;
    const long long warp = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long col_groups = (f + 255) / 256;
    const long long row_chunks = (d + kFoldRows - 1) / kFoldRows;
    if (warp >= col_groups * row_chunks) return;
    const int cg = static_cast<int>(warp % col_groups);
    const int rc = static_cast<int>(warp / col_groups);
    const int col = cg * 256 + lane * 8;
    if (col >= f) return;  // f is a multiple of 8: a lane's 8 columns are all in or all out
    float cs[8] = {0, 0, 0, 0, 0, 0, 0, 0}, bs[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    const int k_end = min(d, (rc + 1) * kFoldRows);
    for (int k = rc * kFoldRows; k < k_end; ++k) {
        float w[8];
        load8(W + static_cast<long long>(k) * f + col, w, bf16);
        const float g = dec(gamma[k], bf16), be = dec(beta[k], bf16);
        float wf[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            wf[j] = dec(enc(g * w[j], bf16), bf16);  // the 16-bit value the GEMM will read
            cs[j] += wf[j];
            bs[j] = fmaf(be, w[j], bs[j]);
        }
        store8(Wf + static_cast<long long>(k) * f + col, wf, bf16);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        atomicAdd(colsum + col + j, cs[j]);
        atomicAdd(bias_f + col + j, rc == 0 ? bs[j] + dec(b[col + j], bf16) : bs[j]);
    }
}

unsigned grid_for_rows(long long rows, int sm_count)
{
    long long blocks = (rows + 7) / 8;  // 8 warps (rows) per block
    const long long cap = static_cast<long long>(sm_count) * 8;
    if (blocks > cap) blocks = cap;
    return static_cast<unsigned>(blocks < 1 ? 1 : blocks);
}

}  // namespace

cudaError_t layernorm_stats_launch(const void* X, int t, int d, int bf16, float eps,
                                   float* stats, int sm_count, cudaStream_t stream)
{
    if (d <= kRegVec * 256)
        layernorm_stats_kernel<true><<<grid_for_rows(t, sm_count), 256, 0, stream>>>(
            static_cast<const uint16_t*>(X), t, d, bf16, eps, stats);
    else
        layernorm_stats_kernel<false><<<grid_for_rows(t, sm_count), 256, 0, stream>>>(
            static_cast<const uint16_t*>(X), t, d, bf16, eps, stats);
    return cudaGetLastError();
}

cudaError_t layernorm_launch(const void* X, const void* residual, const void* gamma,
                             const void* beta, void* Y, int t, int d, int bf16, float eps,
                             int sm_count, cudaStream_t stream)
{
    layernorm_kernel<<<grid_for_rows(t, sm_count), 256, 0, stream>>>(
        static_cast<const uint16_t*>(X), static_cast<const uint16_t*>(residual),
        static_cast<const uint16_t*>(gamma), static_cast<const uint16_t*>(beta),
        static_cast<uint16_t*>(Y), t, d, bf16, eps);
    return cudaGetLastError();
}

cudaError_t layernorm_fold_launch(const void* gamma, const void* beta, const void* W,
                                  const void* b, void* Wf, float* colsum, float* bias_f, int d,
                                  int f, int bf16, int sm_count, cudaStream_t stream)
{
    (void)sm_count;
    cudaError_t e = cudaMemsetAsync(colsum, 0, sizeof(float) * static_cast<size_t>(f), stream);
    if (e == cudaSuccess)
        e = cudaMemsetAsync(bias_f, 0, sizeof(float) * static_cast<size_t>(f), stream);
    if (e != cudaSuccess) return e;
    const long long warps = ((f + 255) / 256) * static_cast<long long>((d + kFoldRows - 1) / kFoldRows);
    const long long blocks = (warps + 7) / 8;
    layernorm_fold_kernel<<<static_cast<unsigned>(blocks < 1 ? 1 : blocks), 256, 0, stream>>>(
        static_cast<const uint16_t*>(gamma), static_cast<const uint16_t*>(beta),
        static_cast<const uint16_t*>(W), static_cast<const uint16_t*>(b),
        static_cast<uint16_t*>(Wf), colsum, bias_f, d, f, bf16);
    return cudaGetLastError();
}

}  // namespace gemm_epi
