// Elementwise epilogue over a stored 16-bit pre-activation: the second kernel of the
// unfused baseline, which "Fusing bias into cuBLASLt matmul with nvmath-python for PyTorch
// inference" (blog.hotdry.top, 2025-09-22) describes as the separate bias-add and
// activation launches that cost one extra global-memory write and read of the matrix.
// With pre == nullptr the matrix product is taken as zero (the k == 0 problem).  For the
// backward epilogs the bias gradient must be zero on entry; it is accumulated atomically.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gelu.cuh"
#include "kernel_params.h"

namespace gemm_epi {

namespace {

__device__ __forceinline__ float ld16(const uint16_t* p, long long i, int bf16)
{
    const uint16_t h = p[i];
    if (bf16) return __uint_as_float(static_cast<uint32_t>(h) << 16);
    return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ uint16_t st16(float a, int bf16)
{
    if (bf16) return __bfloat16_as_ushort(__float2bfloat16_rn(a));
    return __half_as_ushort(__float2half_rn(a));
}

// One block task = 32 rows x 256 columns; warp w of the block takes columns 32 w .. 32 w + 31
// of it (lane = column) and walks the 32 rows, so each row's 32 columns sit on the lanes:
// one ballot gives an aux word, one warp sum a row's share of a bias gradient, and a
// column's share of a bias gradient stays in its lane's register until the task ends.
__global__ void __launch_bounds__(256) elementwise_epilogue_kernel(
    const uint16_t* __restrict__ pre, const uint16_t* __restrict__ bias,
    const uint16_t* __restrict__ residual, uint16_t* __restrict__ D, void* __restrict__ aux,
    const void* __restrict__ aux_in, float* __restrict__ dbias, int m, int n, int epilog,
    int bias_layout, int bf16, int aux_ld)
{
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const bool bwd = is_backward(epilog);
    const bool has_bias = epilog != EPI_NONE && !bwd;
    const long long groups_per_row = (n + 255) / 256;
    const long long tasks = static_cast<long long>((m + 31) / 32) * groups_per_row;
    for (long long task = blockIdx.x; task < tasks; task += gridDim.x) {
        const int rt = static_cast<int>(task / groups_per_row);
        const int g = static_cast<int>(task - static_cast<long long>(rt) * groups_per_row);
        const int col32 = g * 256 + warp * 32;  // first column of this warp
        const int col = col32 + lane;
        const bool ok = col < n;
        const int rows = min(32, m - rt * 32);
        float col_sum = 0.0f;
        for (int r = 0; r < rows; ++r) {
            const int row = rt * 32 + r;
            const long long idx = static_cast<long long>(row) * n + col;
            float v = 0.0f;
            if (ok) {
                if (pre) v = ld16(pre, idx, bf16);
                if (has_bias) v += ld16(bias, bias_layout == 0 ? row : col, bf16);
            }
            if (epilog == EPI_RELU_AUX_BIAS) {
                const uint32_t word = __ballot_sync(0xFFFFFFFFu, ok && v > 0.0f);
                if (lane == 0 && col32 < n)
                    static_cast<uint32_t*>(aux)[static_cast<long long>(row) * aux_ld + col32 / 32] = word;
            } else if (epilog == EPI_GELU_AUX_BIAS) {
                if (ok) static_cast<uint16_t*>(aux)[idx] = st16(v, bf16);
            } else if (epilog == EPI_DRELU_BGRAD) {
                uint32_t mw = 0;
                if (col32 < n)
                    mw = static_cast<const uint32_t*>(aux_in)[static_cast<long long>(row) * aux_ld + col32 / 32];
                v = (ok && ((mw >> lane) & 1u)) ? v : 0.0f;
            } else if (epilog == EPI_DGELU_BGRAD) {
                v = ok ? v * gelu_grad_fast(ld16(static_cast<const uint16_t*>(aux_in), idx, bf16)) : 0.0f;
            }
            float o = v;
            if (epilog == EPI_RELU_BIAS || epilog == EPI_RELU_AUX_BIAS)
                o = o > 0.0f ? o : 0.0f;
            else if (epilog == EPI_GELU_BIAS || epilog == EPI_GELU_AUX_BIAS)
                o = gelu_erf_fast(o);
            else if (epilog == EPI_TANH_BIAS)
                o = tanh_fast(o);
            if (ok) {
                if (epilog == EPI_BIAS_RESIDUAL) o += ld16(residual, idx, bf16);
                D[idx] = st16(o, bf16);
            }
            if (bwd) {
                if (bias_layout == 0) {
                    float s = v;
#pragma unroll
                    for (int o2 = 16; o2 >= 1; o2 >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, o2);
                    if (lane == 0 && col32 < n) atomicAdd(dbias + row, s);
                } else {
                    col_sum += v;
                }
            }
        }
        if (bwd && bias_layout == 1 && ok) atomicAdd(dbias + col, col_sum);
    }
}

}  // namespace

cudaError_t elementwise_launch(const void* pre, const void* bias, const void* residual, void* D,
                               void* aux, const void* aux_in, float* dbias, int m, int n,
                               int epilog, int bias_layout, int bf16, int aux_ld, int sm_count,
                               cudaStream_t stream)
{
    long long blocks = static_cast<long long>((m + 31) / 32) * ((n + 255) / 256);
    const long long cap = static_cast<long long>(sm_count) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    elementwise_epilogue_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const uint16_t*>(pre), static_cast<const uint16_t*>(bias),
        static_cast<const uint16_t*>(residual), static_cast<uint16_t*>(D), aux, aux_in, dbias, m,
        n, epilog, bias_layout, bf16, aux_ld);
    return cudaGetLastError();
}

}  // namespace gemm_epi
