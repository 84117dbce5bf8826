// Elementwise epilogue over a stored 16-bit pre-activation: the second kernel of the
// unfused baseline, which "Fusing bias into cuBLASLt matmul with nvmath-python for PyTorch
// inference" (blog.hotdry.top, 2025-09-22) describes as the separate bias-add and
// activation launches that cost one extra global-memory write and read of the matrix.
// With pre == nullptr the matrix product is taken as zero (the k == 0 problem).
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

// One warp task = one row x 256 columns; lane l handles columns 32 s + l (s = 0..7), so
// each 32-column group sits on the 32 lanes and one ballot gives its aux word.
__global__ void __launch_bounds__(256) elementwise_epilogue_kernel(
    const uint16_t* __restrict__ pre, const uint16_t* __restrict__ bias,
    const uint16_t* __restrict__ residual, uint16_t* __restrict__ D, uint32_t* __restrict__ aux,
    int m, int n, int epilog, int bias_layout, int bf16, int aux_ld)
{
    const int lane = threadIdx.x & 31;
    const long long groups_per_row = (n + 255) / 256;
    const long long tasks = static_cast<long long>(m) * groups_per_row;
    const long long warp_global = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    const long long warps_total = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    for (long long task = warp_global; task < tasks; task += warps_total) {
        const int row = static_cast<int>(task / groups_per_row);
        const int g = static_cast<int>(task - static_cast<long long>(row) * groups_per_row);
        float x[8];
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const int col = g * 256 + s * 32 + lane;
            const long long idx = static_cast<long long>(row) * n + col;
            float v = 0.0f;
            if (col < n) {
                if (pre) v = ld16(pre, idx, bf16);
                if (epilog != EPI_NONE) v += ld16(bias, bias_layout == 0 ? row : col, bf16);
            }
            x[s] = v;
        }
        uint32_t my_word = 0;
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const int col = g * 256 + s * 32 + lane;
            const bool ok = col < n;
            const uint32_t word = __ballot_sync(0xFFFFFFFFu, ok && x[s] > 0.0f);
            if (lane == s) my_word = word;
            float o = x[s];
            if (epilog == EPI_RELU_BIAS || epilog == EPI_RELU_AUX_BIAS)
                o = o > 0.0f ? o : 0.0f;
            else if (epilog == EPI_GELU_BIAS)
                o = gelu_erf_fast(o);
            else if (epilog == EPI_TANH_BIAS)
                o = tanh_fast(o);
            const long long idx = static_cast<long long>(row) * n + col;
            if (ok) {
                if (epilog == EPI_BIAS_RESIDUAL) o += ld16(residual, idx, bf16);
                D[idx] = st16(o, bf16);
            }
        }
        if (epilog == EPI_RELU_AUX_BIAS && lane < 8 && g * 8 + lane < aux_ld)
            aux[static_cast<long long>(row) * aux_ld + g * 8 + lane] = my_word;
    }
}

}  // namespace

cudaError_t elementwise_launch(const void* pre, const void* bias, const void* residual, void* D,
                               uint32_t* aux, int m, int n, int epilog, int bias_layout, int bf16,
                               int aux_ld, int sm_count, cudaStream_t stream)
{
    const long long tasks = static_cast<long long>(m) * ((n + 255) / 256);
    long long blocks = (tasks + 7) / 8;  // 8 warps per block
    const long long cap = static_cast<long long>(sm_count) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    elementwise_epilogue_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        static_cast<const uint16_t*>(pre), static_cast<const uint16_t*>(bias),
        static_cast<const uint16_t*>(residual), static_cast<uint16_t*>(D), aux, m, n, epilog,
        bias_layout, bf16, aux_ld);
    return cudaGetLastError();
}

}  // namespace gemm_epi
