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

__device__ __forceinline__ float dec16(uint32_t h, int bf16)
{
    if (bf16) return __uint_as_float(h << 16);
    return __half2float(__ushort_as_half(static_cast<uint16_t>(h)));
}

// 8 consecutive 16-bit values (one 16-byte load) to fp32.
__device__ __forceinline__ void load8(const uint16_t* p, float (&x)[8], int bf16)
{
    const uint4 w = *reinterpret_cast<const uint4*>(p);
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        x[2 * h] = dec16(ww[h] & 0xFFFFu, bf16);
        x[2 * h + 1] = dec16(ww[h] >> 16, bf16);
    }
}

__device__ __forceinline__ uint32_t pack2_16(float a, float b, int bf16)
{
    if (bf16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void store8(uint16_t* p, const float (&x)[8], int bf16)
{
    uint4 w;
    w.x = pack2_16(x[0], x[1], bf16);
    w.y = pack2_16(x[2], x[3], bf16);
    w.z = pack2_16(x[4], x[5], bf16);
    w.w = pack2_16(x[6], x[7], bf16);
    *reinterpret_cast<uint4*>(p) = w;
}

constexpr int kRows = 32;        // rows per block task
constexpr int kCols = 256;       // columns per block task: 8 per lane
constexpr int kWarps = 8;

// One block task = 32 rows x 256 columns.  Lane l of every warp owns columns 8l .. 8l + 7 of
// the task (one 16-byte access per row for each 16-bit matrix: a warp reads or writes 512
// contiguous bytes of a row); warp w takes rows w, w + 8, w + 16, w + 24.  n is a multiple
// of 8, so a lane's 8 columns are all inside the matrix or all outside.  A mask word
// (32 columns) is spread over 4 lanes, 8 bits each, combined with two shuffles.  Bias
// gradient: an (m,1) row's share is a warp sum; a (1,n) column's share is summed in the
// lane over its rows, then over the 8 warps through shared memory, then one atomic per
// column and task.
__global__ void __launch_bounds__(256) elementwise_epilogue_kernel(const ElementwiseArgs a)
{
    __shared__ float col_part[kWarps][kCols];
    const uint16_t* __restrict__ pre = static_cast<const uint16_t*>(a.pre);
    const uint16_t* __restrict__ bias = static_cast<const uint16_t*>(a.bias);
    const uint16_t* __restrict__ residual = static_cast<const uint16_t*>(a.residual);
    uint16_t* __restrict__ D = static_cast<uint16_t*>(a.D);
    void* aux = a.aux;
    const void* aux_in = a.aux_in;
    float* dbias = a.dbias;
    const int m = a.m, n = a.n, epilog = a.epilog, bias_layout = a.bias_layout, bf16 = a.bf16,
              aux_ld = a.aux_ld;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const bool bwd = is_backward(epilog);
    const bool ln = epilog == EPI_LN_GELU_BIAS;
    const bool has_bias = epilog != EPI_NONE && !bwd && !ln;
    const long long groups_per_row = (n + kCols - 1) / kCols;
    const long long tasks = static_cast<long long>((m + kRows - 1) / kRows) * groups_per_row;
    for (long long task = blockIdx.x; task < tasks; task += gridDim.x) {
        const int rt = static_cast<int>(task / groups_per_row);
        const int g = static_cast<int>(task - static_cast<long long>(rt) * groups_per_row);
        const int col = g * kCols + lane * 8;  // this lane's first column
        const bool ok = col < n;
        float cb[8];                           // (1,n) bias of the lane's columns
        float lc[8];                           // LayerNorm: c_j (and b'_j in cb)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            cb[j] = (has_bias && bias_layout == 1 && ok) ? ld16(bias, col + j, bf16) : 0.0f;
            lc[j] = 0.0f;
            if (ln && ok) {
                lc[j] = a.ln_colsum[col + j];
                cb[j] = a.ln_bias[col + j];
            }
        }
        float csum[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int r = warp; r < kRows; r += kWarps) {
            const int row = rt * kRows + r;
            if (row >= m) break;
            const long long idx = static_cast<long long>(row) * n + col;
            float v[8];
            if (ok && pre) {
                load8(pre + idx, v, bf16);
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = 0.0f;
            }
            if (has_bias) {
                const float rb = bias_layout == 0 ? ld16(bias, row, bf16) : 0.0f;
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] += bias_layout == 0 ? rb : cb[j];
            }
            if (ln) {
                const float mu = a.ln_stats[2 * row], rs = a.ln_stats[2 * row + 1];
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = ok ? fmaf(rs, fmaf(-mu, lc[j], v[j]), cb[j]) : 0.0f;
            }
            if (epilog == EPI_RELU_AUX_BIAS) {
                uint32_t bits = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) bits |= (ok && v[j] > 0.0f) ? (1u << j) : 0u;
                bits <<= 8 * (lane & 3);
                bits |= __shfl_xor_sync(0xFFFFFFFFu, bits, 1);
                bits |= __shfl_xor_sync(0xFFFFFFFFu, bits, 2);
                if ((lane & 3) == 0 && ok)
                    static_cast<uint32_t*>(aux)[static_cast<long long>(row) * aux_ld + col / 32] = bits;
            } else if (epilog == EPI_GELU_AUX_BIAS) {
                if (ok) store8(static_cast<uint16_t*>(aux) + idx, v, bf16);
            } else if (epilog == EPI_DRELU_BGRAD) {
                uint32_t mw = 0;
                if (ok)
                    mw = static_cast<const uint32_t*>(aux_in)[static_cast<long long>(row) * aux_ld + col / 32];
                mw >>= 8 * (lane & 3);
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = ((mw >> j) & 1u) ? v[j] : 0.0f;
            } else if (epilog == EPI_DGELU_BGRAD) {
                if (ok) {
                    float pv[8];
                    load8(static_cast<const uint16_t*>(aux_in) + idx, pv, bf16);
#pragma unroll
                    for (int j = 0; j < 8; ++j) v[j] *= gelu_grad_fast(pv[j]);
                }
            }
            if (bwd) {
                if (bias_layout == 0) {
                    float sr = 0.0f;
#pragma unroll
                    for (int j = 0; j < 8; ++j) sr += v[j];
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) sr += __shfl_xor_sync(0xFFFFFFFFu, sr, o);
                    if (lane == 0) atomicAdd(dbias + row, sr);
                } else {
#pragma unroll
                    for (int j = 0; j < 8; ++j) csum[j] += v[j];
                }
            }
            if (epilog == EPI_RELU_BIAS || epilog == EPI_RELU_AUX_BIAS) {
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = v[j] > 0.0f ? v[j] : 0.0f;
            } else if (epilog == EPI_GELU_BIAS || epilog == EPI_GELU_AUX_BIAS || ln) {
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = gelu_erf_fast(v[j]);
            } else if (epilog == EPI_TANH_BIAS) {
#pragma unroll
                for (int j = 0; j < 8; ++j) v[j] = tanh_fast(v[j]);
            }
            if (ok) {
                if (epilog == EPI_BIAS_RESIDUAL) {
                    float rv[8];
                    load8(residual + idx, rv, bf16);
#pragma unroll
                    for (int j = 0; j < 8; ++j) v[j] += rv[j];
                }
                store8(D + idx, v, bf16);
            }
        }
        if (bwd && bias_layout == 1) {
            // this task's column sums: over the warp's rows (registers), then the 8 warps
#pragma unroll
            for (int j = 0; j < 8; ++j) col_part[warp][lane * 8 + j] = csum[j];
            __syncthreads();
            const int c = g * kCols + static_cast<int>(threadIdx.x);
            if (c < n) {
                float t = 0.0f;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) t += col_part[w][threadIdx.x];
                atomicAdd(dbias + c, t);
            }
            __syncthreads();
        }
    }
}

}  // namespace

cudaError_t elementwise_launch(const ElementwiseArgs& a, int sm_count, cudaStream_t stream)
{
    long long blocks = static_cast<long long>((a.m + kRows - 1) / kRows) * ((a.n + kCols - 1) / kCols);
    const long long cap = static_cast<long long>(sm_count) * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    elementwise_epilogue_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace gemm_epi
