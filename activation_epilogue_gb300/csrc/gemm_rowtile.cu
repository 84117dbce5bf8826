// Row-tile kernel instantiations: 128 x BN output tiles, BN in {64, 128, 256}, with the epilog
// read from the parameters; and the dispatch to the single-CTA kernels built for one
// forward epilog (gemm_fwd_*.cu).
//
// A kernel that carries every epilog's unrolled epilogue fetches its path cold from memory:
// measured on GB300 with ncu (caches flushed before the launch), 1024 x 512 x 2048 BIAS fp16
// took 19.1-19.9 us in the all-epilog kernel and 13.6-14.1 us in the BIAS-only one (its
// leading stall was instruction fetch: 9.6 cycles per issued instruction); with hot caches
// (CUDA graph replay) 11.59 against 11.16 us.
#include "gemm_single.cuh"

namespace gemm_epi {

cudaError_t fwd_prepare_bias(int bn, bool swap);
cudaError_t fwd_prepare_relu(int bn, bool swap);
cudaError_t fwd_prepare_gelu(int bn, bool swap);
cudaError_t fwd_prepare_relu_aux(int bn, bool swap);
cudaError_t fwd_prepare_residual(int bn, bool swap);
cudaError_t fwd_launch_bias(int bn, bool swap, const GemmParams& p, int grid, cudaStream_t stream, bool pdl);
cudaError_t fwd_launch_relu(int bn, bool swap, const GemmParams& p, int grid, cudaStream_t stream, bool pdl);
cudaError_t fwd_launch_gelu(int bn, bool swap, const GemmParams& p, int grid, cudaStream_t stream, bool pdl);
cudaError_t fwd_launch_relu_aux(int bn, bool swap, const GemmParams& p, int grid, cudaStream_t stream, bool pdl);
cudaError_t fwd_launch_residual(int bn, bool swap, const GemmParams& p, int grid, cudaStream_t stream, bool pdl);

bool fwd_specialised(int epilog)
{
    return epilog == EPI_BIAS || epilog == EPI_RELU_BIAS || epilog == EPI_GELU_BIAS ||
           epilog == EPI_RELU_AUX_BIAS || epilog == EPI_BIAS_RESIDUAL;
}

cudaError_t fwd_prepare(int bn, bool swap)
{
    const cudaError_t e[] = {fwd_prepare_bias(bn, swap), fwd_prepare_relu(bn, swap),
                             fwd_prepare_gelu(bn, swap), fwd_prepare_relu_aux(bn, swap),
                             fwd_prepare_residual(bn, swap)};
    for (cudaError_t x : e)
        if (x != cudaSuccess) return x;
    return cudaSuccess;
}

cudaError_t fwd_launch(int bn, bool swap, const GemmParams& p, int grid, cudaStream_t stream,
                       bool pdl)
{
    switch (p.epilog) {
    case EPI_BIAS: return fwd_launch_bias(bn, swap, p, grid, stream, pdl);
    case EPI_RELU_BIAS: return fwd_launch_relu(bn, swap, p, grid, stream, pdl);
    case EPI_GELU_BIAS: return fwd_launch_gelu(bn, swap, p, grid, stream, pdl);
    case EPI_RELU_AUX_BIAS: return fwd_launch_relu_aux(bn, swap, p, grid, stream, pdl);
    case EPI_BIAS_RESIDUAL: return fwd_launch_residual(bn, swap, p, grid, stream, pdl);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t rowtile_prepare(int bn)
{
    cudaError_t e;
    switch (bn) {
#define F(X) case X: e = single_prepare<X, false, -1>(); break;
        GEMM_EPI_ROWTILE_CASES(F)
#undef F
    default: return cudaErrorInvalidValue;
    }
    return e != cudaSuccess ? e : fwd_prepare(bn, false);
}

cudaError_t rowtile_launch(int bn, const GemmParams& p, int grid, cudaStream_t stream, bool pdl)
{
    if (fwd_specialised(p.epilog)) return fwd_launch(bn, false, p, grid, stream, pdl);
    switch (bn) {
#define F(X) case X: return single_launch<X, false, -1>(p, grid, stream, pdl);
        GEMM_EPI_ROWTILE_CASES(F)
#undef F
    default: return cudaErrorInvalidValue;
    }
}

int rowtile_max_clusters(int bn, int split)
{
    switch (bn) {
#define F(X) case X: return single_max_clusters<X, false, -1>(split);
        GEMM_EPI_ROWTILE_CASES(F)
#undef F
    default: return 0;
    }
}

int rowtile_smem_bytes(int bn)
{
    switch (bn) {
#define F(X) case X: return TileCfg<X>::kSmemBytes;
        GEMM_EPI_ROWTILE_CASES(F)
#undef F
    default: return 0;
    }
}

int rowtile_stages(int bn)
{
    switch (bn) {
#define F(X) case X: return TileCfg<X>::kStages;
        GEMM_EPI_ROWTILE_CASES(F)
#undef F
    default: return 0;
    }
}

}  // namespace gemm_epi
