// Swapped small-m kernel instantiations: D^T tiles of 128 columns of D by BN rows of D,
// BN in {16, 32, 64, 128, 256}, with the epilog read from the parameters; the forward epilogs
// with kernels of their own (gemm_fwd_*.cu) launch those.
#include "gemm_single.cuh"

namespace gemm_epi {

cudaError_t swapped_prepare(int bn)
{
    cudaError_t e;
    switch (bn) {
#define F(X) case X: e = single_prepare<X, true, -1>(); break;
        GEMM_EPI_SWAPPED_CASES(F)
#undef F
    default: return cudaErrorInvalidValue;
    }
    return e != cudaSuccess ? e : fwd_prepare(bn, true);
}

cudaError_t swapped_launch(int bn, const GemmParams& p, int grid, cudaStream_t stream, bool pdl)
{
    if (fwd_specialised(p.epilog)) return fwd_launch(bn, true, p, grid, stream, pdl);
    switch (bn) {
#define F(X) case X: return single_launch<X, true, -1>(p, grid, stream, pdl);
        GEMM_EPI_SWAPPED_CASES(F)
#undef F
    default: return cudaErrorInvalidValue;
    }
}

int swapped_smem_bytes(int bn)
{
    switch (bn) {
#define F(X) case X: return TileCfg<X>::kSmemBytes;
        GEMM_EPI_SWAPPED_CASES(F)
#undef F
    default: return 0;
    }
}

int swapped_stages(int bn)
{
    switch (bn) {
#define F(X) case X: return TileCfg<X>::kStages;
        GEMM_EPI_SWAPPED_CASES(F)
#undef F
    default: return 0;
    }
}

}  // namespace gemm_epi
