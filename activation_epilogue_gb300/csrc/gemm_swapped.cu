// Swapped small-m kernel instantiations: D^T tiles of 128 columns of D by BN rows of D,
// BN in {16, 32, 64, 128, 256}.
#include "gemm_kernel.cuh"

namespace gemm_epi {

namespace {
template <int BN>
cudaError_t prepare_one()
{
    return cudaFuncSetAttribute(gemm_epi_kernel<BN, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                TileCfg<BN>::kSmemBytes);
}

template <int BN>
cudaError_t launch_one(const GemmParams& p, int grid, cudaStream_t stream, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = TileCfg<BN>::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    if (p.split > 1 && !p.split_global) {  // split-K: one cluster of `split` CTAs per tile
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = static_cast<unsigned>(p.split);
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = na ? attr : nullptr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, gemm_epi_kernel<BN, true>, p);
}
}  // namespace

#define GEMM_EPI_SWAPPED_CASES(F) F(16) F(32) F(64) F(128) F(256)

cudaError_t swapped_prepare(int bn)
{
    switch (bn) {
#define F(X) case X: return prepare_one<X>();
        GEMM_EPI_SWAPPED_CASES(F)
#undef F
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t swapped_launch(int bn, const GemmParams& p, int grid, cudaStream_t stream, bool pdl)
{
    switch (bn) {
#define F(X) case X: return launch_one<X>(p, grid, stream, pdl);
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
