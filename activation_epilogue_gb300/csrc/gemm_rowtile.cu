// Row-tile kernel instantiations: 128 x BN output tiles, BN in {64, 128, 256}.
#include "gemm_kernel.cuh"

namespace gemm_epi {

namespace {
template <int BN>
cudaError_t prepare_one()
{
    return cudaFuncSetAttribute(gemm_epi_kernel<BN, false>,
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
    return cudaLaunchKernelEx(&cfg, gemm_epi_kernel<BN, false>, p);
}
}  // namespace

cudaError_t rowtile_prepare(int bn)
{
    switch (bn) {
    case 64: return prepare_one<64>();
    case 128: return prepare_one<128>();
    case 256: return prepare_one<256>();
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t rowtile_launch(int bn, const GemmParams& p, int grid, cudaStream_t stream, bool pdl)
{
    switch (bn) {
    case 64: return launch_one<64>(p, grid, stream, pdl);
    case 128: return launch_one<128>(p, grid, stream, pdl);
    case 256: return launch_one<256>(p, grid, stream, pdl);
    default: return cudaErrorInvalidValue;
    }
}

int rowtile_smem_bytes(int bn)
{
    switch (bn) {
    case 64: return TileCfg<64>::kSmemBytes;
    case 128: return TileCfg<128>::kSmemBytes;
    case 256: return TileCfg<256>::kSmemBytes;
    default: return 0;
    }
}

int rowtile_stages(int bn)
{
    switch (bn) {
    case 64: return TileCfg<64>::kStages;
    case 128: return TileCfg<128>::kStages;
    case 256: return TileCfg<256>::kStages;
    default: return 0;
    }
}


}  // namespace gemm_epi
