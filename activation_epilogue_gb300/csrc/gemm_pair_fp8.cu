// CTA-pair kernel on E4M3 inputs: 256 x BN tiles (BN 256 or 224), one instantiation per
// forward epilog without a 16-bit auxiliary output (BIAS, RELU_BIAS, GELU_BIAS,
// RELU_AUX_BIAS, BIAS_RESIDUAL, NONE).  The plan takes the width that needs fewer waves of
// tiles over the pairs, as for 16-bit inputs: 4096 x 4096 is 256 tiles of 256 x 256 on 76
// pairs (3.4 waves, paid as 4) but 304 tiles of 256 x 224 (4 waves exactly).
#include "gemm_kernel.cuh"

namespace gemm_epi {

namespace {

template <int BN, int EPI>
cudaError_t fp8_prepare_one()
{
    return cudaFuncSetAttribute(gemm_epi_kernel<BN, false, true, EPI, true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                TileCfg<BN, true>::kSmemBytes);
}

template <int BN, int EPI>
cudaError_t fp8_launch_one(const GemmParams& p, int grid, cudaStream_t stream, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = TileCfg<BN, true>::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = 2;  // one CTA pair
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, gemm_epi_kernel<BN, false, true, EPI, true>, p);
}

template <int BN>
cudaError_t fp8_prepare_bn()
{
    const cudaError_t e[] = {fp8_prepare_one<BN, EPI_BIAS>(), fp8_prepare_one<BN, EPI_RELU_BIAS>(),
                             fp8_prepare_one<BN, EPI_GELU_BIAS>(),
                             fp8_prepare_one<BN, EPI_RELU_AUX_BIAS>(),
                             fp8_prepare_one<BN, EPI_BIAS_RESIDUAL>(),
                             fp8_prepare_one<BN, EPI_NONE>()};
    for (cudaError_t x : e)
        if (x != cudaSuccess) return x;
    return cudaSuccess;
}

template <int BN>
cudaError_t fp8_launch_bn(const GemmParams& p, int grid, cudaStream_t stream, bool pdl)
{
    switch (p.epilog) {
    case EPI_BIAS: return fp8_launch_one<BN, EPI_BIAS>(p, grid, stream, pdl);
    case EPI_RELU_BIAS: return fp8_launch_one<BN, EPI_RELU_BIAS>(p, grid, stream, pdl);
    case EPI_GELU_BIAS: return fp8_launch_one<BN, EPI_GELU_BIAS>(p, grid, stream, pdl);
    case EPI_RELU_AUX_BIAS: return fp8_launch_one<BN, EPI_RELU_AUX_BIAS>(p, grid, stream, pdl);
    case EPI_BIAS_RESIDUAL: return fp8_launch_one<BN, EPI_BIAS_RESIDUAL>(p, grid, stream, pdl);
    case EPI_NONE: return fp8_launch_one<BN, EPI_NONE>(p, grid, stream, pdl);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t fp8_pair_prepare()
{
    const cudaError_t e = fp8_prepare_bn<256>();
    return e != cudaSuccess ? e : fp8_prepare_bn<224>();
}

cudaError_t fp8_pair_launch(int bn, const GemmParams& p, int grid, cudaStream_t stream, bool pdl)
{
    switch (bn) {
    case 224: return fp8_launch_bn<224>(p, grid, stream, pdl);
    case 256: return fp8_launch_bn<256>(p, grid, stream, pdl);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gemm_epi
