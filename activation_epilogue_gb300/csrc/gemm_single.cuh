// Launch helpers of the single-CTA kernels (row-tile: SWAP = false, BN 64/128/256; swapped
// small-m: SWAP = true, BN 16/32/64/128/256), shared by the instantiations that read the
// epilog from the parameters (EPI = -1) and those built for one forward epilog.
#pragma once

#include "gemm_kernel.cuh"

namespace gemm_epi {

template <int BN, bool SWAP, int EPI>
cudaError_t single_prepare()
{
    return cudaFuncSetAttribute(gemm_epi_kernel<BN, SWAP, false, EPI>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                TileCfg<BN>::kSmemBytes);
}

template <int BN, bool SWAP, int EPI>
cudaError_t single_launch(const GemmParams& p, int grid, cudaStream_t stream, bool pdl)
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
    return cudaLaunchKernelEx(&cfg, gemm_epi_kernel<BN, SWAP, false, EPI>, p);
}

// Clusters of `split` CTAs of this kernel that the GPU holds at once (0 if the query fails).
template <int BN, bool SWAP, int EPI>
int single_max_clusters(int split)
{
    if (single_prepare<BN, SWAP, EPI>() != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(split), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = TileCfg<BN>::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_epi_kernel<BN, SWAP, false, EPI>, &cfg) !=
        cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

#define GEMM_EPI_ROWTILE_CASES(F) F(64) F(128) F(256)
#define GEMM_EPI_SWAPPED_CASES(F) F(16) F(32) F(64) F(128) F(256)

// The row-tile and swapped kernels of one epilog: prepare and launch by (bn, swap).
template <int EPI>
cudaError_t single_prepare_epi(int bn, bool swap)
{
    if (swap) {
        switch (bn) {
#define F(X) case X: return single_prepare<X, true, EPI>();
            GEMM_EPI_SWAPPED_CASES(F)
#undef F
        default: return cudaErrorInvalidValue;
        }
    }
    switch (bn) {
#define F(X) case X: return single_prepare<X, false, EPI>();
        GEMM_EPI_ROWTILE_CASES(F)
#undef F
    default: return cudaErrorInvalidValue;
    }
}

template <int EPI>
cudaError_t single_launch_epi(int bn, bool swap, const GemmParams& p, int grid,
                              cudaStream_t stream, bool pdl)
{
    if (swap) {
        switch (bn) {
#define F(X) case X: return single_launch<X, true, EPI>(p, grid, stream, pdl);
            GEMM_EPI_SWAPPED_CASES(F)
#undef F
        default: return cudaErrorInvalidValue;
        }
    }
    switch (bn) {
#define F(X) case X: return single_launch<X, false, EPI>(p, grid, stream, pdl);
        GEMM_EPI_ROWTILE_CASES(F)
#undef F
    default: return cudaErrorInvalidValue;
    }
}

// One translation unit per forward epilog instantiates its kernels (they compile in
// parallel): fwd_prepare_<name> / fwd_launch_<name>, dispatched by fwd_prepare / fwd_launch.
#define GEMM_EPI_FORWARD_INSTANCES(EPI, NAME)                                                  \
    cudaError_t fwd_prepare_##NAME(int bn, bool swap) { return single_prepare_epi<EPI>(bn, swap); } \
    cudaError_t fwd_launch_##NAME(int bn, bool swap, const GemmParams& p, int grid,            \
                                  cudaStream_t stream, bool pdl)                                \
    {                                                                                          \
        return single_launch_epi<EPI>(bn, swap, p, grid, stream, pdl);                         \
    }

}  // namespace gemm_epi
