// CTA-pair kernel instantiations: 256 x BN tiles (BN 224 or 256) computed by two CTAs with
// cta_group::2 MMAs, one instantiation per epilog.  With the epilog fixed at compile time a
// kernel carries only its own epilogue code: measured on GB300, the kernel that held every
// epilog's fully unrolled code stalled its warps on instruction fetch (ncu: no_instruction
// about 1.3 cycles per issued instruction in the GELU epilogue).  One more instantiation runs
// a whole FFN block (GELU GEMM, then bias + residual GEMM) in a single launch.
#include "gemm_kernel.cuh"

namespace gemm_epi {

namespace {

// Epilogue warps per CTA: 8, and 16 for GELU_BIAS and TANH_BIAS when a tile has at most 8
// K blocks (K <= 512), where the activation's epilogue outlasts the tile's MMAs.  Measured on
// GB300 (GELU, CUDA graph, hot L2): 8192 x 4096 x 512 40.1 us with 8 warps, 36.7 with 12,
// 35.1 with 16; at K = 1024 more warps gain nothing (16384 x 4096 x 1024: 91.1 / 92.2 /
// 92.5 us), nor at 4096^3.
constexpr int kShortKBlocks = 8;

template <int EPI>
constexpr bool short_k_variant() { return EPI == EPI_GELU_BIAS || EPI == EPI_TANH_BIAS; }

template <int BN, int EPI, int EW = 8>
cudaError_t prepare_one()
{
    return cudaFuncSetAttribute(gemm_epi_kernel<BN, false, true, EPI, false, EW>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                TileCfg<BN, true, EW>::kSmemBytes);
}

template <int BN>
cudaError_t prepare_all()
{
    const cudaError_t e[] = {prepare_one<BN, EPI_BIAS>(),          prepare_one<BN, EPI_RELU_BIAS>(),
                             prepare_one<BN, EPI_GELU_BIAS>(),     prepare_one<BN, EPI_RELU_AUX_BIAS>(),
                             prepare_one<BN, EPI_BIAS_RESIDUAL>(), prepare_one<BN, EPI_NONE>(),
                             prepare_one<BN, EPI_TANH_BIAS>(),     prepare_one<BN, EPI_GELU_AUX_BIAS>(),
                             prepare_one<BN, EPI_DRELU_BGRAD>(),   prepare_one<BN, EPI_DGELU_BGRAD>(),
                             prepare_one<BN, EPI_LN_GELU_BIAS>(), prepare_one<BN, EPI_GELU_BIAS, 16>(),
                             prepare_one<BN, EPI_TANH_BIAS, 16>()};
    for (cudaError_t x : e)
        if (x != cudaSuccess) return x;
    return cudaSuccess;
}

template <int BN, int EPI, int EW = 8>
cudaError_t launch_one(const GemmParams& p, int grid, cudaStream_t stream, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(64 + 32 * EW, 1, 1);
    cfg.dynamicSmemBytes = TileCfg<BN, true, EW>::kSmemBytes;
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
    return cudaLaunchKernelEx(&cfg, gemm_epi_kernel<BN, false, true, EPI, false, EW>, p);
}

template <int BN>
cudaError_t launch_bn(const GemmParams& p, int grid, cudaStream_t stream, bool pdl)
{
    switch (p.epilog) {
    case EPI_BIAS: return launch_one<BN, EPI_BIAS>(p, grid, stream, pdl);
    case EPI_RELU_BIAS: return launch_one<BN, EPI_RELU_BIAS>(p, grid, stream, pdl);
    case EPI_GELU_BIAS:
        if (p.k_blocks <= kShortKBlocks) return launch_one<BN, EPI_GELU_BIAS, 16>(p, grid, stream, pdl);
        return launch_one<BN, EPI_GELU_BIAS>(p, grid, stream, pdl);
    case EPI_RELU_AUX_BIAS: return launch_one<BN, EPI_RELU_AUX_BIAS>(p, grid, stream, pdl);
    case EPI_BIAS_RESIDUAL: return launch_one<BN, EPI_BIAS_RESIDUAL>(p, grid, stream, pdl);
    case EPI_NONE: return launch_one<BN, EPI_NONE>(p, grid, stream, pdl);
    case EPI_TANH_BIAS:
        if (p.k_blocks <= kShortKBlocks) return launch_one<BN, EPI_TANH_BIAS, 16>(p, grid, stream, pdl);
        return launch_one<BN, EPI_TANH_BIAS>(p, grid, stream, pdl);
    case EPI_GELU_AUX_BIAS: return launch_one<BN, EPI_GELU_AUX_BIAS>(p, grid, stream, pdl);
    case EPI_DRELU_BGRAD: return launch_one<BN, EPI_DRELU_BGRAD>(p, grid, stream, pdl);
    case EPI_DGELU_BGRAD: return launch_one<BN, EPI_DGELU_BGRAD>(p, grid, stream, pdl);
    case EPI_LN_GELU_BIAS: return launch_one<BN, EPI_LN_GELU_BIAS>(p, grid, stream, pdl);
    default: return cudaErrorInvalidValue;
    }
}

template <int BN>
int max_clusters_one()
{
    constexpr unsigned size = 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(size, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = TileCfg<BN, true>::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = size;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_epi_kernel<BN, false, true, EPI_BIAS>, &cfg) !=
        cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace

cudaError_t rowpair_prepare(int bn)
{
    switch (bn) {
    case 224: return prepare_all<224>();
    case 256: return prepare_all<256>();
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t rowpair_launch(int bn, const GemmParams& p, int grid, cudaStream_t stream, bool pdl)
{
    switch (bn) {
    case 224: return launch_bn<224>(p, grid, stream, pdl);
    case 256: return launch_bn<256>(p, grid, stream, pdl);
    default: return cudaErrorInvalidValue;
    }
}

int rowpair_smem_bytes(int bn)
{
    switch (bn) {
    case 224: return TileCfg<224, true>::kSmemBytes;
    case 256: return TileCfg<256, true>::kSmemBytes;
    default: return 0;
    }
}

int rowpair_stages(int bn)
{
    switch (bn) {
    case 224: return TileCfg<224, true>::kStages;
    case 256: return TileCfg<256, true>::kStages;
    default: return 0;
    }
}

cudaError_t ffn_pair_prepare()
{
    const cudaError_t e = prepare_one<256, kEpiFfn>();
    return e != cudaSuccess ? e : prepare_one<256, kEpiFfnSplit>();
}

cudaError_t ffn_pair_launch(const GemmParams& p, int grid, cudaStream_t stream)
{
    if (p.ffn_split2 > 1) return launch_one<256, kEpiFfnSplit>(p, grid, stream, false);
    return launch_one<256, kEpiFfn>(p, grid, stream, false);
}

int rowpair_max_clusters(int bn)
{
    switch (bn) {
    case 224: return max_clusters_one<224>();
    case 256: return max_clusters_one<256>();
    default: return 0;
    }
}

}  // namespace gemm_epi
