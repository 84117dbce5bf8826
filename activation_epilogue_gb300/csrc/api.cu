// Host side of the C ABI in gemm_epi.h: plans, argument checks, tensor-map encoding and
// kernel launches.
//
// The plan/execute/free split follows the stateful Matmul API of "Fusing bias into cuBLASLt
// matmul with nvmath-python for PyTorch inference" (blog.hotdry.top, 2025-09-22, code
// example and the paragraph on operational parameters): the plan fixes shape, dtype, epilog
// and bias layout and chooses the kernel configuration ("nvmath-python: cuBLAS and cuSOLVER
// bindings", matmul-planning checklist: plan() picks the algorithm); execute() is
// asynchronous; free() releases the plan.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "gemm_epi.h"
#include "kernel_params.h"

using namespace gemm_epi;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

EncodeTiledFn encode_fn()
{
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    });
    return g_encode;
}

enum Variant { kEmpty = 0, kRowTile = 1, kSwapped = 2, kBiasOnly = 3, kRowPair = 4 };

constexpr int kSwappedMaxM = 256;
constexpr unsigned long long kDefaultWaitNs = 2000ull * 1000 * 1000;  // 2 s

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Epilogs built for E4M3 inputs (forward, no 16-bit auxiliary output).
bool fp8_epilog(int e)
{
    return e == GEMM_EPI_BIAS || e == GEMM_EPI_RELU_BIAS || e == GEMM_EPI_GELU_BIAS ||
           e == GEMM_EPI_RELU_AUX_BIAS || e == GEMM_EPI_BIAS_RESIDUAL || e == GEMM_EPI_NONE;
}

}  // namespace

struct HostPipe;

struct gemm_epi_plan_s {
    int64_t m, n, k;
    int dtype, epilog, bias_layout;
    int device, sm_count;
    // chosen configuration
    int variant, bn, stages, smem, grid, group_m, tiles_m, tiles_n, k_blocks;
    int split, kb_per_split;  // split-K across a cluster (split == 1: persistent kernel)
    // options (0 = automatic)
    int opt_variant, opt_bn, opt_split_k, opt_grid, opt_group_m;
    int prefetch;  // L2 prefetch distance in K blocks (GEMM_EPI_OPT_PREFETCH)
    int no_pdl;    // 1: launch without programmatic dependent launch (GEMM_EPI_OPT_PDL = 0)
    unsigned long long wait_limit_ns;
    int debug_stall;
    int* d_status;
    // tensor maps for the last (A, B, D) pointers
    const void* key_A;
    const void* key_B;
    const void* key_D;
    bool maps_valid;
    CUtensorMap tm_A, tm_B, tm_D;
    char desc[320];
    HostPipe* host;  // gemm_epi_execute_host's streams, buffers and chunk plans
};

namespace {

// Split-K is used only when GEMM_EPI_OPT_SPLIT_K asks for it.  Measured on GB300, the
// cluster launch, the two cluster barriers and the partial-sum exchange cost more than the
// shorter K loop saves on every under-filled shape tried (1024x512x2048: 15.5 us unsplit vs
// 19-20 us split; GELU T=16/64/256 x 3072 x 768: 9.2/11.1/16.8 us unsplit vs 10.2/22/28 us
// with split 4), so a plan does not split by itself.

int normalise_split(int split, int k_blocks, int* kb_per_split)
{
    if (split > k_blocks) split = k_blocks;
    if (split < 1) split = 1;
    const int kpb = (k_blocks + split - 1) / split;
    *kb_per_split = kpb;
    return (k_blocks + kpb - 1) / kpb;
}

// N tile of the row-tile kernel.  When the widest tile already gives every SM a tile, that
// one (fewest operand bytes per flop).  Otherwise the width whose busiest CTA moves the
// fewest operand bytes (waves of tiles x K blocks x stage bytes).
int pick_rowtile_bn(int64_t m, int64_t n, int k_blocks, int sm_count)
{
    const int64_t tm = (m + 127) / 128;
    if (tm * ((n + 255) / 256) >= sm_count) return 256;
    int best = 256;
    double best_cost = 1e300;
    for (int bn : {64, 128, 256}) {
        const long long tiles = tm * ((n + bn - 1) / bn);
        const long long waves = (tiles + sm_count - 1) / sm_count;
        const double cost = static_cast<double>(waves) * k_blocks * (16384.0 + bn * 128.0);
        if (cost < best_cost) {
            best_cost = cost;
            best = bn;
        }
    }
    return best;
}

// N tile of the CTA-pair kernel: 224 when it needs fewer 256-row tile waves over the resident
// pairs than 256 does, else 256.  Both stage the same 32 KB of operands per CTA and K block
// (224 wide leaves part of the second 64-column B panel unused), and measured on GB300 a
// 224-wide tile costs about what a 256-wide one does, so only the wave count decides:
// 4096 x 4096 on 76 pairs is 4 waves either way (256: 3.4 paid as 4), and 224 gives the
// shorter last tile (4096 x 4096 x 1024 GELU: 38.5 us against 41.0 us).
int pick_pair_bn(int64_t m, int64_t n, long long pairs)
{
    const int64_t tm = (m + 255) / 256;
    const long long w256 = (tm * ((n + 255) / 256) + pairs - 1) / pairs;
    const long long w224 = (tm * ((n + 223) / 224) + pairs - 1) / pairs;
    return w224 <= w256 ? 224 : 256;
}

gemm_epi_status configure(gemm_epi_plan_s* p)
{
    p->maps_valid = false;
    p->bn = p->stages = p->smem = p->grid = p->tiles_m = p->tiles_n = p->k_blocks = 0;
    p->group_m = 1;
    p->split = 1;
    p->kb_per_split = 0;
    if (p->m == 0 || p->n == 0) {
        p->variant = kEmpty;
    } else if (p->k == 0) {
        p->variant = kBiasOnly;
    } else if (p->dtype == GEMM_EPI_E4M3) {
        // E4M3: the CTA-pair kernel with 256 x 256 tiles and 128-deep K blocks, any shape
        if ((p->opt_variant != 0 && p->opt_variant != 3) || (p->opt_bn != 0 && p->opt_bn != 256))
            return GEMM_EPI_ERR_INVALID_ARG;
        if (fp8_pair_prepare() != cudaSuccess || rowpair_prepare(256) != cudaSuccess)
            return GEMM_EPI_ERR_LAUNCH;
        p->variant = kRowPair;
        p->bn = 256;
        p->k_blocks = static_cast<int>((p->k + 127) / 128);
        p->tiles_m = static_cast<int>((p->m + 255) / 256);
        p->tiles_n = static_cast<int>((p->n + 255) / 256);
        p->stages = rowpair_stages(256);
        p->smem = rowpair_smem_bytes(256);
        long long pairs = rowpair_max_clusters(256);
        if (pairs > p->sm_count / 2) pairs = p->sm_count / 2;
        if (p->opt_grid > 0 && p->opt_grid / 2 < pairs) pairs = p->opt_grid / 2;
        if (pairs < 1) return GEMM_EPI_ERR_LAUNCH;
        const long long tiles = static_cast<long long>(p->tiles_m) * p->tiles_n;
        if (pairs > tiles) pairs = tiles;
        p->kb_per_split = p->k_blocks;
        p->grid = static_cast<int>(2 * pairs);
        int gm = p->opt_group_m ? p->opt_group_m : 8;
        if (gm > p->tiles_m) gm = p->tiles_m;
        p->group_m = gm < 1 ? 1 : gm;
    } else {
        int v = p->opt_variant;
        if (v == 0) {
            // small m: swapped; enough 256 x 256 tiles for most CTA pairs: the pair kernel
            // (half the operand bytes per flop in every SM); else the single-CTA row tiles
            const long long pair_tiles = ((p->m + 255) / 256) * ((p->n + 255) / 256);
            if (p->m <= kSwappedMaxM && p->epilog != GEMM_EPI_LN_GELU_BIAS)
                v = kSwapped;
            else if (pair_tiles * 10 >= static_cast<long long>(p->sm_count / 2) * 8)
                v = kRowPair;
            else
                v = kRowTile;
        }
        if (v == 3) v = kRowPair;  // option value 3 selects the CTA-pair kernel
        if (v == kSwapped && p->m > kSwappedMaxM) return GEMM_EPI_ERR_INVALID_ARG;
        // the swapped kernel has no LayerNorm epilogue
        if (v == kSwapped && p->epilog == GEMM_EPI_LN_GELU_BIAS) return GEMM_EPI_ERR_INVALID_ARG;
        p->variant = v;
        p->k_blocks = static_cast<int>((p->k + 63) / 64);
        if (v == kRowPair) {
            // CTA pairs on 256 x BN tiles, persistent, no split
            if (p->opt_bn && p->opt_bn != 224 && p->opt_bn != 256)
                return GEMM_EPI_ERR_INVALID_ARG;
            if (rowpair_prepare(256) != cudaSuccess) return GEMM_EPI_ERR_LAUNCH;
            long long pairs = rowpair_max_clusters(256);  // same shared memory for every BN
            if (pairs > p->sm_count / 2) pairs = p->sm_count / 2;
            if (p->opt_grid > 0 && p->opt_grid / 2 < pairs) pairs = p->opt_grid / 2;
            if (pairs < 1) return GEMM_EPI_ERR_LAUNCH;
            p->bn = p->opt_bn ? p->opt_bn : pick_pair_bn(p->m, p->n, pairs);
            p->tiles_m = static_cast<int>((p->m + 255) / 256);
            p->tiles_n = static_cast<int>((p->n + p->bn - 1) / p->bn);
            p->stages = rowpair_stages(p->bn);
            p->smem = rowpair_smem_bytes(p->bn);
            if (rowpair_prepare(p->bn) != cudaSuccess) return GEMM_EPI_ERR_LAUNCH;
            const long long tiles = static_cast<long long>(p->tiles_m) * p->tiles_n;
            if (pairs > tiles) pairs = tiles;
            p->kb_per_split = p->k_blocks;
            p->grid = static_cast<int>(2 * pairs);
            int gm = p->opt_group_m ? p->opt_group_m : 8;
            if (gm > p->tiles_m) gm = p->tiles_m;
            p->group_m = gm < 1 ? 1 : gm;
        } else if (v == kRowTile) {
            if (p->opt_bn && p->opt_bn != 64 && p->opt_bn != 128 && p->opt_bn != 256)
                return GEMM_EPI_ERR_INVALID_ARG;
            p->bn = p->opt_bn ? p->opt_bn : pick_rowtile_bn(p->m, p->n, p->k_blocks, p->sm_count);
            p->tiles_m = static_cast<int>((p->m + 127) / 128);
            p->tiles_n = static_cast<int>((p->n + p->bn - 1) / p->bn);
            p->stages = rowtile_stages(p->bn);
            p->smem = rowtile_smem_bytes(p->bn);
        } else {
            int bn = 16;
            while (bn < p->m) bn *= 2;
            p->bn = bn;
            p->tiles_m = static_cast<int>((p->n + 127) / 128);
            p->tiles_n = static_cast<int>((p->m + bn - 1) / bn);
            p->stages = swapped_stages(bn);
            p->smem = swapped_smem_bytes(bn);
        }
    }
    if (p->variant == kRowTile || p->variant == kSwapped) {
        const int v = p->variant;
        const long long tiles = static_cast<long long>(p->tiles_m) * p->tiles_n;
        cudaError_t e = v == kRowTile ? rowtile_prepare(p->bn) : swapped_prepare(p->bn);
        if (e != cudaSuccess) return GEMM_EPI_ERR_LAUNCH;
        const int want_split = p->opt_split_k > 0 ? p->opt_split_k : 1;
        p->split = normalise_split(want_split, p->k_blocks, &p->kb_per_split);
        long long grid;
        if (p->split > 1) {
            grid = tiles * p->split;  // one cluster per tile, not persistent
            if (grid > (1ll << 30)) return GEMM_EPI_ERR_UNSUPPORTED_SHAPE;
        } else {
            p->kb_per_split = p->k_blocks;
            grid = tiles < p->sm_count ? tiles : p->sm_count;
            if (p->opt_grid > 0 && p->opt_grid < grid) grid = p->opt_grid;
        }
        p->grid = static_cast<int>(grid);
        int gm = p->opt_group_m ? p->opt_group_m : 16;
        if (gm > p->tiles_m) gm = p->tiles_m;
        p->group_m = gm < 1 ? 1 : gm;
    }
    static const char* vname[] = {"empty", "row-tile", "swapped", "bias-only", "row-pair"};
    static const char* ename[] = {"BIAS",          "RELU_BIAS",     "GELU_BIAS",
                                  "RELU_AUX_BIAS", "BIAS_RESIDUAL", "NONE",
                                  "TANH_BIAS",     "GELU_AUX_BIAS", "DRELU_BGRAD",
                                  "DGELU_BGRAD",   "LN_GELU_BIAS"};
    snprintf(p->desc, sizeof(p->desc),
             "m=%lld n=%lld k=%lld dtype=%s epilog=%s bias=%s variant=%s tile=%dx%d bk=%d "
             "stages=%d smem=%d tiles=%dx%d k_blocks=%d split_k=%d grid=%d group_m=%d sms=%d",
             static_cast<long long>(p->m), static_cast<long long>(p->n),
             static_cast<long long>(p->k),
             p->dtype == GEMM_EPI_E4M3 ? "e4m3" : p->dtype == GEMM_EPI_BF16 ? "bf16" : "f16",
             ename[p->epilog], p->bias_layout == GEMM_EPI_BIAS_M1 ? "(m,1)" : "(1,n)",
             vname[p->variant], p->variant == kRowPair ? 256 : 128, p->bn,
             p->dtype == GEMM_EPI_E4M3 ? 128 : 64, p->stages, p->smem, p->tiles_m, p->tiles_n,
             p->k_blocks,
             p->split, p->grid, p->group_m, p->sm_count);
    const char* log = getenv("GEMM_EPI_LOG");
    if (log && log[0] == '1') fprintf(stderr, "[gemm_epi] plan: %s\n", p->desc);
    return GEMM_EPI_OK;
}

bool encode_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, uint64_t inner,
               uint64_t outer, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw,
               uint64_t elem_bytes = 2)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * elem_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

gemm_epi_status ensure_maps(gemm_epi_plan_s* p, const void* A, const void* B, void* D)
{
    if (p->maps_valid && p->key_A == A && p->key_B == B && p->key_D == D) return GEMM_EPI_OK;
    p->maps_valid = false;
    if (p->dtype == GEMM_EPI_E4M3) {
        // A [m][k] and B transposed [n][k], bytes, K-major boxes {128 k, 128 rows}; D bf16
        const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
        if (!encode_2d(&p->tm_A, A, u8, p->k, p->m, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B, 1) ||
            !encode_2d(&p->tm_B, B, u8, p->k, p->n, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B, 1) ||
            !encode_2d(&p->tm_D, D, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, p->n, p->m, 32, 32,
                       CU_TENSOR_MAP_SWIZZLE_64B))
            return GEMM_EPI_ERR_LAUNCH;
        p->key_A = A;
        p->key_B = B;
        p->key_D = D;
        p->maps_valid = true;
        return GEMM_EPI_OK;
    }
    const CUtensorMapDataType dt = p->dtype == GEMM_EPI_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const bool rows_of_a = p->variant == kRowTile || p->variant == kRowPair;
    const uint32_t a_rows = rows_of_a ? 128u : static_cast<uint32_t>(p->bn);
    if (!encode_2d(&p->tm_A, A, dt, p->k, p->m, 64, a_rows, CU_TENSOR_MAP_SWIZZLE_128B))
        return GEMM_EPI_ERR_LAUNCH;
    if (!encode_2d(&p->tm_B, B, dt, p->n, p->k, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B))
        return GEMM_EPI_ERR_LAUNCH;
    if (rows_of_a) {
        if (!encode_2d(&p->tm_D, D, dt, p->n, p->m, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
            return GEMM_EPI_ERR_LAUNCH;
    } else {
        // swapped kernel: boxes of 32 columns x (up to) 32 rows of D, transposed on chip
        const uint32_t rows = p->bn < 32 ? static_cast<uint32_t>(p->bn) : 32u;
        if (!encode_2d(&p->tm_D, D, dt, p->n, p->m, 32, rows, CU_TENSOR_MAP_SWIZZLE_NONE))
            return GEMM_EPI_ERR_LAUNCH;
    }
    p->key_A = A;
    p->key_B = B;
    p->key_D = D;
    p->maps_valid = true;
    return GEMM_EPI_OK;
}

gemm_epi_status check_device(const gemm_epi_plan_s* p)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_EPI_ERR_NO_DEVICE;
    if (dev != p->device) return GEMM_EPI_ERR_INVALID_ARG;
    return GEMM_EPI_OK;
}

gemm_epi_status launch_gemm(gemm_epi_plan_s* p, const gemm_epi_operands& ops, int epilog,
                            cudaStream_t stream, bool pdl = false)
{
    gemm_epi_status st = ensure_maps(p, ops.A, ops.B, ops.D);
    if (st != GEMM_EPI_OK) return st;
    GemmParams prm;
    memset(&prm, 0, sizeof(prm));
    prm.tm_A = p->tm_A;
    prm.tm_B = p->tm_B;
    prm.tm_D = p->tm_D;
    prm.bias = ops.bias;
    prm.residual = ops.residual;
    prm.D = ops.D;
    prm.aux = ops.aux;
    prm.aux_in = ops.aux_in;
    prm.dbias = ops.dbias;
    prm.ln_stats = ops.ln_stats;
    prm.ln_colsum = ops.ln_colsum;
    prm.ln_bias = ops.ln_bias;
    prm.scale_a = ops.scale_a;
    prm.scale_b = ops.scale_b;
    prm.status = p->d_status;
    prm.wait_limit_ns = p->wait_limit_ns;
    prm.m = static_cast<int>(p->m);
    prm.n = static_cast<int>(p->n);
    prm.k = static_cast<int>(p->k);
    prm.tiles_m = p->tiles_m;
    prm.tiles_n = p->tiles_n;
    prm.k_blocks = p->k_blocks;
    prm.group_m = p->group_m;
    prm.epilog = epilog;
    prm.bias_layout = p->bias_layout;
    prm.bf16 = p->dtype == GEMM_EPI_F16 ? 0 : 1;  // E4M3 plans write bf16
    prm.aux_ld = static_cast<int>((p->n + 31) / 32);
    prm.debug_stall = p->debug_stall;
    prm.split = p->split;
    prm.kb_per_split = p->kb_per_split;
    prm.prefetch = p->prefetch;
    cudaError_t e;
    if (p->variant == kRowPair && p->dtype == GEMM_EPI_E4M3)
        e = fp8_pair_launch(prm, p->grid, stream, pdl);
    else if (p->variant == kRowPair)
        e = rowpair_launch(p->bn, prm, p->grid, stream, pdl);
    else if (p->variant == kRowTile)
        e = rowtile_launch(p->bn, prm, p->grid, stream, pdl);
    else
        e = swapped_launch(p->bn, prm, p->grid, stream, pdl);
    if (e != cudaSuccess) {
        const char* log = getenv("GEMM_EPI_LOG");
        if (log && log[0] == '1')
            fprintf(stderr, "[gemm_epi] launch failed: %s (%s)\n", cudaGetErrorString(e), p->desc);
        return GEMM_EPI_ERR_LAUNCH;
    }
    return GEMM_EPI_OK;
}

gemm_epi_status check_device(const gemm_epi_plan_s* p);

bool backward(int epilog) { return epilog == GEMM_EPI_DRELU_BGRAD || epilog == GEMM_EPI_DGELU_BGRAD; }

int64_t dbias_len(const gemm_epi_plan_s* p) { return p->bias_layout == GEMM_EPI_BIAS_M1 ? p->m : p->n; }

// Backward calls: dbias is accumulated atomically, so it starts from zero on the stream.
gemm_epi_status zero_dbias(const gemm_epi_plan_s* p, const gemm_epi_operands& ops,
                           cudaStream_t stream)
{
    if (!backward(p->epilog) || dbias_len(p) == 0) return GEMM_EPI_OK;
    return cudaMemsetAsync(ops.dbias, 0, sizeof(float) * static_cast<size_t>(dbias_len(p)),
                           stream) == cudaSuccess
               ? GEMM_EPI_OK
               : GEMM_EPI_ERR_LAUNCH;
}

cudaError_t run_elementwise(const gemm_epi_plan_s* p, const void* pre,
                            const gemm_epi_operands& ops, cudaStream_t stream)
{
    ElementwiseArgs a;
    a.pre = pre;
    a.bias = ops.bias;
    a.residual = ops.residual;
    a.D = ops.D;
    a.aux = ops.aux;
    a.aux_in = ops.aux_in;
    a.dbias = ops.dbias;
    a.ln_stats = ops.ln_stats;
    a.ln_colsum = ops.ln_colsum;
    a.ln_bias = ops.ln_bias;
    a.m = static_cast<int>(p->m);
    a.n = static_cast<int>(p->n);
    a.epilog = p->epilog;
    a.bias_layout = p->bias_layout;
    a.bf16 = p->dtype == GEMM_EPI_F16 ? 0 : 1;  // E4M3 plans write bf16
    a.aux_ld = static_cast<int>((p->n + 31) / 32);
    return elementwise_launch(a, p->sm_count, stream);
}

// One fused call on an already-checked plan: empty problems launch nothing, k == 0 runs the
// elementwise epilogue on the bias alone, everything else the GEMM kernel.
gemm_epi_status run_plan(gemm_epi_plan_s* p, const gemm_epi_operands& ops, cudaStream_t stream,
                         bool pdl)
{
    gemm_epi_status st = zero_dbias(p, ops, stream);
    if (st != GEMM_EPI_OK || p->variant == kEmpty) return st;
    if (p->variant == kBiasOnly)
        return run_elementwise(p, nullptr, ops, stream) == cudaSuccess ? GEMM_EPI_OK
                                                                        : GEMM_EPI_ERR_LAUNCH;
    // (a backward launch follows the memset of dbias: plain stream order)
    return launch_gemm(p, ops, p->epilog, stream, pdl && !p->no_pdl && !backward(p->epilog));
}

gemm_epi_status check_operands(const gemm_epi_plan_s* p, const gemm_epi_operands& o)
{
    const int e = p->epilog;
    const bool bwd = backward(e);
    if (bwd && o.bias) return GEMM_EPI_ERR_INVALID_ARG;
    if (bwd && dbias_len(p) > 0 && !o.dbias) return GEMM_EPI_ERR_INVALID_ARG;
    if (o.dbias && !aligned(o.dbias, 4)) return GEMM_EPI_ERR_MISALIGNED;
    // An empty problem touches no operand but dbias (its matrices may have no storage).
    if (p->variant == kEmpty) return GEMM_EPI_OK;
    const bool f8 = p->dtype == GEMM_EPI_E4M3;
    if ((o.scale_a != nullptr) != f8 || (o.scale_b != nullptr) != f8) return GEMM_EPI_ERR_INVALID_ARG;
    if (f8 && (!aligned(o.scale_a, 4) || !aligned(o.scale_b, 4))) return GEMM_EPI_ERR_MISALIGNED;
    const bool ln = e == GEMM_EPI_LN_GELU_BIAS;
    if (((o.ln_stats != nullptr) != ln) || ((o.ln_colsum != nullptr) != ln) ||
        ((o.ln_bias != nullptr) != ln))
        return GEMM_EPI_ERR_INVALID_ARG;
    if (ln && (!aligned(o.ln_stats, 8) || !aligned(o.ln_colsum, 4) || !aligned(o.ln_bias, 4)))
        return GEMM_EPI_ERR_MISALIGNED;
    const bool needs_res = e == GEMM_EPI_BIAS_RESIDUAL;
    const bool needs_aux = e == GEMM_EPI_RELU_AUX_BIAS || e == GEMM_EPI_GELU_AUX_BIAS;
    if ((o.aux != nullptr) != needs_aux) return GEMM_EPI_ERR_INVALID_ARG;
    if ((o.residual != nullptr) != needs_res) return GEMM_EPI_ERR_INVALID_ARG;
    if ((o.aux_in != nullptr) != bwd || (o.dbias != nullptr) != bwd) return GEMM_EPI_ERR_INVALID_ARG;
    if (!o.D) return GEMM_EPI_ERR_INVALID_ARG;
    if (p->k > 0 && (!o.A || !o.B)) return GEMM_EPI_ERR_INVALID_ARG;
    if (e != GEMM_EPI_NONE && !bwd && !ln && !o.bias) return GEMM_EPI_ERR_INVALID_ARG;
    if (ln && o.bias) return GEMM_EPI_ERR_INVALID_ARG;
    const uintptr_t aux_align = e == GEMM_EPI_GELU_AUX_BIAS ? 16 : 4;
    const uintptr_t aux_in_align = e == GEMM_EPI_DGELU_BGRAD ? 16 : 4;
    if (!aligned(o.D, 16) || (o.A && !aligned(o.A, 16)) || (o.B && !aligned(o.B, 16)) ||
        (o.residual && !aligned(o.residual, 16)) || (o.bias && !aligned(o.bias, 2)) ||
        (o.aux && !aligned(o.aux, aux_align)) || (o.aux_in && !aligned(o.aux_in, aux_in_align)))
        return GEMM_EPI_ERR_MISALIGNED;
    return GEMM_EPI_OK;
}

gemm_epi_operands make_operands(const void* A, const void* B, const void* bias,
                                const void* residual, void* D, void* aux)
{
    gemm_epi_operands o;
    memset(&o, 0, sizeof(o));
    o.A = A;
    o.B = B;
    o.bias = bias;
    o.residual = residual;
    o.D = D;
    o.aux = aux;
    return o;
}

}  // namespace

// ---- host buffers: row chunks, pipelined copies and GEMMs ---------------------------------

// gemm_epi_execute_host: A, D (and residual, aux) are split into row chunks; chunk j's
// host-to-device copy, GEMM and device-to-host copy run on three streams, each waiting only
// for what it needs, with two device slots per chunked operand, so the copies of chunks
// j+1 and j-1 overlap the GEMM of chunk j.  B and the bias are copied once per call.
struct HostPipe {
    int64_t chunk = 0;  // rows per chunk (the last may be shorter)
    cudaStream_t s_in = nullptr, s_comp = nullptr, s_out = nullptr;
    cudaEvent_t ev_start = nullptr, ev_shared = nullptr;
    cudaEvent_t ev_in[2] = {nullptr, nullptr}, ev_comp[2] = {nullptr, nullptr},
                ev_out[2] = {nullptr, nullptr};
    void* dA[2] = {nullptr, nullptr};
    void* dD[2] = {nullptr, nullptr};
    void* dR[2] = {nullptr, nullptr};
    void* dAux[2] = {nullptr, nullptr};
    void* dB = nullptr;
    void* dBias = nullptr;
    gemm_epi_plan_s full{}, last{};  // the chunk plans (sharing the parent's status word)
    bool has_last = false;
};

namespace {

void destroy_host_pipe(gemm_epi_plan_s* p)
{
    HostPipe* h = p->host;
    if (!h) return;
    for (cudaStream_t st : {h->s_in, h->s_comp, h->s_out})
        if (st) {
            cudaStreamSynchronize(st);
            cudaStreamDestroy(st);
        }
    for (cudaEvent_t e : {h->ev_start, h->ev_shared, h->ev_in[0], h->ev_in[1], h->ev_comp[0],
                          h->ev_comp[1], h->ev_out[0], h->ev_out[1]})
        if (e) cudaEventDestroy(e);
    for (void* b : {h->dA[0], h->dA[1], h->dD[0], h->dD[1], h->dR[0], h->dR[1], h->dAux[0],
                    h->dAux[1], h->dB, h->dBias})
        if (b) cudaFree(b);
    delete h;
    p->host = nullptr;
}

// Rows per chunk: about 1024-row chunks, at most 16 of them (a chunk of a large problem still
// fills the machine), whole 128-row tiles.  The copies out cannot start before the first
// chunk's inputs are in and its GEMM is done, so more, smaller chunks shorten that fill;
// measured on GB300 with ~190 GB/s each way to pinned host memory, the 65536 x 16384 x 8192
// step is then bound by the 2 GiB copy of D out.
int64_t host_chunk_rows(int64_t m)
{
    int64_t chunks = m / 1024;
    if (chunks < 1) chunks = 1;
    if (chunks > 16) chunks = 16;
    int64_t rows = (m + chunks - 1) / chunks;
    rows = (rows + 127) / 128 * 128;
    return rows < m ? rows : m;
}

gemm_epi_status chunk_plan(const gemm_epi_plan_s* p, int64_t rows, gemm_epi_plan_s* c)
{
    memset(c, 0, sizeof(*c));
    c->m = rows;
    c->n = p->n;
    c->k = p->k;
    c->dtype = p->dtype;
    c->epilog = p->epilog;
    c->bias_layout = p->bias_layout;
    c->device = p->device;
    c->sm_count = p->sm_count;
    c->opt_variant = p->opt_variant;
    c->opt_bn = p->opt_bn;
    c->opt_split_k = p->opt_split_k;
    c->opt_grid = p->opt_grid;
    c->opt_group_m = p->opt_group_m;
    c->prefetch = p->prefetch;
    c->no_pdl = p->no_pdl;
    c->wait_limit_ns = p->wait_limit_ns;
    c->d_status = p->d_status;
    return configure(c);
}

gemm_epi_status make_host_pipe(gemm_epi_plan_s* p)
{
    if (p->host) return GEMM_EPI_OK;
    HostPipe* h = new (std::nothrow) HostPipe();
    if (!h) return GEMM_EPI_ERR_ALLOC;
    p->host = h;
    h->chunk = host_chunk_rows(p->m);
    gemm_epi_status st = chunk_plan(p, h->chunk, &h->full);
    const int64_t rem = p->m % h->chunk;
    h->has_last = rem != 0;
    if (st == GEMM_EPI_OK && h->has_last) st = chunk_plan(p, rem, &h->last);
    if (st != GEMM_EPI_OK) {
        destroy_host_pipe(p);
        return st;
    }
    bool ok = true;
    for (cudaStream_t* st2 : {&h->s_in, &h->s_comp, &h->s_out})
        ok = ok && cudaStreamCreateWithFlags(st2, cudaStreamNonBlocking) == cudaSuccess;
    for (cudaEvent_t* e : {&h->ev_start, &h->ev_shared, &h->ev_in[0], &h->ev_in[1], &h->ev_comp[0],
                           &h->ev_comp[1], &h->ev_out[0], &h->ev_out[1]})
        ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
    const size_t e2 = 2;
    const size_t a_bytes = static_cast<size_t>(h->chunk) * p->k * e2;
    const size_t d_bytes = static_cast<size_t>(h->chunk) * p->n * e2;
    const size_t aux_bytes = static_cast<size_t>(h->chunk) * ((p->n + 31) / 32) * 4;
    const size_t b_bytes = static_cast<size_t>(p->k) * p->n * e2;
    const size_t bias_bytes = static_cast<size_t>(p->bias_layout == GEMM_EPI_BIAS_M1 ? p->m : p->n) * e2;
    auto alloc = [&](void** ptr, size_t bytes) {
        if (!ok || bytes == 0) return;
        ok = cudaMalloc(ptr, bytes) == cudaSuccess;
    };
    for (int s = 0; s < 2; ++s) {
        alloc(&h->dA[s], a_bytes);
        alloc(&h->dD[s], d_bytes);
        if (p->epilog == GEMM_EPI_BIAS_RESIDUAL) alloc(&h->dR[s], d_bytes);
        if (p->epilog == GEMM_EPI_RELU_AUX_BIAS || p->epilog == GEMM_EPI_GELU_AUX_BIAS)
            alloc(&h->dAux[s], p->epilog == GEMM_EPI_GELU_AUX_BIAS ? d_bytes : aux_bytes);
    }
    alloc(&h->dB, b_bytes);
    if (p->epilog != GEMM_EPI_NONE) alloc(&h->dBias, bias_bytes);
    if (!ok) {
        cudaGetLastError();
        destroy_host_pipe(p);
        return GEMM_EPI_ERR_ALLOC;
    }
    return GEMM_EPI_OK;
}

gemm_epi_status run_host(gemm_epi_plan_s* p, const gemm_epi_operands& o, cudaStream_t stream)
{
    gemm_epi_status st = make_host_pipe(p);
    if (st != GEMM_EPI_OK) return st;
    HostPipe* h = p->host;
    const size_t e2 = 2;
    const int64_t ldw = (p->n + 31) / 32;
    const size_t aux_row = p->epilog == GEMM_EPI_GELU_AUX_BIAS ? static_cast<size_t>(p->n) * e2
                                                             : static_cast<size_t>(ldw) * 4;
    const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
    bool ok = cudaEventRecord(h->ev_start, stream) == cudaSuccess;
    for (cudaStream_t s : {h->s_in, h->s_comp, h->s_out})
        ok = ok && cudaStreamWaitEvent(s, h->ev_start, 0) == cudaSuccess;
    // operands every chunk needs
    if (ok && h->dB)
        ok = cudaMemcpyAsync(h->dB, o.B, static_cast<size_t>(p->k) * p->n * e2, h2d, h->s_in) ==
             cudaSuccess;
    if (ok && h->dBias)
        ok = cudaMemcpyAsync(h->dBias, o.bias,
                             static_cast<size_t>(p->bias_layout == GEMM_EPI_BIAS_M1 ? p->m : p->n) * e2,
                             h2d, h->s_in) == cudaSuccess;
    ok = ok && cudaEventRecord(h->ev_shared, h->s_in) == cudaSuccess;
    const int64_t nchunks = (p->m + h->chunk - 1) / h->chunk;
    int last_slot = 0;
    for (int64_t j = 0; ok && j < nchunks; ++j) {
        const int s = static_cast<int>(j & 1);
        const int64_t r0 = j * h->chunk;
        const int64_t rows = p->m - r0 < h->chunk ? p->m - r0 : h->chunk;
        gemm_epi_plan_s* c = rows == h->chunk ? &h->full : &h->last;
        // in: slot s is free once the GEMM of chunk j - 2 has read it
        ok = cudaStreamWaitEvent(h->s_in, h->ev_comp[s], 0) == cudaSuccess;
        if (ok && p->k > 0)
            ok = cudaMemcpyAsync(h->dA[s], static_cast<const char*>(o.A) + r0 * p->k * e2,
                                 static_cast<size_t>(rows) * p->k * e2, h2d, h->s_in) == cudaSuccess;
        if (ok && h->dR[s])
            ok = cudaMemcpyAsync(h->dR[s], static_cast<const char*>(o.residual) + r0 * p->n * e2,
                                 static_cast<size_t>(rows) * p->n * e2, h2d, h->s_in) == cudaSuccess;
        ok = ok && cudaEventRecord(h->ev_in[s], h->s_in) == cudaSuccess;
        // the GEMM: after its inputs, and after chunk j - 2's results left slot s
        ok = ok && cudaStreamWaitEvent(h->s_comp, h->ev_in[s], 0) == cudaSuccess &&
             cudaStreamWaitEvent(h->s_comp, h->ev_shared, 0) == cudaSuccess &&
             cudaStreamWaitEvent(h->s_comp, h->ev_out[s], 0) == cudaSuccess;
        if (!ok) break;
        gemm_epi_operands co = make_operands(
            h->dA[s], h->dB,
            h->dBias ? static_cast<const char*>(h->dBias) +
                           (p->bias_layout == GEMM_EPI_BIAS_M1 ? r0 * static_cast<int64_t>(e2) : 0)
                     : nullptr,
            h->dR[s], h->dD[s], h->dAux[s]);
        st = run_plan(c, co, h->s_comp, false);
        if (st != GEMM_EPI_OK) return st;
        ok = cudaEventRecord(h->ev_comp[s], h->s_comp) == cudaSuccess;
        // out
        ok = ok && cudaStreamWaitEvent(h->s_out, h->ev_comp[s], 0) == cudaSuccess;
        if (ok)
            ok = cudaMemcpyAsync(static_cast<char*>(o.D) + r0 * p->n * e2, h->dD[s],
                                 static_cast<size_t>(rows) * p->n * e2, d2h, h->s_out) == cudaSuccess;
        if (ok && h->dAux[s])
            ok = cudaMemcpyAsync(static_cast<char*>(o.aux) + r0 * aux_row, h->dAux[s],
                                 static_cast<size_t>(rows) * aux_row, d2h, h->s_out) == cudaSuccess;
        ok = ok && cudaEventRecord(h->ev_out[s], h->s_out) == cudaSuccess;
        last_slot = s;
    }
    // the caller's stream continues once the last results are in host memory (the copies
    // on s_out run in order, so the last one is the end of all of them)
    ok = ok && cudaStreamWaitEvent(stream, h->ev_out[last_slot], 0) == cudaSuccess;
    if (!ok) {
        cudaGetLastError();
        return GEMM_EPI_ERR_LAUNCH;
    }
    return GEMM_EPI_OK;
}

}  // namespace

extern "C" {

gemm_epi_status gemm_epi_plan(gemm_epi_plan_t* out, int64_t m, int64_t n, int64_t k,
                              gemm_epi_dtype dtype, gemm_epi_epilog epilog,
                              gemm_epi_bias_layout bias_layout)
{
    if (!out) return GEMM_EPI_ERR_INVALID_ARG;
    *out = nullptr;
    if (dtype != GEMM_EPI_F16 && dtype != GEMM_EPI_BF16 && dtype != GEMM_EPI_E4M3)
        return GEMM_EPI_ERR_INVALID_ARG;
    if (epilog < GEMM_EPI_BIAS || epilog > GEMM_EPI_LN_GELU_BIAS) return GEMM_EPI_ERR_INVALID_ARG;
    if (dtype == GEMM_EPI_E4M3 && !fp8_epilog(epilog)) return GEMM_EPI_ERR_INVALID_ARG;
    if (bias_layout != GEMM_EPI_BIAS_M1 && bias_layout != GEMM_EPI_BIAS_1N)
        return GEMM_EPI_ERR_INVALID_ARG;
    const int64_t kMax = (1ll << 31) - 1;
    if (m < 0 || n < 0 || k < 0 || m > kMax || n > kMax || k > kMax)
        return GEMM_EPI_ERR_UNSUPPORTED_SHAPE;
    if (n % 8 != 0 || k % 8 != 0) return GEMM_EPI_ERR_UNSUPPORTED_SHAPE;
    // E4M3 rows are k bytes long: a multiple of 16 for the tensor-memory-access unit
    if (dtype == GEMM_EPI_E4M3 && k % 16 != 0) return GEMM_EPI_ERR_UNSUPPORTED_SHAPE;
    if (epilog == GEMM_EPI_LN_GELU_BIAS && k == 0) return GEMM_EPI_ERR_UNSUPPORTED_SHAPE;

    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev < 1) {
        cudaGetLastError();
        return GEMM_EPI_ERR_NO_DEVICE;
    }
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_EPI_ERR_NO_DEVICE;
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (major != 10 || minor != 3) return GEMM_EPI_ERR_ARCH;

    gemm_epi_plan_s* p = new (std::nothrow) gemm_epi_plan_s();
    if (!p) return GEMM_EPI_ERR_ALLOC;
    p->m = m;
    p->n = n;
    p->k = k;
    p->dtype = dtype;
    p->epilog = epilog;
    p->bias_layout = bias_layout;
    p->device = dev;
    p->sm_count = sms;
    p->wait_limit_ns = kDefaultWaitNs;
    if (cudaMalloc(reinterpret_cast<void**>(&p->d_status), sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        delete p;
        return GEMM_EPI_ERR_ALLOC;
    }
    if (cudaMemset(p->d_status, 0, sizeof(int)) != cudaSuccess) {
        cudaFree(p->d_status);
        delete p;
        return GEMM_EPI_ERR_ALLOC;
    }
    gemm_epi_status st = configure(p);
    if (st != GEMM_EPI_OK) {
        cudaFree(p->d_status);
        delete p;
        return st;
    }
    *out = p;
    return GEMM_EPI_OK;
}

gemm_epi_status gemm_epi_plan_set_option(gemm_epi_plan_t p, gemm_epi_option opt, int64_t value)
{
    if (!p) return GEMM_EPI_ERR_INVALID_ARG;
    gemm_epi_plan_s saved = *p;
    switch (opt) {
    case GEMM_EPI_OPT_VARIANT:
        if (value < 0 || value > 3) return GEMM_EPI_ERR_INVALID_ARG;
        p->opt_variant = static_cast<int>(value);
        break;
    case GEMM_EPI_OPT_TILE_N:
        if (value != 0 && value != 64 && value != 128 && value != 224 && value != 256)
            return GEMM_EPI_ERR_INVALID_ARG;
        p->opt_bn = static_cast<int>(value);
        break;
    case GEMM_EPI_OPT_SPLIT_K:
        if (value < 0 || value > 8) return GEMM_EPI_ERR_INVALID_ARG;
        p->opt_split_k = static_cast<int>(value);
        break;
    case GEMM_EPI_OPT_GRID:
        if (value < 0 || value > (1 << 20)) return GEMM_EPI_ERR_INVALID_ARG;
        p->opt_grid = static_cast<int>(value);
        break;
    case GEMM_EPI_OPT_GROUP_M:
        if (value < 0 || value > (1 << 20)) return GEMM_EPI_ERR_INVALID_ARG;
        p->opt_group_m = static_cast<int>(value);
        break;
    case GEMM_EPI_OPT_WAIT_LIMIT_US:
        if (value < 0 || value > 600ll * 1000 * 1000) return GEMM_EPI_ERR_INVALID_ARG;
        p->wait_limit_ns = value == 0 ? kDefaultWaitNs : static_cast<unsigned long long>(value) * 1000ull;
        return GEMM_EPI_OK;
    case GEMM_EPI_OPT_PREFETCH:
        if (value < 0 || value > 64) return GEMM_EPI_ERR_INVALID_ARG;
        p->prefetch = static_cast<int>(value);
        return GEMM_EPI_OK;
    case GEMM_EPI_OPT_PDL:
        if (value != 0 && value != 1) return GEMM_EPI_ERR_INVALID_ARG;
        p->no_pdl = value ? 0 : 1;
        return GEMM_EPI_OK;
    case GEMM_EPI_OPT_DEBUG_STALL:
        if (value != 0 && value != 1) return GEMM_EPI_ERR_INVALID_ARG;
        p->debug_stall = static_cast<int>(value);
        return GEMM_EPI_OK;
    default:
        return GEMM_EPI_ERR_INVALID_ARG;
    }
    gemm_epi_status st = configure(p);
    if (st != GEMM_EPI_OK) {
        *p = saved;  // keep the previous, valid configuration
        p->maps_valid = false;
    } else {
        destroy_host_pipe(p);  // its chunk plans follow the options: rebuilt on next use
    }
    return st;
}

gemm_epi_status gemm_epi_execute_operands(gemm_epi_plan_t p, const gemm_epi_operands* ops,
                                          cudaStream_t stream)
{
    if (!p || !ops) return GEMM_EPI_ERR_INVALID_ARG;
    gemm_epi_status st = check_operands(p, *ops);
    if (st != GEMM_EPI_OK) return st;
    if (p->variant == kEmpty && (!backward(p->epilog) || dbias_len(p) == 0)) return GEMM_EPI_OK;
    st = check_device(p);
    if (st != GEMM_EPI_OK) return st;
    // Every global access of the fused kernel waits for the previous grid on the stream
    // (griddepcontrol.wait), so it is launched as a programmatic dependent: its launch and
    // set-up overlap the tail of whatever runs before it.
    return run_plan(p, *ops, stream, true);
}

gemm_epi_status gemm_epi_execute_ex(gemm_epi_plan_t p, const void* A, const void* B,
                                    const void* bias, const void* residual, void* D,
                                    uint32_t* aux, cudaStream_t stream)
{
    const gemm_epi_operands o = make_operands(A, B, bias, residual, D, aux);
    return gemm_epi_execute_operands(p, &o, stream);
}

gemm_epi_status gemm_epi_execute(gemm_epi_plan_t p, const void* A, const void* B,
                                 const void* bias, void* D, uint32_t* aux, cudaStream_t stream)
{
    if (p && p->epilog == GEMM_EPI_BIAS_RESIDUAL) return GEMM_EPI_ERR_INVALID_ARG;
    return gemm_epi_execute_ex(p, A, B, bias, nullptr, D, aux, stream);
}

gemm_epi_status gemm_epi_execute_operands_unfused(gemm_epi_plan_t p,
                                                  const gemm_epi_operands* ops, void* pre,
                                                  cudaStream_t stream)
{
    if (!p || !ops) return GEMM_EPI_ERR_INVALID_ARG;
    gemm_epi_status st = check_operands(p, *ops);
    if (st != GEMM_EPI_OK) return st;
    if (p->variant != kEmpty) {
        if (!pre) return GEMM_EPI_ERR_INVALID_ARG;
        if (!aligned(pre, 16)) return GEMM_EPI_ERR_MISALIGNED;
    } else if (!backward(p->epilog) || dbias_len(p) == 0) {
        return GEMM_EPI_OK;
    }
    st = check_device(p);
    if (st != GEMM_EPI_OK) return st;
    st = zero_dbias(p, *ops, stream);
    if (st != GEMM_EPI_OK || p->variant == kEmpty) return st;
    const void* pre_in = nullptr;
    if (p->variant != kBiasOnly) {
        gemm_epi_operands g = make_operands(ops->A, ops->B, nullptr, nullptr, pre, nullptr);
        g.scale_a = ops->scale_a;  // E4M3: the GEMM applies the scales
        g.scale_b = ops->scale_b;
        st = launch_gemm(p, g, EPI_NONE, stream);
        if (st != GEMM_EPI_OK) return st;
        pre_in = pre;
    }
    return run_elementwise(p, pre_in, *ops, stream) == cudaSuccess ? GEMM_EPI_OK
                                                                   : GEMM_EPI_ERR_LAUNCH;
}

gemm_epi_status gemm_epi_execute_host(gemm_epi_plan_t p, const gemm_epi_operands* ops,
                                      cudaStream_t stream)
{
    if (!p || !ops) return GEMM_EPI_ERR_INVALID_ARG;
    const int e = p->epilog;
    if (p->dtype == GEMM_EPI_E4M3 || backward(e) || e == GEMM_EPI_LN_GELU_BIAS)
        return GEMM_EPI_ERR_INVALID_ARG;
    gemm_epi_status st = check_operands(p, *ops);
    if (st != GEMM_EPI_OK) return st;
    if (p->variant == kEmpty) return GEMM_EPI_OK;
    st = check_device(p);
    if (st != GEMM_EPI_OK) return st;
    return run_host(p, *ops, stream);
}

gemm_epi_status gemm_epi_execute_unfused(gemm_epi_plan_t p, const void* A, const void* B,
                                         const void* bias, const void* residual, void* pre,
                                         void* D, uint32_t* aux, cudaStream_t stream)
{
    const gemm_epi_operands o = make_operands(A, B, bias, residual, D, aux);
    return gemm_epi_execute_operands_unfused(p, &o, pre, stream);
}

gemm_epi_status gemm_epi_free(gemm_epi_plan_t p)
{
    if (!p) return GEMM_EPI_OK;
    destroy_host_pipe(p);
    if (p->d_status) cudaFree(p->d_status);
    delete p;
    return GEMM_EPI_OK;
}

gemm_epi_status gemm_epi_sync_status(gemm_epi_plan_t p, cudaStream_t stream)
{
    if (!p) return GEMM_EPI_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return GEMM_EPI_ERR_LAUNCH;
    int h = 0;
    if (cudaMemcpy(&h, p->d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return GEMM_EPI_ERR_LAUNCH;
    if (h != 0) {
        cudaMemset(p->d_status, 0, sizeof(int));
        return GEMM_EPI_ERR_DEVICE_TIMEOUT;
    }
    return GEMM_EPI_OK;
}

const char* gemm_epi_status_string(gemm_epi_status s)
{
    switch (s) {
    case GEMM_EPI_OK: return "GEMM_EPI_OK";
    case GEMM_EPI_ERR_INVALID_ARG: return "GEMM_EPI_ERR_INVALID_ARG: invalid argument";
    case GEMM_EPI_ERR_UNSUPPORTED_SHAPE:
        return "GEMM_EPI_ERR_UNSUPPORTED_SHAPE: sizes must be >= 0 and n, k multiples of 8";
    case GEMM_EPI_ERR_MISALIGNED: return "GEMM_EPI_ERR_MISALIGNED: pointer alignment";
    case GEMM_EPI_ERR_NO_DEVICE: return "GEMM_EPI_ERR_NO_DEVICE: no CUDA device";
    case GEMM_EPI_ERR_ARCH: return "GEMM_EPI_ERR_ARCH: the current device is not sm_103";
    case GEMM_EPI_ERR_ALLOC: return "GEMM_EPI_ERR_ALLOC: allocation failed";
    case GEMM_EPI_ERR_LAUNCH: return "GEMM_EPI_ERR_LAUNCH: CUDA launch or encode failed";
    case GEMM_EPI_ERR_DEVICE_TIMEOUT:
        return "GEMM_EPI_ERR_DEVICE_TIMEOUT: a kernel gave up on a device-side wait";
    case GEMM_EPI_ERR_SCRATCH_LIMIT:
        return "GEMM_EPI_ERR_SCRATCH_LIMIT: t*f exceeds the static scratch of the "
               "allocation-free FFN call (GEMM_EPI_FFN_NOALLOC_MAX_HIDDEN elements)";
    default: return "GEMM_EPI_ERR_UNKNOWN";
    }
}

const char* gemm_epi_plan_describe(gemm_epi_plan_t p) { return p ? p->desc : ""; }

}  // extern "C"

// ---- the FFN block ----------------------------------------------------------------------

struct gemm_epi_ffn_plan_s {
    int64_t t, d, f;
    int dtype;
    gemm_epi_plan_t g1;  // H = GELU(X.W1 + b1):   t x f, k = d
    gemm_epi_plan_t g2;  // Y = H.W2 + b2 + R:     t x d, k = f
    void* H;
    bool layernorm;      // GEMM 1 is LN_GELU_BIAS on the raw X; stats holds (mu, rstd) per row
    float* stats;
    // one-launch mode: both GEMMs in one CTA-pair kernel (256 x 256 tiles)
    int opt_launches;  // GEMM_EPI_FFN_OPT_LAUNCHES value (0 = automatic)
    bool one_launch;   // the mode in use
    int* ready;        // per 256-row block of H: epilogue warps done with it
    int tiles_m, tiles_n1, tiles_n2, grid;
    const void* key_X;
    const void* key_W1;
    const void* key_W2;
    const void* key_Y;
    bool maps_valid;
    CUtensorMap tm_X, tm_W1, tm_Hs, tm_Hl, tm_W2, tm_Y;
    char desc[400];
};

namespace {

// One launch pays off on long walks: there the second GEMM's K loops run beside the first
// GEMM's last tiles and their GELU epilogues instead of after them.  Measured on GB300
// (bf16, hot L2): t x d x f = 8192 x 1024 x 4096, 640 tiles of 256 x 256: 100.8 us in one
// launch, 102.7 us in two; 4096 x 2048 x 8192: 170.6 against 173.8 us; but 4096 x 1024 x 4096,
// 320 tiles: 65.6 against 60.5 us, where the two-launch plan's 224-wide first GEMM fills
// its four waves exactly.  So: one launch from six waves of tiles over the resident pairs.
bool pick_one_launch(const gemm_epi_ffn_plan_s* p, long long pairs)
{
    if (p->opt_launches == 1) return true;
    if (p->opt_launches == 2) return false;
    if (p->g1->variant != kRowPair || p->g2->variant != kRowPair) return false;
    const long long tiles = ((p->t + 255) / 256) * ((p->f + 255) / 256 + (p->d + 255) / 256);
    return tiles >= 6 * pairs;
}

gemm_epi_status configure_ffn(gemm_epi_ffn_plan_s* p)
{
    p->maps_valid = false;
    if (p->layernorm) {  // the one-launch kernel runs GELU_BIAS only
        p->one_launch = false;
        snprintf(p->desc, sizeof(p->desc), "two launches after the row statistics: [%s] then [%s]",
                 p->g1->desc, p->g2->desc);
        return GEMM_EPI_OK;
    }
    p->tiles_m = static_cast<int>((p->t + 255) / 256);
    p->tiles_n1 = static_cast<int>((p->f + 255) / 256);
    p->tiles_n2 = static_cast<int>((p->d + 255) / 256);
    p->grid = 0;
    if (ffn_pair_prepare() != cudaSuccess || rowpair_prepare(256) != cudaSuccess)
        return GEMM_EPI_ERR_LAUNCH;
    long long pairs = rowpair_max_clusters(256);
    if (pairs > p->g1->sm_count / 2) pairs = p->g1->sm_count / 2;
    p->one_launch = p->t > 0 && p->d > 0 && p->f > 0 && pick_one_launch(p, pairs);
    if (p->one_launch) {
        const long long tiles = static_cast<long long>(p->tiles_m) * (p->tiles_n1 + p->tiles_n2);
        if (pairs > tiles) pairs = tiles;
        if (pairs < 1) return GEMM_EPI_ERR_LAUNCH;
        p->grid = static_cast<int>(2 * pairs);
        if (!p->ready && cudaMalloc(reinterpret_cast<void**>(&p->ready),
                                    sizeof(int) * static_cast<size_t>(p->tiles_m)) != cudaSuccess) {
            cudaGetLastError();
            p->ready = nullptr;
            return GEMM_EPI_ERR_ALLOC;
        }
        snprintf(p->desc, sizeof(p->desc),
                 "one launch: t=%lld d=%lld f=%lld, CTA pairs on 256x256 tiles: %dx%d GEMM-1 tiles "
                 "then %dx%d GEMM-2 tiles, grid=%d",
                 static_cast<long long>(p->t), static_cast<long long>(p->d),
                 static_cast<long long>(p->f), p->tiles_m, p->tiles_n1, p->tiles_m, p->tiles_n2,
                 p->grid);
    } else {
        snprintf(p->desc, sizeof(p->desc), "two launches: [%s] then [%s]", p->g1->desc,
                 p->g2->desc);
    }
    return GEMM_EPI_OK;
}

gemm_epi_status ensure_ffn_maps(gemm_epi_ffn_plan_s* p, const void* X, const void* W1,
                                const void* W2, void* Y)
{
    if (p->maps_valid && p->key_X == X && p->key_W1 == W1 && p->key_W2 == W2 && p->key_Y == Y)
        return GEMM_EPI_OK;
    p->maps_valid = false;
    const CUtensorMapDataType dt = p->dtype == GEMM_EPI_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const uint64_t t = static_cast<uint64_t>(p->t), d = static_cast<uint64_t>(p->d),
                   f = static_cast<uint64_t>(p->f);
    const CUtensorMapSwizzle sw128 = CU_TENSOR_MAP_SWIZZLE_128B, sw64 = CU_TENSOR_MAP_SWIZZLE_64B;
    if (!encode_2d(&p->tm_X, X, dt, d, t, 64, 128, sw128) ||
        !encode_2d(&p->tm_W1, W1, dt, f, d, 64, 64, sw128) ||
        !encode_2d(&p->tm_Hs, p->H, dt, f, t, 32, 32, sw64) ||
        !encode_2d(&p->tm_Hl, p->H, dt, f, t, 64, 128, sw128) ||
        !encode_2d(&p->tm_W2, W2, dt, d, f, 64, 64, sw128) ||
        !encode_2d(&p->tm_Y, Y, dt, d, t, 32, 32, sw64))
        return GEMM_EPI_ERR_LAUNCH;
    p->key_X = X;
    p->key_W1 = W1;
    p->key_W2 = W2;
    p->key_Y = Y;
    p->maps_valid = true;
    return GEMM_EPI_OK;
}

gemm_epi_status run_ffn_one_launch(gemm_epi_ffn_plan_s* p, const void* X, const void* W1,
                                   const void* b1, const void* W2, const void* b2, const void* R,
                                   void* Y, cudaStream_t stream)
{
    gemm_epi_status st = ensure_ffn_maps(p, X, W1, W2, Y);
    if (st != GEMM_EPI_OK) return st;
    if (cudaMemsetAsync(p->ready, 0, sizeof(int) * static_cast<size_t>(p->tiles_m), stream) !=
        cudaSuccess)
        return GEMM_EPI_ERR_LAUNCH;
    const gemm_epi_plan_s* g1 = p->g1;
    GemmParams prm;
    memset(&prm, 0, sizeof(prm));
    prm.tm_A = p->tm_X;
    prm.tm_B = p->tm_W1;
    prm.tm_D = p->tm_Hs;
    prm.bias = b1;
    prm.D = p->H;
    prm.status = g1->d_status;
    prm.wait_limit_ns = g1->wait_limit_ns;
    prm.m = static_cast<int>(p->t);
    prm.n = static_cast<int>(p->f);
    prm.k = static_cast<int>(p->d);
    prm.tiles_m = p->tiles_m;
    prm.tiles_n = p->tiles_n1;
    prm.k_blocks = static_cast<int>((p->d + 63) / 64);
    prm.group_m = p->tiles_m < 8 ? p->tiles_m : 8;
    prm.epilog = EPI_GELU_BIAS;
    prm.bias_layout = GEMM_EPI_BIAS_1N;
    prm.bf16 = p->dtype == GEMM_EPI_BF16 ? 1 : 0;
    prm.aux_ld = static_cast<int>((p->f + 31) / 32);
    prm.split = 1;
    prm.kb_per_split = prm.k_blocks;
    prm.tm_A2 = p->tm_Hl;
    prm.tm_B2 = p->tm_W2;
    prm.tm_D2 = p->tm_Y;
    prm.bias2 = b2;
    prm.residual2 = R;
    prm.ffn_ready = p->ready;
    prm.ffn_ready_target = p->tiles_n1 * 2 * kEpilogueWarps;
    prm.ffn_tiles2 = p->tiles_m * p->tiles_n2;
    prm.n2 = static_cast<int>(p->d);
    prm.tiles_n2 = p->tiles_n2;
    prm.k_blocks2 = static_cast<int>((p->f + 63) / 64);
    const cudaError_t e = ffn_pair_launch(prm, p->grid, stream);
    if (e != cudaSuccess) {
        const char* log = getenv("GEMM_EPI_LOG");
        if (log && log[0] == '1')
            fprintf(stderr, "[gemm_epi] FFN launch failed: %s (%s)\n", cudaGetErrorString(e),
                    p->desc);
        return GEMM_EPI_ERR_LAUNCH;
    }
    return GEMM_EPI_OK;
}

}  // namespace

extern "C" {

}  // extern "C"

namespace {

gemm_epi_status make_ffn_plan(gemm_epi_ffn_plan_t* out, int64_t t, int64_t d, int64_t f,
                              gemm_epi_dtype dtype, bool layernorm)
{
    if (!out) return GEMM_EPI_ERR_INVALID_ARG;
    *out = nullptr;
    if (dtype != GEMM_EPI_F16 && dtype != GEMM_EPI_BF16) return GEMM_EPI_ERR_INVALID_ARG;
    gemm_epi_plan_t g1 = nullptr, g2 = nullptr;
    gemm_epi_status st = gemm_epi_plan(&g1, t, f, d, dtype,
                                       layernorm ? GEMM_EPI_LN_GELU_BIAS : GEMM_EPI_GELU_BIAS,
                                       GEMM_EPI_BIAS_1N);
    if (st != GEMM_EPI_OK) return st;
    st = gemm_epi_plan(&g2, t, d, f, dtype, GEMM_EPI_BIAS_RESIDUAL, GEMM_EPI_BIAS_1N);
    if (st != GEMM_EPI_OK) {
        gemm_epi_free(g1);
        return st;
    }
    gemm_epi_ffn_plan_s* p = new (std::nothrow) gemm_epi_ffn_plan_s();
    if (!p) {
        gemm_epi_free(g1);
        gemm_epi_free(g2);
        return GEMM_EPI_ERR_ALLOC;
    }
    p->t = t;
    p->d = d;
    p->f = f;
    p->dtype = dtype;
    p->g1 = g1;
    p->g2 = g2;
    p->H = nullptr;
    p->ready = nullptr;
    p->stats = nullptr;
    p->layernorm = layernorm;
    if (t > 0 && f > 0) {
        if (cudaMalloc(&p->H, static_cast<size_t>(t) * static_cast<size_t>(f) * 2) != cudaSuccess) {
            cudaGetLastError();
            gemm_epi_ffn_free(p);
            return GEMM_EPI_ERR_ALLOC;
        }
    }
    if (layernorm && t > 0) {
        if (cudaMalloc(reinterpret_cast<void**>(&p->stats), sizeof(float) * 2 * static_cast<size_t>(t)) !=
            cudaSuccess) {
            cudaGetLastError();
            p->stats = nullptr;
            gemm_epi_ffn_free(p);
            return GEMM_EPI_ERR_ALLOC;
        }
    }
    st = configure_ffn(p);
    if (st != GEMM_EPI_OK) {
        gemm_epi_ffn_free(p);
        return st;
    }
    *out = p;
    return GEMM_EPI_OK;
}

// The current device, checked to be sm_103, and its SM count.
gemm_epi_status current_device(int* sms)
{
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev < 1) {
        cudaGetLastError();
        return GEMM_EPI_ERR_NO_DEVICE;
    }
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_EPI_ERR_NO_DEVICE;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
    if (major != 10 || minor != 3) return GEMM_EPI_ERR_ARCH;
    return GEMM_EPI_OK;
}

bool ln_shape_ok(int64_t t, int64_t d)
{
    const int64_t kMax = (1ll << 31) - 1;
    return t >= 0 && d >= 8 && d % 8 == 0 && t <= kMax && d <= kMax && t * d <= (1ll << 40);
}

}  // namespace

extern "C" {

gemm_epi_status gemm_epi_ffn_plan(gemm_epi_ffn_plan_t* out, int64_t t, int64_t d, int64_t f,
                                  gemm_epi_dtype dtype)
{
    return make_ffn_plan(out, t, d, f, dtype, false);
}

gemm_epi_status gemm_epi_ffn_plan_layernorm(gemm_epi_ffn_plan_t* out, int64_t t, int64_t d,
                                            int64_t f, gemm_epi_dtype dtype)
{
    if (d == 0) return GEMM_EPI_ERR_UNSUPPORTED_SHAPE;
    return make_ffn_plan(out, t, d, f, dtype, true);
}

gemm_epi_status gemm_epi_ffn_execute_layernorm(gemm_epi_ffn_plan_t p, const void* X, float eps,
                                               const void* W1_folded, const float* colsum,
                                               const float* b1_folded, const void* W2,
                                               const void* b2, const void* R, void* Y,
                                               cudaStream_t stream)
{
    if (!p || !p->layernorm || !(eps >= 0.0f)) return GEMM_EPI_ERR_INVALID_ARG;
    gemm_epi_operands o1 = make_operands(X, W1_folded, nullptr, nullptr, p->H ? p->H : Y, nullptr);
    o1.ln_stats = p->stats ? p->stats : colsum;  // (t == 0: never read)
    o1.ln_colsum = colsum;
    o1.ln_bias = b1_folded;
    const gemm_epi_operands o2 = make_operands(p->H, W2, b2, R, Y, nullptr);
    gemm_epi_status st = check_operands(p->g1, o1);
    if (st != GEMM_EPI_OK) return st;
    st = check_operands(p->g2, o2);
    if (st != GEMM_EPI_OK) return st;
    if (p->t == 0) return GEMM_EPI_OK;
    st = check_device(p->g1);
    if (st != GEMM_EPI_OK) return st;
    if (layernorm_stats_launch(X, static_cast<int>(p->t), static_cast<int>(p->d),
                               p->dtype == GEMM_EPI_BF16 ? 1 : 0, eps, p->stats,
                               p->g1->sm_count, stream) != cudaSuccess)
        return GEMM_EPI_ERR_LAUNCH;
    st = run_plan(p->g1, o1, stream, true);
    if (st != GEMM_EPI_OK) return st;
    return run_plan(p->g2, o2, stream, p->g1->variant != kEmpty);
}

gemm_epi_status gemm_epi_layernorm(int64_t t, int64_t d, gemm_epi_dtype dtype, const void* X,
                                   const void* residual, const void* gamma, const void* beta,
                                   float eps, void* Y, cudaStream_t stream)
{
    if (dtype != GEMM_EPI_F16 && dtype != GEMM_EPI_BF16) return GEMM_EPI_ERR_INVALID_ARG;
    if (!ln_shape_ok(t, d)) return GEMM_EPI_ERR_UNSUPPORTED_SHAPE;
    if (!(eps >= 0.0f) || !(eps < 1e30f)) return GEMM_EPI_ERR_INVALID_ARG;
    if (t == 0) return GEMM_EPI_OK;
    if (!X || !gamma || !beta || !Y) return GEMM_EPI_ERR_INVALID_ARG;
    if (!aligned(X, 16) || !aligned(Y, 16) || (residual && !aligned(residual, 16)) ||
        !aligned(gamma, 2) || !aligned(beta, 2))
        return GEMM_EPI_ERR_MISALIGNED;
    int sms = 0;
    gemm_epi_status st = current_device(&sms);
    if (st != GEMM_EPI_OK) return st;
    return layernorm_launch(X, residual, gamma, beta, Y, static_cast<int>(t), static_cast<int>(d),
                            dtype == GEMM_EPI_BF16 ? 1 : 0, eps, sms, stream) == cudaSuccess
               ? GEMM_EPI_OK
               : GEMM_EPI_ERR_LAUNCH;
}

gemm_epi_status gemm_epi_layernorm_stats(int64_t t, int64_t d, gemm_epi_dtype dtype,
                                         const void* X, float eps, float* stats,
                                         cudaStream_t stream)
{
    if (dtype != GEMM_EPI_F16 && dtype != GEMM_EPI_BF16) return GEMM_EPI_ERR_INVALID_ARG;
    if (!ln_shape_ok(t, d)) return GEMM_EPI_ERR_UNSUPPORTED_SHAPE;
    if (!(eps >= 0.0f) || !(eps < 1e30f)) return GEMM_EPI_ERR_INVALID_ARG;
    if (t == 0) return GEMM_EPI_OK;
    if (!X || !stats) return GEMM_EPI_ERR_INVALID_ARG;
    if (!aligned(X, 16) || !aligned(stats, 8)) return GEMM_EPI_ERR_MISALIGNED;
    int sms = 0;
    gemm_epi_status st = current_device(&sms);
    if (st != GEMM_EPI_OK) return st;
    return layernorm_stats_launch(X, static_cast<int>(t), static_cast<int>(d),
                                  dtype == GEMM_EPI_BF16 ? 1 : 0, eps, stats, sms, stream) ==
                   cudaSuccess
               ? GEMM_EPI_OK
               : GEMM_EPI_ERR_LAUNCH;
}

gemm_epi_status gemm_epi_layernorm_fold(int64_t d, int64_t f, gemm_epi_dtype dtype,
                                        const void* gamma, const void* beta, const void* W,
                                        const void* b, void* W_folded, float* colsum,
                                        float* bias_folded, cudaStream_t stream)
{
    if (dtype != GEMM_EPI_F16 && dtype != GEMM_EPI_BF16) return GEMM_EPI_ERR_INVALID_ARG;
    if (!ln_shape_ok(f, d) || f % 8 != 0) return GEMM_EPI_ERR_UNSUPPORTED_SHAPE;
    if (f == 0) return GEMM_EPI_OK;
    if (!gamma || !beta || !W || !b || !W_folded || !colsum || !bias_folded)
        return GEMM_EPI_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(W_folded, 16) || !aligned(gamma, 2) || !aligned(beta, 2) ||
        !aligned(b, 2) || !aligned(colsum, 4) || !aligned(bias_folded, 4))
        return GEMM_EPI_ERR_MISALIGNED;
    int sms = 0;
    gemm_epi_status st = current_device(&sms);
    if (st != GEMM_EPI_OK) return st;
    return layernorm_fold_launch(gamma, beta, W, b, W_folded, colsum, bias_folded,
                                 static_cast<int>(d), static_cast<int>(f),
                                 dtype == GEMM_EPI_BF16 ? 1 : 0, sms, stream) == cudaSuccess
               ? GEMM_EPI_OK
               : GEMM_EPI_ERR_LAUNCH;
}

gemm_epi_status gemm_epi_ffn_set_option(gemm_epi_ffn_plan_t p, gemm_epi_ffn_option opt,
                                        int64_t value)
{
    if (!p) return GEMM_EPI_ERR_INVALID_ARG;
    if (opt != GEMM_EPI_FFN_OPT_LAUNCHES || value < 0 || value > 2) return GEMM_EPI_ERR_INVALID_ARG;
    const int saved = p->opt_launches;
    p->opt_launches = static_cast<int>(value);
    gemm_epi_status st = configure_ffn(p);
    if (st != GEMM_EPI_OK) {
        p->opt_launches = saved;
        configure_ffn(p);
    }
    return st;
}

const char* gemm_epi_ffn_plan_describe(gemm_epi_ffn_plan_t p) { return p ? p->desc : ""; }

gemm_epi_status gemm_epi_ffn_execute(gemm_epi_ffn_plan_t p, const void* X, const void* W1,
                                     const void* b1, const void* W2, const void* b2,
                                     const void* R, void* Y, cudaStream_t stream)
{
    if (!p || p->layernorm) return GEMM_EPI_ERR_INVALID_ARG;
    const gemm_epi_operands o1 = make_operands(X, W1, b1, nullptr, p->H ? p->H : Y, nullptr);
    const gemm_epi_operands o2 = make_operands(p->H, W2, b2, R, Y, nullptr);
    gemm_epi_status st = check_operands(p->g1, o1);
    if (st != GEMM_EPI_OK) return st;
    st = check_operands(p->g2, o2);
    if (st != GEMM_EPI_OK) return st;
    if (p->t == 0 || p->d == 0) return GEMM_EPI_OK;
    st = check_device(p->g1);
    if (st != GEMM_EPI_OK) return st;
    if (p->one_launch) return run_ffn_one_launch(p, X, W1, b1, W2, b2, R, Y, stream);
    st = run_plan(p->g1, o1, stream, true);
    if (st != GEMM_EPI_OK) return st;
    // GEMM 2 reads H only after GEMM 1 has completed (griddepcontrol.wait in its producer).
    return run_plan(p->g2, o2, stream, p->g1->variant != kEmpty);
}

const void* gemm_epi_ffn_hidden(gemm_epi_ffn_plan_t p) { return p ? p->H : nullptr; }

gemm_epi_status gemm_epi_ffn_sync_status(gemm_epi_ffn_plan_t p, cudaStream_t stream)
{
    if (!p) return GEMM_EPI_ERR_INVALID_ARG;
    gemm_epi_status s1 = gemm_epi_sync_status(p->g1, stream);
    gemm_epi_status s2 = gemm_epi_sync_status(p->g2, stream);
    return s1 != GEMM_EPI_OK ? s1 : s2;
}

gemm_epi_status gemm_epi_ffn_free(gemm_epi_ffn_plan_t p)
{
    if (!p) return GEMM_EPI_OK;
    if (p->H) cudaFree(p->H);
    if (p->ready) cudaFree(p->ready);
    if (p->stats) cudaFree(p->stats);
    gemm_epi_free(p->g1);
    gemm_epi_free(p->g2);
    delete p;
    return GEMM_EPI_OK;
}

int64_t gemm_epi_aux_words_per_row(int64_t n) { return n <= 0 ? 0 : (n + 31) / 32; }

}  // extern "C"

// ---- the FFN block without allocation ------------------------------------------------------
//
// For callers that cannot allocate device memory.  The hidden activation and the status
// words of the two launches live in one file-scope device array; its device address is
// looked up once per device (with that device current) and then passed to the kernels.

namespace {

constexpr size_t kNoAllocStatusBytes = 256;  // two status words, padded to 256 bytes
constexpr size_t kNoAllocHiddenBytes = static_cast<size_t>(GEMM_EPI_FFN_NOALLOC_MAX_HIDDEN) * 2;

// In host code this name is only a stand-in; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char
    g_ffn_noalloc_scratch[kNoAllocStatusBytes + kNoAllocHiddenBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
unsigned char* g_noalloc_addr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on device `dev` (the current device); the first call
// per device looks it up and zeroes the status words.
gemm_epi_status noalloc_scratch(int dev, unsigned char** out)
{
    if (dev < 0 || dev >= kNoAllocMaxDevices) return GEMM_EPI_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_ffn_noalloc_scratch) != cudaSuccess || !ptr) {
            cudaGetLastError();
            return GEMM_EPI_ERR_LAUNCH;
        }
        if (cudaMemset(ptr, 0, kNoAllocStatusBytes) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_EPI_ERR_LAUNCH;
        }
        g_noalloc_addr[dev] = static_cast<unsigned char*>(ptr);
    }
    *out = g_noalloc_addr[dev];
    return GEMM_EPI_OK;
}

// A plan on the caller's stack whose status word points into the static scratch.
gemm_epi_status stack_plan(gemm_epi_plan_s* p, int64_t m, int64_t n, int64_t k, int dtype,
                           int epilog, int dev, int sms, int* status)
{
    memset(p, 0, sizeof(*p));
    p->m = m;
    p->n = n;
    p->k = k;
    p->dtype = dtype;
    p->epilog = epilog;
    p->bias_layout = GEMM_EPI_BIAS_1N;
    p->device = dev;
    p->sm_count = sms;
    p->wait_limit_ns = kDefaultWaitNs;
    p->d_status = status;
    return configure(p);
}

}  // namespace

extern "C" gemm_epi_status gemm_epi_ffn_execute_noalloc(int64_t t, int64_t d, int64_t f,
                                                        gemm_epi_dtype dtype, const void* X,
                                                        const void* W1, const void* b1,
                                                        const void* W2, const void* b2,
                                                        const void* R, void* Y,
                                                        cudaStream_t stream)
{
    if (dtype != GEMM_EPI_F16 && dtype != GEMM_EPI_BF16) return GEMM_EPI_ERR_INVALID_ARG;
    const int64_t kMax = (1ll << 31) - 1;
    if (t < 0 || d < 0 || f < 0 || t > kMax || d > kMax || f > kMax)
        return GEMM_EPI_ERR_UNSUPPORTED_SHAPE;
    if (d % 8 != 0 || f % 8 != 0) return GEMM_EPI_ERR_UNSUPPORTED_SHAPE;
    if (f > 0 && t > GEMM_EPI_FFN_NOALLOC_MAX_HIDDEN / f) return GEMM_EPI_ERR_SCRATCH_LIMIT;

    int dev = 0, major = 0, minor = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return GEMM_EPI_ERR_NO_DEVICE;
    }
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (major != 10 || minor != 3) return GEMM_EPI_ERR_ARCH;

    unsigned char* scratch = nullptr;
    gemm_epi_status st = noalloc_scratch(dev, &scratch);
    if (st != GEMM_EPI_OK) return st;
    int* status = reinterpret_cast<int*>(scratch);
    void* H = scratch + kNoAllocStatusBytes;

    gemm_epi_plan_s g1, g2;
    st = stack_plan(&g1, t, f, d, dtype, GEMM_EPI_GELU_BIAS, dev, sms, status);
    if (st != GEMM_EPI_OK) return st;
    st = stack_plan(&g2, t, d, f, dtype, GEMM_EPI_BIAS_RESIDUAL, dev, sms, status + 1);
    if (st != GEMM_EPI_OK) return st;
    const gemm_epi_operands o1 = make_operands(X, W1, b1, nullptr, H, nullptr);
    const gemm_epi_operands o2 = make_operands(H, W2, b2, R, Y, nullptr);
    st = check_operands(&g1, o1);
    if (st != GEMM_EPI_OK) return st;
    st = check_operands(&g2, o2);
    if (st != GEMM_EPI_OK) return st;
    if (t == 0 || d == 0) return GEMM_EPI_OK;
    st = run_plan(&g1, o1, stream, false);
    if (st != GEMM_EPI_OK) return st;
    return run_plan(&g2, o2, stream, g1.variant != kEmpty);
}
