// The FFN block as one plan ("Operator fusion in model inference, from LayerNorm to residual
// connections" (wmrh.cn/news/429806), section 1 and its flowchart; section 3 for the
// residual): GEMM 1 with bias + GELU, GEMM 2 with bias + residual, run as two fused launches
// or as one persistent CTA-pair kernel; optionally behind a LayerNorm folded into GEMM 1's
// epilogue (section 2); and an allocation-free form of the plain block.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "plan.h"

using namespace gemm_epi;
using namespace gemm_epi_impl;

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
    int opt_split2;    // GEMM_EPI_FFN_OPT_SPLIT2 value
    int opt_order;     // GEMM_EPI_FFN_OPT_TILE_ORDER value
    bool one_launch;   // the mode in use: one CTA-pair launch, H through L2
    bool onchip;       // ... or one launch with H kept on chip (opt_launches == 3)
    // per (256-row block of H, GEMM-2 K slice): epilogue warps done with it; then the
    // GEMM-2 slice counts (per tile, CTA of the pair and epilogue warp), zeroed together
    int* ready;
    size_t ready_bytes;
    int split2, kb2;   // GEMM-2 K slices and K blocks per slice
    float* ws;         // the slices' fp32 partial sums (split2 > 1)
    size_t ws_bytes;
    bool dynamic;      // one launch: units from the device counter
    int tiles_m, tiles_n1, tiles_n2, grid;
    const void* key_X;
    const void* key_W1;
    const void* key_W2;
    const void* key_Y;
    bool maps_valid;
    CUtensorMap tm_X, tm_W1, tm_Hs, tm_Hl, tm_W2, tm_Y;
    char desc[720];  // room for both GEMM plans' descriptions (320 bytes each) and the text
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

// K blocks per GEMM-2 slice for `want` slices of k_blocks2 (whole 256-column tiles of H).
// Splitting is never automatic: each slice's fp32 partial sums (128 KiB per CTA) go out to
// L2 and the last slice reads all of them back, on the same per-SM path that feeds the
// MMAs their operands.  Measured on GB300 (bf16, hot L2, dynamic order), 4096 x 1024 x 4096:
// 94 us in 4 slices against 66 us unsplit (a copy-out took 3.0 us per unit, the last
// slice's read-back and epilogue 8.7 us, and the epilogue warps fell behind the MMAs);
// 8192 x 1024 x 4096: 173 against 104 us; 512 x 1024 x 4096: 39 against 43 us, but two
// launches take 31 us there.
int slice_kblocks(int k_blocks2, int want)
{
    const int kb = (k_blocks2 + want - 1) / want;
    return (kb + 3) / 4 * 4;
}

gemm_epi_status configure_ffn(gemm_epi_ffn_plan_s* p)
{
    p->maps_valid = false;
    if (p->layernorm) {  // the one-launch kernel runs GELU_BIAS only
        p->one_launch = false;
        p->onchip = false;
        if (p->opt_launches == 3) return GEMM_EPI_ERR_INVALID_ARG;
        snprintf(p->desc, sizeof(p->desc), "two launches after the row statistics: [%s] then [%s]",
                 p->g1->desc, p->g2->desc);
        return GEMM_EPI_OK;
    }
    p->tiles_m = static_cast<int>((p->t + 255) / 256);
    p->tiles_n1 = static_cast<int>((p->f + 255) / 256);
    p->tiles_n2 = static_cast<int>((p->d + 255) / 256);
    p->grid = 0;
    p->onchip = p->opt_launches == 3;
    if (p->onchip) {
        // H kept on chip: one CTA per (128 tokens, 256 columns of Y), chunks of 256 of H
        p->one_launch = false;
        if (p->d % 256 != 0 || p->f % 256 != 0) return GEMM_EPI_ERR_UNSUPPORTED_SHAPE;
        if (ffn_onchip_prepare() != cudaSuccess) return GEMM_EPI_ERR_LAUNCH;
        const long long grid = ((p->t + 127) / 128) * (p->d / 256);
        if (grid > (1ll << 30)) return GEMM_EPI_ERR_UNSUPPORTED_SHAPE;
        p->grid = static_cast<int>(grid);
        snprintf(p->desc, sizeof(p->desc),
                 "one launch, H on chip: t=%lld d=%lld f=%lld, one CTA per 128 tokens x 256 columns "
                 "of Y, %lld chunks of 256 of H, grid=%d",
                 static_cast<long long>(p->t), static_cast<long long>(p->d),
                 static_cast<long long>(p->f), static_cast<long long>(p->f / 256), p->grid);
        return GEMM_EPI_OK;
    }
    if (ffn_pair_prepare() != cudaSuccess || rowpair_prepare(256) != cudaSuccess)
        return GEMM_EPI_ERR_LAUNCH;
    long long pairs = rowpair_max_clusters(256);
    if (pairs > p->g1->sm_count / 2) pairs = p->g1->sm_count / 2;
    const int k_blocks2 = static_cast<int>((p->f + 63) / 64);
    const bool shape_ok = p->t > 0 && p->d > 0 && p->f > 0;
    const int want2 = p->opt_split2 > 1 ? p->opt_split2 : 1;
    p->kb2 = want2 > 1 ? slice_kblocks(k_blocks2, want2) : k_blocks2;
    p->split2 = shape_ok ? (k_blocks2 + p->kb2 - 1) / p->kb2 : 1;
    if (p->split2 <= 1) {
        p->split2 = 1;
        p->kb2 = k_blocks2;
    }
    p->one_launch = shape_ok && pick_one_launch(p, pairs);
    if (p->one_launch) {
        const long long tiles2 = static_cast<long long>(p->tiles_m) * p->tiles_n2;
        const long long units = static_cast<long long>(p->tiles_m) * p->tiles_n1 + tiles2 * p->split2;
        if (pairs > units) pairs = units;
        if (pairs < 1) return GEMM_EPI_ERR_LAUNCH;
        p->grid = static_cast<int>(2 * pairs);
        // automatic: static (units of equal size in order; the dynamic order measured 1-4 us
        // slower unsplit), dynamic when GEMM 2 is split
        p->dynamic = p->g1->d_sched != nullptr &&
                     (p->opt_order == 2 || (p->opt_order == 0 && p->split2 > 1));
        // counters: ready (row block x slice), then the slice counts (tile x CTA x warp)
        const size_t ready_bytes =
            sizeof(int) * static_cast<size_t>(p->tiles_m) * static_cast<size_t>(p->split2) +
            (p->split2 > 1 ? sizeof(unsigned) * static_cast<size_t>(tiles2) * 2 * kEpilogueWarps : 0);
        if (p->ready && p->ready_bytes < ready_bytes) {
            cudaFree(p->ready);
            p->ready = nullptr;
        }
        if (!p->ready) {
            if (cudaMalloc(reinterpret_cast<void**>(&p->ready), ready_bytes) != cudaSuccess) {
                cudaGetLastError();
                p->ready = nullptr;
                p->ready_bytes = 0;
                return GEMM_EPI_ERR_ALLOC;
            }
            p->ready_bytes = ready_bytes;
        }
        const size_t ws_bytes = p->split2 > 1 ? static_cast<size_t>(tiles2) * p->split2 * 2 * 128 * 256 * 4 : 0;
        if (p->ws && p->ws_bytes < ws_bytes) {
            cudaFree(p->ws);
            p->ws = nullptr;
            p->ws_bytes = 0;
        }
        if (ws_bytes && !p->ws) {
            if (cudaMalloc(reinterpret_cast<void**>(&p->ws), ws_bytes) != cudaSuccess) {
                cudaGetLastError();
                p->ws = nullptr;
                return GEMM_EPI_ERR_ALLOC;
            }
            p->ws_bytes = ws_bytes;
        }
        snprintf(p->desc, sizeof(p->desc),
                 "one launch: t=%lld d=%lld f=%lld, CTA pairs on 256x256 tiles: %dx%d GEMM-1 tiles "
                 "then %dx%d GEMM-2 tiles in %d K slice%s of %d blocks, grid=%d order=%s",
                 static_cast<long long>(p->t), static_cast<long long>(p->d),
                 static_cast<long long>(p->f), p->tiles_m, p->tiles_n1, p->tiles_m, p->tiles_n2,
                 p->split2, p->split2 > 1 ? "s" : "", p->kb2, p->grid,
                 p->dynamic ? "dynamic" : "static");
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

gemm_epi_status run_ffn_onchip(gemm_epi_ffn_plan_s* p, const void* X, const void* W1,
                               const void* b1, const void* W2, const void* b2, const void* R,
                               void* Y, cudaStream_t stream)
{
    gemm_epi_status st = ensure_ffn_maps(p, X, W1, W2, Y);
    if (st != GEMM_EPI_OK) return st;
    OnchipFfnParams prm;
    memset(&prm, 0, sizeof(prm));
    prm.tm_X = p->tm_X;
    prm.tm_W1 = p->tm_W1;
    prm.tm_W2 = p->tm_W2;
    prm.b1 = b1;
    prm.b2 = b2;
    prm.R = R;
    prm.Y = Y;
    prm.status = p->g1->d_status;
    prm.wait_limit_ns = p->g1->wait_limit_ns;
    prm.t = static_cast<int>(p->t);
    prm.d = static_cast<int>(p->d);
    prm.f = static_cast<int>(p->f);
    prm.bf16 = p->dtype == GEMM_EPI_BF16 ? 1 : 0;
    return ffn_onchip_launch(prm, p->grid, stream) == cudaSuccess ? GEMM_EPI_OK : GEMM_EPI_ERR_LAUNCH;
}

gemm_epi_status run_ffn_one_launch(gemm_epi_ffn_plan_s* p, const void* X, const void* W1,
                                   const void* b1, const void* W2, const void* b2, const void* R,
                                   void* Y, cudaStream_t stream)
{
    gemm_epi_status st = ensure_ffn_maps(p, X, W1, W2, Y);
    if (st != GEMM_EPI_OK) return st;
    if (cudaMemsetAsync(p->ready, 0, p->ready_bytes, stream) != cudaSuccess)
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
    prm.sched = p->dynamic ? g1->d_sched : nullptr;
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
    prm.ffn_ready_target = 2 * kEpilogueWarps;
    prm.ffn_tiles2 = p->tiles_m * p->tiles_n2 * p->split2;
    prm.n2 = static_cast<int>(p->d);
    prm.tiles_n2 = p->tiles_n2;
    prm.k_blocks2 = static_cast<int>((p->f + 63) / 64);
    prm.ffn_split2 = p->split2;
    prm.ffn_kb2 = p->kb2;
    prm.ffn_ws = p->ws;
    prm.ffn_count = p->split2 > 1 ? reinterpret_cast<unsigned*>(p->ready + static_cast<size_t>(p->tiles_m) * p->split2)
                                  : nullptr;
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
    p->ready_bytes = 0;
    p->ws = nullptr;
    p->ws_bytes = 0;
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

gemm_epi_status gemm_epi_ffn_set_option(gemm_epi_ffn_plan_t p, gemm_epi_ffn_option opt,
                                        int64_t value)
{
    if (!p) return GEMM_EPI_ERR_INVALID_ARG;
    int* field = nullptr;
    switch (opt) {
    case GEMM_EPI_FFN_OPT_LAUNCHES:
        if (value < 0 || value > 3) return GEMM_EPI_ERR_INVALID_ARG;
        field = &p->opt_launches;
        break;
    case GEMM_EPI_FFN_OPT_SPLIT2:
        if (!(value == 0 || value == 1 || value == 2 || value == 4)) return GEMM_EPI_ERR_INVALID_ARG;
        field = &p->opt_split2;
        break;
    case GEMM_EPI_FFN_OPT_TILE_ORDER:
        if (value < 0 || value > 2) return GEMM_EPI_ERR_INVALID_ARG;
        field = &p->opt_order;
        break;
    case GEMM_EPI_FFN_OPT_B_READY:
        // (launch-time only: the GEMM plans' configuration does not change)
        if (value != 0 && value != 1) return GEMM_EPI_ERR_INVALID_ARG;
        p->g1->b_ready = static_cast<int>(value);
        p->g2->b_ready = static_cast<int>(value);
        return GEMM_EPI_OK;
    default: return GEMM_EPI_ERR_INVALID_ARG;
    }
    const int saved = *field;
    *field = static_cast<int>(value);
    gemm_epi_status st = configure_ffn(p);
    if (st != GEMM_EPI_OK) {
        *field = saved;
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
    if (p->onchip) return run_ffn_onchip(p, X, W1, b1, W2, b2, R, Y, stream);
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
    if (p->ws) cudaFree(p->ws);
    if (p->stats) cudaFree(p->stats);
    gemm_epi_free(p->g1);
    gemm_epi_free(p->g2);
    delete p;
    return GEMM_EPI_OK;
}

}  // extern "C"

// ---- the FFN block without allocation ------------------------------------------------------
//
// For callers that cannot allocate device memory.  The hidden activation, and the status
// words and tile counters of the two launches, live in one file-scope device array; its
// device address is looked up on every call (with the device current) and passed to the
// kernels.

namespace {

// two status words (bytes 0 and 4) and two tile counters (bytes 8 and 16), padded to 256
constexpr size_t kNoAllocStatusBytes = 256;
constexpr size_t kNoAllocHiddenBytes = static_cast<size_t>(GEMM_EPI_FFN_NOALLOC_MAX_HIDDEN) * 2;

// In host code this name is only a stand-in; the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char
    g_ffn_noalloc_scratch[kNoAllocStatusBytes + kNoAllocHiddenBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
unsigned char* g_noalloc_addr[kNoAllocMaxDevices] = {};

// Device address of the scratch array on device `dev` (the current device), looked up on
// every call (the lookup allocates nothing).  When it differs from the last one seen on the
// device (the first call, or the module was loaded again after a cudaDeviceReset), the
// status words and tile counters are zeroed.
gemm_epi_status noalloc_scratch(int dev, unsigned char** out)
{
    if (dev < 0 || dev >= kNoAllocMaxDevices) return GEMM_EPI_ERR_INVALID_ARG;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_ffn_noalloc_scratch) != cudaSuccess || !ptr) {
        cudaGetLastError();
        return GEMM_EPI_ERR_LAUNCH;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_addr[dev] != ptr) {
        if (cudaMemset(ptr, 0, kNoAllocStatusBytes) != cudaSuccess) {
            cudaGetLastError();
            return GEMM_EPI_ERR_LAUNCH;
        }
        g_noalloc_addr[dev] = static_cast<unsigned char*>(ptr);
    }
    *out = static_cast<unsigned char*>(ptr);
    return GEMM_EPI_OK;
}

// A plan on the caller's stack whose status word and tile counter point into the static
// scratch.
gemm_epi_status stack_plan(gemm_epi_plan_s* p, int64_t m, int64_t n, int64_t k, int dtype,
                           int epilog, int dev, int sms, int* status, unsigned* sched)
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
    p->d_sched = sched;
    p->opt_split_k = 1;  // no split-K workspace to allocate
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
    unsigned* sched = reinterpret_cast<unsigned*>(scratch + 8);
    void* H = scratch + kNoAllocStatusBytes;

    gemm_epi_plan_s g1, g2;
    st = stack_plan(&g1, t, f, d, dtype, GEMM_EPI_GELU_BIAS, dev, sms, status, sched);
    if (st != GEMM_EPI_OK) return st;
    st = stack_plan(&g2, t, d, f, dtype, GEMM_EPI_BIAS_RESIDUAL, dev, sms, status + 1, sched + 2);
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
