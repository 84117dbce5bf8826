// Host side of the C ABI in gemm_epi.h: plans, argument checks, tensor-map encoding and
// kernel launches.
//
// The plan/execute/free split follows the stateful Matmul API of "Fusing bias into cuBLASLt
// matmul with nvmath-python for PyTorch inference" (blog.hotdry.top, 2025-09-22, code
// example and the paragraph on operational parameters): the plan fixes shape, dtype, epilog
// and bias layout and chooses the kernel configuration ("nvmath-python: cuBLAS and cuSOLVER
// bindings", matmul-planning checklist: plan() picks the algorithm); execute() is
// asynchronous; free() releases the plan.
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <new>

#include "plan.h"

using namespace gemm_epi;
using namespace gemm_epi_impl;

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

// Split-K on the swapped kernel is used only when GEMM_EPI_OPT_SPLIT_K asks for it: measured
// on GB300 it did not pay there.  GELU T=16/64/256 x 3072 x 768 through a cluster (DSMEM):
// 9.2/11.1/16.8 us unsplit vs 10.2/22/28 us with split 4 (T=16 graph-replayed: 6.5 us
// against 6.8 us, the one gain); through device memory with 2/4/6 slices at T=16:
// 13.0/13.0/13.5 us cold, 8.1/7.5/7.5 us hot, against 11.0 / 6.8 us unsplit (narrower
// swapped tiles, below, add CTAs without any exchange; m <= 64 now runs the small-m
// kernel).  Row tiles take 2 to 4 K slices through a cluster by themselves where the time
// model says so, the partial sums meeting in L2 (pick_auto_split), and so do plans of
// m <= 256 with a long K that would otherwise run the swapped kernel.
constexpr int kMaxClusterSplit = 4;  // CTAs per cluster (kernel: kMaxSplit)
constexpr int kMaxGlobalSplit = 8;   // K slices through device memory (kernel: kMaxGSplit)

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

// Time model of the busiest CTA, used to choose K splits and between the swapped and the
// row-tile kernel for small m.  These kernels are bound by streaming their operand slabs
// into the SMs and, when K is split, by sending partial sums out; measured on GB300: ~84 GB/s
// per SM into row tiles 64 wide, ~110 GB/s into wider ones, ~62 GB/s into swapped tiles
// (W streamed as 128-column panels) and ~50 GB/s per SM of fp32 partial sums out through
// L2; a K split adds ~3 us of fixed cost (the cluster barrier, the partial sums' reload,
// the epilogue starting after both).  Fitted on 1024 x 512 x 2048, 512 x 512 x 4096,
// 1024 x 1024 x 2048, 2048 x 512 x 2048, 256 x 1024 x 8192, 768 x 768 x 3072 and
// 1024 x 256 x 4096 (CUDA graph, hot L2).
double slab_us(int k_blocks, int bn, double bytes_per_us)
{
    return k_blocks * (16384.0 + 128.0 * bn) / bytes_per_us;
}

double rowtile_rate(int bn) { return bn == 64 ? 84e3 : 110e3; }

constexpr double kSwappedRate = 62e3;
constexpr double kPartialOutRate = 50e3;
constexpr double kSplitFixedUs = 3.0;

// Unsplit row tiles: waves of tiles, each a whole K loop.
double rowtile_us(int64_t m, int64_t n, int k_blocks, int sm_count, int bn)
{
    const int64_t tiles = ((m + 127) / 128) * ((n + bn - 1) / bn);
    const int64_t waves = (tiles + sm_count - 1) / sm_count;
    return static_cast<double>(waves) * slab_us(k_blocks, bn, rowtile_rate(bn));
}

// Row tiles with K split over a cluster, partial sums through L2: over the tile widths
// (fixed_bn, or 64, 128 and 256) and 2 to 4 slices whose clusters are all resident at once
// (cudaOccupancyMaxActiveClusters: clusters of 3 leave SMs of a GPC unused, so 48 of them
// did not fit and ran as two waves, 15.7 against 9.2 us at 256 x 3072 x 768) and whose
// slices are at least 4 K blocks deep, the fastest in the model.  At 1024 x 512 x 2048
// BIAS fp16 (hot / L2 flushed): 128 x 128 tiles in 4 slices 9.8 / 9.9 us (the choice), in 3
// 10.2 / 10.6, 128 x 256 in 4 10.5 / 11.1, 128 x 64 in 2 10.8 / 11.3, unsplit 12.2 / 12.7;
// the same 4 slices over distributed shared memory 15.2 / 16.1 us.
// rowtile_max_clusters per (width, slices), queried once per process (every device of a
// process is taken to be the same GPU model, as elsewhere in the planner)
int max_clusters_cached(int bn, int split)
{
    static std::atomic<int> cache[3][kMaxClusterSplit + 1];
    static std::atomic<bool> known[3][kMaxClusterSplit + 1];
    const int w = bn == 64 ? 0 : bn == 128 ? 1 : 2;
    if (!known[w][split].load()) {
        cache[w][split].store(rowtile_max_clusters(bn, split));
        known[w][split].store(true);
    }
    return cache[w][split].load();
}

bool pick_auto_split(int64_t m, int64_t n, int k_blocks, int sm_count, int fixed_bn, int* bn_out,
                     int* split_out, double* us_out)
{
    const int64_t tm = (m + 127) / 128;
    double best = 1e300;
    for (int bn : {64, 128, 256}) {
        if (fixed_bn && bn != fixed_bn) continue;
        const int64_t tiles = tm * ((n + bn - 1) / bn);
        for (int s = 2; s <= kMaxClusterSplit; ++s) {
            const int kpb = (k_blocks + s - 1) / s;
            if (tiles * s > sm_count || kpb < 4) continue;
            if (tiles > max_clusters_cached(bn, s)) continue;
            const double t = slab_us(kpb, bn, rowtile_rate(bn)) +
                             (s - 1.0) / s * 128.0 * bn * 4.0 / kPartialOutRate + kSplitFixedUs;
            if (t < best) {
                best = t;
                *bn_out = bn;
                *split_out = s;
            }
        }
    }
    *us_out = best;
    return best < 1e300;
}

// Tile width (rows of D) of the swapped small-m kernel: the narrowest that still gives
// every tile its own SM, else one tile over all m rows.  The operand W is then read by
// several tiles (the later reads hit L2), but more SMs stream it: measured on GB300 at
// 256 x 3072 x 768 GELU, 64-row tiles (96 CTAs) take 12.9 us cold / 8.2 us hot against
// 17.2 / 11.5 us for one 256-row tile (24 CTAs); at 64 x 3072 x 768, 16-row tiles 7.0 us
// hot against 7.8 us.
int pick_swapped_bn(int64_t m, int64_t n, int sm_count)
{
    int full = 16;
    while (full < m) full *= 2;
    const int64_t tiles_n = (n + 127) / 128;
    for (int bn = 16; bn < full; bn *= 2)
        if (tiles_n * ((m + bn - 1) / bn) <= sm_count) return bn;
    return full;
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

// Small-m kernel configuration: rows-of-D tile bn (16, 32 or 64, at least m), `split` K
// slices of kb 64-deep blocks each (a cluster of `split` CTAs per 128-column tile), copies of
// B box_k rows deep, and the shared memory per CTA.  Takes the most slices whose CTAs all run
// at once (one CTA per SM: the shared memory is padded so that two never share one, which
// would halve the copy bandwidth each gets) and fit in shared memory; want_split > 0 asks for
// that many (lowered, like the other kernels' splits, until no slice is empty).  False if no
// configuration fits (k too long for one slab per CTA).
struct SmallMCfg {
    int bn, split, kb, box_k, smem;
};
constexpr int kSmallMMaxM = 64;
constexpr int kSmallMMinSmem = 116 * 1024;
constexpr int kSmemLimit = 227 * 1024;

bool smallm_epilog(int e)
{
    return e == GEMM_EPI_BIAS || e == GEMM_EPI_RELU_BIAS || e == GEMM_EPI_GELU_BIAS ||
           e == GEMM_EPI_RELU_AUX_BIAS || e == GEMM_EPI_BIAS_RESIDUAL || e == GEMM_EPI_NONE ||
           e == GEMM_EPI_TANH_BIAS || e == GEMM_EPI_GELU_AUX_BIAS;
}

bool pick_smallm_bn(int64_t n, int64_t k, int want_split, SmallMCfg* c);

// The narrowest tile of rows that holds m (or want_bn), else a wider one: a wider tile lets
// the K slab be cut into more slices (each rank's rows of the tile come in fours), which is
// what fits a long K into shared memory (16 x 768 x 3072: no 16-row configuration fits; 32
// rows in 8 slices measured 6.5 us against 9.6 for the row tiles it replaced, graph, hot L2).
bool pick_smallm(int64_t m, int64_t n, int64_t k, int want_split, int want_bn, SmallMCfg* c)
{
    if (m < 1 || m > kSmallMMaxM || n < 1 || k < 1) return false;
    const int natural = m <= 16 ? 16 : m <= 32 ? 32 : 64;
    if (want_bn) {
        if (want_bn < natural) return false;
        c->bn = want_bn;
        return pick_smallm_bn(n, k, want_split, c);
    }
    for (int bn = natural; bn <= 64; bn *= 2) {
        c->bn = bn;
        if (pick_smallm_bn(n, k, want_split, c)) return true;
    }
    return false;
}

bool pick_smallm_bn(int64_t n, int64_t k, int want_split, SmallMCfg* c)
{
    const int64_t tiles = (n + 127) / 128;
    const int kblocks = static_cast<int>((k + 63) / 64);
    const int top = want_split > 0 ? want_split : (kblocks < 8 ? kblocks : 8);
    for (int s = top; s >= 1; --s) {
        const int kb = (kblocks + s - 1) / s;
        const int split = (kblocks + kb - 1) / kb;  // no empty slice
        const int need = smallm_smem_bytes(c->bn, kb * 64, split);
        if (need <= 0) continue;  // the split does not divide the rows: a smaller one
        if (need > kSmemLimit) {
            if (want_split > 0) return false;  // (fewer slices need more)
            continue;
        }
        const int smem = need > kSmallMMinSmem ? need : kSmallMMinSmem;
        if (want_split == 0 && split > 1) {
            const int clusters = smallm_max_clusters(c->bn, split, smem);
            if (clusters < 1 || tiles > clusters) continue;  // every cluster resident at once
        }
        c->split = split;
        c->kb = kb;
        c->smem = smem;
        const int kc = kb * 64;
        c->box_k = kc % 256 == 0 ? 256 : kc % 192 == 0 ? 192 : kc % 128 == 0 ? 128 : 64;
        return true;
    }
    return false;
}

}  // namespace

namespace gemm_epi_impl {

bool fp8_epilog(int e)
{
    return e == GEMM_EPI_BIAS || e == GEMM_EPI_RELU_BIAS || e == GEMM_EPI_GELU_BIAS ||
           e == GEMM_EPI_RELU_AUX_BIAS || e == GEMM_EPI_BIAS_RESIDUAL || e == GEMM_EPI_NONE;
}

// The split-K workspace for the configured shape: kept when large enough, else replaced
// (the old buffers stay if an allocation fails).  The counts start at zero; each launch
// leaves them at zero.
gemm_epi_status ensure_split_ws(gemm_epi_plan_s* p)
{
    const size_t tiles = static_cast<size_t>(p->tiles_m) * p->tiles_n;
    const size_t ws_bytes = tiles * p->split * 128 * p->bn * sizeof(float);
    if (p->d_split_ws && p->split_ws_bytes >= ws_bytes && p->split_count_len >= tiles)
        return GEMM_EPI_OK;
    float* ws = nullptr;
    unsigned* cnt = nullptr;
    if (cudaMalloc(reinterpret_cast<void**>(&ws), ws_bytes) != cudaSuccess ||
        cudaMalloc(reinterpret_cast<void**>(&cnt), tiles * sizeof(unsigned)) != cudaSuccess) {
        cudaGetLastError();
        if (ws) cudaFree(ws);
        return GEMM_EPI_ERR_ALLOC;
    }
    // (the legacy stream orders the memset; synchronise so that launches on any stream see it)
    if (cudaMemset(cnt, 0, tiles * sizeof(unsigned)) != cudaSuccess ||
        cudaStreamSynchronize(nullptr) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(ws);
        cudaFree(cnt);
        return GEMM_EPI_ERR_ALLOC;
    }
    release_split_ws(p);
    p->d_split_ws = ws;
    p->d_split_count = cnt;
    p->split_ws_bytes = ws_bytes;
    p->split_count_len = tiles;
    return GEMM_EPI_OK;
}

gemm_epi_status configure(gemm_epi_plan_s* p)
{
    p->maps_valid = false;
    p->bn = p->stages = p->smem = p->grid = p->tiles_m = p->tiles_n = p->k_blocks = 0;
    p->group_m = 1;
    p->split = 1;
    p->split_global = 0;
    p->split_l2 = 0;
    p->dyn_order = 0;
    p->swap_m64 = 0;
    p->box_k = 0;
    p->kb_per_split = 0;
    if (p->m == 0 || p->n == 0) {
        p->variant = kEmpty;
    } else if (p->k == 0) {
        p->variant = kBiasOnly;
    } else if (p->dtype == GEMM_EPI_E4M3) {
        // E4M3: the CTA-pair kernel with 256 x 256 or 256 x 224 tiles (the width with fewer
        // waves, as for 16-bit inputs) and 128-deep K blocks, any shape
        if ((p->opt_variant != 0 && p->opt_variant != 3) ||
            (p->opt_bn != 0 && p->opt_bn != 256 && p->opt_bn != 224))
            return GEMM_EPI_ERR_INVALID_ARG;
        if (fp8_pair_prepare() != cudaSuccess || rowpair_prepare(256) != cudaSuccess)
            return GEMM_EPI_ERR_LAUNCH;
        long long pairs = rowpair_max_clusters(256);  // same shared memory for both widths
        if (pairs > p->sm_count / 2) pairs = p->sm_count / 2;
        if (p->opt_grid > 0 && p->opt_grid / 2 < pairs) pairs = p->opt_grid / 2;
        if (pairs < 1) return GEMM_EPI_ERR_LAUNCH;
        p->variant = kRowPair;
        p->bn = p->opt_bn ? p->opt_bn : pick_pair_bn(p->m, p->n, pairs);
        p->k_blocks = static_cast<int>((p->k + 127) / 128);
        p->tiles_m = static_cast<int>((p->m + 255) / 256);
        p->tiles_n = static_cast<int>((p->n + p->bn - 1) / p->bn);
        p->stages = rowpair_stages(p->bn);
        p->smem = rowpair_smem_bytes(p->bn);
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
            // m <= 64 with a forward epilog and a K slab that fits a CTA: the small-m kernel
            SmallMCfg sc;
            if (v == kSwapped && smallm_epilog(p->epilog) && p->opt_split_k == 0 &&
                smallm_prepare() == cudaSuccess &&
                pick_smallm(p->m, p->n, p->k, 0, 0, &sc))
                v = kSmallM;
            // otherwise, over a long K loop: row tiles with K split over a cluster when the
            // model puts them well ahead of the swapped kernel, which streams each 128-column
            // panel of B through one SM (256 x 1024 x 8192 BIAS: 37.8 us swapped, 15.5 us as
            // 128 x 64 row tiles in 4 slices; the swapped kernel keeps T x 3072 x 768)
            if (v == kSwapped && p->opt_split_k == 0 && p->opt_bn == 0 && p->opt_split_mode != 2) {
                const int kb = static_cast<int>((p->k + 63) / 64);
                const int sbn = pick_swapped_bn(p->m, p->n, p->sm_count);
                const int64_t sw_tiles = ((p->n + 127) / 128) * ((p->m + sbn - 1) / sbn);
                const double sw_us = static_cast<double>((sw_tiles + p->sm_count - 1) / p->sm_count) *
                                     slab_us(kb, sbn, kSwappedRate);
                int sp_bn = 0, sp_split = 0;
                double sp_us = 0.0;
                if (pick_auto_split(p->m, p->n, kb, p->sm_count, 0, &sp_bn, &sp_split, &sp_us) &&
                    sp_us < 0.7 * sw_us)
                    v = kRowTile;
            }
        }
        // (option values: 1 row-tile, 2 swapped, 3 CTA pairs, 5 small-m; the internal
        // Variant codes differ)
        if (p->opt_variant == 3) v = kRowPair;  // option value 3: the CTA-pair kernel
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
        } else if (v == kSmallM) {
            // one K slab per CTA, split over a cluster (the rows of D are one tile)
            SmallMCfg sc;
            if (smallm_prepare() != cudaSuccess) return GEMM_EPI_ERR_LAUNCH;
            if (!smallm_epilog(p->epilog) || p->opt_split_k > 8 ||
                (p->opt_bn && p->opt_bn != 16 && p->opt_bn != 32 && p->opt_bn != 64))
                return GEMM_EPI_ERR_INVALID_ARG;
            if (!pick_smallm(p->m, p->n, p->k, p->opt_split_k, p->opt_bn, &sc))
                return GEMM_EPI_ERR_INVALID_ARG;
            const int need = smallm_smem_bytes(sc.bn, sc.kb * 64, sc.split);
            if (need > kSmemLimit) return GEMM_EPI_ERR_INVALID_ARG;
            if (need > sc.smem) sc.smem = need;
            p->bn = sc.bn;
            p->tiles_m = static_cast<int>((p->n + 127) / 128);
            p->tiles_n = static_cast<int>((p->m + sc.bn - 1) / sc.bn);
            p->split = sc.split;
            p->kb_per_split = sc.kb;
            p->box_k = sc.box_k;
            p->smem = sc.smem;
            p->stages = 1;
            const long long grid = static_cast<long long>(p->tiles_m) * p->tiles_n * sc.split;
            if (grid > (1ll << 30)) return GEMM_EPI_ERR_UNSUPPORTED_SHAPE;
            p->grid = static_cast<int>(grid);
        } else if (v == kRowTile) {
            if (p->opt_bn && p->opt_bn != 64 && p->opt_bn != 128 && p->opt_bn != 256)
                return GEMM_EPI_ERR_INVALID_ARG;
            p->bn = p->opt_bn ? p->opt_bn : pick_rowtile_bn(p->m, p->n, p->k_blocks, p->sm_count);
            p->tiles_m = static_cast<int>((p->m + 127) / 128);
            p->tiles_n = static_cast<int>((p->n + p->bn - 1) / p->bn);
            p->stages = rowtile_stages(p->bn);
            p->smem = rowtile_smem_bytes(p->bn);
        } else {
            if (p->opt_bn && p->opt_bn != 16 && p->opt_bn != 32 && p->opt_bn != 64 &&
                p->opt_bn != 128 && p->opt_bn != 256)
                return GEMM_EPI_ERR_INVALID_ARG;
            int bn = p->opt_bn ? p->opt_bn : pick_swapped_bn(p->m, p->n, p->sm_count);
            p->bn = bn;
            p->tiles_m = static_cast<int>((p->n + 127) / 128);
            p->tiles_n = static_cast<int>((p->m + bn - 1) / bn);
            // 64 columns of D per tile (64-row MMAs), on request only: twice the CTAs copy B,
            // but the K loop is bound by the copies' round trips, not by the SMs' copy rate.
            // Measured on GB300 (CUDA graph, L2 flushed / hot, two runs): 16x3072x768
            // GELU_BIAS 7.2-7.5 / 6.9 us against 6.6-7.5 / 7.0 us with 128 columns; at m = 64
            // and 256 (152 CTAs) 10.8 and 12.3 us against 7.5-7.8 and 8.3-8.5 us.
            const bool m64_epilog = p->epilog == GEMM_EPI_BIAS || p->epilog == GEMM_EPI_RELU_BIAS ||
                                    p->epilog == GEMM_EPI_GELU_BIAS || p->epilog == GEMM_EPI_NONE ||
                                    p->epilog == GEMM_EPI_TANH_BIAS ||
                                    p->epilog == GEMM_EPI_BIAS_RESIDUAL ||
                                    p->epilog == GEMM_EPI_GELU_AUX_BIAS;
            const bool m64_split = p->opt_split_k > 1;
            if (p->opt_tile_m == 64) {
                if (!m64_epilog || m64_split) return GEMM_EPI_ERR_INVALID_ARG;
                p->swap_m64 = 1;
            }
            if (p->swap_m64) p->tiles_m = static_cast<int>((p->n + 63) / 64);
            p->stages = swapped_stages(bn);
            p->smem = swapped_smem_bytes(bn);
        }
    }
    if (p->variant == kRowTile || p->variant == kSwapped) {
        const int v = p->variant;
        int want_split = p->opt_split_k > 0 ? p->opt_split_k : 1;
        bool via_cluster = p->opt_split_mode == 1 || p->opt_split_mode == 3;
        bool via_l2 = p->opt_split_mode == 3;
        int auto_bn = 0, auto_split = 0;
        double split_us = 0.0;
        if (p->opt_split_k == 0 && v == kRowTile && p->opt_split_mode != 2 &&
            pick_auto_split(p->m, p->n, p->k_blocks, p->sm_count, p->opt_bn, &auto_bn, &auto_split,
                            &split_us) &&
            split_us < rowtile_us(p->m, p->n, p->k_blocks, p->sm_count, p->bn)) {
            // Row tiles whose K loop is long against the work's spread over the SMs: K slices
            // through a cluster, the partial sums through L2 unless SPLIT_MODE asks for
            // distributed shared memory (pick_auto_split); through device memory alone (no
            // cluster) 1024 x 512 x 2048 took 15.0 / 17.2 us.
            want_split = auto_split;
            via_cluster = true;
            via_l2 = p->opt_split_mode != 1;
            p->bn = auto_bn;
            p->tiles_n = static_cast<int>((p->n + p->bn - 1) / p->bn);
            p->stages = rowtile_stages(p->bn);
            p->smem = rowtile_smem_bytes(p->bn);
        }
        const long long tiles = static_cast<long long>(p->tiles_m) * p->tiles_n;
        cudaError_t e = v == kRowTile ? rowtile_prepare(p->bn) : swapped_prepare(p->bn);
        if (e != cudaSuccess) return GEMM_EPI_ERR_LAUNCH;
        if (want_split > (via_cluster ? kMaxClusterSplit : kMaxGlobalSplit))
            return GEMM_EPI_ERR_INVALID_ARG;
        p->split = normalise_split(want_split, p->k_blocks, &p->kb_per_split);
        long long grid;
        if (p->split > 1) {
            // one CTA per (tile, K slice), not persistent; in clusters of `split` CTAs when
            // the slices meet on chip
            p->split_global = via_cluster ? 0 : 1;
            p->split_l2 = via_cluster && via_l2 ? 1 : 0;
            grid = tiles * p->split;
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
    // CTA pairs take their tiles from the plan's device counter on long walks (eight or more
    // waves of tiles over the pairs), where a static order lets the pairs drift apart and
    // lose the operand panels they share in L2; on a few waves the static order keeps the
    // tiles per pair equal, where handing them out as pairs free up can give one pair a tile
    // more than another.  Measured on GB300 (hot L2): 65536 x 16384 x 8192 (215 waves)
    // 10.9 GB read and 8.98 ms dynamic against 26.4 GB and 9.89 ms static; 4096^3 (4 waves)
    // 87.4 us dynamic against 86.0 static; FFN GEMM 1 4096 x 4096 x 1024 GELU (4 waves) 35.2
    // against 32.4 us.  A plan on the caller's stack may have no counter: static.
    if (p->variant == kRowPair) {
        const long long tiles = static_cast<long long>(p->tiles_m) * p->tiles_n;
        const long long pairs = p->grid / 2;
        const bool want = p->opt_tile_order == 2 || (p->opt_tile_order == 0 && tiles >= 8 * pairs);
        p->dyn_order = want && p->d_sched != nullptr;
    }
    static const char* vname[] = {"empty", "row-tile", "swapped", "bias-only", "row-pair",
                                  "small-m"};
    static const char* ename[] = {"BIAS",          "RELU_BIAS",     "GELU_BIAS",
                                  "RELU_AUX_BIAS", "BIAS_RESIDUAL", "NONE",
                                  "TANH_BIAS",     "GELU_AUX_BIAS", "DRELU_BGRAD",
                                  "DGELU_BGRAD",   "LN_GELU_BIAS"};
    snprintf(p->desc, sizeof(p->desc),
             "m=%lld n=%lld k=%lld dtype=%s epilog=%s bias=%s variant=%s tile=%dx%d bk=%d "
             "stages=%d smem=%d tiles=%dx%d k_blocks=%d split_k=%d%s grid=%d group_m=%d%s sms=%d",
             static_cast<long long>(p->m), static_cast<long long>(p->n),
             static_cast<long long>(p->k),
             p->dtype == GEMM_EPI_E4M3 ? "e4m3" : p->dtype == GEMM_EPI_BF16 ? "bf16" : "f16",
             ename[p->epilog], p->bias_layout == GEMM_EPI_BIAS_M1 ? "(m,1)" : "(1,n)",
             vname[p->variant],
             p->variant == kRowPair ? 256 : p->swap_m64 ? 64 : 128, p->bn,
             p->dtype == GEMM_EPI_E4M3 ? 128 : 64, p->stages, p->smem, p->tiles_m, p->tiles_n,
             p->k_blocks,
             p->split,
             p->split > 1 ? (p->split_global ? "(device memory)"
                             : p->split_l2   ? "(cluster+L2)"
                                             : "(cluster)")
                          : "",
             p->grid, p->group_m,
             p->variant != kRowPair ? "" : p->dyn_order ? " order=dynamic" : " order=static",
             p->sm_count);
    const char* log = getenv("GEMM_EPI_LOG");
    if (log && log[0] == '1') fprintf(stderr, "[gemm_epi] plan: %s\n", p->desc);
    if (p->split_global || p->split_l2) return ensure_split_ws(p);
    return GEMM_EPI_OK;
}

void release_split_ws(gemm_epi_plan_s* p)
{
    if (p->d_split_ws) cudaFree(p->d_split_ws);
    if (p->d_split_count) cudaFree(p->d_split_count);
    p->d_split_ws = nullptr;
    p->d_split_count = nullptr;
    p->split_ws_bytes = 0;
    p->split_count_len = 0;
}

bool encode_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, uint64_t inner,
               uint64_t outer, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw,
               uint64_t elem_bytes, uint64_t row_elems)
{
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {(row_elems ? row_elems : inner) * elem_bytes};
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
        // A [m][k] and B transposed [n][k], bytes, K-major boxes {128 k, 128 rows} (A) and
        // {128 k, bn / 2 rows} (B: each CTA's half of a tile's columns); D bf16
        const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
        const uint32_t b_rows = static_cast<uint32_t>(p->bn / 2);
        if (!encode_2d(&p->tm_A, A, u8, p->k, p->m, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B, 1) ||
            !encode_2d(&p->tm_B, B, u8, p->k, p->n, 128, b_rows, CU_TENSOR_MAP_SWIZZLE_128B, 1) ||
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
    if (p->variant == kSmallM) {
        // A: K-major boxes {64 k, bn rows}; B: N-major boxes {64 n, box_k k}; D is stored
        // without a map
        if (!encode_2d(&p->tm_A, A, dt, p->k, p->m, 64, static_cast<uint32_t>(p->bn),
                       CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_2d(&p->tm_B, B, dt, p->n, p->k, 64, static_cast<uint32_t>(p->box_k),
                       CU_TENSOR_MAP_SWIZZLE_128B))
            return GEMM_EPI_ERR_LAUNCH;
        p->key_A = A;
        p->key_B = B;
        p->key_D = D;
        p->maps_valid = true;
        return GEMM_EPI_OK;
    }
    const bool rows_of_a = p->variant == kRowTile || p->variant == kRowPair;
    const uint32_t a_rows = rows_of_a ? 128u : static_cast<uint32_t>(p->bn);
    if (!encode_2d(&p->tm_A, A, dt, p->k, p->m, 64, a_rows, CU_TENSOR_MAP_SWIZZLE_128B))
        return GEMM_EPI_ERR_LAUNCH;
    if (!encode_2d(&p->tm_B, B, dt, p->n, p->k, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B, 2,
                   static_cast<uint64_t>(p->ldb)))
        return GEMM_EPI_ERR_LAUNCH;
    if (rows_of_a) {
        if (!encode_2d(&p->tm_D, D, dt, p->n, p->m, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B, 2,
                       static_cast<uint64_t>(p->ldd)))
            return GEMM_EPI_ERR_LAUNCH;
    } else {
        // swapped kernel: boxes of 32 columns (16 with 64-column tiles) x (up to) 32 rows
        // of D, transposed on chip
        const uint32_t rows = p->bn < 32 ? static_cast<uint32_t>(p->bn) : 32u;
        const uint32_t cols = p->swap_m64 ? 16u : 32u;
        if (!encode_2d(&p->tm_D, D, dt, p->n, p->m, cols, rows, CU_TENSOR_MAP_SWIZZLE_NONE))
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

gemm_epi_status launch_gemm(gemm_epi_plan_s* p, const gemm_epi_operands& ops, int epilog,
                            cudaStream_t stream, bool pdl)
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
    prm.split_global = p->split_global;
    prm.split_ws = p->d_split_ws;
    prm.split_count = p->d_split_count;
    prm.split_l2 = p->split_l2;
    prm.sched = p->dyn_order ? p->d_sched : nullptr;
    prm.swap_m64 = p->swap_m64;
    prm.box_k = p->box_k;
    prm.prefetch = p->prefetch;
    // Under a programmatic dependent launch: B copied before the wait (b_ready), or, on the
    // small-m kernel, brought into L2 before it.
    prm.b_ready = pdl && p->b_ready ? 1 : 0;
    if (pdl && !p->b_ready && p->variant == kSmallM) {
        prm.b_l2 = ops.B;
        prm.b_ld = p->ldb ? p->ldb : p->n;
    }
    cudaError_t e;
    if (p->variant == kRowPair && p->dtype == GEMM_EPI_E4M3)
        e = fp8_pair_launch(p->bn, prm, p->grid, stream, pdl);
    else if (p->variant == kRowPair)
        e = rowpair_launch(p->bn, prm, p->grid, stream, pdl);
    else if (p->variant == kRowTile)
        e = rowtile_launch(p->bn, prm, p->grid, stream, pdl);
    else if (p->variant == kSmallM)
        e = smallm_launch(p->bn, prm, p->grid, p->smem, stream, pdl);
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

}  // namespace gemm_epi_impl

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
    // status word at byte 0, the CTA pairs' tile counter (two words) at byte 8
    if (cudaMalloc(reinterpret_cast<void**>(&p->d_status), kPlanWordsBytes) != cudaSuccess) {
        cudaGetLastError();
        delete p;
        return GEMM_EPI_ERR_ALLOC;
    }
    if (cudaMemset(p->d_status, 0, kPlanWordsBytes) != cudaSuccess) {
        cudaFree(p->d_status);
        delete p;
        return GEMM_EPI_ERR_ALLOC;
    }
    p->d_sched = reinterpret_cast<unsigned*>(reinterpret_cast<char*>(p->d_status) + 8);
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
        if (value < 0 || value > 5 || value == 4) return GEMM_EPI_ERR_INVALID_ARG;
        p->opt_variant = static_cast<int>(value);
        break;
    case GEMM_EPI_OPT_TILE_N:
        if (value != 0 && value != 16 && value != 32 && value != 64 && value != 128 &&
            value != 224 && value != 256)
            return GEMM_EPI_ERR_INVALID_ARG;
        p->opt_bn = static_cast<int>(value);
        break;
    case GEMM_EPI_OPT_SPLIT_K:
        if (value < 0 || value > kMaxGlobalSplit) return GEMM_EPI_ERR_INVALID_ARG;
        p->opt_split_k = static_cast<int>(value);
        break;
    case GEMM_EPI_OPT_SPLIT_MODE:
        if (value < 0 || value > 3) return GEMM_EPI_ERR_INVALID_ARG;
        p->opt_split_mode = static_cast<int>(value);
        break;
    case GEMM_EPI_OPT_TILE_M:
        if (value != 0 && value != 64 && value != 128) return GEMM_EPI_ERR_INVALID_ARG;
        p->opt_tile_m = static_cast<int>(value);
        break;
    case GEMM_EPI_OPT_TILE_ORDER:
        if (value < 0 || value > 2) return GEMM_EPI_ERR_INVALID_ARG;
        p->opt_tile_order = static_cast<int>(value);
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
    case GEMM_EPI_OPT_B_READY:
        if (value != 0 && value != 1) return GEMM_EPI_ERR_INVALID_ARG;
        p->b_ready = static_cast<int>(value);
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
    release_split_ws(p);
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

int64_t gemm_epi_aux_words_per_row(int64_t n) { return n <= 0 ? 0 : (n + 31) / 32; }

}  // extern "C"
