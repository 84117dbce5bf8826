// Parameters shared by the host API and the kernels (internal; not part of the C ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gemm_epi {

enum Epilog : int {
    EPI_BIAS = 0,
    EPI_RELU_BIAS = 1,
    EPI_GELU_BIAS = 2,
    EPI_RELU_AUX_BIAS = 3,
    EPI_BIAS_RESIDUAL = 4,
    EPI_NONE = 5,
    EPI_TANH_BIAS = 6,
    EPI_GELU_AUX_BIAS = 7,  // as GELU_BIAS, and the pre-activation written to aux (16-bit)
    EPI_DRELU_BGRAD = 8,    // D = A.B * mask bit (aux_in), dbias = sums of D
    EPI_DGELU_BGRAD = 9,    // D = A.B * GELU'(aux_in pre), dbias = sums of D
    EPI_LN_GELU_BIAS = 10   // D = GELU(rstd_i (A.B - mu_i c_j) + b'_j): LayerNorm folded in
};

// Template values of the CTA-pair kernel that runs a whole FFN block (two GEMMs) in one
// launch: GEMM 2 whole, or in K slices (ffn_split2 > 1; only that instantiation carries the
// slices' partial-sum code, which cost the other one 32 registers and ~1.2 us per call).
constexpr int kEpiFfn = 100;
constexpr int kEpiFfnSplit = 101;
__host__ __device__ constexpr bool is_ffn(int epi) { return epi == kEpiFfn || epi == kEpiFfnSplit; }

// Epilogue warps per CTA (two per 32-lane quarter of tensor memory).
constexpr int kEpilogueWarps = 8;

__host__ __device__ constexpr bool is_backward(int epilog)
{
    return epilog == EPI_DRELU_BGRAD || epilog == EPI_DGELU_BGRAD;
}

// Device status word values: 0 = fine, else (kCodeTimeout | role).
enum : int {
    kCodeTimeout = 0x100,
    kRoleProducer = 1,
    kRoleMma = 2,
    kRoleEpilogue = 3,
    kRoleStallTest = 4
};

// One launch of the fused kernel.  The MMA tile is 128 rows (MMA M) by BN columns (MMA N)
// with an fp32 accumulator in tensor memory.
//   row-tile kernel:  MMA rows = rows of D (from A), MMA columns = columns of D (from B);
//   swapped kernel:   MMA rows = columns of D (from B), MMA columns = rows of D (from A),
//                     i.e. it computes D^T = B^T A^T, for small m.
struct GemmParams {
    CUtensorMap tm_A;  // A[m][k]: K-major boxes {64 k, rows}, 128-byte swizzle
    CUtensorMap tm_B;  // B[k][n]: N-major boxes {64 n, 64 k}, 128-byte swizzle
    CUtensorMap tm_D;  // D[m][n]: store boxes {32 n, 32 m} with the 64-byte swizzle (row-tile
                       // kernel) or {32 n, min(BN, 32) m} unswizzled (swapped kernel)
    const void* bias;
    const void* residual;
    void* D;
    void* aux;            // RELU_AUX_BIAS: uint32 mask words; GELU_AUX_BIAS: 16-bit pre-activation
    const void* aux_in;   // DRELU_BGRAD: mask words; DGELU_BGRAD: 16-bit pre-activation
    float* dbias;         // backward epilogs: bias gradient (zeroed before the launch)
    const float* ln_stats;   // LN_GELU_BIAS: (mu, rstd) per row of D (per row of A)
    const float* ln_colsum;  // LN_GELU_BIAS: c_j, column sums of the folded weight
    const float* ln_bias;    // LN_GELU_BIAS: b'_j = beta . W + b (fp32)
    // FP8 (E4M3) inputs (CTA-pair kernel instantiated for them): tm_B maps B transposed
    // (n x k, K-major boxes {128 k, 128 n}); K blocks are 128 deep; the accumulator is
    // multiplied by *scale_a * *scale_b before the bias.
    const float* scale_a;
    const float* scale_b;
    int* status;
    unsigned long long wait_limit_ns;
    int m, n, k;
    int tiles_m;    // tiles along the MMA rows (128 each)
    int tiles_n;    // tiles along the MMA columns (BN each)
    int k_blocks;   // 64-deep K blocks per tile
    int group_m;    // raster: MMA-row tiles per group
    int epilog;
    int bias_layout;  // 0 = (m,1), 1 = (1,n)
    int bf16;         // 1 = bfloat16, 0 = binary16
    int aux_ld;       // uint32 words per aux row
    int debug_stall;
    // Split-K across a thread-block cluster: split > 1 launches tiles * split CTAs in
    // clusters of `split`; rank r of a cluster accumulates K blocks
    // [r * kb_per_split, (r + 1) * kb_per_split) of the cluster's tile, and the partial
    // sums are added before the epilogue (over distributed shared memory, or through L2
    // with split_l2 below).
    int split;
    int kb_per_split;
    // Split-K through device memory instead (split_global == 1, split > 1): tiles * split
    // CTAs, no cluster; CTA b takes K slice b % split of tile b / split, writes its fp32
    // partial tile to split_ws ([tile][slice][128 x BN]) and counts itself in
    // split_count[tile]; the CTA that arrives last adds the slices in slice order (the
    // result does not depend on the arrival order), runs the epilogue and sets the count
    // back to zero for the next launch.
    int split_global;
    float* split_ws;
    unsigned* split_count;
    // Split-K across a cluster whose partial sums meet in split_ws instead of in the peers'
    // shared memory (split_l2 == 1, split_global == 0), laid out as blocks of 32 rows x one
    // chunk (4 KB at 32 columns), [tile][rank][lane quarter][chunk], each [16-byte unit][lane],
    // so that a warp's stores and copies of a block are contiguous 512-byte runs.
    // Each CTA writes the partials of the chunks it does not own, the cluster barrier orders
    // them, and each owner reads its peers' partials from L2 (split_count is not used).
    int split_l2;
    // CTA-pair kernels: order of the tiles.  sched == nullptr: static, pair q takes tiles
    // q, q + pairs, q + 2 pairs, ...  Otherwise each pair takes tile q first and then the
    // tile pairs + atomicAdd(&sched[0], 1) each time it starts one, until the walk ends;
    // sched[1] counts the pairs that have finished, and the last one sets both words back
    // to zero, so every launch finds them at zero.  Handing out tiles in raster order keeps
    // the tiles in flight a contiguous window of the walk (pairs that run slower do not
    // fall behind the others), so the operand panels they share are still in L2.
    unsigned* sched;
    // Swapped kernel with 64 MMA rows per tile (swap_m64 == 1): each tile is 64 columns of
    // D (one 64-column box of B per stage), the MMA runs M = 64, and its rows sit in TMEM
    // lanes 0-15 of each lane quarter (row r in lane 32 (r / 16) + r % 16), so every
    // epilogue warp owns 16 columns of D.  Only for epilogs whose outputs are per element
    // (no mask words, no backward) and without a K split.
    int swap_m64;
    // Small-m kernel: rows of k per copy of B (divides the K slice kb_per_split * 64).
    int box_k;
    // Launched as a programmatic dependent, the kernel may start while the previous grid on
    // the stream still runs.  b_ready == 1: nothing that grid does writes B (a weight that
    // stays in place), so the small-m kernel and the single-CTA producers copy B's first K
    // blocks into shared memory before waiting for that grid, and A after.  b_l2 != nullptr
    // (small-m kernel, without b_ready): B's element (0, 0), with row stride b_ld elements;
    // the CTA's threads bring its slab of B into L2 at entry (L2 is coherent with that grid's
    // writes, so this needs no promise) and the copies into shared memory follow the wait.
    int b_ready;
    const void* b_l2;
    long long b_ld;
    // The producer also prefetches into L2 the operand boxes of the K block this many
    // blocks ahead of the one it loads (0 = off), so that a first touch of a panel in
    // device memory overlaps the loads of the blocks before it.
    int prefetch;
    // FFN block in one launch (CTA-pair kernel, kEpiFfn): tiles [0, tiles_m * tiles_n) are
    // GEMM 1, H = GELU(X.W1 + b1), described by the fields above (A = X, B = W1, D = H; 256
    // columns of H per tile); the next ffn_tiles2 = tiles_m * tiles_n2 * ffn_split2 work units
    // are GEMM 2, Y = H.W2 + b2 + R, with the maps and sizes below.  Unit u is K slice
    // s = u % ffn_split2 (K blocks [s * ffn_kb2, (s + 1) * ffn_kb2) of H's columns) of output
    // tile u / ffn_split2 (row order).  A unit loads its slice of H only once
    // ffn_ready[row tile * ffn_split2 + s] has reached ffn_ready_target times the number of
    // GEMM-1 tiles in that slice: every epilogue warp of both CTAs adds 1 to its tile's
    // counter when its stores of H are done, so ffn_ready_target = 2 x epilogue warps.
    // ffn_split2 > 1 (ffn_kb2 a multiple of 4, so each GEMM-1 tile lies in one slice): every
    // epilogue warp writes the fp32 partial sums of its rows and chunks of a unit to ffn_ws
    // ([tile][slice][CTA of the pair][16-byte column unit][128 rows]) and counts itself in
    // ffn_count[(tile * 2 + CTA) * epilogue warps + warp]; the warp that completes the count
    // (the slice that finished last) adds the slices in slice order, so the sum does not
    // depend on the arrival order, and runs the epilogue.  ffn_ready and ffn_count are zero
    // at the launch.  ffn_tiles2 == 0 for every other launch.
    CUtensorMap tm_A2, tm_B2, tm_D2;
    const void* bias2;
    const void* residual2;
    int* ffn_ready;
    int ffn_ready_target;
    int ffn_tiles2;
    int n2, tiles_n2, k_blocks2;
    int ffn_split2, ffn_kb2;
    float* ffn_ws;
    unsigned* ffn_count;
};

// Most K slices of the FFN kernel's second GEMM.
constexpr int kFfnMaxSplit2 = 4;

// Row-tile kernel (BN in {64, 128, 256}) and swapped small-m kernel (BN in {16 ... 256}).
cudaError_t rowtile_prepare(int bn);
// pdl: launch as a programmatic dependent of the previous grid on the stream.
cudaError_t rowtile_launch(int bn, const GemmParams& p, int grid, cudaStream_t stream, bool pdl);
int rowtile_smem_bytes(int bn);
// Clusters of `split` row-tile CTAs of width bn that the GPU holds at once.
int rowtile_max_clusters(int bn, int split);
int rowtile_stages(int bn);

// Row-tile (swap = false) and swapped (swap = true) kernels built for one forward epilog:
// BIAS, RELU_BIAS, GELU_BIAS, RELU_AUX_BIAS, BIAS_RESIDUAL (fwd_specialised).  rowtile_* and
// swapped_* launch them for those epilogs and the all-epilog kernels for the others.
bool fwd_specialised(int epilog);
cudaError_t fwd_prepare(int bn, bool swap);
cudaError_t fwd_launch(int bn, bool swap, const GemmParams& p, int grid, cudaStream_t stream,
                       bool pdl);

cudaError_t swapped_prepare(int bn);
cudaError_t swapped_launch(int bn, const GemmParams& p, int grid, cudaStream_t stream, bool pdl);
int swapped_smem_bytes(int bn);
int swapped_stages(int bn);

// Small-m kernel (m <= 64): 128 columns of D per CTA, K split over a cluster of `split` CTAs
// (GemmParams::split, kb_per_split, box_k; tiles_m = column tiles, tiles_n = row tiles of bn);
// grid = tiles_m * tiles_n * split.  smem: smallm_smem_bytes for the configuration.
cudaError_t smallm_prepare();
cudaError_t smallm_launch(int bn, const GemmParams& p, int grid, int smem, cudaStream_t stream,
                          bool pdl);
int smallm_smem_bytes(int bn, int kc, int split);
int smallm_max_clusters(int bn, int split, int smem);

// Row-tile kernel run by CTA pairs (cta_group::2): 256 x 256 tiles, clusters of 2.
cudaError_t rowpair_prepare(int bn);
cudaError_t rowpair_launch(int bn, const GemmParams& p, int grid, cudaStream_t stream, bool pdl);
int rowpair_smem_bytes(int bn);
int rowpair_stages(int bn);
int rowpair_max_clusters(int bn);

// CTA-pair kernel on E4M3 inputs (256 x bn tiles, bn 256 or 224), epilogs BIAS, RELU_BIAS,
// GELU_BIAS, RELU_AUX_BIAS, BIAS_RESIDUAL, NONE.
cudaError_t fp8_pair_prepare();
cudaError_t fp8_pair_launch(int bn, const GemmParams& p, int grid, cudaStream_t stream, bool pdl);

// The FFN block in one CTA-pair launch (256 x 256 tiles); never a programmatic dependent.
cudaError_t ffn_pair_prepare();
cudaError_t ffn_pair_launch(const GemmParams& p, int grid, cudaStream_t stream);

// The FFN block with H kept on chip (csrc/ffn_onchip.cu): CTA (r, q) owns rows
// [128 r, 128 r + 128) of X and Y and columns [256 q, 256 q + 256) of Y.  For each 256-wide
// chunk of H: GEMM 1 H_c = X W1[:, chunk] into tensor memory, bias + GELU into a 16-bit
// copy in shared memory (the layout GEMM 2 reads), GEMM 2 Y += H_c W2[chunk, cols] into
// tensor memory; then Y + b2 + R.  d and f are multiples of 256.
struct OnchipFfnParams {
    CUtensorMap tm_X;   // X[t][d]: K-major boxes {64 k, 128 rows}, 128-byte swizzle
    CUtensorMap tm_W1;  // W1[d][f]: N-major boxes {64 n, 64 k}, 128-byte swizzle
    CUtensorMap tm_W2;  // W2[f][d]: N-major boxes {64 n, 64 k}, 128-byte swizzle
    const void* b1;
    const void* b2;
    const void* R;
    void* Y;
    int* status;
    unsigned long long wait_limit_ns;
    int t, d, f;
    int bf16;
};
cudaError_t ffn_onchip_prepare();
cudaError_t ffn_onchip_launch(const OnchipFfnParams& p, int grid, cudaStream_t stream);


// Elementwise epilogue over a 16-bit pre-activation (the unfused baseline's second kernel;
// pre == nullptr means pre = 0, which serves k == 0).
struct ElementwiseArgs {
    const void* pre;       // 16-bit A.B (nullptr: zero, the k == 0 problem)
    const void* bias;
    const void* residual;
    void* D;
    void* aux;
    const void* aux_in;
    float* dbias;
    const float* ln_stats;
    const float* ln_colsum;
    const float* ln_bias;
    int m, n, epilog, bias_layout, bf16, aux_ld;
};
cudaError_t elementwise_launch(const ElementwiseArgs& a, int sm_count, cudaStream_t stream);

// LayerNorm kernels (csrc/layernorm.cu); d must be a multiple of 8.
// stats[2i], stats[2i+1] = mean and 1/sqrt(var + eps) of row i of X (t x d).
cudaError_t layernorm_stats_launch(const void* X, int t, int d, int bf16, float eps,
                                   float* stats, int sm_count, cudaStream_t stream);
// Y = LayerNorm(X) * gamma + beta (+ residual when not nullptr), one pass per row.
cudaError_t layernorm_launch(const void* X, const void* residual, const void* gamma,
                             const void* beta, void* Y, int t, int d, int bf16, float eps,
                             int sm_count, cudaStream_t stream);
// Folding LayerNorm's affine part into the following GEMM (W: d x f):
// Wf[k][j] = 16-bit(gamma_k W[k][j]), colsum_j = sum_k Wf[k][j], bias_f_j = sum_k beta_k W[k][j] + b_j.
cudaError_t layernorm_fold_launch(const void* gamma, const void* beta, const void* W,
                                  const void* b, void* Wf, float* colsum, float* bias_f, int d,
                                  int f, int bf16, int sm_count, cudaStream_t stream);

}  // namespace gemm_epi
