// Internal to the library (not part of the C ABI): the plan object and the helpers the C
// entry points share.  api.cu holds the GEMM plans and their launches, host_exec.cu the
// host-buffer call, ffn_api.cu the FFN block (and its allocation-free form),
// layernorm_api.cu the LayerNorm calls.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "gemm_epi.h"
#include "kernel_params.h"

namespace gemm_epi_impl {

enum Variant { kEmpty = 0, kRowTile = 1, kSwapped = 2, kBiasOnly = 3, kRowPair = 4, kSmallM = 5 };

constexpr int kSwappedMaxM = 256;
// A plan's own device words: the status word (byte 0) and the tile counter (bytes 8-15).
constexpr size_t kPlanWordsBytes = 16;
constexpr unsigned long long kDefaultWaitNs = 2000ull * 1000 * 1000;  // 2 s

struct HostPipe;

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace gemm_epi_impl

struct gemm_epi_plan_s {
    int64_t m, n, k;
    int dtype, epilog, bias_layout;
    int device, sm_count;
    // chosen configuration
    int variant, bn, stages, smem, grid, group_m, tiles_m, tiles_n, k_blocks;
    int split, kb_per_split;  // split-K slices (split == 1: persistent kernel)
    int split_global;         // 1: the slices meet in device memory, 0: in a cluster
    int split_l2;             // cluster slices whose partial sums meet in device memory
    int dyn_order;            // CTA-pair kernel: tiles handed out by the device counter
    int swap_m64;             // swapped kernel with 64 MMA rows (columns of D) per tile
    int box_k;                // small-m kernel: rows of k per copy of B
    // Row strides of B and D in elements (0: n, the dense layout).  Set only on the host
    // pipeline's column-panel plans (a panel of B and of D inside the full matrices).
    int64_t ldb, ldd;
    // options (0 = automatic)
    int opt_variant, opt_bn, opt_split_k, opt_grid, opt_group_m, opt_split_mode, opt_tile_m;
    int opt_tile_order;
    // split-K through device memory: fp32 partial tiles [tile][slice][128 x bn] and the
    // per-tile arrival counts (zero between launches), allocated when the plan is configured
    float* d_split_ws;
    unsigned* d_split_count;
    size_t split_ws_bytes, split_count_len;
    int prefetch;  // L2 prefetch distance in K blocks (GEMM_EPI_OPT_PREFETCH)
    int no_pdl;    // 1: launch without programmatic dependent launch (GEMM_EPI_OPT_PDL = 0)
    int b_ready;   // 1: no earlier work on the stream writes B (GEMM_EPI_OPT_B_READY)
    unsigned long long wait_limit_ns;
    int debug_stall;
    int* d_status;
    // CTA-pair kernels' tile counter (two words, zero between launches; see GemmParams::sched),
    // in the same allocation as the status word; NULL: static tile order only
    unsigned* d_sched;
    // tensor maps for the last (A, B, D) pointers
    const void* key_A;
    const void* key_B;
    const void* key_D;
    bool maps_valid;
    CUtensorMap tm_A, tm_B, tm_D;
    char desc[320];
    gemm_epi_impl::HostPipe* host;  // gemm_epi_execute_host's streams, buffers and chunk plans
};

namespace gemm_epi_impl {

// Epilogs built for E4M3 inputs (forward, no 16-bit auxiliary output).
bool fp8_epilog(int e);
bool backward(int epilog);
int64_t dbias_len(const gemm_epi_plan_s* p);

// Pick the kernel and its configuration for the plan's shape and options (allocates the
// split-K workspace when the configuration needs one).
gemm_epi_status configure(gemm_epi_plan_s* p);
// Free the split-K workspace of a plan (NULL-safe on its fields).
void release_split_ws(gemm_epi_plan_s* p);
bool encode_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dt, uint64_t inner,
               uint64_t outer, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw,
               uint64_t elem_bytes = 2, uint64_t row_elems = 0);
gemm_epi_status ensure_maps(gemm_epi_plan_s* p, const void* A, const void* B, void* D);
gemm_epi_status check_device(const gemm_epi_plan_s* p);
// The current device, checked to be sm_103, and its SM count.
gemm_epi_status current_device(int* sms);
gemm_epi_status check_operands(const gemm_epi_plan_s* p, const gemm_epi_operands& o);
gemm_epi_operands make_operands(const void* A, const void* B, const void* bias,
                                const void* residual, void* D, void* aux);
gemm_epi_status launch_gemm(gemm_epi_plan_s* p, const gemm_epi_operands& ops, int epilog,
                            cudaStream_t stream, bool pdl = false);
gemm_epi_status zero_dbias(const gemm_epi_plan_s* p, const gemm_epi_operands& ops,
                           cudaStream_t stream);
cudaError_t run_elementwise(const gemm_epi_plan_s* p, const void* pre,
                            const gemm_epi_operands& ops, cudaStream_t stream);
// One fused call on an already-checked plan (empty problems launch nothing, k == 0 runs the
// elementwise epilogue on the bias alone).
gemm_epi_status run_plan(gemm_epi_plan_s* p, const gemm_epi_operands& ops, cudaStream_t stream,
                         bool pdl);
// host_exec.cu
void destroy_host_pipe(gemm_epi_plan_s* p);
gemm_epi_status run_host(gemm_epi_plan_s* p, const gemm_epi_operands& o, cudaStream_t stream);

}  // namespace gemm_epi_impl
