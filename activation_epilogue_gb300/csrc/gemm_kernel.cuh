// Fused GEMM + bias/activation epilogue for sm_103a.
//
// D = epi(A . B + bias), computed as in "Fusing bias into cuBLASLt matmul with
// nvmath-python for PyTorch inference" (blog.hotdry.top, 2025-09-22): the bias is added and
// the activation applied right after the core GEMM, inside the same thread block, and the
// intermediate matrix is never written back to device memory.
//
// One persistent CTA per SM (or per SM of a CTA pair), with warps in fixed roles:
//   warp 0      TMA producer: one thread streams 64-deep K blocks of both operands into a
//               ring of shared-memory stages (128-byte swizzle), arming a "full" mbarrier
//               with the byte count of each stage.  In a CTA pair, the even CTA's producer
//               also decides the pair's next tile (statically, or from a device-wide
//               counter) and hands the tile indices to the other roles of both CTAs.
//   warp 1      allocates tensor memory; one thread issues tcgen05.mma (fp32 accumulate)
//               into one of two TMEM accumulators and commits each consumed stage back to
//               its "empty" mbarrier, and each finished tile to a "tmem full" mbarrier.
//   warps 2..   epilogue (EW warps: 8, or 16 for GELU/TANH pair tiles on short K): EW / 4
//               warps per 32-lane quarter of the accumulator, taking every (EW / 4)-th
//               32-column chunk (several warps per scheduler hide the latency of the
//               activation arithmetic); a warp reads a chunk from TMEM, adds the bias
//               (staged per warp in shared memory, or shuffled between lanes with more
//               warps, when it varies along the columns), applies the activation, builds
//               the ReLU mask words, rounds to 16 bits and writes D through a swizzled
//               shared-memory box and a TMA store.  While it drains one accumulator the
//               MMA warp fills the other, so the epilogue overlaps the next tile's GEMM.
//
// Backward epilogues (DRELU_BGRAD, DGELU_BGRAD): the accumulator is multiplied by the
// stored ReLU mask bit or by GELU' of the stored pre-activation, written as D, and reduced
// on chip into the bias gradient: sums along a thread's own row of the chunk stay in
// registers until the tile is done, sums across the 32 lanes of a warp come from one
// transpose-and-add butterfly; either way one fp32 atomic per warp and bias entry per tile.
//
// Split-K (small grids), three forms.  Cluster: the CTAs of a cluster share one output tile,
// each accumulating a slice of K in its own TMEM.  The tile's (lane quarter, 32-column
// chunk) blocks are owned by the ranks in a cycle along each epilogue warp's chunks
// (split_owner); every CTA publishes the blocks it does not own, the cluster synchronises,
// and each owner adds the peers' blocks in rank order before running the epilogue on its
// chunks.  The blocks meet either in a device-memory workspace (split_l2: stored with
// st.global, copied back into the owner's idle stage ring with cp.async right after the
// barrier; an SM moves data to and from L2 several times faster than over distributed
// shared memory) or in the publishing CTA's idle stage ring, read by the owners over
// distributed shared memory.  Device memory alone: independent CTAs write their fp32
// partial tiles to a workspace (it stays in L2) and count themselves per tile; the CTA that
// arrives last adds the slices in slice order and runs the epilogue.  No CTA waits for
// another.
//
// Every mbarrier wait is bounded by a time limit; on expiry the waiting thread records the
// failure in the plan's status word and raises a shared abort flag, every role leaves its
// loop, in-flight copies and MMAs are drained, tensor memory is freed and the kernel returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "gelu.cuh"
#include "kernel_params.h"
#include "ptx.cuh"

namespace gemm_epi {

constexpr int kBM = 128;        // MMA M: TMEM lanes
constexpr int kBK = 64;         // K block: one 128-byte swizzle row of 16-bit elements
constexpr int kUmmaK = 16;      // K of one tcgen05.mma.kind::f16
constexpr int kEpiWarps = kEpilogueWarps;  // two per TMEM lane quarter, alternating chunks
constexpr int kThreads = 64 + 32 * kEpiWarps;   // producer, MMA, epilogue warps
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kPipeBudget = 192 * 1024;
constexpr int kMaxSplit = 4;    // split-K: CTAs per cluster at most
constexpr int kMaxGSplit = 8;   // split-K through device memory: K slices per tile at most

constexpr int pow2_at_least(int x, int p = 32) { return p >= x ? p : pow2_at_least(x, 2 * p); }

// PAIR: a CTA pair computes a 256 x BN tile with cta_group::2 MMAs; each CTA holds 128 rows
// of A and BN/2 rows (columns of D) of B per stage, staged as whole 64-row panels (for BN
// 224 or 192 the last panel is partly unused).
// EW: epilogue warps (8, or 16 for the CTA-pair kernels of the costlier activations on short
// K; with more than 8 the bias is shuffled between lanes instead of staged in shared memory).
template <int BN, bool PAIR = false, int EW = 8>
struct TileCfg {
    static constexpr int kBRows = PAIR ? (BN / 2 + 63) / 64 * 64 : BN;
    static constexpr int kABytes = kBM * kBK * 2;      // MMA-A operand: 128 rows x 64 k
    static constexpr int kBBytes = kBRows * kBK * 2;   // MMA-B operand: kBRows rows x 64 k
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kStagesRaw = kPipeBudget / kStageBytes;
    static constexpr int kStages = kStagesRaw > 8 ? 8 : kStagesRaw;
    static constexpr int kChunk = BN < 32 ? BN : 32;            // columns per TMEM load
    static constexpr int kTmemCols = pow2_at_least(2 * BN);  // two accumulators
    static constexpr int kOffEpi = kStages * kStageBytes;        // one 2 KB box per warp
    static constexpr int kEpiBytes = EW * 2048;
    static constexpr int kOffBias = kOffEpi + kEpiBytes;         // 2 x 256 fp32 per warp
    static constexpr int kBiasBytes = EW == 8 ? EW * 512 * 4 : 0;
    static constexpr int kOffBar = kOffBias + kBiasBytes;
    static constexpr int kBarBytes = 512;
    static constexpr int kSmemBytes = 1024 + kOffBar + kBarBytes;  // + alignment slack
    static constexpr int kRedBytes = kBM * BN * 4;  // one fp32 partial tile (split-K)
    static_assert(kStages >= 2, "pipeline needs two stages");
    static_assert(kRedBytes <= kStages * kStageBytes, "partial tile must fit the stage ring");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
    static_assert(kOffBias % 16 == 0, "per-warp bias staging is read with 16-byte loads");
};

// mbarrier slots in the barrier area
constexpr int kBarFull = 0;        // [8]
constexpr int kBarEmpty = 8;       // [8]
constexpr int kBarTmemFull = 16;   // [2]
constexpr int kBarTmemEmpty = 18;  // [2]
constexpr int kBarStall = 20;
constexpr int kBarDrain = 21;
constexpr int kOffHolder = 22 * 8;  // TMEM base address written by tcgen05.alloc
constexpr int kOffAbort = kOffHolder + 4;
constexpr int kOffLast = kOffAbort + 4;  // split-K through device memory: "this CTA is last"
// CTA pairs: the ring of tile indices (see sched_publish)
constexpr int kSchedSlots = 8;
constexpr int kBarSchedFull = 24;         // [8] in each CTA: slot written
constexpr int kBarSchedEmpty = 32;        // [8] in the even CTA: slot read by every consumer
constexpr int kOffSchedSlot = 40 * 8;     // int[8] in each CTA: the tile indices
static_assert(kOffLast + 4 <= kBarSchedFull * 8, "barrier area layout");
// Split-K across a cluster through L2 (single CTAs): the shared memory each epilogue warp
// receives its peers' partial sums in (in the idle stage ring)
constexpr int kL2SlotBytes = 16 * 1024;

constexpr unsigned long long kDrainLimitNs = 20ull * 1000 * 1000;  // 20 ms

// Wait for the phase of `bar` with parity `parity` to complete.  Gives up (returns false)
// when the abort flag is raised or after limit_ns nanoseconds; also after limit_ns / 8
// polls, in case the global timer does not advance.  CLUSTER: acquire at cluster scope (the
// barrier is signalled from the other CTA of a pair, after it wrote data read here).
template <bool CLUSTER = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity,
                                             const volatile int* abort_flag,
                                             unsigned long long limit_ns, bool honour_abort = true)
{
    if (CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    const unsigned long long max_polls = limit_ns / 8 + 1024;
    for (unsigned long long poll = 1; poll < max_polls; ++poll) {
        if (CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if ((poll & 63) == 0) {
            if (honour_abort && *abort_flag) return false;
            if (globaltimer_ns() - t0 > limit_ns) return false;
        }
    }
    return false;
}

__device__ __forceinline__ void record_failure(int* status, volatile int* abort_flag, int role)
{
    *abort_flag = 1;
    __threadfence_block();
    atomicCAS(status, 0, kCodeTimeout | role);
}

__device__ __forceinline__ void tile_coords(int tile, const GemmParams& p, int& tm, int& tn)
{
    // Groups of group_m MMA-row tiles; inside a group the row tile varies fastest, so the
    // CTAs running at one time share a few B panels and a few A panels in L2.
    const int per_group = p.group_m * p.tiles_n;
    const int g = tile / per_group;
    const int first = g * p.group_m;
    const int rows_in_group = min(p.tiles_m - first, p.group_m);
    const int r = tile - g * per_group;
    tm = first + r % rows_in_group;
    tn = r / rows_in_group;
    // Odd groups walk the column tiles backwards, so a group starts on the B panels the
    // previous one read last (still in L2).  Measured on GB300 at 65536 x 16384 x 8192
    // RELU_BIAS: DRAM reads 26.5-27.4 -> 21.3-24.3 GB per launch, 1755 -> 1762 TFLOP/s.
    if (g & 1) tn = p.tiles_n - 1 - tn;
}

// The tiles and K blocks one CTA works on.
struct WorkRange {
    int first, stride, end;  // tiles first, first + stride, ... below end
    int kb_begin, kb_end;    // K blocks [kb_begin, kb_end) of each tile
    int rank, split;         // split-K: cluster rank and size (split == 1: no split)
    int grank, gsplit;       // split-K through device memory: K slice and slices (1: none)
    int pair_rank;           // CTA pairs: 0 = the even CTA (issues the MMAs), 1 = the odd
};

template <bool PAIR = false>
__device__ __forceinline__ WorkRange work_range(const GemmParams& p)
{
    WorkRange w;
    if (PAIR) {
        // persistent CTA pairs (clusters of 2) walking 256-row tiles: first tile and the
        // static stride (the tiles after the first come through the pair's tile ring)
        const int cr = static_cast<int>(cluster_ctarank());
        w.first = static_cast<int>(cluster_id_x());
        w.stride = static_cast<int>(gridDim.x / 2);
        w.end = p.tiles_m * p.tiles_n + p.ffn_tiles2;
        w.rank = 0;
        w.split = 1;
        w.pair_rank = cr & 1;
        w.kb_begin = 0;
        w.kb_end = p.k_blocks;
        w.grank = 0;
        w.gsplit = 1;
    } else if (p.split > 1 && p.split_global) {
        // one (tile, K slice) per CTA
        const int tile = static_cast<int>(blockIdx.x) / p.split;
        w.first = tile;
        w.stride = 1;
        w.end = tile + 1;
        w.rank = 0;
        w.split = 1;
        w.grank = static_cast<int>(blockIdx.x) - tile * p.split;
        w.gsplit = p.split;
        w.pair_rank = 0;
        w.kb_begin = w.grank * p.kb_per_split;
        w.kb_end = min(p.k_blocks, w.kb_begin + p.kb_per_split);
        return w;
    } else if (p.split > 1) {
        const int tile = static_cast<int>(cluster_id_x());
        w.first = tile;
        w.stride = 1;
        w.end = tile + 1;
        w.rank = static_cast<int>(cluster_ctarank());
        w.split = p.split;
        w.grank = 0;
        w.gsplit = 1;
        w.pair_rank = 0;
        w.kb_begin = w.rank * p.kb_per_split;
        w.kb_end = min(p.k_blocks, w.kb_begin + p.kb_per_split);
    } else {
        w.first = blockIdx.x;
        w.stride = gridDim.x;
        w.end = p.tiles_m * p.tiles_n;
        w.rank = 0;
        w.split = 1;
        w.grank = 0;
        w.gsplit = 1;
        w.pair_rank = 0;
        w.kb_begin = 0;
        w.kb_end = p.k_blocks;
    }
    return w;
}

// Split-K: the rank of the cluster that owns (reduces, then runs the epilogue of) chunk c
// of TMEM lane quarter q.  Spreading (quarter, chunk) units over the ranks shares the
// reduction among the CTAs even when a tile has a single chunk.  The epilogue warp of
// quarter q with index `part` takes chunks part, part + 2, ...; as it walks them the owner
// steps through the ranks, so every warp both publishes and reduces, about 1/split of its
// chunks each (the warp index 4 part + q offsets the cycle).
__device__ __forceinline__ int split_owner(int q, int c, int split)
{
    return (4 * (c & 1) + q + (c >> 1)) % split;
}

// One tile of the walk: which GEMM (0, or 1 = the second GEMM of a fused FFN block), its
// coordinates, its K blocks [kb_begin, kb_end) and (second GEMM) its K slice.
struct TileInfo {
    int prob, tm, tn, kb_begin, kb_end, slice, tile2;
};

template <bool FFN>
__device__ __forceinline__ TileInfo tile_info(const GemmParams& p, int tile, const WorkRange& w)
{
    TileInfo t;
    const int tiles1 = p.tiles_m * p.tiles_n;
    if (!FFN || tile < tiles1) {
        tile_coords(tile, p, t.tm, t.tn);
        t.prob = 0;
        t.kb_begin = w.kb_begin;
        t.kb_end = w.kb_end;
        t.slice = 0;
        t.tile2 = 0;
    } else {
        // GEMM 2 in row order (the row blocks of H finish roughly in that order), the K
        // slices of a tile next to each other
        const int u = tile - tiles1;
        t.tile2 = u / p.ffn_split2;
        t.slice = u - t.tile2 * p.ffn_split2;
        t.tm = t.tile2 / p.tiles_n2;
        t.tn = t.tile2 - t.tm * p.tiles_n2;
        t.prob = 1;
        t.kb_begin = t.slice * p.ffn_kb2;
        t.kb_end = min(p.k_blocks2, t.kb_begin + p.ffn_kb2);
    }
    return t;
}

// FFN: the counter of H's row block tm and GEMM-2 K slice s, and the count that means "all
// of it stored": GEMM-1 tile tn (columns [256 tn, 256 tn + 256) of H, GEMM-2 K blocks
// [4 tn, 4 tn + 4)) lies in slice 4 tn / ffn_kb2.
__device__ __forceinline__ int ffn_ready_index(const GemmParams& p, int tm, int s)
{
    return tm * p.ffn_split2 + s;
}
__device__ __forceinline__ int ffn_slice_of_tile1(const GemmParams& p, int tn)
{
    return 4 * tn / p.ffn_kb2;
}
__device__ __forceinline__ int ffn_ready_count(const GemmParams& p, int s)
{
    const int lo = (s * p.ffn_kb2 + 3) / 4;
    const int hi = min(p.tiles_n, ((s + 1) * p.ffn_kb2 + 3) / 4);
    return p.ffn_ready_target * (hi - lo);
}

// FFN: wait until the slice of H a GEMM-2 unit reads is complete (bounded like the
// mbarrier waits; false on abort or time-out).  The acquire load orders the TMA loads that
// follow (after a proxy fence) behind the GEMM-1 stores it observes.
__device__ __forceinline__ bool wait_ffn_ready(const GemmParams& p, int tm, int s,
                                               const volatile int* abort_flag)
{
    const int* flag = p.ffn_ready + ffn_ready_index(p, tm, s);
    const int target = ffn_ready_count(p, s);
    if (ld_acquire_gpu(flag) >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    const unsigned long long max_polls = p.wait_limit_ns / 32 + 1024;
    for (unsigned long long poll = 1; poll < max_polls; ++poll) {
        __nanosleep(32);
        if (ld_acquire_gpu(flag) >= target) return true;
        if ((poll & 15) == 0) {
            if (*abort_flag) return false;
            if (globaltimer_ns() - t0 > p.wait_limit_ns) return false;
        }
    }
    return false;
}

// ---- tile order of the CTA-pair kernels ---------------------------------------------------
// Every role of both CTAs starts with the pair's first tile, the cluster index.  The even
// CTA's producer thread decides the later ones: statically (+ the number of pairs), or from
// the device-wide counter p.sched (tiles handed out in raster order, as pairs become free).
// It hands each index, in order, to the other roles of both CTAs through a ring of
// kSchedSlots words that exists in both CTAs: slot s has a "full" barrier in each CTA (one
// arrival, the even producer's) and an "empty" barrier in the even CTA that counts the
// consumers (the even CTA's MMA thread, the odd CTA's producer, and every epilogue warp of
// both CTAs).  The pair's tile j >= 1 travels in slot (j - 1) mod kSchedSlots; an index at
// or past the end of the walk ends it.
template <int EW>
__host__ __device__ constexpr uint32_t sched_consumers() { return 2u + 2u * EW; }

// Even producer: publish `tile` as the pair's tile j (j >= 1) to both CTAs.
__device__ __forceinline__ bool sched_publish(uint32_t bar0, int j, int tile,
                                              const volatile int* abort_flag,
                                              unsigned long long limit_ns)
{
    const int s = (j - 1) % kSchedSlots;
    const uint32_t ph = static_cast<uint32_t>(((j - 1) / kSchedSlots) & 1);
    // every consumer has read this slot's previous index
    if (!wait_bounded<true>(bar0 + 8u * (kBarSchedEmpty + s), ph ^ 1u, abort_flag, limit_ns))
        return false;
    const uint32_t slot = bar0 + kOffSchedSlot + 4u * static_cast<uint32_t>(s);
    const uint32_t full = bar0 + 8u * (kBarSchedFull + s);
    const uint32_t peer = cluster_ctarank() ^ 1u;
    st_shared_u32(slot, static_cast<uint32_t>(tile));
    st_shared_cluster_u32(map_shared_rank(slot, peer), static_cast<uint32_t>(tile));
    mbar_arrive(full);                                 // release: the local write above
    mbar_arrive_cluster(map_shared_rank(full, peer));  // release.cluster: the remote write
    return true;
}

// Consumer (one thread): the pair's tile j (j >= 1); releases the slot after reading it.
__device__ __forceinline__ bool sched_take(uint32_t bar0, int j, int& tile,
                                           const volatile int* abort_flag,
                                           unsigned long long limit_ns)
{
    const int s = (j - 1) % kSchedSlots;
    const uint32_t ph = static_cast<uint32_t>(((j - 1) / kSchedSlots) & 1);
    if (!wait_bounded<true>(bar0 + 8u * (kBarSchedFull + s), ph, abort_flag, limit_ns))
        return false;
    tile = static_cast<int>(ld_shared_u32(bar0 + kOffSchedSlot + 4u * static_cast<uint32_t>(s)));
    const uint32_t empty = bar0 + 8u * (kBarSchedEmpty + s);
    const uint32_t cr = cluster_ctarank();
    if (cr & 1u)
        mbar_arrive_cluster(map_shared_rank(empty, cr & ~1u));
    else
        mbar_arrive(empty);
    return true;
}

// The whole warp: the pair's tile j (j >= 1), taken by lane 0 and broadcast.
__device__ __forceinline__ bool sched_take_warp(uint32_t bar0, int j, int& tile,
                                                const volatile int* abort_flag,
                                                unsigned long long limit_ns)
{
    int ok = 0, t = 0;
    if ((threadIdx.x & 31) == 0) ok = sched_take(bar0, j, t, abort_flag, limit_ns) ? 1 : 0;
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    tile = __shfl_sync(0xFFFFFFFFu, t, 0);
    return ok != 0;
}

// Run by each pair's even CTA, thread 0 (the producer, after its last use of the counter):
// count the pair as done; the last pair sets the counter and the count back to zero, so the
// next launch finds them at zero.  Every pair reaches this whether or not it aborted.
__device__ __forceinline__ void sched_finish(const GemmParams& p)
{
    __threadfence();
    const unsigned pairs = gridDim.x / 2;
    if (atomicAdd(p.sched + 1, 1u) == pairs - 1) {
        __threadfence();
        atomicExch(p.sched, 0u);
        atomicExch(p.sched + 1, 0u);
    }
}

// Byte offset, in the partial-tile buffer, of 16-byte unit `unit` (4 fp32 columns) of
// accumulator row `row`; units are XOR-swizzled by the row so that the 8 rows a quarter
// warp touches land in different banks.
template <int BN>
__device__ __forceinline__ uint32_t red_offset(int row, int unit)
{
    constexpr int kUnits = BN / 4;
    constexpr int kSw = kUnits < 8 ? kUnits - 1 : 7;
    return static_cast<uint32_t>(row * (BN * 4) + ((unit ^ (row & kSw)) << 4));
}

__device__ __forceinline__ float load_16bit(const void* base, long long idx, int bf16)
{
    const uint16_t h = static_cast<const uint16_t*>(base)[idx];
    if (bf16) return __uint_as_float(static_cast<uint32_t>(h) << 16);
    return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ float decode16(uint32_t h, int bf16)
{
    if (bf16) return __uint_as_float(h << 16);
    return __half2float(__ushort_as_half(static_cast<uint16_t>(h)));
}

__device__ __forceinline__ uint32_t pack2(float a, float b, int bf16)
{
    if (bf16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&v);
    }
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint16_t to16(float a, int bf16)
{
    if (bf16) return __bfloat16_as_ushort(__float2bfloat16_rn(a));
    return __half_as_ushort(__float2half_rn(a));
}


// ------------------------------------------------------------------------------------------
// producer: TMA loads
// ------------------------------------------------------------------------------------------
// Arm stage `stage` for K block `kb` of tile (tm, tn) and issue its TMA loads.  Single
// CTAs only, PART = 1: arm the stage and copy B alone; PART = 2: copy A alone (into a stage
// that PART 1 armed).
template <int BN, bool SWAP, bool PAIR = false, bool F8 = false, int PART = 0>
__device__ __forceinline__ void issue_stage(const GemmParams& p, uint32_t sbase, uint32_t bar0,
                                            int stage, int tm, int tn, int kb, int prob = 0)
{
    static_assert(PART == 0 || !PAIR, "CTA pairs copy a stage in one part");
    constexpr bool kArm = PART != 2, kCopyA = PART != 1, kCopyB = PART != 2;
    using C = TileCfg<BN, PAIR>;
    const uint32_t fb = bar0 + 8u * (kBarFull + stage);
    const uint32_t sa = sbase + stage * C::kStageBytes;
    const uint32_t sb = sa + C::kABytes;
    const int k0 = kb * kBK;
    if constexpr (PAIR && F8) {
        // E4M3: a K block is 128 elements (one 128-byte swizzle row); A rows and the rows of
        // B transposed (columns of D) are K-major boxes of 128-byte rows: A {128 k, 128
        // rows}, B {128 k, BN / 2 rows} (each CTA's half of the tile's columns: 112 rows at
        // BN = 224, laid out like the first 112 of a 128-row box).  The copy bytes are what
        // bounds this kernel, so the box holds only the rows the MMA (N = BN) reads.
        static_assert(BN == 256 || BN == 224, "the FP8 pair kernel runs 256- or 224-wide tiles");
        constexpr uint32_t kF8StageBytes = C::kABytes + (BN / 2) * 128;
        const uint32_t cr = cluster_ctarank();
        const uint32_t rank = cr & 1u;
        if (rank == 0) mbar_arrive_expect_tx(fb, 2 * kF8StageBytes);
        const uint32_t fb0 = map_shared_rank(fb, cr & ~1u);
        const int k8 = kb * 128;
        const int brow = tn * BN + static_cast<int>(rank) * (BN / 2);
        tma_load_2d_pair(sa, &p.tm_A, fb0, k8, tm * 2 * kBM + static_cast<int>(rank) * kBM);
        tma_load_2d_pair(sb, &p.tm_B, fb0, k8, brow);
        return;
    }
    if constexpr (PAIR) {
        // Both CTAs' halves are counted on the even CTA's "full" barrier, which that CTA
        // arms with the bytes of both (the odd CTA's bytes may land first: the
        // transaction count is signed).
        const uint32_t cr = cluster_ctarank();
        const uint32_t rank = cr & 1u;
        if (rank == 0) mbar_arrive_expect_tx(fb, 2 * C::kStageBytes);
        const uint32_t fb0 = map_shared_rank(fb, cr & ~1u);
        const CUtensorMap* mA = prob ? &p.tm_A2 : &p.tm_A;
        const CUtensorMap* mB = prob ? &p.tm_B2 : &p.tm_B;
        tma_load_2d_pair(sa, mA, fb0, k0, tm * 2 * kBM + static_cast<int>(rank) * kBM);
#pragma unroll
        for (int q = 0; q < C::kBRows / 64; ++q)
            tma_load_2d_pair(sb + q * 8192, mB, fb0,
                             tn * BN + static_cast<int>(rank) * (BN / 2) + q * 64, k0);
        return;
    }
    if (!SWAP) {
        if (kArm) mbar_arrive_expect_tx(fb, C::kStageBytes);
        if (kCopyA) tma_load_2d(sa, &p.tm_A, fb, k0, tm * kBM);
        if (kCopyB) {
#pragma unroll
            for (int q = 0; q < BN / 64; ++q)
                tma_load_2d(sb + q * 8192, &p.tm_B, fb, tn * BN + q * 64, k0);
        }
    } else if (p.swap_m64) {
        // 64 MMA rows: one 64-column box of B (the second half of the A area stays unused)
        if (kArm) mbar_arrive_expect_tx(fb, C::kStageBytes - 8192);
        if (kCopyB) tma_load_2d(sa, &p.tm_B, fb, tm * 64, k0);
        if (kCopyA) tma_load_2d(sb, &p.tm_A, fb, k0, tn * BN);
    } else {
        if (kArm) mbar_arrive_expect_tx(fb, C::kStageBytes);
        if (kCopyB) {
            tma_load_2d(sa, &p.tm_B, fb, tm * kBM, k0);
            tma_load_2d(sa + 8192, &p.tm_B, fb, tm * kBM + 64, k0);
        }
        if (kCopyA) tma_load_2d(sb, &p.tm_A, fb, k0, tn * BN);
    }
}

// L2 prefetch of the operand boxes of K block `kb` of tile (tm, tn).
template <int BN, bool SWAP>
__device__ __forceinline__ void prefetch_stage(const GemmParams& p, int tm, int tn, int kb)
{
    const int k0 = kb * kBK;
    if (!SWAP) {
        tma_prefetch_2d(&p.tm_A, k0, tm * kBM);
#pragma unroll
        for (int q = 0; q < BN / 64; ++q) tma_prefetch_2d(&p.tm_B, tn * BN + q * 64, k0);
    } else if (p.swap_m64) {
        tma_prefetch_2d(&p.tm_B, tm * 64, k0);
        tma_prefetch_2d(&p.tm_A, k0, tn * BN);
    } else {
        tma_prefetch_2d(&p.tm_B, tm * kBM, k0);
        tma_prefetch_2d(&p.tm_B, tm * kBM + 64, k0);
        tma_prefetch_2d(&p.tm_A, k0, tn * BN);
    }
}

// Before the CTA-wide set-up barrier, the thread that initialised the mbarriers fills the
// fresh stage ring for the first tile (no "empty" wait is needed yet), so the first loads
// overlap the tensor-memory allocation.  Returns the number of stages issued.
template <int BN, bool SWAP>
__device__ __forceinline__ int producer_prologue(const GemmParams& p, uint32_t sbase,
                                                 uint32_t bar0)
{
    using C = TileCfg<BN>;
    const WorkRange w = work_range(p);
    if (w.first >= w.end || p.debug_stall) return 0;
    int tm, tn;
    tile_coords(w.first, p, tm, tn);
    const int n = min(C::kStages, w.kb_end - w.kb_begin);
    // Under a programmatic dependent launch the operands may come from the previous grid;
    // B not, when the plan was told so (b_ready): its stages are copied before the wait.
    if (p.b_ready) {
        for (int i = 0; i < n; ++i)
            issue_stage<BN, SWAP, false, false, 1>(p, sbase, bar0, i, tm, tn, w.kb_begin + i);
        grid_dependency_wait();
        for (int i = 0; i < n; ++i)
            issue_stage<BN, SWAP, false, false, 2>(p, sbase, bar0, i, tm, tn, w.kb_begin + i);
    } else {
        grid_dependency_wait();
        for (int i = 0; i < n; ++i) issue_stage<BN, SWAP>(p, sbase, bar0, i, tm, tn, w.kb_begin + i);
    }
    for (int i = 0; i < p.prefetch && w.kb_begin + n + i < w.kb_end; ++i)
        prefetch_stage<BN, SWAP>(p, tm, tn, w.kb_begin + n + i);
    return n;
}

// The producer loop, continuing after the `pre` stages the prologue issued.
template <int BN, bool SWAP, bool PAIR = false, bool FFN = false, bool F8 = false>
__device__ __forceinline__ void run_producer(const GemmParams& p, uint32_t sbase, uint32_t bar0,
                                             volatile int* abort_flag, int pre)
{
    using C = TileCfg<BN, PAIR>;
    const WorkRange w = work_range<PAIR>(p);
    int stage = pre % C::kStages;
    uint32_t phase = static_cast<uint32_t>((pre / C::kStages) & 1);
    long long issued = pre;
    bool ok = true;
    grid_dependency_wait();
    const bool even = !PAIR || w.pair_rank == 0;
    const bool dyn = PAIR && even && p.sched != nullptr;
    // A pair's even producer publishes tile j + 1 while it issues tile j's loads (after its
    // third K block), so that the odd producer and the other roles never wait for it.
    const bool publisher = PAIR && even;
    int tile = w.first;
    int next = w.end;  // publisher: tile j + 1, published during tile j
    for (int j = 0; ok; ++j) {
        if (PAIR && j > 0) {
            if (even) {
                tile = next;
            } else if (!sched_take(bar0, j, tile, abort_flag, p.wait_limit_ns)) {
                if (!*abort_flag) record_failure(p.status, abort_flag, kRoleProducer);
                ok = false;
                break;
            }
        }
        if (tile >= w.end) break;
        // The next tile: asked for now, its index is needed only a few K blocks later.
        unsigned ticket = 0;
        if (dyn) ticket = atomicAdd(p.sched, 1u);
        bool published = !publisher;
        auto publish_next = [&]() -> bool {
            if (dyn) {
                const long long nxt = static_cast<long long>(w.stride) + ticket;
                next = nxt < w.end ? static_cast<int>(nxt) : w.end;
            } else {
                next = tile + w.stride < w.end ? tile + w.stride : w.end;
            }
            published = true;
            return sched_publish(bar0, j + 1, next, abort_flag, p.wait_limit_ns);
        };
        const TileInfo t = tile_info<FFN>(p, tile, w);
        if (FFN && t.prob == 1) {
            if (!wait_ffn_ready(p, t.tm, t.slice, abort_flag)) {
                if (!*abort_flag) record_failure(p.status, abort_flag, kRoleProducer);
                ok = false;
                break;
            }
            fence_proxy_async_global();
        }
        const int kb0 = j == 0 ? t.kb_begin + pre : t.kb_begin;
        const int kb_pub = kb0 + 2 < t.kb_end - 1 ? kb0 + 2 : t.kb_end - 1;
        for (int kb = kb0; kb < t.kb_end; ++kb) {
            if (!wait_bounded(bar0 + 8u * (kBarEmpty + stage), phase ^ 1u, abort_flag,
                              p.wait_limit_ns)) {
                if (!*abort_flag) record_failure(p.status, abort_flag, kRoleProducer);
                ok = false;
                break;
            }
            issue_stage<BN, SWAP, PAIR, F8>(p, sbase, bar0, stage, t.tm, t.tn, kb, t.prob);
            if (!PAIR && p.prefetch && kb + p.prefetch < t.kb_end)
                prefetch_stage<BN, SWAP>(p, t.tm, t.tn, kb + p.prefetch);
            ++issued;
            if (++stage == C::kStages) {
                stage = 0;
                phase ^= 1u;
            }
            if (!published && kb == kb_pub && !publish_next()) {
                if (!*abort_flag) record_failure(p.status, abort_flag, kRoleProducer);
                ok = false;
                break;
            }
        }
        if (ok && !published && !publish_next()) {  // (a tile without K blocks)
            if (!*abort_flag) record_failure(p.status, abort_flag, kRoleProducer);
            ok = false;
        }
        if (!PAIR) tile = tile + w.stride < w.end ? tile + w.stride : w.end;
    }
    if (!ok && !(PAIR && w.pair_rank != 0)) {
        // Let the copies already issued land before the CTA can exit (in a pair, the even
        // CTA's barriers count both CTAs' copies).
        const long long back = issued < C::kStages ? issued : C::kStages;
        for (long long j = 1; j <= back; ++j) {
            const long long f = issued - j;
            const int s = static_cast<int>(f % C::kStages);
            const uint32_t ph = static_cast<uint32_t>((f / C::kStages) & 1);
            wait_bounded(bar0 + 8u * (kBarFull + s), ph, abort_flag, kDrainLimitNs, false);
        }
    }
}

// ------------------------------------------------------------------------------------------
// MMA issuer
// ------------------------------------------------------------------------------------------
template <int BN, bool SWAP, bool PAIR = false, bool FFN = false, bool F8 = false>
__device__ __forceinline__ void run_mma(const GemmParams& p, uint32_t sbase, uint32_t bar0,
                                        uint32_t tmem_base, volatile int* abort_flag)
{
    using C = TileCfg<BN, PAIR>;
    // Row-tile: A operand K-major (rows of A), B operand N-major (rows of B).
    // Swapped:  A operand N-major (rows of B), B operand K-major (rows of A).
    // Pair: M = 256 across the two CTAs; only the even CTA issues.
    // E4M3 (F8): both operands K-major, 32 K elements (32 bytes) per MMA.
    const uint32_t idesc = F8 ? make_idesc_e4m3(2 * kBM, BN)
                              : make_idesc_f16(static_cast<uint32_t>(p.bf16), SWAP ? 1u : 0u,
                                               SWAP ? 0u : 1u,
                                               PAIR ? 2 * kBM : (SWAP && p.swap_m64 ? 64 : kBM), BN);
    const WorkRange w = work_range<PAIR>(p);
    if (PAIR && w.pair_rank != 0) return;
    // commit targets: this (even) CTA, its pair, every CTA whose stages these MMAs read from
    const uint32_t self = PAIR ? cluster_ctarank() : 0u;
    const uint16_t mask_self = static_cast<uint16_t>(1u << self);
    const uint16_t mask_pair = static_cast<uint16_t>(3u << self);
    int stage = 0;
    uint32_t phase = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool issued_any = false;
    bool ok = true;
    int tile = w.first;
    for (int j = 0; ok; ++j) {
        if (j > 0) {
            if (!PAIR) {
                tile += w.stride;
            } else if (!sched_take(bar0, j, tile, abort_flag, p.wait_limit_ns)) {
                if (!*abort_flag) record_failure(p.status, abort_flag, kRoleMma);
                ok = false;
                break;
            }
        }
        if (tile >= w.end) break;
        if (!wait_bounded(bar0 + 8u * (kBarTmemEmpty + acc), acc_phase ^ 1u, abort_flag,
                          p.wait_limit_ns)) {
            if (!*abort_flag) record_failure(p.status, abort_flag, kRoleMma);
            ok = false;
            break;
        }
        tcgen05_fence_after_sync();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        const TileInfo t = tile_info<FFN>(p, tile, w);
        const int kb_begin = t.kb_begin, kb_end = t.kb_end;
        for (int kb = kb_begin; kb < kb_end; ++kb) {
            if (!wait_bounded(bar0 + 8u * (kBarFull + stage), phase, abort_flag,
                              p.wait_limit_ns)) {
                if (!*abort_flag) record_failure(p.status, abort_flag, kRoleMma);
                ok = false;
                break;
            }
            tcgen05_fence_after_sync();
            const uint32_t sa = sbase + stage * C::kStageBytes;
            const uint32_t sb = sa + C::kABytes;
#pragma unroll
            for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
                uint64_t ad, bd;
                if (F8) {
                    ad = make_sdesc_sw128(sa + kk * 32, 0, 1024);
                    bd = make_sdesc_sw128(sb + kk * 32, 0, 1024);
                } else if (!SWAP) {
                    // K-major: +32 bytes per 16-element K step inside the swizzled row;
                    // 8-row groups 1024 bytes apart.
                    ad = make_sdesc_sw128(sa + kk * 32, 0, 1024);
                    // N-major: 64-column panels 8 KB apart, 8-row K groups 1 KB apart;
                    // a 16-deep K step is 16 rows of 128 bytes.
                    bd = make_sdesc_sw128(sb + kk * 2048, 8192, 1024);
                } else {
                    ad = make_sdesc_sw128(sa + kk * 2048, 8192, 1024);
                    bd = make_sdesc_sw128(sb + kk * 32, 0, 1024);
                }
                const uint32_t accum = (kb > kb_begin || kk > 0) ? 1u : 0u;
                if constexpr (PAIR && F8)
                    mma_f8_ss_pair(d_tmem, ad, bd, idesc, accum);
                else if constexpr (PAIR)
                    mma_f16_ss_pair(d_tmem, ad, bd, idesc, accum);
                else
                    mma_f16_ss(d_tmem, ad, bd, idesc, accum);
            }
            issued_any = true;
            // stage free (in both CTAs of a pair) once these MMAs finish
            if constexpr (PAIR)
                mma_commit_pair(bar0 + 8u * (kBarEmpty + stage), mask_pair);
            else
                mma_commit(bar0 + 8u * (kBarEmpty + stage));
            if (++stage == C::kStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) break;
        // accumulator ready for the epilogue (of both CTAs of a pair)
        if constexpr (PAIR)
            mma_commit_pair(bar0 + 8u * (kBarTmemFull + acc), mask_pair);
        else
            mma_commit(bar0 + 8u * (kBarTmemFull + acc));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
    }
    if (!ok && issued_any) {
        // Wait for every MMA this thread issued before tensor memory is released.
        if constexpr (PAIR)
            mma_commit_pair(bar0 + 8u * kBarDrain, mask_self);
        else
            mma_commit(bar0 + 8u * kBarDrain);
        wait_bounded(bar0 + 8u * kBarDrain, 0, abort_flag, kDrainLimitNs, false);
    }
}

// ------------------------------------------------------------------------------------------
// epilogue
// ------------------------------------------------------------------------------------------

// Add the bias to N consecutive accumulator columns: the staged per-column values (four at
// a time, 16-byte broadcast loads: sb is 16-byte aligned, as the staging area and every
// chunk's offset are) or one per-lane value.
template <int N>
__device__ __forceinline__ void add_bias(float (&v)[N], const float* sb, bool col_bias, float lb)
{
    if (col_bias) {
        const float4* s4 = reinterpret_cast<const float4*>(sb);
#pragma unroll
        for (int q = 0; q < N / 4; ++q) {
            const float4 b = s4[q];
            v[4 * q] += b.x;
            v[4 * q + 1] += b.y;
            v[4 * q + 2] += b.z;
            v[4 * q + 3] += b.w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < N; ++j) v[j] += lb;
    }
}

// Apply the activation to one chunk in place: v[] holds acc + bias on entry.
template <int N>
__device__ __forceinline__ void activate(float (&v)[N], int epilog)
{
    if (epilog == EPI_RELU_BIAS || epilog == EPI_RELU_AUX_BIAS) {
#pragma unroll
        for (int j = 0; j < N; ++j) v[j] = v[j] > 0.0f ? v[j] : 0.0f;
    } else if (epilog == EPI_GELU_BIAS || epilog == EPI_GELU_AUX_BIAS || epilog == EPI_LN_GELU_BIAS) {
#pragma unroll
        for (int j = 0; j < N; ++j) v[j] = gelu_erf_fast(v[j]);
    } else if (epilog == EPI_TANH_BIAS) {
#pragma unroll
        for (int j = 0; j < N; ++j) v[j] = tanh_fast(v[j]);
    }
}

// Sums over the 32 lanes of a warp of each of 32 columns: on entry lane l holds x[j], the
// element (l, j) of a 32 x 32 block; on return lane l holds the sum of column l.  Each of
// five rounds halves the columns a lane keeps and adds its partner's half of them
// (16 + 8 + 4 + 2 + 1 = 31 shuffles, against 32 x 5 for 32 separate warp reductions).
__device__ __forceinline__ float warp_column_sums(float (&x)[32], int lane)
{
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < o; ++i) {
            const float send = upper ? x[i] : x[i + o];
            const float keep = upper ? x[i + o] : x[i];
            x[i] = keep + __shfl_xor_sync(0xFFFFFFFFu, send, o);
        }
    }
    return x[0];
}

// Row-tile backward factor: v[j] (row `row`, column col0 + j) times the ReLU mask bit or
// GELU' of the stored pre-activation; 0 outside the matrix.
__device__ __forceinline__ void backward_factor_row(const GemmParams& p, int epilog, float (&v)[32],
                                                    int row, int col0)
{
    const int valid = row < p.m ? min(32, p.n - col0) : 0;
    if (epilog == EPI_DRELU_BGRAD) {
        uint32_t mw = 0;
        if (valid > 0)
            mw = __ldg(static_cast<const uint32_t*>(p.aux_in) + static_cast<long long>(row) * p.aux_ld +
                       col0 / 32);
        if (valid < 32) mw &= (1u << valid) - 1u;  // valid == 0 clears every bit
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = ((mw >> j) & 1u) ? v[j] : 0.0f;
        return;
    }
    const uint16_t* src = static_cast<const uint16_t*>(p.aux_in) + static_cast<long long>(row) * p.n + col0;
    if (valid == 32) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 w = __ldg(reinterpret_cast<const uint4*>(src) + q);
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                v[8 * q + 2 * h] *= gelu_grad_fast(decode16(ww[h] & 0xFFFFu, p.bf16));
                v[8 * q + 2 * h + 1] *= gelu_grad_fast(decode16(ww[h] >> 16, p.bf16));
            }
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            v[j] = j < valid ? v[j] * gelu_grad_fast(decode16(src[j], p.bf16)) : 0.0f;
    }
}

// Row-tile GELU_AUX_BIAS: the 32 pre-activation values of one row, rounded to 16 bits.
__device__ __forceinline__ void store_pre_row(const GemmParams& p, const float (&v)[32], int row,
                                              int col0)
{
    if (row >= p.m) return;
    uint16_t* dst = static_cast<uint16_t*>(p.aux) + static_cast<long long>(row) * p.n + col0;
    const int valid = min(32, p.n - col0);
    if (valid == 32) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack2(v[8 * q + 0], v[8 * q + 1], p.bf16);
            w.y = pack2(v[8 * q + 2], v[8 * q + 3], p.bf16);
            w.z = pack2(v[8 * q + 4], v[8 * q + 5], p.bf16);
            w.w = pack2(v[8 * q + 6], v[8 * q + 7], p.bf16);
            reinterpret_cast<uint4*>(dst)[q] = w;
        }
    } else {
#pragma unroll
        for (int j = 0; j < 32; ++j)
            if (j < valid) dst[j] = to16(v[j], p.bf16);
    }
}

// Split-K through device memory: float4 index of 16-byte unit u (4 fp32 columns) of chunk c
// of accumulator row `row` in K slice s of tile `tile`.  One unit of a warp's 32 rows is
// 512 contiguous bytes.
template <int BN>
__device__ __forceinline__ long long gsplit_index(const GemmParams& p, int tile, int s, int c,
                                                  int u, int row)
{
    constexpr int CH = TileCfg<BN>::kChunk;
    return ((static_cast<long long>(tile) * p.split + s) * (BN / 4) + c * (CH / 4) + u) * kBM + row;
}

// Split-K across a cluster through L2 (split_l2): float4 index, in the workspace, of 16-byte
// unit u of lane `lane` in the block (lane quarter q, chunk c) of cluster rank s's partial
// sums of tile `tile`.  A block (32 rows x CH columns, 128 * CH bytes) is contiguous; in
// it, unit u of the 32 lanes is 512 contiguous bytes (one warp-wide store or copy).
template <int BN>
__device__ __forceinline__ long long l2split_index(const GemmParams& p, int tile, int s, int q,
                                                   int c, int u, int lane)
{
    constexpr int CH = TileCfg<BN>::kChunk;
    return ((((static_cast<long long>(tile) * p.split + s) * 4 + q) * (BN / CH) + c) * (CH / 4) + u) *
               32 + lane;
}

// Split-K across a cluster through L2, an owning epilogue warp (quarter, part) right after
// the cluster barrier: copy the peers' partial sums of its chunks into its slots in the
// idle stage ring (at `slots` from the start of shared memory), each lane its own 16-byte
// units, every copy in flight at once; the lane waits for its copies before reading them
// (cp_async_wait_all) and reads only what it copied.  The cluster barrier (release /
// acquire) has ordered the peers' stores before these loads.
template <int BN>
__device__ __forceinline__ void fetch_peer_partials(const GemmParams& p, uint32_t sbase,
                                                    uint32_t slots, int tile, int rank, int split,
                                                    int quarter, int part, int nchunks)
{
    constexpr int CH = TileCfg<BN>::kChunk;
    constexpr uint32_t kBlk = 128u * CH;
    // A warp takes J = ceil(chunks / 2) chunks and owns at most ceil(J / split) of them (the
    // owner cycles through the ranks), each with split - 1 peer blocks: within its slots.
    constexpr int J = (BN / CH + 1) / 2;
    static_assert(((J + 1) / 2) * 1 * kBlk <= kL2SlotBytes && ((J + 2) / 3) * 2 * kBlk <= kL2SlotBytes &&
                      ((J + 3) / 4) * 3 * kBlk <= kL2SlotBytes,
                  "a warp's peer blocks fit its slots for 2, 3 and 4 slices");
    const int lane = threadIdx.x & 31;
    const float4* ws = reinterpret_cast<const float4*>(p.split_ws);
    int oi = 0;
    for (int c = part; c < nchunks; c += 2) {
        if (split_owner(quarter, c, split) != rank) continue;
        for (int pi = 0; pi < split - 1; ++pi) {
            const int peer = pi < rank ? pi : pi + 1;
            const float4* src = ws + l2split_index<BN>(p, tile, peer, quarter, c, 0, lane);
            const uint32_t dst = sbase + slots + (oi * (split - 1) + pi) * kBlk + lane * 16;
#pragma unroll
            for (int u = 0; u < CH / 4; ++u) cp_async_16(dst + u * 512, src + u * 32);
        }
        ++oi;
    }
}

// Split-K, before the cluster synchronises: write this CTA's partial sums of the chunks
// it does not own into its partial-tile buffer (the stage ring, idle once every MMA of the
// tile has completed).
template <int BN, bool SWAP>
__device__ __forceinline__ void publish_partials(const GemmParams& p, uint8_t* smem,
                                                 uint32_t bar0, uint32_t tmem_base,
                                                 volatile int* abort_flag)
{
    using C = TileCfg<BN>;
    constexpr int CH = C::kChunk;
    const WorkRange w = work_range(p);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;  // which warp of this quarter's pair
    const int row = quarter * 32 + lane;
    int tm, tn;
    tile_coords(w.first, p, tm, tn);
    const int col_limit = SWAP ? p.m : p.n;
    const int nchunks = (min(BN, col_limit - tn * BN) + CH - 1) / CH;
    if (!wait_bounded(bar0 + 8u * kBarTmemFull, 0, abort_flag, p.wait_limit_ns)) {
        if (!*abort_flag) record_failure(p.status, abort_flag, kRoleEpilogue);
        return;
    }
    tcgen05_fence_after_sync();
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    // The workspace may still be read by a programmatic predecessor grid.
    if (p.split_l2) grid_dependency_wait();
    // The bias is read after the cluster barrier: start bringing it into L2 now.
    if (p.epilog != EPI_NONE) {
        const int nb = (SWAP ? p.bias_layout == 0 : p.bias_layout == 1) ? col_limit : (SWAP ? p.n : p.m);
        const int idx = (SWAP ? p.bias_layout == 0 : p.bias_layout == 1) ? tn * BN + lane * 8
                                                                          : tm * kBM + row;
        if (idx < nb) prefetch_global_l2(static_cast<const uint16_t*>(p.bias) + idx);
    }
    for (int c = half; c < nchunks; c += 2) {
        if (split_owner(quarter, c, w.split) == w.rank) continue;
        uint32_t r[32];
        __syncwarp();
        if constexpr (CH == 32)
            tmem_load_32cols(t_lane + c * 32, r);
        else
            tmem_load_16cols(t_lane + c * 16, r);
        if (p.split_l2) {
            // (one block of the workspace: 512 contiguous bytes per unit for the warp)
            float4* ws = reinterpret_cast<float4*>(p.split_ws);
#pragma unroll
            for (int u = 0; u < CH / 4; ++u)
                __stcg(ws + l2split_index<BN>(p, w.first, w.rank, quarter, c, u, lane),
                       make_float4(__uint_as_float(r[4 * u]), __uint_as_float(r[4 * u + 1]),
                                   __uint_as_float(r[4 * u + 2]), __uint_as_float(r[4 * u + 3])));
        } else {
#pragma unroll
            for (int u = 0; u < CH / 4; ++u) {
                uint4 q = make_uint4(r[4 * u], r[4 * u + 1], r[4 * u + 2], r[4 * u + 3]);
                *reinterpret_cast<uint4*>(smem + red_offset<BN>(row, c * (CH / 4) + u)) = q;
            }
        }
    }
    tcgen05_fence_before_sync();
}

// Split-K through device memory, every epilogue thread of every CTA: write this CTA's
// partial tile (all its chunks) to the workspace, then count the CTA for its tile.  Returns
// true in the CTA that arrived last, which then reduces and runs the epilogue.  A CTA that
// gave up on a wait still counts itself (so the count returns to zero); its status word
// entry reports the failure.
template <int BN, bool SWAP>
__device__ __noinline__ bool publish_partials_global(const GemmParams& p, uint8_t* smem,
                                                        uint32_t bar0, uint32_t tmem_base,
                                                        volatile int* abort_flag)
{
    using C = TileCfg<BN>;
    constexpr int CH = C::kChunk;
    const WorkRange w = work_range(p);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;  // which warp of this quarter's pair
    const int row = quarter * 32 + lane;
    const int tile = w.first;
    int tm, tn;
    tile_coords(tile, p, tm, tn);
    const int col_limit = SWAP ? p.m : p.n;
    const int nchunks = (min(BN, col_limit - tn * BN) + CH - 1) / CH;
    // The workspace and the counts may still be in use by a programmatic predecessor.
    grid_dependency_wait();
    bool ok = !*abort_flag;
    if (ok && !wait_bounded(bar0 + 8u * kBarTmemFull, 0, abort_flag, p.wait_limit_ns)) {
        if (!*abort_flag) record_failure(p.status, abort_flag, kRoleEpilogue);
        ok = false;
    }
    if (ok) {
        tcgen05_fence_after_sync();
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
        float4* ws = reinterpret_cast<float4*>(p.split_ws);
        for (int c = half; c < nchunks; c += 2) {
            uint32_t r[32];
            __syncwarp();
            if constexpr (CH == 32)
                tmem_load_32cols(t_lane + c * 32, r);
            else
                tmem_load_16cols(t_lane + c * 16, r);
#pragma unroll
            for (int u = 0; u < CH / 4; ++u)
                __stcg(ws + gsplit_index<BN>(p, tile, w.grank, c, u, row),
                       make_float4(__uint_as_float(r[4 * u]), __uint_as_float(r[4 * u + 1]),
                                   __uint_as_float(r[4 * u + 2]), __uint_as_float(r[4 * u + 3])));
        }
        tcgen05_fence_before_sync();
    }
    // Count the CTA with one acquire-release atomic after the barrier: the release makes the
    // stores of every epilogue thread (ordered before it by the barrier) visible to the CTA
    // that sees the final count, and in that CTA the acquire orders the workspace loads
    // (after the second barrier) behind the other slices' stores.
    named_barrier_sync(1, kEpiThreads);
    volatile int* last_flag = reinterpret_cast<volatile int*>(smem + C::kOffBar + kOffLast);
    if (threadIdx.x == 64) {
        const unsigned before = atom_add_acq_rel_gpu(p.split_count + tile, 1u);
        const bool last = before + 1 == static_cast<unsigned>(p.split);
        if (last) p.split_count[tile] = 0u;  // every CTA of the tile has counted itself
        *last_flag = last ? 1 : 0;
    }
    named_barrier_sync(1, kEpiThreads);
    const bool last = *last_flag != 0;
    if (!last || !ok) return last;
    // The last CTA: add the K slices of each of its chunks in slice order (its own from
    // tensor memory, the others from the workspace, every load of a batch issued first) and
    // put the sum back into tensor memory, where the epilogue reads it.
    tcgen05_fence_after_sync();
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    const float4* ws = reinterpret_cast<const float4*>(p.split_ws);
    constexpr int kUB = CH == 16 ? 4 : 2;  // 16-byte units per batch
    for (int c = half; c < nchunks; c += 2) {
        uint32_t r[32];
        __syncwarp();
        if constexpr (CH == 32)
            tmem_load_32cols(t_lane + c * 32, r);
        else
            tmem_load_16cols(t_lane + c * 16, r);
#pragma unroll
        for (int u0 = 0; u0 < CH / 4; u0 += kUB) {
            float4 part[kMaxGSplit - 1][kUB];
#pragma unroll
            for (int pi = 0; pi < kMaxGSplit - 1; ++pi) {
                if (pi < w.gsplit - 1) {
                    const int s = pi < w.grank ? pi : pi + 1;
#pragma unroll
                    for (int uu = 0; uu < kUB; ++uu)
                        part[pi][uu] = __ldcg(ws + gsplit_index<BN>(p, tile, s, c, u0 + uu, row));
                }
            }
#pragma unroll
            for (int uu = 0; uu < kUB; ++uu) {
                const int j = 4 * (u0 + uu);
                const float4 own = make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                               __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
                float4 a = w.grank == 0 ? own : part[0][uu];
#pragma unroll
                for (int s = 1; s < kMaxGSplit; ++s) {
                    if (s < w.gsplit) {
                        // (indices fixed at compile time: part stays in registers)
                        const float4 b = s == w.grank ? own
                                         : s < w.grank && s < kMaxGSplit - 1 ? part[s][uu]
                                                                              : part[s - 1][uu];
                        a.x += b.x;
                        a.y += b.y;
                        a.z += b.z;
                        a.w += b.w;
                    }
                }
                r[j] = __float_as_uint(a.x);
                r[j + 1] = __float_as_uint(a.y);
                r[j + 2] = __float_as_uint(a.z);
                r[j + 3] = __float_as_uint(a.w);
            }
        }
        if constexpr (CH == 32)
            tmem_store_32cols(t_lane + c * 32, r);
        else
            tmem_store_16cols(t_lane + c * 16, r);
    }
    tcgen05_fence_before_sync();
    return true;
}

// FFN kernel, GEMM 2 split along K (ffn_split2 > 1): float4 index, in the workspace, of
// 16-byte unit u (4 fp32 columns) of 32-column chunk c of accumulator row `row` (0..127 of
// the pair's CTA `pair_rank`) in K slice s of GEMM-2 tile `tile2`.  A warp's 32 rows of one
// unit are 512 contiguous bytes.
template <int BN>
__device__ __forceinline__ long long ffn_ws_index(const GemmParams& p, int tile2, int s,
                                                  int pair_rank, int c, int u, int row)
{
    return (((static_cast<long long>(tile2) * p.ffn_split2 + s) * 2 + pair_rank) * (BN / 4) + c * 8 + u) *
               kBM + row;
}

// One epilogue warp, one K slice of a GEMM-2 tile: copy the warp's accumulator chunks
// (part, part + kParts, ...) to the slice's place in the workspace.  Tensor memory is free
// again once this returns.
template <int BN, int EW>
__device__ __forceinline__ void ffn_write_slice(const GemmParams& p, int tile2, int slice,
                                                int pair_rank, int quarter, int part, int nchunks,
                                                uint32_t t_lane)
{
    constexpr int kParts = EW / 4;
    const int row = quarter * 32 + (threadIdx.x & 31);
    float4* ws = reinterpret_cast<float4*>(p.ffn_ws);
    for (int c = part; c < nchunks; c += kParts) {
        uint32_t r[32];
        __syncwarp();
        tmem_load_32cols(t_lane + c * 32, r);
#pragma unroll
        for (int u = 0; u < 8; ++u)
            __stcg(ws + ffn_ws_index<BN>(p, tile2, slice, pair_rank, c, u, row),
                   make_float4(__uint_as_float(r[4 * u]), __uint_as_float(r[4 * u + 1]),
                               __uint_as_float(r[4 * u + 2]), __uint_as_float(r[4 * u + 3])));
    }
}

// Count this warp's slice for its share of the tile (one acquire-release atomic per warp:
// the release publishes every lane's workspace stores, ordered before it by the warp
// barrier; in the warp that completes the count, the acquire orders its workspace loads
// behind the other slices' stores).  True in the warp of the slice that finished last.
template <int EW>
__device__ __forceinline__ bool ffn_count_slice(const GemmParams& p, int tile2, int pair_rank, int ew)
{
    __syncwarp();
    unsigned before = 0;
    if ((threadIdx.x & 31) == 0)
        before = atom_add_acq_rel_gpu(p.ffn_count + (static_cast<long long>(tile2) * 2 + pair_rank) * EW + ew, 1u);
    before = __shfl_sync(0xFFFFFFFFu, before, 0);
    __syncwarp();
    return before + 1 == static_cast<unsigned>(p.ffn_split2);
}

// The last slice's warp: chunk c of its rows summed over the K slices in slice order (the
// sum does not depend on which slice finished last), from the workspace.  Loads are issued
// 16 columns (every slice) at a time before any is added, so a round trip to L2 serves 16
// columns.
template <int BN>
__device__ __forceinline__ void ffn_sum_chunk(const GemmParams& p, int tile2, int pair_rank,
                                              int quarter, int c, uint32_t (&r)[32])
{
    const int row = quarter * 32 + (threadIdx.x & 31);
    const int S = p.ffn_split2;
    const float4* ws = reinterpret_cast<const float4*>(p.ffn_ws);
#pragma unroll
    for (int u0 = 0; u0 < 8; u0 += 4) {
        float4 part[kFfnMaxSplit2][4];
#pragma unroll
        for (int s = 0; s < kFfnMaxSplit2; ++s) {
            if (s < S) {
#pragma unroll
                for (int uu = 0; uu < 4; ++uu)
                    part[s][uu] = __ldcg(ws + ffn_ws_index<BN>(p, tile2, s, pair_rank, c, u0 + uu, row));
            }
        }
#pragma unroll
        for (int uu = 0; uu < 4; ++uu) {
            float4 a = part[0][uu];
#pragma unroll
            for (int s = 1; s < kFfnMaxSplit2; ++s) {
                if (s < S) {
                    a.x += part[s][uu].x;
                    a.y += part[s][uu].y;
                    a.z += part[s][uu].z;
                    a.w += part[s][uu].w;
                }
            }
            const int j = 4 * (u0 + uu);
            r[j] = __float_as_uint(a.x);
            r[j + 1] = __float_as_uint(a.y);
            r[j + 2] = __float_as_uint(a.z);
            r[j + 3] = __float_as_uint(a.w);
        }
    }
}

// EPI >= 0 fixes the epilog at compile time (only its code is in the kernel); -1 reads it
// from the parameters.
template <int BN, bool SWAP, bool PAIR = false, int EPI = -1, bool F8 = false, int EW = 8>
__device__ __forceinline__ void run_epilogue(const GemmParams& p, uint8_t* smem, uint32_t sbase,
                                             uint32_t bar0, uint32_t tmem_base,
                                             volatile int* abort_flag)
{
    // The FFN kernel runs GELU_BIAS on GEMM-1 tiles and BIAS_RESIDUAL on GEMM-2 tiles.
    constexpr bool FFN = is_ffn(EPI);
    constexpr bool FFN_SPLIT = EPI == kEpiFfnSplit;
    const int epilog0 = FFN ? EPI_GELU_BIAS : (EPI >= 0 ? EPI : p.epilog);
    using C = TileCfg<BN, PAIR, EW>;
    constexpr int CH = C::kChunk;
    constexpr int kParts = EW / 4;       // warps per TMEM lane quarter
    constexpr int kOwn = (BN / CH + kParts - 1) / kParts;  // most chunks a warp takes
    static_assert(EW == 8 || (PAIR && CH == 32 && EW % 4 == 0), "more warps: CTA-pair kernels only");
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int ew = warp - 2;             // epilogue warp 0 .. EW-1
    const int quarter = warp & 3;        // the TMEM lane quarter this warp may access
    const int part = ew >> 2;            // a quarter's warps take every kParts-th chunk
    WorkRange w = work_range<PAIR>(p);
    if (PAIR) w.split = 1;  // (compile-time: the pair kernel never splits K)
    // This warp's own staging area for per-column values (bias; LayerNorm: two arrays of
    // 256): no other warp reads it, so a __syncwarp orders it.  (None with more warps.)
    float* sbias = EW == 8 ? reinterpret_cast<float*>(smem + C::kOffBias) + ew * 512 : nullptr;
    uint8_t* epi_buf = smem + C::kOffEpi + ew * 2048;
    const uint32_t epi_buf_u32 = sbase + C::kOffEpi + ew * 2048;
    // Split-K across a cluster through L2 (one tile per CTA): start copying the peers'
    // partial sums of this warp's chunks (written by this grid) before anything else.
    const uint32_t l2_slots = static_cast<uint32_t>(ew) * kL2SlotBytes;  // (from shared memory)
    if constexpr (!PAIR) {
        static_assert(PAIR || kEpiWarps * kL2SlotBytes <= C::kStages * C::kStageBytes,
                      "every warp's slots fit the stage ring");
        if (w.split > 1 && p.split_l2) {
            int tm0, tn0;
            tile_coords(w.first, p, tm0, tn0);
            const int nch = (min(BN, (SWAP ? p.m : p.n) - tn0 * BN) + CH - 1) / CH;
            fetch_peer_partials<BN>(p, sbase, l2_slots, w.first, w.rank, w.split, quarter, part, nch);
        }
    }
    // Bias, residual and the outputs may belong to a programmatic predecessor grid.
    grid_dependency_wait();
    // E4M3 inputs: the per-tensor dequantisation scales
    const float fp8_scale = F8 ? __ldg(p.scale_a) * __ldg(p.scale_b) : 1.0f;

    int acc = 0;
    uint32_t acc_phase = 0;
    int tile = w.first;
    for (int j = 0;; ++j) {
        if (j > 0) {
            if (!PAIR) {
                tile += w.stride;
            } else if (!sched_take_warp(bar0, j, tile, abort_flag, p.wait_limit_ns)) {
                if (!*abort_flag) record_failure(p.status, abort_flag, kRoleEpilogue);
                break;
            }
        }
        if (tile >= w.end) break;
        const TileInfo t = tile_info<FFN>(p, tile, w);
        const int tm = t.tm, tn = t.tn;
        const bool second = FFN && t.prob == 1;  // GEMM 2 of the FFN block
        const int epilog = second ? static_cast<int>(EPI_BIAS_RESIDUAL) : epilog0;
        const int ncols = second ? p.n2 : p.n;    // columns of this tile's output
        const void* bias_ptr = second ? p.bias2 : p.bias;
        const uint16_t* R = static_cast<const uint16_t*>(second ? p.residual2 : p.residual);
        const CUtensorMap* tmD = second ? &p.tm_D2 : &p.tm_D;
        const bool bwd = is_backward(epilog);
        // LayerNorm folded into the GEMM: pre = rstd_i (acc - mu_i c_j) + b'_j, with (mu, rstd)
        // per row of D and (c, b') per column of D, in fp32
        // (row-tile and pair kernels only: the planner never runs it on the swapped kernel)
        const bool ln = EW == 8 && !SWAP && epilog == EPI_LN_GELU_BIAS;
        const bool has_bias = epilog != EPI_NONE && !bwd && !ln;
        // Bias (and, backward, bias gradient) that varies along the accumulator's columns
        // (staged in shared memory; column sums) or along its lanes (one value per thread).
        const bool along_cols = SWAP ? p.bias_layout == 0 : p.bias_layout == 1;
        const bool col_bias = has_bias && along_cols;
        const bool lane_bias = has_bias && !col_bias;
        const int col_limit = SWAP ? p.m : ncols;   // extent of the accumulator-column coordinate
        const int lane_limit = SWAP ? ncols : p.m;  // extent of the accumulator-lane coordinate
        const int col_base = tn * BN;                          // first accumulator column
        // this warp's first lane coordinate (a pair's odd CTA holds rows 128..255 of the tile)
        // (64-row swapped tiles: 16 columns of D per warp, in lanes 0-15)
        const bool m64 = SWAP && p.swap_m64;
        const int lane_base = PAIR  ? tm * 2 * kBM + w.pair_rank * kBM + quarter * 32
                              : m64 ? tm * 64 + quarter * 16
                                    : tm * kBM + quarter * 32;
        const int lane_idx = m64 && lane >= 16 ? lane_limit : lane_base + lane;
        if (*abort_flag) break;
        if (EW == 8 && col_bias) {
            __syncwarp();  // every lane is done reading the previous tile's values
            const uint16_t* bsrc = static_cast<const uint16_t*>(bias_ptr) + col_base;
            if (col_base + BN <= col_limit && (reinterpret_cast<uintptr_t>(bsrc) & 15) == 0) {
                // whole tile in range and 16-byte aligned: one 8-element load per lane
                for (int i8 = lane; i8 < BN / 8; i8 += 32) {
                    const uint4 w8 = __ldg(reinterpret_cast<const uint4*>(bsrc) + i8);
                    const uint32_t ww[4] = {w8.x, w8.y, w8.z, w8.w};
                    float f[8];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const uint16_t lo = static_cast<uint16_t>(ww[h] & 0xFFFFu);
                        const uint16_t hi = static_cast<uint16_t>(ww[h] >> 16);
                        f[2 * h] = p.bf16 ? __uint_as_float(static_cast<uint32_t>(lo) << 16)
                                          : __half2float(__ushort_as_half(lo));
                        f[2 * h + 1] = p.bf16 ? __uint_as_float(static_cast<uint32_t>(hi) << 16)
                                              : __half2float(__ushort_as_half(hi));
                    }
                    reinterpret_cast<float4*>(sbias)[2 * i8] = make_float4(f[0], f[1], f[2], f[3]);
                    reinterpret_cast<float4*>(sbias)[2 * i8 + 1] = make_float4(f[4], f[5], f[6], f[7]);
                }
            } else {
                for (int i = lane; i < BN; i += 32) {
                    const int c = col_base + i;
                    sbias[i] = c < col_limit ? load_16bit(bias_ptr, c, p.bf16) : 0.0f;
                }
            }
            __syncwarp();
        }
        const float lb = (lane_bias && lane_idx < lane_limit) ? load_16bit(bias_ptr, lane_idx, p.bf16)
                                                              : 0.0f;
        // LayerNorm values: staged per accumulator column (row-tile: c_j and b'_j; swapped:
        // mu_i and rstd_i) and one pair per lane (row-tile: mu_i, rstd_i; swapped: c_j, b'_j)
        float ln_la = 0.0f, ln_lb = 0.0f;
        if (ln) {
            __syncwarp();
            for (int i = lane; i < BN; i += 32) {
                const int ci = col_base + i;
                float va = 0.0f, vb = 0.0f;
                if (ci < col_limit) {
                    va = SWAP ? p.ln_stats[2 * ci] : p.ln_colsum[ci];
                    vb = SWAP ? p.ln_stats[2 * ci + 1] : p.ln_bias[ci];
                }
                sbias[i] = va;
                sbias[256 + i] = vb;
            }
            __syncwarp();
            if (lane_idx < lane_limit) {
                ln_la = SWAP ? p.ln_colsum[lane_idx] : p.ln_stats[2 * lane_idx];
                ln_lb = SWAP ? p.ln_bias[lane_idx] : p.ln_stats[2 * lane_idx + 1];
            }
        }

        const int valid_cols = min(BN, col_limit - col_base);
        const int nchunks = (valid_cols + CH - 1) / CH;
        // more warps: lane l holds the bias of column l of each of its chunks (shuffled out)
        float bl[EW == 8 ? 1 : kOwn];
        if constexpr (EW != 8) {
#pragma unroll
            for (int i = 0; i < kOwn; ++i) {
                const int col = col_base + (part + i * kParts) * CH + lane;
                bl[i] = col_bias && col < col_limit ? load_16bit(bias_ptr, col, p.bf16) : 0.0f;
            }
        }
        if (!SWAP && (epilog == EPI_BIAS_RESIDUAL || epilog == EPI_DGELU_BGRAD) &&
            lane_idx < lane_limit) {
            // While the MMAs of the tile finish, bring this thread's row segments of the
            // 16-bit per-element input (residual, or stored pre-activation) into L2.
            const uint16_t* src = epilog == EPI_BIAS_RESIDUAL
                                      ? R
                                      : static_cast<const uint16_t*>(p.aux_in);
            for (int c = part; c < nchunks; c += kParts)
                if (split_owner(quarter, c, w.split) == w.rank)
                    prefetch_global_l2(src + static_cast<long long>(lane_idx) * ncols + col_base + c * CH);
        }
        if (!wait_bounded(bar0 + 8u * (kBarTmemFull + acc), acc_phase, abort_flag,
                          p.wait_limit_ns)) {
            if (!*abort_flag) record_failure(p.status, abort_flag, kRoleEpilogue);
            break;
        }
        tcgen05_fence_after_sync();
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                static_cast<uint32_t>(acc * BN);
        const bool warp_live = lane_base < lane_limit;
        float lane_sum = 0.0f;  // backward, bias gradient along the lanes: this tile's sum
        // FFN, GEMM 2 split along K: the slice's partial sums go to the workspace and tensor
        // memory is released at once; only the warp of the slice that finished last goes on,
        // with the sums of all slices read back from the workspace.
        bool reduce_done = true;  // this warp runs the epilogue of the tile
        bool from_ws = false;     // ... on values from the workspace, not tensor memory
        bool tmem_released = false;
        if constexpr (FFN_SPLIT) {
            if (second && p.ffn_split2 > 1) {
                ffn_write_slice<BN, EW>(p, t.tile2, t.slice, w.pair_rank, quarter, part, nchunks, t_lane);
                tcgen05_fence_before_sync();
                mbar_arrive_cluster(map_shared_rank(bar0 + 8u * (kBarTmemEmpty + acc),
                                                    cluster_ctarank() & ~1u));
                tmem_released = true;
                reduce_done = ffn_count_slice<EW>(p, t.tile2, w.pair_rank, ew);
                from_ws = reduce_done;
            }
        }

        // CTA-pair kernels, plain forward epilogs: each 32-column chunk in two 16-column
        // halves, the second half's TMEM load in flight while the first is processed (fewer
        // live registers, so the activations of 16 values interleave).
        constexpr bool kHalves = PAIR && CH == 32 &&
                                 (FFN || EPI == EPI_BIAS || EPI == EPI_RELU_BIAS ||
                                  EPI == EPI_GELU_BIAS || EPI == EPI_NONE || EPI == EPI_TANH_BIAS);
        const bool halves = kHalves && (epilog == EPI_BIAS || epilog == EPI_RELU_BIAS ||
                                        epilog == EPI_GELU_BIAS || epilog == EPI_NONE ||
                                        epilog == EPI_TANH_BIAS);
        // Split-K across a cluster through L2: the peers' partial sums of this warp's chunks,
        // copied into its slots in shared memory at the start (below), have landed.
        if (!PAIR && w.split > 1 && p.split_l2) cp_async_wait_all();
        int own_index = -1;  // owned chunks so far (split-K)
        for (int c = part; c < (reduce_done ? nchunks : 0); c += kParts) {
            if (split_owner(quarter, c, w.split) != w.rank) continue;
            ++own_index;
            if constexpr (kHalves) {
                if (halves) {
                    float bcur = 0.0f;  // more warps: this lane's bias value for the chunk
                    if constexpr (EW != 8) {
                        const int oi = (c - part) / kParts;
                        bcur = bl[0];
#pragma unroll
                        for (int i = 1; i < kOwn; ++i) bcur = oi == i ? bl[i] : bcur;
                    }
                    uint8_t* rowp = epi_buf + lane * 64;
                    uint32_t ra[16], rb[16];
                    __syncwarp();
                    tmem_load_16cols_async(t_lane + c * CH, ra);
                    tmem_wait_ld(ra);
                    tmem_load_16cols_async(t_lane + c * CH + 16, rb);
                    if (warp_live && lane == 0) bulk_wait_group_read<0>();  // last box read
                    __syncwarp();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (h == 1) tmem_wait_ld(rb);
                        float v[16];
#pragma unroll
                        for (int j = 0; j < 16; ++j) {
                            v[j] = __uint_as_float(h == 0 ? ra[j] : rb[j]);
                            if (F8) v[j] *= fp8_scale;
                            if constexpr (EW != 8)
                                v[j] += col_bias ? __shfl_sync(0xFFFFFFFFu, bcur, 16 * h + j) : lb;
                        }
                        if constexpr (EW == 8) add_bias<16>(v, sbias + c * CH + 16 * h, col_bias, lb);
                        activate(v, epilog);
                        if (warp_live) {
#pragma unroll
                            for (int qq = 0; qq < 2; ++qq) {
                                const int q = 2 * h + qq;
                                uint4 w4;
                                w4.x = pack2(v[8 * qq + 0], v[8 * qq + 1], p.bf16);
                                w4.y = pack2(v[8 * qq + 2], v[8 * qq + 3], p.bf16);
                                w4.z = pack2(v[8 * qq + 4], v[8 * qq + 5], p.bf16);
                                w4.w = pack2(v[8 * qq + 6], v[8 * qq + 7], p.bf16);
                                *reinterpret_cast<uint4*>(rowp + ((q ^ ((lane >> 1) & 3)) << 4)) = w4;
                            }
                        }
                    }
                    if (warp_live) {
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tma_store_2d(tmD, epi_buf_u32, col_base + c * CH, lane_base);
                            bulk_commit_group();
                        }
                    }
                    continue;
                }
            }
            if constexpr (EW != 8) continue;  // (more warps: plain forward epilogs only)
            // Row-tile residual: this thread's 32 values, requested before the TMEM read so
            // that the load latency overlaps it.
            uint4 rres[4];
            bool rfull = false;
            if constexpr (!SWAP && CH == 32) {
                if (epilog == EPI_BIAS_RESIDUAL) {
                    const int col0 = col_base + c * CH;
                    rfull = lane_idx < p.m && col0 + CH <= ncols;
                    if (rfull) {
                        const uint4* rp = reinterpret_cast<const uint4*>(
                            R + static_cast<long long>(lane_idx) * ncols + col0);
#pragma unroll
                        for (int q = 0; q < 4; ++q) rres[q] = __ldg(rp + q);
                    }
                }
            }
            uint32_t r[32];
            __syncwarp();
            if constexpr (FFN_SPLIT && CH == 32) {
                if (from_ws)
                    ffn_sum_chunk<BN>(p, t.tile2, w.pair_rank, quarter, c, r);
                else
                    tmem_load_32cols(t_lane + c * 32, r);
            } else if constexpr (CH == 32) {
                tmem_load_32cols(t_lane + c * 32, r);
            } else {
                tmem_load_16cols(t_lane + c * 16, r);
            }
            float v[CH];
#pragma unroll
            for (int j = 0; j < CH; ++j) v[j] = __uint_as_float(r[j]);
            if (w.split > 1) {
                // Add the other ranks' partial sums of this chunk (over distributed shared
                // memory, or from this warp's slots, which hold the blocks copied from L2) in
                // batches of 16-byte units: every load of a batch (units x peers) is issued
                // before any is consumed, so one remote round trip serves a whole 16-column
                // chunk (two units per trip for 32-column chunks, whose registers are needed
                // elsewhere).
                const int row = quarter * 32 + lane;
                constexpr int kUB = CH == 16 ? 4 : 2;
#pragma unroll
                for (int u0 = 0; u0 < CH / 4; u0 += kUB) {
                    float4 part[kMaxSplit - 1][kUB];
#pragma unroll
                    for (int pi = 0; pi < kMaxSplit - 1; ++pi) {
                        if (pi < w.split - 1) {
                            const uint32_t peer = static_cast<uint32_t>(pi < w.rank ? pi : pi + 1);
#pragma unroll
                            for (int uu = 0; uu < kUB; ++uu)
                                part[pi][uu] =
                                    p.split_l2
                                        ? *reinterpret_cast<const float4*>(
                                              smem + l2_slots +
                                              (own_index * (w.split - 1) + pi) * (128 * CH) +
                                              ((u0 + uu) * 32 + lane) * 16)
                                        : ld_shared_cluster_v4(map_shared_rank(
                                              sbase + red_offset<BN>(row, c * (CH / 4) + u0 + uu),
                                              peer));
                        }
                    }
#pragma unroll
                    for (int pi = 0; pi < kMaxSplit - 1; ++pi) {
                        if (pi < w.split - 1) {
#pragma unroll
                            for (int uu = 0; uu < kUB; ++uu) {
                                v[4 * (u0 + uu)] += part[pi][uu].x;
                                v[4 * (u0 + uu) + 1] += part[pi][uu].y;
                                v[4 * (u0 + uu) + 2] += part[pi][uu].z;
                                v[4 * (u0 + uu) + 3] += part[pi][uu].w;
                            }
                        }
                    }
                }
            }
            if (F8) {
#pragma unroll
                for (int j = 0; j < CH; ++j) v[j] *= fp8_scale;
            }
            if (!ln) {
                add_bias<CH>(v, sbias + c * CH, col_bias, lb);
            } else {
#pragma unroll
                for (int j = 0; j < CH; ++j) {
                    const float sa = sbias[c * CH + j], sb = sbias[256 + c * CH + j];
                    const float mu = SWAP ? sa : ln_la, rs = SWAP ? sb : ln_lb;
                    const float cc = SWAP ? ln_la : sa, bb = SWAP ? ln_lb : sb;
                    v[j] = fmaf(rs, fmaf(-mu, cc, v[j]), bb);
                }
            }

            if constexpr (!SWAP) {
                // ---- rows of D on lanes: thread = one row, 32 consecutive columns ----
                const int row = lane_idx;
                const int col0 = col_base + c * CH;
                if (epilog == EPI_RELU_AUX_BIAS) {
                    uint32_t word = 0;
#pragma unroll
                    for (int j = 0; j < CH; ++j)
                        word |= (v[j] > 0.0f && col0 + j < p.n) ? (1u << j) : 0u;
                    if (row < p.m)
                        static_cast<uint32_t*>(p.aux)[static_cast<long long>(row) * p.aux_ld + col0 / 32] = word;
                } else if (epilog == EPI_GELU_AUX_BIAS) {
                    store_pre_row(p, v, row, col0);
                } else if (bwd) {
                    backward_factor_row(p, epilog, v, row, col0);
                }
                activate(v, epilog);
                if (epilog == EPI_BIAS_RESIDUAL && row < p.m) {
                    const uint16_t* rrow = R + static_cast<long long>(row) * ncols + col0;
                    if (rfull) {
#pragma unroll
                        for (int j8 = 0; j8 < CH / 8; ++j8) {
                            const uint4 w = rres[j8];
                            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                const uint32_t lo = ww[h] & 0xFFFFu, hi = ww[h] >> 16;
                                if (p.bf16) {
                                    v[j8 * 8 + 2 * h] += __uint_as_float(lo << 16);
                                    v[j8 * 8 + 2 * h + 1] += __uint_as_float(hi << 16);
                                } else {
                                    v[j8 * 8 + 2 * h] +=
                                        __half2float(__ushort_as_half(static_cast<uint16_t>(lo)));
                                    v[j8 * 8 + 2 * h + 1] +=
                                        __half2float(__ushort_as_half(static_cast<uint16_t>(hi)));
                                }
                            }
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < CH; ++j)
                            if (col0 + j < ncols) v[j] += load_16bit(rrow, j, p.bf16);
                    }
                }
                if (warp_live) {
                    // 32 rows x 32 columns of 16-bit = one 2 KB box, 64-byte rows, stored
                    // with the 64-byte swizzle (16-byte chunk q of row r at q ^ ((r>>1)&3)).
                    if (lane == 0) bulk_wait_group_read<0>();  // this warp's last box is read
                    __syncwarp();
                    uint8_t* rowp = epi_buf + lane * 64;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint4 w;
                        w.x = pack2(v[8 * q + 0], v[8 * q + 1], p.bf16);
                        w.y = pack2(v[8 * q + 2], v[8 * q + 3], p.bf16);
                        w.z = pack2(v[8 * q + 4], v[8 * q + 5], p.bf16);
                        w.w = pack2(v[8 * q + 6], v[8 * q + 7], p.bf16);
                        *reinterpret_cast<uint4*>(rowp + ((q ^ ((lane >> 1) & 3)) << 4)) = w;
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(tmD, epi_buf_u32, col0, lane_base);
                        bulk_commit_group();
                    }
                }
            } else {
                // ---- columns of D on lanes: thread = one column, CH consecutive rows ----
                const int col = lane_idx;
                const bool col_ok = col < p.n;
                const int t0 = col_base + c * CH;
                const int word_idx = lane_base / 32;
                if (epilog == EPI_RELU_AUX_BIAS) {
#pragma unroll
                    for (int j = 0; j < CH; ++j) {
                        const uint32_t word = __ballot_sync(0xFFFFFFFFu, col_ok && v[j] > 0.0f);
                        if (lane == 0 && t0 + j < p.m && word_idx < p.aux_ld)
                            static_cast<uint32_t*>(p.aux)[static_cast<long long>(t0 + j) * p.aux_ld + word_idx] = word;
                    }
                } else if (epilog == EPI_GELU_AUX_BIAS) {
                    uint16_t* pre16 = static_cast<uint16_t*>(p.aux);
#pragma unroll
                    for (int j = 0; j < CH; ++j)
                        if (col_ok && t0 + j < p.m)
                            pre16[static_cast<long long>(t0 + j) * p.n + col] = to16(v[j], p.bf16);
                } else if (epilog == EPI_DRELU_BGRAD) {
                    // lane j < CH fetches the mask word of row t0 + j; bit `lane` of it
                    uint32_t mrow = 0;
                    if (lane < CH && t0 + lane < p.m && word_idx < p.aux_ld)
                        mrow = __ldg(static_cast<const uint32_t*>(p.aux_in) +
                                     static_cast<long long>(t0 + lane) * p.aux_ld + word_idx);
#pragma unroll
                    for (int j = 0; j < CH; ++j) {
                        const uint32_t mw = __shfl_sync(0xFFFFFFFFu, mrow, j);
                        v[j] = (col_ok && ((mw >> lane) & 1u)) ? v[j] : 0.0f;
                    }
                } else if (epilog == EPI_DGELU_BGRAD) {
#pragma unroll
                    for (int j = 0; j < CH; ++j) {
                        float g = 0.0f;
                        if (col_ok && t0 + j < p.m)
                            g = gelu_grad_fast(load_16bit(p.aux_in, static_cast<long long>(t0 + j) * p.n + col,
                                                          p.bf16));
                        v[j] *= g;
                    }
                }
                activate(v, epilog);
                if (epilog == EPI_BIAS_RESIDUAL) {
#pragma unroll
                    for (int j = 0; j < CH; ++j)
                        if (col_ok && t0 + j < p.m)
                            v[j] += load_16bit(R, static_cast<long long>(t0 + j) * p.n + col, p.bf16);
                }
                if (warp_live) {
                    // Transpose through shared memory: row j of the box holds D[t0 + j][32
                    // columns of this warp] (64 bytes; lane = column, so each row is written
                    // by one conflict-free warp store), then one TMA store of the box.
                    if (lane == 0) bulk_wait_group_read<0>();  // this warp's last box is read
                    __syncwarp();
                    uint16_t* tb = reinterpret_cast<uint16_t*>(epi_buf);
                    if (m64) {
                        // a 16-column box (rows of 32 bytes) from lanes 0-15
                        if (lane < 16) {
#pragma unroll
                            for (int j = 0; j < CH; ++j) tb[j * 16 + lane] = to16(v[j], p.bf16);
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < CH; ++j) tb[j * 32 + lane] = to16(v[j], p.bf16);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&p.tm_D, epi_buf_u32, lane_base, t0);
                        bulk_commit_group();
                    }
                }
            }
            if (bwd && warp_live) {
                // bias gradient of this chunk (entries outside the matrix are 0 here)
                if (along_cols) {
                    float x[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) x[j] = j < CH ? v[j] : 0.0f;
                    const float colsum = warp_column_sums(x, lane);
                    const int ci = col_base + c * CH + lane;
                    if (lane < CH && ci < col_limit) atomicAdd(p.dbias + ci, colsum);
                } else {
#pragma unroll
                    for (int j = 0; j < CH; ++j) lane_sum += v[j];
                }
            }
        }
        if (bwd && !along_cols && lane_idx < lane_limit) {
            bool any_chunk = false;  // this warp owned a chunk of the tile
            for (int c = part; c < nchunks; c += kParts)
                any_chunk = any_chunk || split_owner(quarter, c, w.split) == w.rank;
            if (any_chunk) atomicAdd(p.dbias + lane_idx, lane_sum);
        }
        if (!tmem_released) {
            tcgen05_fence_before_sync();
            if constexpr (PAIR)  // the even CTA's MMAs write both CTAs' accumulators
                mbar_arrive_cluster(map_shared_rank(bar0 + 8u * (kBarTmemEmpty + acc),
                                                    cluster_ctarank() & ~1u));
            else
                mbar_arrive(bar0 + 8u * (kBarTmemEmpty + acc));
        }
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
        if (FFN && t.prob == 0) {
            // This warp's stores of the tile's H are complete (not just read from shared
            // memory): count the warp for the row block, with release semantics.
            if (lane == 0) {
                bulk_wait_group<0>();
                fence_proxy_async_global();
                red_release_gpu_add(p.ffn_ready + ffn_ready_index(p, tm, ffn_slice_of_tile1(p, tn)), 1);
            }
            __syncwarp();
        }
    }
    // Shared memory may be released once the stores have read it, and once this lane's
    // copies of peers' partial sums (split-K through L2) have landed, also when the tile
    // loop was left early; the grid's writes are complete when the grid is.
    if constexpr (!PAIR) cp_async_wait_all();
    if (lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
}

// ------------------------------------------------------------------------------------------
// the kernel
// ------------------------------------------------------------------------------------------
template <int BN, bool SWAP, bool PAIR = false, int EPI = -1, bool F8 = false, int EW = 8>
__global__ void __launch_bounds__(64 + 32 * EW, 1) gemm_epi_kernel(const __grid_constant__ GemmParams p)
{
    using C = TileCfg<BN, PAIR, EW>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + C::kOffBar;
    uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + C::kOffBar + kOffHolder);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffBar + kOffAbort);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    int pre = 0;  // stages the prologue issued (thread 0, which is also the producer)

    constexpr bool FFN = is_ffn(EPI);
    if (threadIdx.x == 0) {
        prefetch_tensormap(&p.tm_A);
        prefetch_tensormap(&p.tm_B);
        prefetch_tensormap(&p.tm_D);
        if (FFN) {
            prefetch_tensormap(&p.tm_A2);
            prefetch_tensormap(&p.tm_B2);
            prefetch_tensormap(&p.tm_D2);
        }
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar0 + 8u * (kBarFull + s), 1);
            mbar_init(bar0 + 8u * (kBarEmpty + s), 1);
        }
        if (PAIR) {
            for (int s = 0; s < kSchedSlots; ++s) {
                mbar_init(bar0 + 8u * (kBarSchedFull + s), 1);
                mbar_init(bar0 + 8u * (kBarSchedEmpty + s), sched_consumers<EW>());
            }
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar0 + 8u * (kBarTmemFull + a), 1);
            mbar_init(bar0 + 8u * (kBarTmemEmpty + a), (PAIR ? 2 : 1) * 32 * EW);
        }
        mbar_init(bar0 + 8u * kBarStall, 1);
        mbar_init(bar0 + 8u * kBarDrain, 1);
        *abort_flag = 0;
        fence_mbar_init();
        // (a pair's first loads wait for both CTAs' barriers, after the cluster barrier)
        if (!PAIR) pre = producer_prologue<BN, SWAP>(p, sbase, bar0);
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(smem_u32(tmem_holder), C::kTmemCols);
            tmem_relinquish_alloc_permit_pair();
        } else {
            tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);
            tmem_relinquish_alloc_permit();
        }
    }
    tcgen05_fence_before_sync();
    __syncthreads();
    // A pair's CTAs signal each other's barriers: both must be initialised first.
    if constexpr (PAIR) cluster_sync_all();
    tcgen05_fence_after_sync();
    const uint32_t tmem_base = *tmem_holder;
    if (threadIdx.x == 0) grid_launch_dependents();

    if (p.debug_stall) {
        // Test of the timeout path: wait on a barrier that nothing arrives at.
        if (threadIdx.x == 0 &&
            !wait_bounded(bar0 + 8u * kBarStall, 0, abort_flag, p.wait_limit_ns, false))
            record_failure(p.status, abort_flag, kRoleStallTest);
        __syncthreads();
    }

    const bool split = !PAIR && p.split > 1 && !p.split_global;  // (pairs never split)
    const bool gsplit = !PAIR && p.split > 1 && p.split_global;
    if constexpr (PAIR) {
        if (!*abort_flag) {
            if (warp == 0) {
                if (lane == 0) run_producer<BN, SWAP, PAIR, FFN, F8>(p, sbase, bar0, abort_flag, pre);
                __syncwarp();
            } else if (warp == 1) {
                if (lane == 0) run_mma<BN, SWAP, PAIR, FFN, F8>(p, sbase, bar0, tmem_base, abort_flag);
                __syncwarp();
            } else if (split) {
                publish_partials<BN, SWAP>(p, smem, bar0, tmem_base, abort_flag);
            } else {
                run_epilogue<BN, SWAP, PAIR, EPI, F8, EW>(p, smem, sbase, bar0, tmem_base, abort_flag);
            }
        }
    } else {
        bool epilogue = false;  // this thread runs the epilogue below
        if (!*abort_flag) {
            if (warp == 0) {
                if (lane == 0) run_producer<BN, SWAP, PAIR, FFN, F8>(p, sbase, bar0, abort_flag, pre);
                __syncwarp();
            } else if (warp == 1) {
                if (lane == 0) run_mma<BN, SWAP, PAIR, FFN, F8>(p, sbase, bar0, tmem_base, abort_flag);
                __syncwarp();
            } else if (split) {
                publish_partials<BN, SWAP>(p, smem, bar0, tmem_base, abort_flag);
            } else {
                epilogue = !gsplit;
            }
        }
        // Split-K through device memory: every epilogue thread, aborted or not, takes part
        // in the count; the last CTA of the tile runs the epilogue.
        if (gsplit && warp >= 2)
            epilogue = publish_partials_global<BN, SWAP>(p, smem, bar0, tmem_base, abort_flag) &&
                       !*abort_flag;
        if (epilogue) run_epilogue<BN, SWAP, PAIR, EPI, F8>(p, smem, sbase, bar0, tmem_base, abort_flag);
    }
    if (split) {
        // Every thread of every CTA of the cluster reaches both barriers: each role above
        // ends in bounded time, on success or on abort.
        __syncwarp();
        cluster_sync_all();  // partial sums written
        if (warp >= 2 && !*abort_flag)
            run_epilogue<BN, SWAP, PAIR, EPI, F8>(p, smem, sbase, bar0, tmem_base, abort_flag);
        __syncwarp();
        // the peers are done reading this CTA's partial sums (in its shared memory; those in
        // the workspace are next written by a later grid, after this one has completed)
        if (!p.split_l2) cluster_sync_all();
    }

    tcgen05_fence_before_sync();
    __syncthreads();
    // In a pair, neither CTA leaves while the other may still signal its barriers or the
    // even CTA's MMAs may still write its tensor memory.
    if constexpr (PAIR) cluster_sync_all();
    if (warp == 1) {
        tcgen05_fence_after_sync();
        if constexpr (PAIR)
            tmem_dealloc_pair(tmem_base, C::kTmemCols);
        else
            tmem_dealloc(tmem_base, C::kTmemCols);
    }
    // The pair's producer is done with the tile counter.
    if (PAIR && p.sched != nullptr && threadIdx.x == 0 && (cluster_ctarank() & 1u) == 0)
        sched_finish(p);
}

}  // namespace gemm_epi
