// Small-m kernel: D[m][n] = epi(A[m][k] . B[k][n] + bias) for m <= 64, the small-batch,
// latency-sensitive inference case that "Fusing bias into cuBLASLt matmul with nvmath-python
// for PyTorch inference" (blog.hotdry.top, 2025-09-22) names in its closing paragraphs, and
// the launch-bound chain of "Operator fusion in model inference" (wmrh.cn/news/429806),
// section 1 flowchart.
//
// The work is all data movement: B (the weight, k x n) is read once and is most of the bytes.
// So the kernel spreads B over as many SMs as it can and asks for every byte at once:
//   * computed as D^T = B^T A^T: an MMA tile is 128 columns of D (M = 128, rows of the
//     N-major B operand) by BN rows of D (N = BN, the K-major rows of A);
//   * K is split S ways over a thread-block cluster of S CTAs, one K slice of one 128-column
//     tile per CTA, so tiles_n * S CTAs each hold a (128 x K/S) slab of B;
//   * one thread issues every copy of its slice at entry (B as 64-column N-major panels as
//     deep as the slice, A as 64-deep K-major boxes), counted on a single mbarrier: no stage
//     ring, no per-block round trips; then it issues all the slice's MMAs and one commit;
//   * the partial sums meet by a reduce-scatter: rank r of the cluster owns rows
//     [r R, (r + 1) R) of the tile (R = BN / S); every rank sends each peer the rows that
//     peer owns with st.async into the peer's shared memory (16 bytes per thread and store),
//     counted in bytes on one mbarrier of the receiver, so every SM takes in the same small
//     share; each rank adds its rows' partials in rank order (the sum does not depend on
//     arrival order), adds the bias, applies the activation and writes its R rows of D (and
//     the mask or the stored pre-activation) with plain coalesced stores, two threads per
//     column of D taking alternate groups of four rows (with one per column, one warp per
//     scheduler, the loop was bound by the latency of its dependent steps).  One kernel per epilog; the exchange and the epilogue are rolled loops
//     over a shared-memory copy of the accumulator (the kernel runs for a few microseconds,
//     and there an instruction-cache miss costs as much as a row's arithmetic).
// The copies, the MMAs and the partial sums are waited for with a time limit; on expiry the
// thread records the failure in the status word and the kernel winds down (MMAs drained,
// tensor memory freed).  A cluster barrier at start-up (waited at only
// before the first remote store) makes sure every CTA of the cluster runs, with its barriers
// initialised, before a peer writes to it; a second one, arrived at once a CTA has received
// its share and waited at just before it leaves, keeps every CTA until all shares landed.
#include "gemm_kernel.cuh"

namespace gemm_epi {

namespace {

constexpr int kSmTN = 128;            // columns of D per tile (MMA M)
// Threads per CTA: one per column of D (TMEM lane) for 16-row tiles, two for wider ones,
// where the first 128 read the accumulator and both halves take part in the exchange and the
// epilogue, taking alternate groups of four rows.  Measured on GB300 (GELU X[T,768].W[768,3072],
// CUDA graph, hot / L2 flushed): T = 32 4.15 -> 4.03 / 5.8 -> 5.7-5.8 us, T = 64 5.35 -> 5.14 /
// 7.0 -> 6.8-6.9 us; at T = 16 (one row group per rank) the extra warps only cost: 3.61 ->
// 3.78 / 5.0 -> 5.4 us.
__host__ __device__ constexpr int sm_threads(int bn) { return bn >= 32 ? 256 : 128; }
constexpr int kSmMaxSplit = 8;        // K slices per cluster at most

// Shared-memory layout of one CTA (offsets from a 1024-byte aligned base):
//   [B panels: 2 x kc rows x 128 B][A boxes: kc/64 x BN rows x 128 B]
//   [this rank's accumulator: BN/4 x 128 lanes x 16 B]
//   [received partials: (S-1) senders x R/4 x 128 lanes x 16 B, R = BN / S][barriers, holder]
struct SmLayout {
    int kc, bn, split;
    __host__ __device__ int rows() const { return bn / split; }
    __host__ __device__ int b_bytes() const { return 2 * kc * 128; }
    __host__ __device__ int a_bytes() const { return (kc / 64) * bn * 128; }
    __host__ __device__ int mine_off() const { return b_bytes() + a_bytes(); }
    __host__ __device__ int part_off() const { return mine_off() + bn * kSmTN * 4; }
    __host__ __device__ int part_bytes() const { return (split - 1) * rows() * kSmTN * 4; }
    __host__ __device__ int bar_off() const { return part_off() + part_bytes(); }
    __host__ __device__ int rowb_off() const { return bar_off() + 64; }   // <= 64 fp32
    __host__ __device__ int total() const { return 1024 + rowb_off() + 256; }
};

// barrier slots (8 bytes each) after bar_off
constexpr int kSmBarFull = 0;     // copies of the slice landed (1 arrival + bytes)
constexpr int kSmBarMma = 1;      // MMAs of the slice done (tcgen05.commit)
constexpr int kSmBarPart = 2;     // the peers' partial sums of this rank's rows landed (bytes)
constexpr int kSmOffHolder = 32;  // TMEM base address

// Bounded wait on a local barrier whose arrivals may come from other CTAs of the cluster.
__device__ __forceinline__ bool sm_wait(uint32_t bar, uint32_t parity, unsigned long long limit_ns)
{
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    const unsigned long long max_polls = limit_ns / 8 + 1024;
    for (unsigned long long poll = 1; poll < max_polls; ++poll) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((poll & 63) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
    }
    return false;
}

__device__ __forceinline__ void sm_fail(int* status)
{
    atomicCAS(status, 0, kCodeTimeout | kRoleEpilogue);
}

// Asynchronous store of 16 bytes into another CTA's shared memory (`addr` from mapa), its
// completion counted in bytes on the mbarrier `bar` of that CTA.
__device__ __forceinline__ void st_async_v4(uint32_t addr, float a, float b, float c, float d,
                                            uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];"
                 ::"r"(addr), "f"(a), "f"(b), "f"(c), "f"(d), "r"(bar)
                 : "memory");
}

// Arrive without release semantics: used where the arrival only says "this thread got here"
// (the barriers' initialisation is published by fence.mbarrier_init in the thread that
// initialised them, and what was received is established by a byte-counting mbarrier).
__device__ __forceinline__ void cluster_arrive_plain()
{
    asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// This thread's BN accumulator values (its TMEM lane, columns 0..BN-1), 16 at a time.
template <int BN>
__device__ __forceinline__ void load_acc(uint32_t taddr, float (&v)[BN])
{
#pragma unroll
    for (int c = 0; c < BN; c += 16) {
        uint32_t r[16];
        tmem_load_16cols_async(taddr + static_cast<uint32_t>(c), r);
        tmem_wait_ld(r);
#pragma unroll
        for (int j = 0; j < 16; ++j) v[c + j] = __uint_as_float(r[j]);
    }
}

template <int BN, int EPI>
__global__ void __launch_bounds__(sm_threads(BN), 1) smallm_kernel(const __grid_constant__ GemmParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const int S = p.split;
    const int kc = p.kb_per_split * 64;
    const SmLayout L{kc, BN, S};
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + static_cast<uint32_t>(L.bar_off());
    uint32_t* holder = reinterpret_cast<uint32_t*>(smem + L.bar_off() + kSmOffHolder);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = static_cast<int>(cluster_ctarank());
    const int tile = static_cast<int>(blockIdx.x) / S;     // (column tile, row tile)
    const int tn = tile % p.tiles_m;                       // 128-column tile of D
    const int tmr = tile / p.tiles_m;                      // BN-row tile of D
    const int n0 = tn * kSmTN;
    const int t0 = tmr * BN;
    const int k0 = rank * kc;
    const uint32_t b_smem = sbase;
    const uint32_t a_smem = sbase + static_cast<uint32_t>(L.b_bytes());
    // The parameters the exchange and the epilogue use, read into registers at entry: a
    // first read of a kernel parameter can miss in the constant cache, and here that
    // latency overlaps the copies instead of sitting in the epilogue.
    int pn = p.n, pm = p.m, pbf16 = p.bf16, playout = p.bias_layout, paux_ld = p.aux_ld;
    const void* pbias = p.bias;
    const void* pres = p.residual;
    void* pD = p.D;
    void* paux = p.aux;
    asm volatile("" : "+r"(pn), "+r"(pm), "+r"(pbf16), "+r"(playout), "+r"(paux_ld), "+l"(pbias),
                 "+l"(pres), "+l"(pD), "+l"(paux));

    if (threadIdx.x == 0) {
        mbar_init(bar0 + 8u * kSmBarFull, 1);
        mbar_init(bar0 + 8u * kSmBarMma, 1);
        mbar_init(bar0 + 8u * kSmBarPart, 1);
        fence_mbar_init();
        // The copies first: everything else of the set-up overlaps their flight.
        // (debug_stall: no copy is issued, so the wait below runs out its time limit)
        if (!p.debug_stall) {
            // Under a programmatic dependent launch the operands may come from the previous
            // grid: B too, unless the plan was told that grid does not write it (b_ready).
            if (!p.b_ready) grid_dependency_wait();
            const uint32_t full = bar0 + 8u * kSmBarFull;
            mbar_arrive_expect_tx(full, static_cast<uint32_t>(L.b_bytes() + L.a_bytes()));
            // B: two 64-column panels of kc rows (k), in boxes of box_k rows (box_k divides kc)
            const int boxk = p.box_k;
            for (int pnl = 0; pnl < 2; ++pnl)
                for (int kk = 0; kk < kc; kk += boxk)
                    tma_load_2d(b_smem + static_cast<uint32_t>(pnl * kc * 128 + kk * 128), &p.tm_B,
                                full, n0 + pnl * 64, k0 + kk);
            if (p.b_ready) grid_dependency_wait();
            // A: kc / 64 boxes of BN rows x 64 k
            for (int b = 0; b < kc / 64; ++b)
                tma_load_2d(a_smem + static_cast<uint32_t>(b * BN * 128), &p.tm_A, full, k0 + b * 64, t0);
        }
        // every peer's partial sums of this rank's rows, on one barrier
        if (S > 1) mbar_arrive_expect_tx(bar0 + 8u * kSmBarPart, static_cast<uint32_t>(L.part_bytes()));
    }
    // Without b_ready under a programmatic dependent launch: this CTA's slab of B (kc rows
    // of 128 columns, up to three 128-byte lines a row) brought into L2 while the previous
    // grid may still run; the copies above then find it there once the wait returns.
    if (p.b_l2 != nullptr && threadIdx.x >= 32) {
        const char* b = static_cast<const char*>(p.b_l2);
        for (int i = static_cast<int>(threadIdx.x) - 32; i < 3 * kc;
             i += static_cast<int>(blockDim.x) - 32) {
            const int r = k0 + i / 3;
            const int c = min(n0 + (i % 3) * 64 - (i % 3 == 2 ? 1 : 0), pn - 1);
            if (r < p.k) prefetch_global_l2(b + (static_cast<long long>(r) * p.b_ld + c) * 2);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(holder), BN < 32 ? 32 : BN);
        tmem_relinquish_alloc_permit();
    }
    // Cluster barrier: every CTA of the cluster has started, its barriers initialised (its
    // shared memory may be written); waited at only just before the first remote store.
    if (S > 1) cluster_arrive_plain();
    tcgen05_fence_before_sync();
    __syncthreads();
    tcgen05_fence_after_sync();
    const uint32_t tmem = *holder;
    if (threadIdx.x == 0) grid_launch_dependents();

    // ---- MMAs of the slice (thread 0) ----------------------------------------------------
    bool ok = true;
    if (threadIdx.x == 0) {
        bool issued = false;
        if (sm_wait(bar0 + 8u * kSmBarFull, 0, p.wait_limit_ns)) {
            tcgen05_fence_after_sync();
            const uint32_t idesc = make_idesc_f16(static_cast<uint32_t>(p.bf16), 1u, 0u, kSmTN, BN);
            for (int kk = 0; kk < kc / kUmmaK; ++kk) {
                // B^T: N-major panels (LBO = one panel, SBO = 8 k rows), +16 rows per K step
                const uint64_t ad = make_sdesc_sw128(b_smem + static_cast<uint32_t>(kk * 2048),
                                                     static_cast<uint32_t>(kc * 128), 1024);
                // A: K-major boxes of 64 k, +32 bytes per K step inside a box
                const uint64_t bd = make_sdesc_sw128(
                    a_smem + static_cast<uint32_t>((kk >> 2) * BN * 128 + (kk & 3) * 32), 0, 1024);
                mma_f16_ss(tmem, ad, bd, idesc, kk > 0 ? 1u : 0u);
            }
            issued = true;
        } else {
            sm_fail(p.status);
        }
        // (also on failure, so that no MMA is in flight when tensor memory is freed)
        mma_commit(bar0 + 8u * kSmBarMma);
        (void)issued;
    }
    __syncwarp();

    // ---- the first 128 threads: their column's BN accumulator values -----------------------
    const int cidx = static_cast<int>(threadIdx.x) & (kSmTN - 1);  // column of the tile
    const int half = static_cast<int>(threadIdx.x) / kSmTN;        // first row group
    constexpr int kHalves = sm_threads(BN) / kSmTN;                // row-group stride
    float v[BN];
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    if (!sm_wait(bar0 + 8u * kSmBarMma, 0, p.wait_limit_ns)) {
        ok = false;
        sm_fail(p.status);
    }
    tcgen05_fence_after_sync();
    if (ok && half == 0) {
        load_acc<BN>(t_lane, v);
    } else {
#pragma unroll
        for (int j = 0; j < BN; ++j) v[j] = 0.0f;
    }
    // The accumulator is in registers: free tensor memory now (it overlaps the exchange).
    tcgen05_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tcgen05_fence_after_sync();
        tmem_dealloc(tmem, BN < 32 ? 32 : BN);
    }
    const int col = n0 + cidx;              // this thread's column of D
    const bool col_ok = col < pn;

    // Bias, residual and the outputs may belong to a programmatic predecessor grid.
    grid_dependency_wait();
    const int R = BN / S;            // rows of D this rank owns: [lo, lo + R) of the tile
    const int lo = rank * R;
    // the bias along the columns (one value per thread), requested before the exchange; the
    // row-wise inputs of this rank's rows (residual, bias along the rows) brought into L2
    const bool col_bias = playout == 1 && EPI != EPI_NONE;
    const bool row_bias = playout == 0 && EPI != EPI_NONE;
    const float cb = col_bias && col_ok ? load_16bit(pbias, col, pbf16) : 0.0f;
    if (EPI == EPI_BIAS_RESIDUAL && col_ok)
        for (int i = 0; i < R && t0 + lo + i < pm; ++i)
            prefetch_global_l2(static_cast<const uint16_t*>(pres) +
                               static_cast<long long>(t0 + lo + i) * pn + col);
    // The residual of this thread's first group of four rows, loaded now so that its latency
    // overlaps the exchange (a thread's further groups, where it has several, load in the
    // epilogue loop); kept as 16-bit words until used.
    uint16_t rr0[4] = {0, 0, 0, 0};
    if constexpr (EPI == EPI_BIAS_RESIDUAL) {
        if (half < R / 4 && col_ok) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int row = t0 + lo + 4 * half + e;
                if (row < pm) rr0[e] = static_cast<const uint16_t*>(pres)[static_cast<long long>(row) * pn + col];
            }
        }
    }
    // Bias along the rows ((m,1) layout): this rank's R values into shared memory now, so
    // that the epilogue loop reads no global memory.
    float* rowb = reinterpret_cast<float*>(smem + L.rowb_off());
    if (row_bias && static_cast<int>(threadIdx.x) < R)
        rowb[threadIdx.x] = t0 + lo + static_cast<int>(threadIdx.x) < pm
                                ? load_16bit(pbias, t0 + lo + static_cast<int>(threadIdx.x), pbf16)
                                : 0.0f;
    // This thread's accumulator column into shared memory, [BN/4][lanes] float4: the
    // exchange and the epilogue below are rolled loops that read it back (unrolled over BN
    // rows with run-time tests of which rows a rank owns, each row ran code fetched for the
    // first time, one instruction-cache miss per row).
    const uint32_t mine = sbase + static_cast<uint32_t>(L.mine_off()) + static_cast<uint32_t>(cidx * 16);
    const uint32_t part = sbase + static_cast<uint32_t>(L.part_off()) + static_cast<uint32_t>(cidx * 16);
    // (the same, for plain loads that the compiler may schedule around the stores to D)
    const float4* mine_p = reinterpret_cast<const float4*>(smem + L.mine_off()) + cidx;
    const float4* part_p = reinterpret_cast<const float4*>(smem + L.part_off()) + cidx;
    if (half == 0) {
#pragma unroll
        for (int j4 = 0; j4 < BN / 4; ++j4)
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(mine + static_cast<uint32_t>(j4 * kSmTN * 16)),
                         "f"(v[4 * j4]), "f"(v[4 * j4 + 1]), "f"(v[4 * j4 + 2]), "f"(v[4 * j4 + 3])
                         : "memory");
    }
    __syncthreads();  // (the second half reads the columns the first half stored)
    if (S > 1) {
        // ---- reduce-scatter: each peer's rows to it, then this rank's rows from them ------
        cluster_wait();
        for (int q = 0; q < S; ++q) {
            if (q == rank) continue;
            const int slot = rank < q ? rank : rank - 1;
            const uint32_t qbar = map_shared_rank(bar0 + 8u * kSmBarPart, static_cast<uint32_t>(q));
            for (int g = half; g < R / 4; g += kHalves) {
                const float4 a = mine_p[(q * (R / 4) + g) * kSmTN];
                const uint32_t dst = part + static_cast<uint32_t>((slot * (R / 4) + g) * kSmTN * 16);
                st_async_v4(map_shared_rank(dst, static_cast<uint32_t>(q)), a.x, a.y, a.z, a.w, qbar);
            }
        }
        if (!sm_wait(bar0 + 8u * kSmBarPart, 0, p.wait_limit_ns)) {
            ok = false;
            sm_fail(p.status);
        }
    }
    __syncthreads();  // (rowb)
    if (ok) {
        // ---- this rank's rows: own partial + the senders' in rank order, then the epilogue ----
        uint16_t* D = static_cast<uint16_t*>(pD);
        for (int g = half; g < R / 4; g += kHalves) {
            float4 a = mine_p[(lo / 4 + g) * kSmTN];
            // the senders' partial sums in rank order (all loads issued before the adds)
            float4 w[kSmMaxSplit - 1];
#pragma unroll
            for (int sl = 0; sl < kSmMaxSplit - 1; ++sl)
                if (sl < S - 1) w[sl] = part_p[(sl * (R / 4) + g) * kSmTN];
#pragma unroll
            for (int sl = 0; sl < kSmMaxSplit - 1; ++sl) {
                if (sl < S - 1) {
                    a.x += w[sl].x;
                    a.y += w[sl].y;
                    a.z += w[sl].z;
                    a.w += w[sl].w;
                }
            }
            const float xs[4] = {a.x, a.y, a.z, a.w};
            float rb[4] = {0.0f, 0.0f, 0.0f, 0.0f}, rr[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (row_bias) {
#pragma unroll
                for (int e = 0; e < 4; ++e) rb[e] = rowb[4 * g + e];
            }
            if constexpr (EPI == EPI_BIAS_RESIDUAL) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int row = t0 + lo + 4 * g + e;
                    if (row < pm && col_ok)
                        rr[e] = g == half ? decode16(rr0[e], pbf16)
                                          : load_16bit(pres, static_cast<long long>(row) * pn + col, pbf16);
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int row = t0 + lo + 4 * g + e;
                float x = xs[e] + cb + rb[e];
                if constexpr (EPI == EPI_RELU_AUX_BIAS) {
                    const uint32_t word = __ballot_sync(0xFFFFFFFFu, col_ok && x > 0.0f);
                    const int widx = (n0 + (warp & 3) * 32) / 32;
                    if (lane == 0 && row < pm && widx < paux_ld)
                        static_cast<uint32_t*>(paux)[static_cast<long long>(row) * paux_ld + widx] = word;
                } else if constexpr (EPI == EPI_GELU_AUX_BIAS) {
                    if (col_ok && row < pm)
                        static_cast<uint16_t*>(paux)[static_cast<long long>(row) * pn + col] = to16(x, pbf16);
                }
                if constexpr (EPI == EPI_RELU_BIAS || EPI == EPI_RELU_AUX_BIAS) {
                    x = x > 0.0f ? x : 0.0f;
                } else if constexpr (EPI == EPI_GELU_BIAS || EPI == EPI_GELU_AUX_BIAS) {
                    x = gelu_erf_fast(x);
                } else if constexpr (EPI == EPI_TANH_BIAS) {
                    x = tanh_fast(x);
                } else if constexpr (EPI == EPI_BIAS_RESIDUAL) {
                    x += rr[e];
                }
                if (col_ok && row < pm) D[static_cast<long long>(row) * pn + col] = to16(x, pbf16);
            }
        }
    }
    // Second cluster barrier: this rank has every byte addressed to it (its mbarrier said so
    // above); a CTA leaves only once every receiver of its stores has them, so nobody writes
    // to a CTA that has left.  (Arrived at after the epilogue: an arrival waits for this
    // thread's own outgoing stores to complete.)
    if (S > 1) {
        cluster_arrive_plain();
        cluster_wait();
    }
}

#define GEMM_EPI_SMALLM_EPILOGS(F, BN)                                                        \
    F(BN, EPI_BIAS) F(BN, EPI_RELU_BIAS) F(BN, EPI_GELU_BIAS) F(BN, EPI_RELU_AUX_BIAS)        \
        F(BN, EPI_BIAS_RESIDUAL) F(BN, EPI_NONE) F(BN, EPI_TANH_BIAS) F(BN, EPI_GELU_AUX_BIAS)

// The kernel for (bn, epilog), or nullptr.
const void* smallm_fn(int bn, int epilog)
{
#define F(B, E) \
    if (bn == B && epilog == E) return reinterpret_cast<const void*>(smallm_kernel<B, E>);
    GEMM_EPI_SMALLM_EPILOGS(F, 16)
    GEMM_EPI_SMALLM_EPILOGS(F, 32)
    GEMM_EPI_SMALLM_EPILOGS(F, 64)
#undef F
    return nullptr;
}

cudaError_t smallm_launch_fn(const void* fn, const GemmParams& p, int grid, int smem, int threads,
                             cudaStream_t stream, bool pdl)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = static_cast<unsigned>(p.split);
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
    void* args[] = {const_cast<GemmParams*>(&p)};
    return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

// Shared memory a CTA needs for rows-of-D tile bn, K slices of kc (a multiple of 64) and
// `split` slices; 0 if bn is not a built width or the split does not give every rank a
// multiple of 4 rows of D (split divides bn / 4).
int smallm_smem_bytes(int bn, int kc, int split)
{
    if (bn != 16 && bn != 32 && bn != 64) return 0;
    if (split < 1 || split > 8 || bn % split != 0 || (bn / split) % 4 != 0) return 0;
    return SmLayout{kc, bn, split}.total();
}

// Allow every instantiation the full shared memory (on the current device).
cudaError_t smallm_prepare()
{
    const int bns[] = {16, 32, 64};
    const int epis[] = {EPI_BIAS, EPI_RELU_BIAS, EPI_GELU_BIAS, EPI_RELU_AUX_BIAS,
                        EPI_BIAS_RESIDUAL, EPI_NONE, EPI_TANH_BIAS, EPI_GELU_AUX_BIAS};
    for (int bn : bns)
        for (int e : epis) {
            const cudaError_t r = cudaFuncSetAttribute(
                smallm_fn(bn, e), cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
            if (r != cudaSuccess) return r;
        }
    return cudaSuccess;
}

// Clusters of `split` CTAs of the bn kernel with `smem` bytes each that the GPU holds at once.
int smallm_max_clusters(int bn, int split, int smem)
{
    const void* f = smallm_fn(bn, EPI_BIAS);
    if (!f) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(split), 1, 1);
    cfg.blockDim = dim3(static_cast<unsigned>(sm_threads(bn)), 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(split);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, f, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t smallm_launch(int bn, const GemmParams& p, int grid, int smem, cudaStream_t stream, bool pdl)
{
    const void* f = smallm_fn(bn, p.epilog);
    if (!f) return cudaErrorInvalidValue;
    return smallm_launch_fn(f, p, grid, smem, sm_threads(bn), stream, pdl);
}

}  // namespace gemm_epi
