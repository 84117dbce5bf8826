// The FFN block with the hidden activation H kept on chip ("Operator fusion in model
// inference, from LayerNorm to residual connections" (wmrh.cn/news/429806), section 1, the
// fused flowchart: H never written to device memory).  Built to measure that layout against
// the plan's default (two fused launches, H through L2); see the FFN option LAUNCHES = 3.
//
// One CTA (320 threads: producer warp, MMA warp, 8 epilogue warps) per (row block r of 128
// tokens, quarter q of d): tensor memory holds Y[128, 256] (columns 0-255) and one 256-wide
// chunk of H (columns 256-511).  For each chunk c of H (f / 256 chunks):
//   GEMM 1  H_c = X[rows, :] W1[:, 256 c ...]     (d / 64 K blocks; stages of X and W1)
//   epilogue: H_c + b1, GELU, rounded to 16 bits into shared memory in the K-major,
//             128-byte-swizzled layout that GEMM 2 reads as its A operand
//   GEMM 2  Y += H_c W2[256 c ..., 256 q ...]     (4 K blocks; stages of W2)
// The MMA warp issues GEMM 1 of chunk c + 1 before GEMM 2 of chunk c, so the tensor pipe
// has work while the epilogue turns H_c into bf16.  Finally Y + b2 + R is stored.
//
// X (its 128 rows, 256 KB at d = 1024) does not fit in shared memory next to the stages,
// so it is streamed again for every chunk of H, and every CTA streams all of W1: the copies
// into each SM, not the MMAs, bound this layout.
#include "gemm_kernel.cuh"

namespace gemm_epi {

namespace {

constexpr int kOcStages = 3;
constexpr int kOcABytes = kBM * kBK * 2;          // X box: 128 rows x 64 k
constexpr int kOcBBytes = 4 * 64 * kBK * 2;       // four N-major boxes {64 n, 64 k}
constexpr int kOcStageBytes = kOcABytes + kOcBBytes;  // 48 KB
constexpr int kOcHBytes = 4 * kBM * kBK * 2;      // H chunk: four K-major boxes of 64 k
constexpr int kOcOffH = kOcStages * kOcStageBytes;
constexpr int kOcOffBar = kOcOffH + kOcHBytes;
constexpr int kOcSmemBytes = 1024 + kOcOffBar + 256;  // + alignment slack
constexpr int kOcChunk = 256;                      // columns of H per chunk; of Y per CTA
static_assert(kOcSmemBytes <= 227 * 1024, "shared memory budget");

// barrier slots
constexpr int kOcFull = 0;      // [kOcStages]
constexpr int kOcEmpty = 4;     // [kOcStages]
constexpr int kOcHcFull = 8;    // GEMM 1 of the chunk done
constexpr int kOcHcEmpty = 9;   // the epilogue has read the chunk's accumulator
constexpr int kOcHReady = 10;   // the chunk's 16-bit H is in shared memory
constexpr int kOcHFree = 11;    // GEMM 2 has read it
constexpr int kOcYFull = 12;    // the last GEMM 2 done
constexpr int kOcDrain = 13;
constexpr int kOcOffHolder = 14 * 8;
constexpr int kOcOffAbort = kOcOffHolder + 4;

// Byte offset in the H buffer of 16-byte piece j (8 consecutive k) of row `row` in K box b:
// the layout a TMA copy of a {64 k, 128 rows} box with the 128-byte swizzle produces.
__device__ __forceinline__ uint32_t oc_h_offset(int b, int row, int j)
{
    return static_cast<uint32_t>(b * (kBM * kBK * 2) + row * 128 + ((j ^ (row & 7)) << 4));
}

// Producer: the stages in the order the MMA warp consumes them: GEMM 1 of chunk 0, then for
// each chunk c >= 1 GEMM 1 of c and GEMM 2 of c - 1, then GEMM 2 of the last chunk.
__device__ __forceinline__ void oc_producer(const OnchipFfnParams& p, uint32_t sbase, uint32_t bar0,
                                            int r, int q, volatile int* abort_flag)
{
    const int chunks = p.f / kOcChunk;
    const int kb1 = p.d / kBK;
    int stage = 0;
    uint32_t phase = 0;
    long long issued = 0;
    bool ok = true;
    auto next_stage = [&](uint32_t bytes) -> uint32_t {
        if (!wait_bounded(bar0 + 8u * (kOcEmpty + stage), phase ^ 1u, abort_flag, p.wait_limit_ns)) {
            if (!*abort_flag) record_failure(p.status, abort_flag, kRoleProducer);
            ok = false;
            return 0;
        }
        const uint32_t fb = bar0 + 8u * (kOcFull + stage);
        mbar_arrive_expect_tx(fb, bytes);
        return fb;
    };
    auto advance = [&]() {
        ++issued;
        if (++stage == kOcStages) {
            stage = 0;
            phase ^= 1u;
        }
    };
    auto gemm1 = [&](int c) {
        for (int kb = 0; kb < kb1 && ok; ++kb) {
            const uint32_t fb = next_stage(kOcStageBytes);
            if (!ok) return;
            const uint32_t sa = sbase + static_cast<uint32_t>(stage * kOcStageBytes);
            const uint32_t sb = sa + kOcABytes;
            tma_load_2d(sa, &p.tm_X, fb, kb * kBK, r * kBM);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                tma_load_2d(sb + j * 8192, &p.tm_W1, fb, c * kOcChunk + j * 64, kb * kBK);
            advance();
        }
    };
    auto gemm2 = [&](int c) {
        for (int kb = 0; kb < kOcChunk / kBK && ok; ++kb) {
            const uint32_t fb = next_stage(kOcBBytes);
            if (!ok) return;
            const uint32_t sb = sbase + static_cast<uint32_t>(stage * kOcStageBytes) + kOcABytes;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                tma_load_2d(sb + j * 8192, &p.tm_W2, fb, q * kOcChunk + j * 64, c * kOcChunk + kb * kBK);
            advance();
        }
    };
    grid_dependency_wait();
    gemm1(0);
    for (int c = 1; c < chunks && ok; ++c) {
        gemm1(c);
        gemm2(c - 1);
    }
    if (ok) gemm2(chunks - 1);
    if (!ok) {
        // let the copies already issued land before the CTA can leave
        const long long back = issued < kOcStages ? issued : kOcStages;
        for (long long j = 1; j <= back; ++j) {
            const long long f = issued - j;
            const int s = static_cast<int>(f % kOcStages);
            const uint32_t ph = static_cast<uint32_t>((f / kOcStages) & 1);
            wait_bounded(bar0 + 8u * (kOcFull + s), ph, abort_flag, kDrainLimitNs, false);
        }
    }
}

// MMA issuer (one thread): GEMM 1 of chunk c into the H accumulator (TMEM columns 256-511)
// once the epilogue has read chunk c - 1 from it; GEMM 2 of chunk c - 1 into Y (columns
// 0-255) once its 16-bit H is in shared memory.
__device__ __forceinline__ void oc_mma(const OnchipFfnParams& p, uint32_t sbase, uint32_t bar0,
                                       uint32_t tmem, volatile int* abort_flag)
{
    const int chunks = p.f / kOcChunk;
    const int kb1 = p.d / kBK;
    const uint32_t idesc = make_idesc_f16(static_cast<uint32_t>(p.bf16), 0u, 1u, kBM, kOcChunk);
    const uint32_t y_tmem = tmem;
    const uint32_t h_tmem = tmem + static_cast<uint32_t>(kOcChunk);
    const uint32_t h_smem = sbase + static_cast<uint32_t>(kOcOffH);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    bool issued_any = false;
    auto wait = [&](int slot, uint32_t parity) {
        if (ok && !wait_bounded(bar0 + 8u * slot, parity, abort_flag, p.wait_limit_ns)) {
            if (!*abort_flag) record_failure(p.status, abort_flag, kRoleMma);
            ok = false;
        }
        if (ok) tcgen05_fence_after_sync();
        return ok;
    };
    auto advance = [&]() {
        if (++stage == kOcStages) {
            stage = 0;
            phase ^= 1u;
        }
    };
    auto gemm1 = [&](int c) {
        if (c > 0 && !wait(kOcHcEmpty, static_cast<uint32_t>((c - 1) & 1))) return;
        for (int kb = 0; kb < kb1; ++kb) {
            if (!wait(kOcFull + stage, phase)) return;
            const uint32_t sa = sbase + static_cast<uint32_t>(stage * kOcStageBytes);
            const uint32_t sb = sa + kOcABytes;
#pragma unroll
            for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
                // A (X) K-major: +32 bytes per 16-deep K step; B (W1) N-major: 64-column
                // panels 8 KB apart, +16 rows (2 KB) per K step
                const uint64_t ad = make_sdesc_sw128(sa + kk * 32, 0, 1024);
                const uint64_t bd = make_sdesc_sw128(sb + kk * 2048, 8192, 1024);
                mma_f16_ss(h_tmem, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
            }
            issued_any = true;
            mma_commit(bar0 + 8u * (kOcEmpty + stage));
            advance();
        }
        mma_commit(bar0 + 8u * kOcHcFull);
    };
    auto gemm2 = [&](int c) {
        if (!wait(kOcHReady, static_cast<uint32_t>(c & 1))) return;
        for (int kb = 0; kb < kOcChunk / kBK; ++kb) {
            if (!wait(kOcFull + stage, phase)) return;
            const uint32_t sb = sbase + static_cast<uint32_t>(stage * kOcStageBytes) + kOcABytes;
#pragma unroll
            for (int kk = 0; kk < kBK / kUmmaK; ++kk) {
                // A (H) K-major from the H buffer's box kb; B (W2) N-major as above
                const uint64_t ad = make_sdesc_sw128(h_smem + kb * (kBM * kBK * 2) + kk * 32, 0, 1024);
                const uint64_t bd = make_sdesc_sw128(sb + kk * 2048, 8192, 1024);
                mma_f16_ss(y_tmem, ad, bd, idesc, (c > 0 || kb > 0 || kk > 0) ? 1u : 0u);
            }
            issued_any = true;
            mma_commit(bar0 + 8u * (kOcEmpty + stage));
            advance();
        }
        mma_commit(bar0 + 8u * kOcHFree);
    };
    gemm1(0);
    for (int c = 1; c < chunks && ok; ++c) {
        gemm1(c);
        if (ok) gemm2(c - 1);
    }
    if (ok) gemm2(chunks - 1);
    if (ok) mma_commit(bar0 + 8u * kOcYFull);
    if (!ok && issued_any) {
        // every MMA this thread issued completes before tensor memory is released
        mma_commit(bar0 + 8u * kOcDrain);
        wait_bounded(bar0 + 8u * kOcDrain, 0, abort_flag, kDrainLimitNs, false);
    }
}

// Epilogue warps (2..9): warp w reads TMEM lane quarter w mod 4 (rows 32 (w mod 4) ... of the
// block) and takes every other 32-column chunk.  Per chunk of H: + b1, GELU, 16 bits into the
// H buffer (after GEMM 2 of the previous chunk has read it); at the end Y + b2 + R.
__device__ __forceinline__ void oc_epilogue(const OnchipFfnParams& p, uint8_t* smem, uint32_t bar0,
                                            uint32_t tmem, int r, int q, volatile int* abort_flag)
{
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int quarter = warp & 3;
    const int part = (warp - 2) >> 2;
    const int row = quarter * 32 + lane;  // accumulator row (TMEM lane)
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int chunks = p.f / kOcChunk;
    bool ok = true;
    auto wait = [&](int slot, uint32_t parity) {
        if (ok && !wait_bounded(bar0 + 8u * slot, parity, abort_flag, p.wait_limit_ns)) {
            if (!*abort_flag) record_failure(p.status, abort_flag, kRoleEpilogue);
            ok = false;
        }
        if (ok) tcgen05_fence_after_sync();
        return ok;
    };
    grid_dependency_wait();
    for (int c = 0; c < chunks && ok; ++c) {
        if (!wait(kOcHcFull, static_cast<uint32_t>(c & 1))) break;
        if (c > 0 && !wait(kOcHFree, static_cast<uint32_t>((c - 1) & 1))) break;
        for (int c32 = part; c32 < kOcChunk / 32; c32 += 2) {
            uint32_t v[32];
            tmem_load_32cols(t_lane + static_cast<uint32_t>(kOcChunk + c32 * 32), v);
            const int col0 = c * kOcChunk + c32 * 32;  // column of H
            float x[32];
#pragma unroll
            for (int j = 0; j < 32; ++j)
                x[j] = gelu_erf_fast(__uint_as_float(v[j]) + load_16bit(p.b1, col0 + j, p.bf16));
            const int b = (c32 * 32) >> 6;            // K box of the H buffer
            const int j0 = ((c32 * 32) & 63) >> 3;    // first 16-byte piece in the box row
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                uint4 w;
                w.x = pack2(x[8 * i + 0], x[8 * i + 1], p.bf16);
                w.y = pack2(x[8 * i + 2], x[8 * i + 3], p.bf16);
                w.z = pack2(x[8 * i + 4], x[8 * i + 5], p.bf16);
                w.w = pack2(x[8 * i + 6], x[8 * i + 7], p.bf16);
                *reinterpret_cast<uint4*>(smem + kOcOffH + oc_h_offset(b, row, j0 + i)) = w;
            }
        }
        // the accumulator is read; the 16-bit H written (and visible to the MMAs' reads)
        tcgen05_fence_before_sync();
        fence_proxy_async_smem();
        mbar_arrive(bar0 + 8u * kOcHcEmpty);
        mbar_arrive(bar0 + 8u * kOcHReady);
    }
    if (ok && wait(kOcYFull, 0)) {
        const int grow = r * kBM + row;
        for (int c32 = part; c32 < kOcChunk / 32; c32 += 2) {
            uint32_t v[32];
            tmem_load_32cols(t_lane + static_cast<uint32_t>(c32 * 32), v);
            const int gcol = q * kOcChunk + c32 * 32;
            if (grow < p.t) {
                const long long base = static_cast<long long>(grow) * p.d + gcol;
                const uint4* rp = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.R) + base);
                uint4* yp = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.Y) + base);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint4 rr = __ldg(rp + i);
                    const uint32_t rw[4] = {rr.x, rr.y, rr.z, rr.w};
                    float y[8];
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const uint32_t lo = rw[h] & 0xFFFFu, hi = rw[h] >> 16;
                        const float r0 = p.bf16 ? __uint_as_float(lo << 16)
                                                : __half2float(__ushort_as_half(static_cast<uint16_t>(lo)));
                        const float r1 = p.bf16 ? __uint_as_float(hi << 16)
                                                : __half2float(__ushort_as_half(static_cast<uint16_t>(hi)));
                        const int j = 8 * i + 2 * h;
                        y[2 * h] = __uint_as_float(v[j]) + load_16bit(p.b2, gcol + j, p.bf16) + r0;
                        y[2 * h + 1] = __uint_as_float(v[j + 1]) + load_16bit(p.b2, gcol + j + 1, p.bf16) + r1;
                    }
                    uint4 w;
                    w.x = pack2(y[0], y[1], p.bf16);
                    w.y = pack2(y[2], y[3], p.bf16);
                    w.z = pack2(y[4], y[5], p.bf16);
                    w.w = pack2(y[6], y[7], p.bf16);
                    yp[i] = w;
                }
            }
        }
    }
    tcgen05_fence_before_sync();
}

__global__ void __launch_bounds__(kThreads, 1) ffn_onchip_kernel(const __grid_constant__ OnchipFfnParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + static_cast<uint32_t>(kOcOffBar);
    uint32_t* holder = reinterpret_cast<uint32_t*>(smem + kOcOffBar + kOcOffHolder);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOcOffBar + kOcOffAbort);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int quarters = p.d / kOcChunk;
    const int r = static_cast<int>(blockIdx.x) / quarters;
    const int q = static_cast<int>(blockIdx.x) - r * quarters;
    if (threadIdx.x == 0) {
        prefetch_tensormap(&p.tm_X);
        prefetch_tensormap(&p.tm_W1);
        prefetch_tensormap(&p.tm_W2);
        for (int s = 0; s < kOcStages; ++s) {
            mbar_init(bar0 + 8u * (kOcFull + s), 1);
            mbar_init(bar0 + 8u * (kOcEmpty + s), 1);
        }
        mbar_init(bar0 + 8u * kOcHcFull, 1);
        mbar_init(bar0 + 8u * kOcHcEmpty, kEpiThreads);
        mbar_init(bar0 + 8u * kOcHReady, kEpiThreads);
        mbar_init(bar0 + 8u * kOcHFree, 1);
        mbar_init(bar0 + 8u * kOcYFull, 1);
        mbar_init(bar0 + 8u * kOcDrain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(holder), 2 * kOcChunk);
        tmem_relinquish_alloc_permit();
    }
    tcgen05_fence_before_sync();
    __syncthreads();
    tcgen05_fence_after_sync();
    const uint32_t tmem = *holder;
    if (warp == 0) {
        if (lane == 0) oc_producer(p, sbase, bar0, r, q, abort_flag);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) oc_mma(p, sbase, bar0, tmem, abort_flag);
        __syncwarp();
    } else {
        oc_epilogue(p, smem, bar0, tmem, r, q, abort_flag);
    }
    tcgen05_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tcgen05_fence_after_sync();
        tmem_dealloc(tmem, 2 * kOcChunk);
    }
}

}  // namespace

cudaError_t ffn_onchip_prepare()
{
    return cudaFuncSetAttribute(ffn_onchip_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kOcSmemBytes);
}

cudaError_t ffn_onchip_launch(const OnchipFfnParams& p, int grid, cudaStream_t stream)
{
    ffn_onchip_kernel<<<grid, kThreads, kOcSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace gemm_epi
