// gemm_epi_execute_host: the fused call on operands in host memory.  A, D (and residual,
// aux) are split into row chunks; chunk j's host-to-device copy, GEMM and device-to-host copy
// run on three streams the plan owns, each waiting (on events) only for what it needs, with
// kHostSlots device slots per chunked operand, so the copies of chunks j+1 and j-1 overlap the
// GEMM of chunk j.  B and the bias are copied once per call.
#include <cstring>
#include <new>

#include "plan.h"

using namespace gemm_epi;

namespace gemm_epi_impl {

// Device slots per chunked operand: the GEMM of chunk j reuses the slot of chunk j - kHostSlots,
// so it waits for that chunk's copy out; with three slots a GEMM that runs late does not hold
// up the copies out (with two, a GEMM only 10 % shorter than a chunk's copy out is all the
// slack there is).
constexpr int kHostSlots = 3;

struct HostPipe {
    int64_t chunk = 0;  // rows per chunk (the last may be shorter)
    cudaStream_t s_in = nullptr, s_comp = nullptr, s_out = nullptr;
    cudaEvent_t ev_start = nullptr, ev_shared = nullptr;
    cudaEvent_t ev_in[kHostSlots] = {}, ev_comp[kHostSlots] = {}, ev_out[kHostSlots] = {};
    void* dA[kHostSlots] = {};
    void* dD[kHostSlots] = {};
    void* dR[kHostSlots] = {};
    void* dAux[kHostSlots] = {};
    void* dB = nullptr;
    void* dBias = nullptr;
    gemm_epi_plan_s full{}, last{};  // the chunk plans (sharing the parent's status word)
    bool has_last = false;
};

void destroy_host_pipe(gemm_epi_plan_s* p)
{
    HostPipe* h = p->host;
    if (!h) return;
    for (cudaStream_t st : {h->s_in, h->s_comp, h->s_out})
        if (st) {
            cudaStreamSynchronize(st);
            cudaStreamDestroy(st);
        }
    for (cudaEvent_t e : {h->ev_start, h->ev_shared})
        if (e) cudaEventDestroy(e);
    for (int s = 0; s < kHostSlots; ++s) {
        for (cudaEvent_t e : {h->ev_in[s], h->ev_comp[s], h->ev_out[s]})
            if (e) cudaEventDestroy(e);
        for (void* b : {h->dA[s], h->dD[s], h->dR[s], h->dAux[s]})
            if (b) cudaFree(b);
    }
    for (void* b : {h->dB, h->dBias})
        if (b) cudaFree(b);
    release_split_ws(&h->full);
    release_split_ws(&h->last);
    delete h;
    p->host = nullptr;
}

namespace {

// Rows per chunk: about 1024-row chunks, at most 32 of them (a chunk of a large problem still
// fills the machine), whole 128-row tiles.  The copies out cannot start before the first
// chunk's inputs are in and its GEMM is done, so more, smaller chunks shorten that fill.
// Measured on GB300, where pinned host memory moves at 193 GB/s to the host and 211 GB/s
// from it (the same for one copy, many, several streams, or SM-driven copies through the
// mapped pointer): the 65536 x 16384 x 8192 step is bound by the 2 GiB copy of D out
// (11.1 ms) plus that fill; 16 chunks and two slots 14.05 ms per step, three slots 13.99,
// 32 chunks and three slots 13.78, 64 chunks 13.80-13.85.
int64_t host_chunk_rows(int64_t m)
{
    int64_t chunks = m / 1024;
    if (chunks < 1) chunks = 1;
    if (chunks > 32) chunks = 32;
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
    c->opt_split_mode = p->opt_split_mode;
    c->opt_tile_m = p->opt_tile_m;
    c->opt_grid = p->opt_grid;
    c->opt_group_m = p->opt_group_m;
    c->prefetch = p->prefetch;
    c->no_pdl = p->no_pdl;
    c->wait_limit_ns = p->wait_limit_ns;
    c->d_status = p->d_status;
    c->d_sched = p->d_sched;  // (the chunk launches run in stream order on one stream)
    c->opt_tile_order = p->opt_tile_order;
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
    for (cudaEvent_t* e : {&h->ev_start, &h->ev_shared})
        ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
    for (int s = 0; s < kHostSlots; ++s)
        for (cudaEvent_t* e : {&h->ev_in[s], &h->ev_comp[s], &h->ev_out[s]})
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
    for (int s = 0; s < kHostSlots; ++s) {
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

}  // namespace

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
        const int s = static_cast<int>(j % kHostSlots);
        const int64_t r0 = j * h->chunk;
        const int64_t rows = p->m - r0 < h->chunk ? p->m - r0 : h->chunk;
        gemm_epi_plan_s* c = rows == h->chunk ? &h->full : &h->last;
        // in: slot s is free once the GEMM of chunk j - kHostSlots has read it
        ok = cudaStreamWaitEvent(h->s_in, h->ev_comp[s], 0) == cudaSuccess;
        if (ok && p->k > 0)
            ok = cudaMemcpyAsync(h->dA[s], static_cast<const char*>(o.A) + r0 * p->k * e2,
                                 static_cast<size_t>(rows) * p->k * e2, h2d, h->s_in) == cudaSuccess;
        if (ok && h->dR[s])
            ok = cudaMemcpyAsync(h->dR[s], static_cast<const char*>(o.residual) + r0 * p->n * e2,
                                 static_cast<size_t>(rows) * p->n * e2, h2d, h->s_in) == cudaSuccess;
        ok = ok && cudaEventRecord(h->ev_in[s], h->s_in) == cudaSuccess;
        // the GEMM: after its inputs, and after chunk j - kHostSlots's results left slot s
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

}  // namespace gemm_epi_impl

using namespace gemm_epi_impl;

extern "C" gemm_epi_status gemm_epi_execute_host(gemm_epi_plan_t p, const gemm_epi_operands* ops,
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
