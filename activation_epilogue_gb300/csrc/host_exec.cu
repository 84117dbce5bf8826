// gemm_epi_execute_host: the fused call on operands in host memory.  A, D (and residual,
// aux) are split into row chunks; chunk j's host-to-device copy, GEMM and device-to-host copy
// run on three streams the plan owns, each waiting (on events) only for what it needs, with
// device slots per chunked operand (kOutSlots for outputs, more for inputs), so the copies of
// chunks j+1 and j-1 overlap the GEMM of chunk j.  B and the bias are copied once per call.
//
// Column panels at the start: no row of D can be computed before all of B is on the device,
// so with a large B the copies out would wait for it.  Instead the first chunks (one per
// slot) are copied in first and B follows in column panels; as each panel lands, those
// chunks' columns of D under it are computed and copied out, so the link to the host starts
// carrying D while B is still coming in.  The rest of the chunks then run as above.
#include <cstring>
#include <new>

#include "plan.h"

using namespace gemm_epi;

namespace gemm_epi_impl {

// Device slots per output (D, mask words): the GEMM of chunk j reuses the slot of chunk
// j - kOutSlots, so it waits for that chunk's copy out; with three slots a GEMM that runs late
// does not hold up the copies out (with two, a GEMM only 10 % shorter than a chunk's copy out
// is all the slack there is).  Inputs (A, residual) get more slots, up to every chunk within
// kInSlotBudget bytes, so that their copies in run ahead and end early: while copies run both
// ways the link to the host carries ~169 GB/s each way, ~192 GB/s device-to-host alone.
constexpr int kOutSlots = 3;
constexpr int kMaxInSlots = 32;  // (the chunk count's cap)
constexpr size_t kInSlotBudget = 2ull << 30;

struct HostPipe {
    int64_t chunk = 0;  // rows per chunk (the last may be shorter)
    cudaStream_t s_in = nullptr, s_comp = nullptr, s_out = nullptr;
    cudaEvent_t ev_start = nullptr, ev_shared = nullptr;
    int nin = kOutSlots;  // input slots
    // per input slot: its copy in done, the GEMM that read it done; per output slot: its copy
    // out done
    cudaEvent_t ev_in[kMaxInSlots] = {}, ev_read[kMaxInSlots] = {}, ev_out[kOutSlots] = {};
    void* dA[kMaxInSlots] = {};
    void* dR[kMaxInSlots] = {};
    void* dD[kOutSlots] = {};
    void* dAux[kOutSlots] = {};
    void* dB = nullptr;
    void* dBias = nullptr;
    gemm_epi_plan_s full{}, last{};  // the chunk plans (sharing the parent's status word)
    bool has_last = false;
    // column panels of the first chunks: panel plans (full chunk rows x panel width, B and
    // D with the full matrices' row stride; the last panel may be narrower)
    int panel_chunks = 0;  // chunks computed panel by panel (0: none)
    int64_t panel_w = 0;
    int npanels = 0;
    gemm_epi_plan_s panel{}, panel_last{};
    cudaEvent_t ev_panel_in = nullptr, ev_panel_done = nullptr;
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
    for (cudaEvent_t e : {h->ev_start, h->ev_shared, h->ev_panel_in, h->ev_panel_done})
        if (e) cudaEventDestroy(e);
    for (int s = 0; s < kMaxInSlots; ++s) {
        for (cudaEvent_t e : {h->ev_in[s], h->ev_read[s]})
            if (e) cudaEventDestroy(e);
        for (void* b : {h->dA[s], h->dR[s]})
            if (b) cudaFree(b);
    }
    for (int s = 0; s < kOutSlots; ++s) {
        if (h->ev_out[s]) cudaEventDestroy(h->ev_out[s]);
        for (void* b : {h->dD[s], h->dAux[s]})
            if (b) cudaFree(b);
    }
    for (void* b : {h->dB, h->dBias})
        if (b) cudaFree(b);
    release_split_ws(&h->full);
    release_split_ws(&h->last);
    release_split_ws(&h->panel);
    release_split_ws(&h->panel_last);
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

// The fields a chunk or panel plan takes from the parent (shape set by the caller); it shares
// the parent's status word and tile counter (its launches run in stream order on one stream).
void derive_plan(const gemm_epi_plan_s* p, int64_t rows, int64_t cols, gemm_epi_plan_s* c)
{
    memset(c, 0, sizeof(*c));
    c->m = rows;
    c->n = cols;
    c->k = p->k;
    c->dtype = p->dtype;
    c->epilog = p->epilog;
    c->bias_layout = p->bias_layout;
    c->device = p->device;
    c->sm_count = p->sm_count;
    c->prefetch = p->prefetch;
    c->no_pdl = p->no_pdl;
    c->wait_limit_ns = p->wait_limit_ns;
    c->d_status = p->d_status;
    c->d_sched = p->d_sched;
}

gemm_epi_status chunk_plan(const gemm_epi_plan_s* p, int64_t rows, gemm_epi_plan_s* c)
{
    derive_plan(p, rows, p->n, c);
    c->opt_variant = p->opt_variant;
    c->opt_bn = p->opt_bn;
    c->opt_split_k = p->opt_split_k;
    c->opt_split_mode = p->opt_split_mode;
    c->opt_tile_m = p->opt_tile_m;
    c->opt_grid = p->opt_grid;
    c->opt_group_m = p->opt_group_m;
    c->opt_tile_order = p->opt_tile_order;
    return configure(c);
}

// Column panels of the first chunks (see the top of this file): for the epilogs whose
// output is D alone (no mask words, no residual) when B is at least 32 MiB and there are two
// or more full chunks; about 32 MiB of B per panel (2 to 8 panels), widths a multiple of
// 256 columns.  Measured on GB300 at 65536 x 16384 x 8192 RELU_BIAS (B 256 MiB, 8 panels of
// 2048 columns over the first three chunks; median of 40 calls): 13.49 ms per call against
// 13.81 with B copied whole first and three input slots (13.68 with the panels alone).  An
// event trace of the call: the first columns of D leave at 0.83 ms (1.7 ms before), B is in
// at 2.2 ms, the inputs at ~8 ms, after which D leaves at ~192 GB/s instead of ~166.
bool panel_epilog(int e)
{
    return e == GEMM_EPI_BIAS || e == GEMM_EPI_RELU_BIAS || e == GEMM_EPI_GELU_BIAS ||
           e == GEMM_EPI_NONE || e == GEMM_EPI_TANH_BIAS;
}

gemm_epi_status panel_plan(const gemm_epi_plan_s* p, int64_t rows, int64_t width, gemm_epi_plan_s* c)
{
    derive_plan(p, rows, width, c);
    c->opt_split_k = 1;  // no split-K workspace
    c->ldb = p->n;
    c->ldd = p->n;
    gemm_epi_status st = configure(c);
    if (st == GEMM_EPI_OK && c->variant != kRowPair && c->variant != kRowTile)
        st = GEMM_EPI_ERR_UNSUPPORTED_SHAPE;  // (the D row stride needs the row-tile store)
    return st;
}

void plan_panels(gemm_epi_plan_s* p, HostPipe* h)
{
    const int64_t b_bytes = p->k * p->n * 2;
    const int64_t full_chunks = p->m / h->chunk;
    if (!panel_epilog(p->epilog) || p->opt_variant != 0 || p->opt_bn != 0 ||
        b_bytes < (32ll << 20) || full_chunks < 2 || p->n < 512)
        return;
    int64_t want = b_bytes / (32ll << 20);
    want = want < 2 ? 2 : want > 8 ? 8 : want;
    int64_t w = (p->n + want - 1) / want;
    w = (w + 255) / 256 * 256;
    const int np = static_cast<int>((p->n + w - 1) / w);
    if (np < 2) return;
    const int64_t w_last = p->n - (np - 1) * w;
    if (panel_plan(p, h->chunk, w, &h->panel) != GEMM_EPI_OK) return;
    if (w_last != w && panel_plan(p, h->chunk, w_last, &h->panel_last) != GEMM_EPI_OK) {
        release_split_ws(&h->panel);
        return;
    }
    h->panel_w = w;
    h->npanels = np;
    h->panel_chunks = static_cast<int>(full_chunks < kOutSlots ? full_chunks : kOutSlots);
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
    for (cudaEvent_t* e : {&h->ev_start, &h->ev_shared, &h->ev_panel_in, &h->ev_panel_done})
        ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
    if (ok) plan_panels(p, h);
    const size_t e2 = 2;
    const size_t a_bytes = static_cast<size_t>(h->chunk) * p->k * e2;
    const size_t d_bytes = static_cast<size_t>(h->chunk) * p->n * e2;
    const size_t in_bytes = a_bytes + (p->epilog == GEMM_EPI_BIAS_RESIDUAL ? d_bytes : 0);
    const int64_t nchunks = (p->m + h->chunk - 1) / h->chunk;
    int64_t nin = in_bytes ? static_cast<int64_t>(kInSlotBudget / in_bytes) : kMaxInSlots;
    if (nin > nchunks) nin = nchunks;
    if (nin > kMaxInSlots) nin = kMaxInSlots;
    if (nin < kOutSlots) nin = kOutSlots;
    h->nin = static_cast<int>(nin);
    for (int s = 0; s < h->nin; ++s)
        for (cudaEvent_t* e : {&h->ev_in[s], &h->ev_read[s]})
            ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
    for (int s = 0; s < kOutSlots; ++s)
        ok = ok && cudaEventCreateWithFlags(&h->ev_out[s], cudaEventDisableTiming) == cudaSuccess;
    const size_t aux_bytes = static_cast<size_t>(h->chunk) * ((p->n + 31) / 32) * 4;
    const size_t b_bytes = static_cast<size_t>(p->k) * p->n * e2;
    const size_t bias_bytes = static_cast<size_t>(p->bias_layout == GEMM_EPI_BIAS_M1 ? p->m : p->n) * e2;
    auto alloc = [&](void** ptr, size_t bytes) {
        if (!ok || bytes == 0) return;
        ok = cudaMalloc(ptr, bytes) == cudaSuccess;
    };
    for (int s = 0; s < h->nin; ++s) {
        alloc(&h->dA[s], a_bytes);
        if (p->epilog == GEMM_EPI_BIAS_RESIDUAL) alloc(&h->dR[s], d_bytes);
    }
    for (int s = 0; s < kOutSlots; ++s) {
        alloc(&h->dD[s], d_bytes);
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
    const int64_t nchunks = (p->m + h->chunk - 1) / h->chunk;
    int last_slot = 0;
    if (ok && h->dBias)
        ok = cudaMemcpyAsync(h->dBias, o.bias,
                             static_cast<size_t>(p->bias_layout == GEMM_EPI_BIAS_M1 ? p->m : p->n) * e2,
                             h2d, h->s_in) == cudaSuccess;
    const int J = h->panel_chunks;
    if (J > 0) {
        // the first J chunks' rows of A, one per slot; then B panel by panel, each followed
        // by those chunks' columns of D under it (computed, then copied out)
        for (int j = 0; ok && j < J; ++j) {
            ok = cudaMemcpyAsync(h->dA[j], static_cast<const char*>(o.A) + j * h->chunk * p->k * e2,
                                 static_cast<size_t>(h->chunk) * p->k * e2, h2d, h->s_in) == cudaSuccess &&
                 cudaEventRecord(h->ev_in[j], h->s_in) == cudaSuccess &&
                 cudaStreamWaitEvent(h->s_comp, h->ev_in[j], 0) == cudaSuccess;
        }
        const size_t row_b = static_cast<size_t>(p->n) * e2;  // bytes per row of B and of D
        for (int i = 0; ok && i < h->npanels; ++i) {
            const int64_t c0 = i * h->panel_w;
            const int64_t wi = p->n - c0 < h->panel_w ? p->n - c0 : h->panel_w;
            gemm_epi_plan_s* c = wi == h->panel_w ? &h->panel : &h->panel_last;
            ok = cudaMemcpy2DAsync(static_cast<char*>(h->dB) + c0 * e2, row_b,
                                   static_cast<const char*>(o.B) + c0 * e2, row_b,
                                   static_cast<size_t>(wi) * e2, static_cast<size_t>(p->k), h2d,
                                   h->s_in) == cudaSuccess &&
                 cudaEventRecord(h->ev_panel_in, h->s_in) == cudaSuccess &&
                 cudaStreamWaitEvent(h->s_comp, h->ev_panel_in, 0) == cudaSuccess;
            for (int j = 0; ok && j < J; ++j) {
                const int64_t r0 = j * h->chunk;
                const char* bias = nullptr;
                if (h->dBias)
                    bias = static_cast<const char*>(h->dBias) +
                           (p->bias_layout == GEMM_EPI_BIAS_M1 ? r0 : c0) * static_cast<int64_t>(e2);
                gemm_epi_operands co = make_operands(
                    h->dA[j], static_cast<const char*>(h->dB) + c0 * e2, bias, nullptr,
                    static_cast<char*>(h->dD[j]) + c0 * e2, nullptr);
                st = run_plan(c, co, h->s_comp, false);
                if (st != GEMM_EPI_OK) return st;
                const bool last_panel = i == h->npanels - 1;
                ok = cudaEventRecord(last_panel ? h->ev_read[j] : h->ev_panel_done, h->s_comp) ==
                         cudaSuccess &&
                     cudaStreamWaitEvent(h->s_out, last_panel ? h->ev_read[j] : h->ev_panel_done, 0) ==
                         cudaSuccess &&
                     cudaMemcpy2DAsync(static_cast<char*>(o.D) + (r0 * p->n + c0) * e2, row_b,
                                       static_cast<char*>(h->dD[j]) + c0 * e2, row_b,
                                       static_cast<size_t>(wi) * e2, static_cast<size_t>(h->chunk),
                                       d2h, h->s_out) == cudaSuccess;
                if (ok && last_panel) ok = cudaEventRecord(h->ev_out[j], h->s_out) == cudaSuccess;
                last_slot = j;
            }
        }
    } else if (ok && h->dB) {
        ok = cudaMemcpyAsync(h->dB, o.B, static_cast<size_t>(p->k) * p->n * e2, h2d, h->s_in) ==
             cudaSuccess;
    }
    // B (and the bias) complete for the chunks below
    ok = ok && cudaEventRecord(h->ev_shared, h->s_in) == cudaSuccess;
    for (int64_t j = J; ok && j < nchunks; ++j) {
        const int a = static_cast<int>(j % h->nin);   // input slot
        const int d = static_cast<int>(j % kOutSlots);  // output slot
        const int64_t r0 = j * h->chunk;
        const int64_t rows = p->m - r0 < h->chunk ? p->m - r0 : h->chunk;
        gemm_epi_plan_s* c = rows == h->chunk ? &h->full : &h->last;
        // in: input slot a is free once the GEMM of chunk j - nin has read it
        ok = cudaStreamWaitEvent(h->s_in, h->ev_read[a], 0) == cudaSuccess;
        if (ok && p->k > 0)
            ok = cudaMemcpyAsync(h->dA[a], static_cast<const char*>(o.A) + r0 * p->k * e2,
                                 static_cast<size_t>(rows) * p->k * e2, h2d, h->s_in) == cudaSuccess;
        if (ok && h->dR[a])
            ok = cudaMemcpyAsync(h->dR[a], static_cast<const char*>(o.residual) + r0 * p->n * e2,
                                 static_cast<size_t>(rows) * p->n * e2, h2d, h->s_in) == cudaSuccess;
        ok = ok && cudaEventRecord(h->ev_in[a], h->s_in) == cudaSuccess;
        // the GEMM: after its inputs, and after chunk j - kOutSlots's results left slot d
        ok = ok && cudaStreamWaitEvent(h->s_comp, h->ev_in[a], 0) == cudaSuccess &&
             cudaStreamWaitEvent(h->s_comp, h->ev_shared, 0) == cudaSuccess &&
             cudaStreamWaitEvent(h->s_comp, h->ev_out[d], 0) == cudaSuccess;
        if (!ok) break;
        gemm_epi_operands co = make_operands(
            h->dA[a], h->dB,
            h->dBias ? static_cast<const char*>(h->dBias) +
                           (p->bias_layout == GEMM_EPI_BIAS_M1 ? r0 * static_cast<int64_t>(e2) : 0)
                     : nullptr,
            h->dR[a], h->dD[d], h->dAux[d]);
        st = run_plan(c, co, h->s_comp, false);
        if (st != GEMM_EPI_OK) return st;
        ok = cudaEventRecord(h->ev_read[a], h->s_comp) == cudaSuccess;
        // out
        ok = ok && cudaStreamWaitEvent(h->s_out, h->ev_read[a], 0) == cudaSuccess;
        if (ok)
            ok = cudaMemcpyAsync(static_cast<char*>(o.D) + r0 * p->n * e2, h->dD[d],
                                 static_cast<size_t>(rows) * p->n * e2, d2h, h->s_out) == cudaSuccess;
        if (ok && h->dAux[d])
            ok = cudaMemcpyAsync(static_cast<char*>(o.aux) + r0 * aux_row, h->dAux[d],
                                 static_cast<size_t>(rows) * aux_row, d2h, h->s_out) == cudaSuccess;
        ok = ok && cudaEventRecord(h->ev_out[d], h->s_out) == cudaSuccess;
        last_slot = d;
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
