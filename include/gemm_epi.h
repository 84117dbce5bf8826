/*
 * gemm_epi.h -- C ABI of the fused GEMM + bias/activation epilogue library (sm_103a).
 *
 *   D[m,n] = epi(A[m,k] . B[k,n] + bias)
 *
 * computed in one kernel, with fp32 accumulation in tensor memory; the pre-activation
 * (A.B + bias) is never written to or read back from device memory.
 *
 * Where the operations come from:
 *   "Fusing bias into cuBLASLt matmul with nvmath-python for PyTorch inference"
 *   (blog.hotdry.top, 2025-09-22):
 *     - code example: a stateful Matmul(a, b) object, .plan(epilog=..., epilog_inputs=
 *       {"bias": bias}), .execute(), .free(); m, n, k = 1024, 512, 2048, fp16, bias (m,1);
 *     - paragraph on the BIAS / RELU_BIAS epilogs: one fused kernel instead of three
 *       (matmul, bias add, activation), no intermediate written back to global memory;
 *     - paragraph on operational parameters: input, weight and bias share one dtype; the
 *       bias is (m,1) or (1,n), any other shape fails; the plan must be freed;
 *     - paragraph on limitations: RELU_AUX_BIAS also produces the mask backward needs;
 *       Tanh is one of the predefined epilogs;
 *     - closing paragraph: GELU and dBias named as further epilogs (the backward epilogs
 *       below consume the mask of RELU_AUX_BIAS, or the pre-activation GELU_AUX_BIAS
 *       keeps, and produce dBias).
 *   "nvmath-python: cuBLAS and cuSOLVER bindings for ML linear algebra"
 *   (blog.hotdry.top, 2025-09-19), matmul-planning checklist: plan() chooses the algorithm,
 *     execute() is non-blocking.
 *   "Operator fusion in model inference, from LayerNorm to residual connections"
 *   (wmrh.cn/news/429806), section 1 flowchart: the FFN chain matmul -> bias -> GELU ->
 *     matmul -> bias; section 3: the residual add folded into the producing op.
 *
 * Conventions for every call:
 *   - A is m x k, B is k x n, D and the residual are m x n: all row-major, contiguous,
 *     of the plan's dtype, in device memory.  The bias has m elements for the (m,1)
 *     layout and n for (1,n), same dtype.  The caller owns all of them; the library never
 *     allocates, frees or keeps them beyond the call.
 *   - aux of RELU_AUX_BIAS is uint32 [m][ceil(n/32)] in device memory: bit (j mod 32)
 *     of word floor(j/32) in row i is 1 iff the fp32 pre-activation at (i, j) is > 0;
 *     bits for columns >= n are written 0.
 *   - Shapes: m, n, k >= 0; n and k must be multiples of 8 (rows of A, B and D start on
 *     16-byte boundaries, which the tensor-memory-access unit needs).  m == 0 or n == 0 is
 *     an empty problem (no kernel is launched; a backward call still zeroes dbias);
 *     k == 0 gives D = epi(bias broadcast) (backward: D = 0, dbias = 0).
 *   - Pointers A, B, D, residual and the unfused pre buffer must be 16-byte aligned; bias
 *     2-byte aligned; aux 4-byte aligned (16 for GELU_AUX_BIAS).  D must not overlap A, B
 *     or bias; D may be the residual buffer itself (an in-place residual add).
 *   - All execute calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and return launch-time errors only; a device-side wait that ran out
 *     its time limit is reported by gemm_epi_sync_status.  The fused kernel is launched as
 *     a programmatic dependent of the stream's previous work: it may start its set-up
 *     early, but reads and writes device memory only after that work has completed (except
 *     B under GEMM_EPI_OPT_B_READY, and prefetches of B into L2, which change no result).
 *   - A plan belongs to the device that was current when it was made; execute with that
 *     device current.  Free it only after the work that uses it has completed.  One plan
 *     must not be executed from several host threads at the same time, and its launches
 *     must not run concurrently on the GPU (two streams without an ordering between them):
 *     they share the plan's status word and tile counter.  Different plans may run
 *     concurrently.
 *   - No call aborts the process; every failure is a status code.
 */
#ifndef GEMM_EPI_H_
#define GEMM_EPI_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t, without requiring the CUDA headers (same definition as cuda_runtime). */
typedef struct CUstream_st* cudaStream_t;

/* Opaque plan: the chosen kernel configuration, cached tensor-memory-access descriptors, a
 * device status word and a device tile counter (zero between launches).  Owned by the
 * library. */
typedef struct gemm_epi_plan_s* gemm_epi_plan_t;

typedef enum {
    GEMM_EPI_F16 = 0,  /* IEEE binary16 inputs and output */
    GEMM_EPI_BF16 = 1, /* bfloat16 inputs and output */
    GEMM_EPI_E4M3 = 2  /* 8-bit floating-point inputs (E4M3: 4 exponent bits, 3 fraction bits,
                          bias 7, no infinities, max 448) with per-tensor fp32 scales; bias,
                          residual and D in bfloat16.  A is m x k row-major; B is given
                          TRANSPOSED, n x k row-major (both operands contiguous along k), and
                          k must be a multiple of 16.  D = epi(scale_a * scale_b * (A.B) +
                          bias), scale_a and scale_b device fp32 scalars in the operands.
                          Epilogs BIAS, RELU_BIAS, GELU_BIAS, RELU_AUX_BIAS, BIAS_RESIDUAL,
                          NONE (gemm_epi_execute_operands); runs on the CTA-pair kernel
                          (256 x 256 or 256 x 224 tiles, whichever takes fewer waves over the
                          pairs); the page names FP8 among the fused matmul's types */
} gemm_epi_dtype;

typedef enum {
    GEMM_EPI_BIAS = 0,          /* D = A.B + bias */
    GEMM_EPI_RELU_BIAS = 1,     /* D = max(A.B + bias, 0)  (+0 for every pre <= 0) */
    GEMM_EPI_GELU_BIAS = 2,     /* D = GELU(A.B + bias), erf form: x * Phi(x) */
    GEMM_EPI_RELU_AUX_BIAS = 3, /* as RELU_BIAS, and writes the aux mask [pre > 0] */
    GEMM_EPI_BIAS_RESIDUAL = 4, /* D = A.B + bias + residual (FFN second GEMM) */
    GEMM_EPI_NONE = 5,          /* D = A.B (no bias; bias pointer ignored) */
    GEMM_EPI_TANH_BIAS = 6,     /* D = tanh(A.B + bias) (the pages list Tanh among the
                                   predefined epilogs) */
    GEMM_EPI_GELU_AUX_BIAS = 7, /* as GELU_BIAS, and writes aux = the pre-activation
                                   A.B + bias rounded to the plan's dtype (m x n, 16-bit),
                                   the input the GELU backward needs */
    GEMM_EPI_DRELU_BGRAD = 8,   /* backward of RELU_AUX_BIAS: D = (A.B) * mask, mask from
                                   aux_in (the RELU_AUX_BIAS layout), and dbias = the sums
                                   of that product along the bias's broadcast direction */
    GEMM_EPI_DGELU_BGRAD = 9,   /* backward of GELU_AUX_BIAS: D = (A.B) * GELU'(pre), pre
                                   from aux_in (the GELU_AUX_BIAS layout), GELU'(x) =
                                   Phi(x) + x phi(x); dbias as for DRELU_BGRAD */
    GEMM_EPI_LN_GELU_BIAS = 10  /* D = GELU(LayerNorm(A) . W + b) with the LayerNorm folded
                                   into the epilogue: B is W' = diag(gamma) W from
                                   gemm_epi_layernorm_fold, and the operands carry ln_stats
                                   (mean, 1/sqrt(var + eps) per row of A, from
                                   gemm_epi_layernorm_stats), ln_colsum and ln_bias; D =
                                   GELU(rstd_i (A.B)_ij - rstd_i mu_i c_j + b'_j).  bias must
                                   be NULL; k >= 1 */
} gemm_epi_epilog;

typedef enum {
    GEMM_EPI_BIAS_M1 = 0, /* bias shape (m,1): bias[i] added to every column of row i */
    GEMM_EPI_BIAS_1N = 1  /* bias shape (1,n): bias[j] added to every row of column j */
} gemm_epi_bias_layout;

typedef enum {
    GEMM_EPI_OK = 0,
    GEMM_EPI_ERR_INVALID_ARG = 1,       /* null handle/pointer, bad enum, operand misuse */
    GEMM_EPI_ERR_UNSUPPORTED_SHAPE = 2, /* negative size, n or k not a multiple of 8 */
    GEMM_EPI_ERR_MISALIGNED = 3,        /* a pointer breaks the alignment rules above */
    GEMM_EPI_ERR_NO_DEVICE = 4,         /* no CUDA device / driver */
    GEMM_EPI_ERR_ARCH = 5,              /* the current device is not sm_103 */
    GEMM_EPI_ERR_ALLOC = 6,             /* the plan's own device or host allocation failed */
    GEMM_EPI_ERR_LAUNCH = 7,            /* a CUDA call failed while encoding or launching */
    GEMM_EPI_ERR_DEVICE_TIMEOUT = 8,    /* a kernel gave up on a wait (see sync_status) */
    GEMM_EPI_ERR_SCRATCH_LIMIT = 9      /* the problem needs more than the fixed static
                                           scratch of gemm_epi_ffn_execute_noalloc */
} gemm_epi_status;

/* Plan-time settings (gemm_epi_plan_set_option).  0 always means "automatic". */
typedef enum {
    GEMM_EPI_OPT_VARIANT = 0,       /* 1 = row-tile kernel, 2 = swapped small-m kernel,
                                       3 = row-tile kernel run by CTA pairs (256-row tiles),
                                       5 = small-m kernel with the K split over a cluster
                                       (m <= 64, forward epilogs, a K slab per CTA that
                                       fits in shared memory; SPLIT_K sets its slices,
                                       TILE_N its rows of D: 16, 32 or 64); E4M3 plans
                                       take 0 or 3 */
    GEMM_EPI_OPT_TILE_N = 1,        /* N tile: 64, 128 or 256 for the row-tile kernel;
                                       224 or 256 for the CTA-pair kernel; 16, 32, 64, 128
                                       or 256 rows of D for the swapped kernel (a width
                                       the chosen kernel lacks is ERR_INVALID_ARG) */
    GEMM_EPI_OPT_SPLIT_K = 2,       /* K slices per output tile, 1..8 (one CTA per tile and
                                       slice; how the partial sums meet: SPLIT_MODE) */
    GEMM_EPI_OPT_GRID = 3,          /* cap on persistent CTAs (<= SM count) */
    GEMM_EPI_OPT_GROUP_M = 4,       /* tile raster: M tiles per group */
    GEMM_EPI_OPT_WAIT_LIMIT_US = 5, /* device-side wait limit, microseconds (default 2 s) */
    GEMM_EPI_OPT_DEBUG_STALL = 6,   /* 1: the next launches wait on a barrier nothing
                                       arrives at, run out the wait limit and report
                                       GEMM_EPI_ERR_DEVICE_TIMEOUT (a test of the timeout
                                       path; no copy or MMA is issued) */
    GEMM_EPI_OPT_PREFETCH = 7,      /* L2 prefetch distance in 64-deep K blocks, 0..64
                                       (0 = none) */
    GEMM_EPI_OPT_PDL = 8,           /* 1 (default): launch the fused kernel as a
                                       programmatic dependent of the previous work on the
                                       stream (its set-up overlaps that work; every global
                                       access still waits for it); 0: plain launch */
    GEMM_EPI_OPT_SPLIT_MODE = 9,    /* how the K slices' partial sums meet.  With SPLIT_K
                                       set: 0 (default) or 2 = through a device-memory
                                       workspace the plan owns (slices 1..8; the last CTA of
                                       a tile adds them in slice order); 1 = within a
                                       thread-block cluster over distributed shared memory
                                       (slices 1..4); 3 = within a cluster, through a
                                       device-memory workspace the plan owns (slices 1..4;
                                       each rank adds the peers' sums of the chunks it
                                       owns, in rank order).  Without SPLIT_K a row-tile
                                       plan (and a plan of m <= 256 that would otherwise
                                       run the swapped kernel) may take 2..4 slices per
                                       tile by itself, with the tile width, where a per-SM
                                       time model puts that ahead: through the cluster
                                       and L2 (0 or 3), over distributed shared memory (1);
                                       2 turns that choice off */
    GEMM_EPI_OPT_TILE_M = 10,       /* swapped kernel: columns of D per tile (MMA rows), 128
                                       (the automatic choice) or 64 (on request; only the
                                       epilogs BIAS, RELU_BIAS, GELU_BIAS, NONE, TANH_BIAS,
                                       BIAS_RESIDUAL and GELU_AUX_BIAS, without a K split,
                                       else ERR_INVALID_ARG); the other kernels ignore it */
    GEMM_EPI_OPT_TILE_ORDER = 11,   /* CTA-pair kernel: 2 = each pair takes its next tile,
                                       in raster order, from a counter in the plan's device
                                       memory as it goes (the automatic choice from eight
                                       waves of tiles over the pairs up); 1 = static, pair q
                                       takes tiles q, q + pairs, ... (the automatic choice
                                       below that); the other kernels ignore it.  With 2 the
                                       plan's launches must not overlap on the GPU (they
                                       share the counter) */
    GEMM_EPI_OPT_B_READY = 12       /* 1: no earlier work on the stream writes B (a weight
                                       that stays in place between calls), so under the
                                       programmatic dependent launch (PDL = 1) the small-m,
                                       swapped and single-CTA row-tile kernels copy B's
                                       first K blocks into shared memory while that work
                                       still runs, and only A's copies wait for it (the
                                       CTA-pair kernels ignore it).  The caller keeps the
                                       promise: B written by the previous kernel on the
                                       stream gives undefined results.  0 (default): every
                                       read waits; the small-m kernel then only brings its
                                       slab of B into L2 ahead of the wait, which needs no
                                       promise.  The host-buffer call ignores it */
} gemm_epi_option;

/*
 * Make a plan for one problem shape, dtype, epilog and bias layout (the page's
 * Matmul(a, b).plan(epilog=..., epilog_inputs={"bias": ...})).  Validates the arguments,
 * checks the current device, picks the kernel configuration and allocates the plan's
 * device status word.  *out is set to NULL on failure.
 */
gemm_epi_status gemm_epi_plan(gemm_epi_plan_t* out, int64_t m, int64_t n, int64_t k,
                              gemm_epi_dtype dtype, gemm_epi_epilog epilog,
                              gemm_epi_bias_layout bias_layout);

/* Override one automatic choice of the plan (benchmarking and tests). */
gemm_epi_status gemm_epi_plan_set_option(gemm_epi_plan_t p, gemm_epi_option opt,
                                         int64_t value);

/*
 * Run the fused kernel: D = epi(A.B + bias), and the aux mask for RELU_AUX_BIAS (the
 * page's .execute()).  aux must be non-NULL exactly for RELU_AUX_BIAS (and GELU_AUX_BIAS,
 * where it points to the 16-bit pre-activation).  Not valid for BIAS_RESIDUAL (use
 * gemm_epi_execute_ex) nor the backward epilogs (use gemm_epi_execute_operands).  bias may
 * be NULL only for NONE.
 */
gemm_epi_status gemm_epi_execute(gemm_epi_plan_t p, const void* A, const void* B,
                                 const void* bias, void* D, uint32_t* aux,
                                 cudaStream_t stream);

/* As gemm_epi_execute, with the residual operand (required for BIAS_RESIDUAL, must be
 * NULL otherwise). */
gemm_epi_status gemm_epi_execute_ex(gemm_epi_plan_t p, const void* A, const void* B,
                                    const void* bias, const void* residual, void* D,
                                    uint32_t* aux, cudaStream_t stream);

/*
 * The unfused baseline, for measuring what the fusion saves: one GEMM kernel writes
 * pre0 = A.B rounded to the plan's dtype into the caller's `pre` buffer (m x n), then one
 * elementwise kernel reads it back with the bias (and residual), applies the epilog and
 * writes D (and aux).  Two launches, one extra round trip of m*n 16-bit values.
 */
gemm_epi_status gemm_epi_execute_unfused(gemm_epi_plan_t p, const void* A, const void* B,
                                         const void* bias, const void* residual, void* pre,
                                         void* D, uint32_t* aux, cudaStream_t stream);

/*
 * Every operand of one call, for the epilogs that need more than execute_ex carries
 * (GELU_AUX_BIAS, DRELU_BGRAD, DGELU_BGRAD; the others are accepted too).  Fields an
 * epilog does not use must be NULL.  All are device pointers owned by the caller.
 *   A, B, bias, residual, D   as in gemm_epi_execute_ex; no bias for the backward epilogs
 *                             (the bias layout of the plan then says which way dbias runs);
 *   aux       output: RELU_AUX_BIAS the uint32 mask words described above; GELU_AUX_BIAS the
 *             16-bit pre-activation, m x n row-major, 16-byte aligned;
 *   aux_in    input: DRELU_BGRAD mask words in the RELU_AUX_BIAS layout (pad bits ignored),
 *             4-byte aligned; DGELU_BGRAD the 16-bit pre-activation in the GELU_AUX_BIAS
 *             layout, 16-byte aligned;
 *   dbias     output, DRELU_BGRAD and DGELU_BGRAD: fp32, m entries (bias layout (m,1): sums
 *             over each row of D before rounding) or n entries ((1,n): sums over each
 *             column), 4-byte aligned.  The call zeroes it on `stream` and the kernel adds
 *             into it, so the summation order, and the last bits of dbias, may vary from
 *             call to call.  D and dbias must not overlap any other operand.
 * Backward calls are launched without the programmatic dependence described above.
 */
typedef struct {
    const void* A;
    const void* B;
    const void* bias;
    const void* residual;
    void* D;
    void* aux;
    const void* aux_in;
    float* dbias;
    const float* ln_stats;   /* LN_GELU_BIAS: m pairs (mean, rstd), 8-byte aligned */
    const float* ln_colsum;  /* LN_GELU_BIAS: n column sums of W' */
    const float* ln_bias;    /* LN_GELU_BIAS: n values beta . W + b */
    const float* scale_a;    /* E4M3 plans: device fp32 scale of A (NULL otherwise) */
    const float* scale_b;    /* E4M3 plans: device fp32 scale of B */
} gemm_epi_operands;

/* The fused kernel on the operands in *ops (any epilog of the plan). */
gemm_epi_status gemm_epi_execute_operands(gemm_epi_plan_t p, const gemm_epi_operands* ops,
                                          cudaStream_t stream);

/*
 * The fused call on operands in HOST memory: A, B, bias (and residual) are read from host
 * memory and D (and aux) written back to host memory, all ordered on `stream` like the
 * other calls (the call returns at once; the host buffers must stay valid and untouched
 * until `stream` reaches this point).  Forward epilogs on fp16/bf16 plans.
 *
 * The rows of A, D, residual and aux are processed in chunks (at most 32, of ~1024 rows or
 * more) on three streams the plan owns: the copies in run ahead, and the GEMM of chunk j
 * and the copy out of chunk j-1 run at the same time, with three device slots per output
 * (D, aux) and up to one per chunk, within 2 GiB, per input (A, residual); B and the bias
 * are copied once per call.  When B is 32 MiB or more and the epilog writes D alone (BIAS,
 * RELU_BIAS, GELU_BIAS, NONE, TANH_BIAS), the first chunks' rows of A are copied first and
 * B follows in column panels, each followed by those chunks' columns of D, so that D starts
 * leaving before all of B has arrived.  The first call allocates the plan's device buffers
 * (the slots, B, bias) and creates its streams and events; a changed plan option rebuilds
 * them.  Host buffers should be page-locked (cudaHostAlloc / pinned): pageable memory
 * works but its copies are slower and less overlapped.
 */
gemm_epi_status gemm_epi_execute_host(gemm_epi_plan_t p, const gemm_epi_operands* host_ops,
                                      cudaStream_t stream);

/* The unfused baseline (as gemm_epi_execute_unfused) on the operands in *ops: the GEMM
 * writes pre0 = A.B to `pre`, the elementwise kernel applies the epilog (and, backward, the
 * mask or GELU' factor and the dbias sums) from there. */
gemm_epi_status gemm_epi_execute_operands_unfused(gemm_epi_plan_t p,
                                                  const gemm_epi_operands* ops, void* pre,
                                                  cudaStream_t stream);

/* ---- LayerNorm ---------------------------------------------------------------------------
 * "Operator fusion in model inference, from LayerNorm to residual connections"
 * (wmrh.cn/news/429806), section 2: y = (x - mu) / sqrt(var + eps) * gamma + beta over each
 * row of X (t x d; var the biased variance of the row), optionally plus a residual, in one
 * pass.  d must be a multiple of 8 and >= 8; X, Y, residual, W and W_folded 16-byte
 * aligned, gamma, beta, b 2-byte aligned, the fp32 outputs 4-byte (stats 8-byte) aligned;
 * eps >= 0.  Asynchronous on `stream`; the caller owns every buffer. */

/* Y = LayerNorm(X) * gamma + beta (+ residual when not NULL; Y may be X or the residual). */
gemm_epi_status gemm_epi_layernorm(int64_t t, int64_t d, gemm_epi_dtype dtype, const void* X,
                                   const void* residual, const void* gamma, const void* beta,
                                   float eps, void* Y, cudaStream_t stream);

/* stats[2i], stats[2i+1] = mean and 1/sqrt(var + eps) of row i of X: the per-row half of a
 * LayerNorm folded into the next GEMM (epilog LN_GELU_BIAS). */
gemm_epi_status gemm_epi_layernorm_stats(int64_t t, int64_t d, gemm_epi_dtype dtype,
                                         const void* X, float eps, float* stats,
                                         cudaStream_t stream);

/* The per-column half, once per weight update, for the GEMM LayerNorm(x) . W + b (W: d x f):
 * W_folded[k][j] = gamma_k W[k][j] rounded to the 16-bit type, colsum[j] = sum_k
 * W_folded[k][j], bias_folded[j] = sum_k beta_k W[k][j] + b[j].  Then
 * LN(x) . W + b = rstd (x . W_folded - mu colsum) + bias_folded. */
gemm_epi_status gemm_epi_layernorm_fold(int64_t d, int64_t f, gemm_epi_dtype dtype,
                                        const void* gamma, const void* beta, const void* W,
                                        const void* b, void* W_folded, float* colsum,
                                        float* bias_folded, cudaStream_t stream);

/* Release the plan (the page's .free()).  NULL is accepted and ignored. */
gemm_epi_status gemm_epi_free(gemm_epi_plan_t p);

/*
 * Wait for `stream`, then read and clear the plan's device status word.  Returns
 * GEMM_EPI_ERR_DEVICE_TIMEOUT if a kernel launched with this plan gave up on a
 * device-side wait since the last call, else GEMM_EPI_OK (or ERR_LAUNCH if the stream
 * itself reports an error).
 */
gemm_epi_status gemm_epi_sync_status(gemm_epi_plan_t p, cudaStream_t stream);

/* Static string for a status code. */
const char* gemm_epi_status_string(gemm_epi_status s);

/* The plan's configuration as text (kernel variant, tiles, stages, grid), owned by the
 * plan; the info log the matmul-planning checklist recommends reading. */
const char* gemm_epi_plan_describe(gemm_epi_plan_t p);

/* Number of uint32 words in one row of the aux mask: ceil(n / 32). */
int64_t gemm_epi_aux_words_per_row(int64_t n);

/* ---- the FFN block ---------------------------------------------------------------------
 * "Operator fusion in model inference, from LayerNorm to residual connections"
 * (wmrh.cn/news/429806), section 1 and its flowchart: the FFN sub-layer is matmul -> bias
 * -> GELU -> matmul -> bias (five launches unfused); section 3: the residual add joins the
 * op before it.  Here it is two fused launches:
 *   GEMM 1:  H = GELU(X . W1 + b1)      X: t x d, W1: d x f, b1: f elements  (bias (1,f))
 *   GEMM 2:  Y = H . W2 + b2 + R        W2: f x d, b2: d elements, R and Y: t x d
 * H (t x f, the plan's dtype) lives in device memory the plan owns; it is written once by
 * GEMM 1 and read once by GEMM 2.  GEMM 2 is launched as a programmatic dependent of GEMM 1
 * on the same stream: its set-up overlaps GEMM 1's tail and it reads H only after GEMM 1
 * has completed.  d and f must be multiples of 8; pointer rules as above. */
typedef struct gemm_epi_ffn_plan_s* gemm_epi_ffn_plan_t;

/* Plan the FFN block for t tokens, model width d and hidden width f; allocates H. */
gemm_epi_status gemm_epi_ffn_plan(gemm_epi_ffn_plan_t* out, int64_t t, int64_t d, int64_t f,
                                  gemm_epi_dtype dtype);

/* How the plan runs the block (gemm_epi_ffn_set_option). */
typedef enum {
    GEMM_EPI_FFN_OPT_LAUNCHES = 0, /* 0 = automatic, 1 = one launch, 2 = two launches,
                                     3 = one launch with H kept on chip (the page's fused
                                     flowchart; for comparison: measured far slower, see
                                     below; d and f multiples of 256, not with LayerNorm).
                                     One launch: a single persistent kernel of CTA pairs
                                     (256 x 256 tiles) takes the GEMM-1 tiles first, then
                                     the GEMM-2 tiles; a GEMM-2 tile (or K slice of one)
                                     starts loading its rows of H once every GEMM-1 tile of
                                     those rows and columns has been stored (counters in
                                     device memory, which the call zeroes on `stream`
                                     first), so GEMM 2
                                     overlaps the end of GEMM 1 and H is read back while it
                                     is still in L2.  Automatic picks one launch when both
                                     GEMMs use the CTA-pair kernel and the block has at
                                     least six waves of tiles over the resident pairs.
                                     H on chip: one CTA per 128 tokens and 256 columns of
                                     Y keeps Y's accumulator and a 256-wide chunk of H in
                                     tensor memory and the chunk's 16-bit H in shared
                                     memory; X and W1 are streamed again for every chunk
                                     (they do not fit on chip), so the copies bound it.
                                     gemm_epi_ffn_hidden's buffer is not written. */
    GEMM_EPI_FFN_OPT_SPLIT2 = 1,  /* one launch: K slices of each GEMM-2 tile, 0 or 1 = none
                                     (the default), 2 or 4.  Each slice is a unit of work of
                                     its own (waiting only for the GEMM-1 tiles of its
                                     columns of H); the fp32 partial sums meet in a
                                     workspace the plan allocates (256 KiB per GEMM-2 tile
                                     and slice) and the slice that finishes last adds them
                                     in slice order, so results do not depend on timing.
                                     Slices are whole multiples of 256 columns of H; a
                                     request the shape cannot meet takes fewer slices.  Not
                                     chosen automatically: on GB300 the partial sums' round
                                     trip through L2 costs more than the more even spread
                                     of work gains (4096 x 1024 x 4096 bf16: 94 us in 4
                                     slices, 66 us unsplit, 62 us in two launches). */
    GEMM_EPI_FFN_OPT_TILE_ORDER = 2, /* one launch: 0 = automatic (static unsplit, dynamic
                                     when GEMM 2 is split), 1 = static (pair q takes units q,
                                     q + pairs, ...), 2 = dynamic (each pair takes the next
                                     unit from a device counter as it becomes free). */
    GEMM_EPI_FFN_OPT_B_READY = 3  /* 1: no earlier work on the stream writes W1 or W2 (the
                                     layer's weights), so in two launches each GEMM copies
                                     its weight ahead of its programmatic dependency (as
                                     GEMM_EPI_OPT_B_READY; GEMM 2's may start before GEMM 1
                                     ends).  0 (default): no promise. */
} gemm_epi_ffn_option;

gemm_epi_status gemm_epi_ffn_set_option(gemm_epi_ffn_plan_t p, gemm_epi_ffn_option opt,
                                        int64_t value);

/* The plan's mode and configuration as text, owned by the plan. */
const char* gemm_epi_ffn_plan_describe(gemm_epi_ffn_plan_t p);

/* Y = GELU(X.W1 + b1).W2 + b2 + R, asynchronous on `stream`.  Y may be R itself (each
 * element of R is read by the thread that then writes that element of Y). */
gemm_epi_status gemm_epi_ffn_execute(gemm_epi_ffn_plan_t p, const void* X, const void* W1,
                                     const void* b1, const void* W2, const void* b2,
                                     const void* R, void* Y, cudaStream_t stream);

/* Device address of the plan's H buffer (t x f), valid until gemm_epi_ffn_free. */
const void* gemm_epi_ffn_hidden(gemm_epi_ffn_plan_t p);

/* As gemm_epi_sync_status, for both GEMMs of the block. */
gemm_epi_status gemm_epi_ffn_sync_status(gemm_epi_ffn_plan_t p, cudaStream_t stream);

/* The pre-LayerNorm FFN block, Y = GELU(LayerNorm(X) . W1 + b1) . W2 + b2 + R (R usually X):
 * a plan whose GEMM 1 uses the LN_GELU_BIAS epilog (two launches plus the row statistics).
 * execute takes the folded W1 (gemm_epi_layernorm_fold) instead of W1, b1, gamma, beta. */
gemm_epi_status gemm_epi_ffn_plan_layernorm(gemm_epi_ffn_plan_t* out, int64_t t, int64_t d,
                                            int64_t f, gemm_epi_dtype dtype);
gemm_epi_status gemm_epi_ffn_execute_layernorm(gemm_epi_ffn_plan_t p, const void* X, float eps,
                                               const void* W1_folded, const float* colsum,
                                               const float* b1_folded, const void* W2,
                                               const void* b2, const void* R, void* Y,
                                               cudaStream_t stream);

/* Release the plan and its H buffer (after the work that uses them has completed). */
gemm_epi_status gemm_epi_ffn_free(gemm_epi_ffn_plan_t p);

/*
 * The FFN block without any allocation.  The pages have no counterpart: this call is for
 * callers that cannot allocate device memory themselves, for instance a serving runtime
 * that hands out all device memory from its own pool and forbids cudaMalloc once it has
 * started, or code that runs in a context where an allocation would stall or fail.  Same
 * computation and arguments as gemm_epi_ffn_plan + gemm_epi_ffn_execute, but there is no
 * plan: the hidden activation H and the two launches' status words live in one static
 * device array inside this library, of GEMM_EPI_FFN_NOALLOC_MAX_HIDDEN 16-bit elements
 * (32 MiB) plus 256 bytes (the launches' status words and tile counters), which every GPU
 * that loads the library keeps until the process exits.
 *   - t * f > GEMM_EPI_FFN_NOALLOC_MAX_HIDDEN returns GEMM_EPI_ERR_SCRATCH_LIMIT and launches
 *     nothing; other argument errors as gemm_epi_ffn_execute.
 *   - No cudaMalloc, cudaFree or other allocating call is made.  Every call looks up the
 *     array's device address (cudaGetSymbolAddress); the first call on a device, and the
 *     first after a cudaDeviceReset has loaded the library's module again at a new
 *     address, also zeroes the status words and tile counters with a synchronous
 *     cudaMemset: make that first call before any stream capture.
 *   - Every call on a device shares the one array, which keeps the last call's H: calls
 *     whose work overlaps on the GPU (different streams, or different host threads) race
 *     on it and give wrong results; order them on one stream.
 *   - A device-side wait that runs out its limit ends the kernels as in the planned path,
 *     but is only recorded in the static status words, which this call does not report.
 */
#define GEMM_EPI_FFN_NOALLOC_MAX_HIDDEN (16ll * 1024 * 1024)
gemm_epi_status gemm_epi_ffn_execute_noalloc(int64_t t, int64_t d, int64_t f,
                                             gemm_epi_dtype dtype, const void* X,
                                             const void* W1, const void* b1, const void* W2,
                                             const void* b2, const void* R, void* Y,
                                             cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_EPI_H_ */
