/*
 * k3moe.h -- C ABI of the GB300 (sm_103a) forward of the Kimi K3 latent
 * routed-MoE layer.
 *
 * The layer (sources: "Kimi K3, as released", sections "The headline
 * correction", "Shape" and "Against the technical report"; the K3 review's
 * "Stable LatentMoE" section and parameter count; the GGUF notes' tensor
 * inventory) computes, for every token x (hidden width H):
 *
 *   l = W_router x                      router logits, fp32-accurate
 *   s = sigmoid(l); key = l, or s + b   b = e_score_correction_bias (selection only)
 *   sel = top-K experts by key (descending; equal keys: lower expert index first)
 *   w_k = s_k / sum_sel s * routed_scaling
 *   h = W_down x                        routed_expert_down_proj, H -> L (latent)
 *   y_e = W2_e (silu(W1_e h) * W3_e h)  GLU expert on the latent, MXFP4 weights
 *   z = sum_k w_k y_{sel_k}
 *   n = z / sqrt(mean(z^2) + eps) * gamma   routed_expert_norm (RMSNorm)
 *   out = W_up n  [+ W2s (silu(W1s x) * W3s x)]   up_proj L -> H, optional shared GLU
 *
 * Conventions for every call:
 *   - Return value: K3MOE_OK (0) or a negative K3MOE_ERR_* code; no exception
 *     or abort crosses the ABI.  k3moe_strerror() names a code.
 *   - Memory: every device buffer (weights, activations, outputs, workspaces)
 *     is allocated and owned by the caller; the library borrows it for the
 *     duration stated per call.  The library itself allocates only the host
 *     handle.  Matrices are row-major ("out x in" for weights, as in the
 *     checkpoint's shard header).
 *   - Streams: device work is enqueued on the caller's stream and is
 *     asynchronous unless a call says otherwise.  One handle serves one stream
 *     at a time.  Device-side failures (bounded-wait timeouts, out-of-range
 *     expert indices, f16 overflow of the GLU activation) are recorded in a
 *     status word read by k3moe_status().
 */
#ifndef K3MOE_H
#define K3MOE_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------ error codes */
#define K3MOE_OK                 0
#define K3MOE_ERR_ARG           -1   /* NULL pointer, negative size, bad enum */
#define K3MOE_ERR_SHAPE         -2   /* dimension not supported (e.g. not a multiple of 32) */
#define K3MOE_ERR_ALIGN         -3   /* pointer alignment below the stated requirement */
#define K3MOE_ERR_BAD_SCALE     -4   /* an E8M0 scale byte equals 255 (NaN) */
#define K3MOE_ERR_ALIAS         -5   /* an output overlaps an input */
#define K3MOE_ERR_WORKSPACE     -6   /* workspace missing or smaller than required */
#define K3MOE_ERR_CUDA          -7   /* a CUDA runtime/driver call failed */
#define K3MOE_ERR_TIMEOUT       -8   /* a device-side bounded wait ran out */
#define K3MOE_ERR_UNSUPPORTED   -9   /* option not implemented for this shape/path */
#define K3MOE_ERR_RANGE        -10   /* device saw an expert index outside [0, E) or an f16 overflow */
#define K3MOE_ERR_STATE        -11   /* call out of order (e.g. forward before load_weights) */

/* ------------------------------------------------------------ enums */
#define K3MOE_ACT_SILU          0    /* a = g * sigmoid(g) * u */
/* SiTU-GLU ("Kimi K3, as released", section "What is new since Kimi-Linear",
 * item 3: hidden_act "situ", activation_situ_beta 4.0, activation_situ_linear_beta
 * 25.0; the K3 report review, section "SiTU-GLU is a soft fuse": sigmoid and tanh
 * soft limits on the two GLU branches, each output coordinate bounded by 100,
 * beta tanh(z / beta) = z + O(z^3 / beta^2) near the origin).  The pages give no
 * formula; this library reads it as
 *   a = sigmoid(g) * beta tanh(g / beta) * linear_beta tanh(u / linear_beta),
 * i.e. SiLU with its linear factor g soft-limited, times the soft-limited up
 * branch (|a| < beta * linear_beta). */
#define K3MOE_ACT_SITU          1

#define K3MOE_ROUTER_F32        0    /* W_router stored fp32 (the K3 checkpoint's router) */
#define K3MOE_ROUTER_BF16       1    /* W_router stored BF16 */

#define K3MOE_PATH_AUTO         0    /* tensor-core path when the shape allows it, else generic */
#define K3MOE_PATH_GENERIC      1    /* CUDA-core kernels only (any shape meeting the basic rules) */
#define K3MOE_PATH_TENSOR       2    /* tcgen05/TMA kernels (requires 16-byte row alignment) */

/* ------------------------------------------------------------ configuration */
typedef struct k3moe_config {
    int hidden;          /* H, e.g. 7168; multiple of 32 */
    int latent;          /* L, e.g. 3584 (routed_expert_hidden_size); multiple of 32 */
    int n_experts;       /* E, e.g. 896; 1..1024 */
    int top_k;           /* K, e.g. 16; 1..min(E, 32) */
    int inter;           /* I, routed expert intermediate, e.g. 3072; multiple of 32 */
    int shared_inter;    /* S, merged shared-expert intermediate (2 x 3072 = 6144), 0 = none */
    float rms_eps;       /* routed_expert_norm epsilon, e.g. 1e-6 */
    float routed_scaling;/* routed_scaling_factor, 1.0 for K3 */
    int act;             /* K3MOE_ACT_* */
    int router_dtype;    /* K3MOE_ROUTER_* */
    int has_select_bias; /* 1: key = sigmoid(l) + b, b given in k3moe_weights.select_bias */
    int path;            /* K3MOE_PATH_* */
    float situ_beta;        /* K3MOE_ACT_SITU gate-branch beta (<= 0: 4.0) */
    float situ_linear_beta; /* K3MOE_ACT_SITU up-branch beta (<= 0: 25.0) */
    int a8;                 /* 1: MXFP8 activations into the routed experts (K3MOE_A8 below) */
} k3moe_config;

/*
 * A8 option (a8 = 1).  The K3 report review's post-training passage: the routed
 * experts were trained and are shipped with MXFP4 weights and MXFP8 input
 * activations, while attention, the latent projections, the shared experts and
 * the router keep higher precision.  With a8 set, the two activation inputs of
 * the routed expert GEMMs are rounded to OCP MXFP8 per token along K -- E4M3
 * elements (nearest even, saturating at +-448) with one E8M0 scale per 32
 * values, scale = 2^(floor(log2 amax) - 8): the latent h from its BF16 value,
 * and the GLU output from its fp32 value.  The GEMMs themselves are unchanged
 * (exact on these values); the shared experts stay A16.
 */

/*
 * Weights, all device pointers, borrowed from load_weights until destroy.
 * MXFP4 matrices are given per expert exactly as the checkpoint's shard header
 * stores them: weight_packed U8 [rows, cols/2] (two E2M1 codes per byte, low
 * nibble = lower column) and weight_scale U8 [rows, cols/32] (E8M0, value
 * 2^(e-127)).  The per-expert arrays below are HOST arrays of n_experts device
 * pointers (copied at load; the host arrays need not outlive the call).
 *   w1 = gate [I, L], w3 = up [I, L], w2 = down [L, I]
 *   ws1 = shared gate [S, H], ws3 = shared up [S, H], ws2 = shared down [H, S]
 */
typedef struct k3moe_weights {
    const void *w_router;          /* [E, H] fp32 or BF16 (router_dtype) */
    const float *select_bias;      /* [E] fp32, or NULL when has_select_bias == 0 */
    const uint16_t *w_down;        /* [L, H] BF16 (routed_expert_down_proj) */
    const uint16_t *w_up;          /* [H, L] BF16 (routed_expert_up_proj) */
    const uint16_t *norm_gamma;    /* [L] BF16 (routed_expert_norm weight) */
    const uint8_t *const *w1_packed, *const *w1_scale;
    const uint8_t *const *w3_packed, *const *w3_scale;
    const uint8_t *const *w2_packed, *const *w2_scale;
    const uint8_t *ws1_packed, *ws1_scale;   /* shared experts; NULL when shared_inter == 0 */
    const uint8_t *ws3_packed, *ws3_scale;
    const uint8_t *ws2_packed, *ws2_scale;
} k3moe_weights;

typedef struct k3moe_handle k3moe_handle;

/* Validate cfg and create a host handle (no device work).  *out is set only on success. */
int k3moe_create(const k3moe_config *cfg, k3moe_handle **out);

/* Bytes of caller-owned persistent device memory that load_weights needs
 * (device copies of the expert pointer tables, TMA descriptors, the status
 * word).  Valid after create. */
size_t k3moe_persistent_bytes(const k3moe_handle *h);

/*
 * Check and record the weights.  `persistent` (>= k3moe_persistent_bytes,
 * 256-byte aligned) must stay valid until destroy.  Scans every scale byte
 * and fails with K3MOE_ERR_BAD_SCALE on a 255.  On the tensor path each
 * packed/scale row must start 16-byte aligned (rows of the K3 shapes are
 * 1792/1536/112/96 bytes, all multiples of 16) or the call fails with
 * K3MOE_ERR_ALIGN.  Synchronises `stream` before returning.
 */
int k3moe_load_weights(k3moe_handle *h, const k3moe_weights *w, void *persistent,
                       size_t persistent_bytes, cudaStream_t stream);

/* Largest T accepted by the per-call entry points (T * top_k stays far inside
 * int range); larger T returns K3MOE_ERR_ARG (workspace_bytes returns 0). */
#define K3MOE_MAX_TOKENS (1 << 24)

/* Bytes of per-call device workspace for T tokens (256-byte aligned base),
 * including the staging used by k3moe_forward_host. */
size_t k3moe_workspace_bytes(const k3moe_handle *h, int T);

/*
 * Forward 0 <= T <= K3MOE_MAX_TOKENS tokens.  x: [T, H] BF16 device; out: [T, H] BF16 device (must
 * not overlap x: K3MOE_ERR_ALIAS).  idx_out [T, K] int32 and w_out [T, K] fp32
 * (optional, may be NULL) receive the selected experts in selection order and
 * their mixture weights.  T == 0 is a no-op.  Asynchronous on `stream`; the
 * workspace must not be used by anything else until the stream reaches this
 * point.  The call only enqueues kernels on `stream` (no host synchronisation,
 * no allocation), so it may be recorded into a CUDA graph by stream capture
 * and replayed while x, out, idx_out, w_out and the workspace stay where they
 * were at capture (the first call per token count should run outside a
 * capture: it sets kernel attributes).
 */
int k3moe_forward(k3moe_handle *h, const void *x, int T, void *out, int32_t *idx_out,
                  float *w_out, void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * Same as k3moe_forward with HOST buffers (x_host [T,H] BF16, out_host [T,H]
 * BF16, idx/w optional host arrays).  Copies in and out through the staging
 * part of `workspace` on `stream` and synchronises before returning.  Host
 * buffers should be pinned for full copy bandwidth.
 */
int k3moe_forward_host(k3moe_handle *h, const void *x_host, int T, void *out_host,
                       int32_t *idx_host, float *w_host, void *workspace, size_t workspace_bytes,
                       cudaStream_t stream);

/* Synchronise `stream`, read and clear the device status word: K3MOE_OK or
 * the first device-side error recorded since the last call.  After an error it
 * also clears the decode-size dense GEMMs' split-K arrival counters (kept in the
 * persistent buffer): a kernel stopped by a timeout may have left them part-way.
 * Forwards enqueued after a failure and before this call may be wrong. */
int k3moe_status(k3moe_handle *h, cudaStream_t stream);

/* Destroy the handle (host only; frees no caller memory).  NULL is allowed. */
void k3moe_destroy(k3moe_handle *h);

/* Static string for an error code. */
const char *k3moe_strerror(int code);

/* Which path k3moe_forward will take for T tokens: K3MOE_PATH_GENERIC or K3MOE_PATH_TENSOR. */
int k3moe_path_for(const k3moe_handle *h, int T);

/* ------------------------------------------------------------ allocation-free routing
 * No counterpart in the sources: an extra entry point for callers that cannot
 * allocate device memory at all (for example plugin hosts that give an
 * operator only its input and output buffers and forbid device allocation
 * while it runs, since cudaMalloc may block and synchronise the device and a
 * caching allocator may already own all free memory).
 *
 * Computes the router logits and the top-K selection (idx_out [T, K] int32 and
 * w_out [T, K] fp32, device memory, as k3moe_forward returns them) for
 * x [T, H] BF16 (device, 16-byte aligned).  The logits come from the fp32
 * CUDA-core GEMM of the generic path (k3moe_forward's tensor path computes them
 * on the tensor cores from BF16 hi + lo weights; the two agree to ~1e-6) and
 * the selection from the same top-K kernel.  The fp32 logits
 * scratch held in a static device array of K3MOE_ROUTE_STATIC_MAX_LOGITS
 * floats (1 MiB) inside the library instead of caller workspace.  That array
 * exists on every GPU that loads the library until the process exits.
 *   - T * n_experts above K3MOE_ROUTE_STATIC_MAX_LOGITS: K3MOE_ERR_WORKSPACE,
 *     nothing is launched.
 *   - Allocates nothing: no cudaMalloc/cudaFree or allocating library call.
 *   - The first call on a device resolves the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call
 *     before any stream capture.
 *   - All calls share the one array, which keeps the previous call's logits;
 *     each call overwrites the T * n_experts values it reads.  Calls whose
 *     work overlaps on the GPU (other streams, other threads, other handles)
 *     race on the array and must be serialised by the caller.
 */
#define K3MOE_ROUTE_STATIC_MAX_LOGITS (256 * 1024)

int k3moe_route_static(k3moe_handle *h, const void *x, int T, int32_t *idx_out, float *w_out,
                       cudaStream_t stream);

/* ------------------------------------------------------------ QB bias update
 * Quantile-Balancing selection-bias update ("the K3 report review", section on
 * Quantile Balancing): the bias each expert should carry at the next step so
 * that about q = T * top_k / n_experts of this batch's tokens select it.  It
 * uses only the handle's configuration (n_experts, top_k); weights need not be
 * loaded.
 *
 *   s[t][j]  = sigmoid(logits[t][j])
 *   alpha[t] = the (top_k + 1)-th largest of s[t][j] + bias_in[j]
 *   m[t][j]  = alpha[t] - s[t][j]   (token t selects j exactly when bias_j > m[t][j])
 *   r        = round(T * top_k / n_experts), kept in [1, T - 1]
 *   bias_out[j] = upper edge of the bin, among nbins equal bins spanning the
 *                 batch's smallest to largest margin, that holds expert j's
 *                 r-th smallest margin: within one bin width above that margin.
 *
 * logits:   device, fp32 [T, n_experts] row-major (the router's logits)
 * bias_in:  device, fp32 [n_experts], or NULL for zeros (the current bias)
 * bias_out: device, fp32 [n_experts]; may equal bias_in
 * nbins:    1 .. 8192 (the source uses 1000)
 * workspace: caller-owned device memory of k3moe_qb_workspace_bytes(h, T, nbins).
 * Asynchronous on `stream`; the result depends only on the inputs (integer
 * histogram counts).  Errors: K3MOE_ERR_ARG (NULL pointers, T < 2,
 * nbins out of range), K3MOE_ERR_UNSUPPORTED (top_k + 1 > n_experts),
 * K3MOE_ERR_WORKSPACE, K3MOE_ERR_CUDA. */
size_t k3moe_qb_workspace_bytes(const k3moe_handle *h, int T, int nbins);
int k3moe_qb_bias(k3moe_handle *h, const float *logits, int T, const float *bias_in, float *bias_out,
                  int nbins, void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------ balanced expert-parallel plan
 * The K3 report review, section "3T pre-training: turning irregular MoE into a
 * static execution plan" (the MoonEP paragraph): with E experts on R
 * expert-parallel ranks and at most E/R redundant expert slots per rank, a
 * plan always exists in which every rank receives exactly S*K routed pairs
 * (S tokens per rank, top-K routing), so the exchange buffers have a fixed
 * size and no host read of token counts sits before the expert kernels.
 * k3moe_ep_plan computes such a plan on the device from all ranks' per-expert
 * counts; k3moe_ep_dispatch gives every routed pair of one source rank its
 * destination rank and row.  The exchange itself (an all-to-all of S*K rows
 * per rank, and the reverse one for the results) is the caller's.  They use
 * the handle's n_experts, top_k and its device status word, which exists once
 * k3moe_load_weights has run (K3MOE_ERR_STATE before).
 *
 * Rank r owns the m = E/R experts r*m .. r*m + m - 1.  The plan (the pages
 * give the guarantee, not an algorithm): R times, the unplanned rank with the
 * smallest remaining home load H (ties: lower rank) takes every remaining
 * token of its home experts, then fills the rest of its C = S*K rows from the
 * largest remaining experts (ties: lower expert index), whole experts first
 * and a part of the last.  It never takes more than m experts for one rank:
 * with n ranks left holding n*C tokens, the other ranks' m largest experts
 * hold at least (n*C - H)/(n-1) >= C - H.  Expert e's pairs are numbered in
 * (source rank, token) order and successive takes of e get successive ranges
 * of that numbering, the home rank's share last.  A rank's C receive rows
 * hold its segments in planning order (home experts in index order, then
 * the takes), each a contiguous run.
 *
 * The plan, in caller-owned device buffers (int32):
 *   seg      [2E][5]  segment i: expert, rank, src (first pair number of the
 *                     expert it holds), count (> 0), dst (first receive row)
 *   rank_seg [R][2]   rank r's segments are seg[first .. first + n)
 *   exp_off  [E + 1]  expert e's segments are exp_seg[exp_off[e] .. exp_off[e + 1])
 *   exp_seg  [2E]     segment ids grouped by expert, increasing src
 *   info     [2]      number of segments; the most redundant experts on one rank
 * A plan has at most 2E segments: one home segment and at most one take per
 * expert and rank pair, at most E takes in all. */
typedef struct {
    int32_t *seg;
    int32_t *rank_seg;
    int32_t *exp_off;
    int32_t *exp_seg;
    int32_t *info;
} k3moe_ep_plan;

/* counts: device int32 [R][E], counts[q][e] = routed pairs of source rank q
 * that select expert e (each rank's counts, all-gathered); their sum must be
 * R * S * K and none negative.  tokens_per_rank: S.  n_ranks: R, 1 .. E with
 * E % R == 0 and R * S * K below 2^31.  E up to 1024.
 * One CTA on the device (its rounds on one warp); asynchronous on `stream`.  Errors: K3MOE_ERR_ARG
 * (NULL pointers, bad sizes), K3MOE_ERR_UNSUPPORTED (E > 1024),
 * K3MOE_ERR_STATE, K3MOE_ERR_CUDA.  Counts that are negative or do not sum to R * S * K are
 * found on the device: the status word gets K3MOE_ERR_RANGE, info gets
 * {0, -1} and the plan is not valid. */
int k3moe_ep_plan_compute(k3moe_handle *h, const int32_t *counts, int n_ranks, int tokens_per_rank,
                          const k3moe_ep_plan *plan, cudaStream_t stream);

/* Destinations of source rank src_rank's routed pairs idx [S][K] (device int32,
 * expert ids; the experts of one token distinct, as top-K gives): dest_rank
 * and dest_row [S][K] (device int32), the rank whose expert copy processes the
 * pair and its row in that rank's C receive rows.  counts and plan as given
 * to k3moe_ep_plan_compute (counts[src_rank] must be this idx's per-expert
 * counts).  workspace: caller-owned device memory of
 * k3moe_ep_dispatch_workspace_bytes(h, S) bytes.  Asynchronous on `stream`.
 * Errors: K3MOE_ERR_ARG, K3MOE_ERR_UNSUPPORTED (E > 1024 or K > 32),
 * K3MOE_ERR_WORKSPACE, K3MOE_ERR_STATE, K3MOE_ERR_CUDA.  An expert id outside [0, E), counts
 * that disagree with idx, or a pair number outside the plan set the status
 * word to K3MOE_ERR_RANGE and that pair's outputs to -1. */
size_t k3moe_ep_dispatch_workspace_bytes(const k3moe_handle *h, int tokens_per_rank);
int k3moe_ep_dispatch(k3moe_handle *h, const int32_t *idx, int tokens_per_rank, int src_rank,
                      const int32_t *counts, int n_ranks, const k3moe_ep_plan *plan, int32_t *dest_rank,
                      int32_t *dest_row, void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------ profiling
 * Stage timing with CUDA events recorded on the launching stream around each
 * stage of k3moe_forward (a ring of 256 forwards), plus a count of kernel
 * launches.  Off by default; enabling creates the events (host call). */
#define K3MOE_STAGE_ROUTER      0   /* router logits (+ latent down-projection when fused) */
#define K3MOE_STAGE_DOWN        1   /* routed_expert_down_proj */
#define K3MOE_STAGE_TOPK        2
#define K3MOE_STAGE_PERMUTE     3
#define K3MOE_STAGE_GATE_UP     4   /* expert w1/w3 + activation */
#define K3MOE_STAGE_EXPERT_DOWN 5   /* expert w2 */
#define K3MOE_STAGE_COMBINE     6   /* combine + RMSNorm */
#define K3MOE_STAGE_UP          7   /* routed_expert_up_proj */
#define K3MOE_STAGE_SHARED      8   /* shared experts: gate/up + activation (the whole GLU on the generic path) */
#define K3MOE_STAGE_FINISH      9   /* output conversion */
#define K3MOE_STAGE_PREP       10   /* activation conversion for the tensor path */
#define K3MOE_STAGE_SHARED_DOWN 11  /* shared experts: down projection (tensor path) */
#define K3MOE_NUM_STAGES       12

int k3moe_profile_enable(k3moe_handle *h, int enable);
/* Synchronise `stream`, then write per-stage milliseconds summed over the
 * forwards recorded since the last read (stage_ms[K3MOE_NUM_STAGES]) and the
 * number of kernel launches per stage (stage_launches, optional); returns the
 * number of forwards covered (>= 0) or an error code.  Resets the ring. */
int k3moe_profile_read(k3moe_handle *h, float *stage_ms, int *stage_launches, cudaStream_t stream);
const char *k3moe_stage_name(int stage);

/* ------------------------------------------------------------ test hooks
 * Entry points that expose one device routine each, for unit tests.  They
 * follow the conventions above. */

/* Decode an MXFP4 matrix [rows, cols] (packed [rows, cols/2], scale
 * [rows, cols/32], device) into fp32 out [rows, cols] with the device decoder
 * the kernels use. */
int k3moe_debug_dequant(const uint8_t *packed, const uint8_t *scale, int rows, int cols,
                        float *out, cudaStream_t stream);

/* Launch one CTA that waits on an mbarrier nothing ever arrives on, with the
 * same bounded-wait helper as the pipelined kernels and `spin_limit`
 * iterations.  The kernel gives up, records K3MOE_ERR_TIMEOUT in the handle's
 * status word and returns; read it with k3moe_status(). */
int k3moe_debug_wait_timeout(k3moe_handle *h, int spin_limit, cudaStream_t stream);

/* Tensor-core peak microbenchmark (the roofline denominator of the expert GEMMs):
 * one CTA per SM issues `iters` x 128 K of back-to-back tcgen05.mma, M = 128 and
 * N = n (16..256, a multiple of 16), on operands resident in shared memory.
 * kind 0: kind::f16 (f16 x f16); 1: kind::mxf8f6f4 E4M3 x E4M3; 2: kind::mxf8f6f4
 * E2M1 x E4M3 (the A8 expert GEMMs' operands), both with E8M0 block scales.
 * Writes the launch's milliseconds to *ms (CUDA events on `stream`; synchronises);
 * its work is SMs x iters x 2 x 128 x n x 128 flops.  A timed-out wait is recorded in
 * status[0] (device int32[4], caller-owned). */
int k3moe_mma_peak(int kind, int n, int iters, int *status, float *ms, cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* K3MOE_H */
