/*
 * moe.h -- C ABI of the B300 (sm_103a) forward pass of a sparse top-k
 * Mixture-of-Experts layer, on one GPU.
 *
 * The layer (pages cited by title and section):
 *   "How Mixture of Experts Works: Sparse Gating, Expert Routing, and the
 *   Architecture Behind Efficient Large Language Models" (letsbuildsolutions),
 *   sections "The Gating Mechanism", "The Load Balancing Problem", "The
 *   Capacity Factor", "Token Dropping and Overflow Handling";
 *   "Mixture of Experts (MoE) -- conditional computation at scale" (getnybble),
 *   sections "The router", "Load balancing and expert collapse", "The shared
 *   expert pattern", "Implementing a complete MoE layer";
 *   "Mixture-of-Experts Routing" (randomcommits), section "How a sparse MoE
 *   layer works" (GELU experts, capacity check, residual add).
 *
 * Stages and the call that runs each:
 *   moe_route         router GEMM, softmax, top-k (ties -> lower index),
 *                     renormalised weights, mean router probability per expert
 *   moe_dispatch      per-expert counts, token-order ranks, capacity drops,
 *                     stable expert-grouped permutation, aux loss
 *   moe_expert_ffn    gather, grouped up-projection + activation, grouped
 *                     down-projection scaled by the gate weight and scattered
 *                     to its assignment slot (+ the shared expert)
 *   moe_combine       y = x + sum of the token's kept slots (+ shared expert)
 *   moe_layer_forward all of the above, in order, on one stream
 *
 * Conventions (every call):
 *  - Pointers are DEVICE pointers unless a parameter says otherwise.  The
 *    caller owns every buffer; the library allocates no device memory and
 *    keeps no state besides per-device attribute caches.
 *  - Matrices are row-major and contiguous.  Weights use the nn.Linear layout
 *    (one row per output unit):  Wr [E,d];  W1, W3 [E,F,d];  W2 [E,d,F];
 *    b1 [E,F];  b2 [E,d];  shared S1, S3 [F_shared,d];  S2 [d,F_shared].
 *  - "Assignment" a = t*k + s is slot s of token t.
 *  - dtype MOE_BF16: x, weights, biases, y and the slot buffer are bf16, router
 *    logits / weights fp32, accumulation fp32.  MOE_F32: everything fp32.
 *    bf16 buffers must be 16-byte aligned; d, F and F_shared multiples of 8;
 *    E * max(d, F) below 2^31 (weight rows take 32-bit coordinates).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  Host-side argument errors are returned before anything
 *    is launched.  Errors found on the device (an expert index out of range, a
 *    bounded wait that ran out) are recorded in a status word inside the
 *    workspace and read with moe_get_device_status; the kernels that find them
 *    skip the offending access and return, so the context stays usable.
 *  - A workspace (moe_workspace_size bytes, device memory) is required by
 *    every call that takes `ws`.  Zero it once with moe_workspace_init after
 *    allocating it; the calls leave it reusable.  Calls that share one
 *    workspace must not overlap in time (use one stream, or one workspace per
 *    stream).
 *  - Return value: MOE_OK or one of the MOE_ERR_* codes below.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,    /* null/misaligned pointer, size out of range */
    MOE_ERR_UNSUPPORTED = 2,    /* combination not implemented (e.g. SwiGLU + bias) */
    MOE_ERR_WORKSPACE = 3,      /* ws_bytes smaller than moe_workspace_size */
    MOE_ERR_CUDA = 4,           /* a CUDA runtime call or launch failed */
    MOE_ERR_DEVICE_TIMEOUT = 5, /* device status: a bounded wait ran out */
    MOE_ERR_DEVICE_BOUNDS = 6,  /* device status: an index was out of range */
    MOE_ERR_NO_DEVICE = 7       /* no usable CUDA device */
};

enum moe_dtype { MOE_F32 = 0, MOE_BF16 = 1 };
enum moe_act { MOE_GELU_ERF = 0, MOE_SWIGLU = 1 };
enum moe_scoring { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 };
enum moe_gemm_kernel { MOE_GEMM_AUTO = 0, MOE_GEMM_TC1 = 1, MOE_GEMM_PAIR = 2, MOE_GEMM_SWAP = 3 };
enum moe_route_path { MOE_ROUTE_AUTO = 0, MOE_ROUTE_SEPARATE = 1 };

/* Layer shape and options.
 *  T        tokens (>= 0; T = 0 is a no-op)
 *  d        model width (d_model), multiple of 8
 *  F        expert hidden width (d_ff), multiple of 8
 *  E        routed experts, 1..256
 *  k        experts per token, 1..min(E, 8)
 *  F_shared hidden width of one always-on shared SwiGLU expert added
 *           unweighted to every token ("The shared expert pattern"); 0 = none
 *  dtype    MOE_F32 or MOE_BF16
 *  act      MOE_GELU_ERF: W2 gelu(W1 x + b1) + b2, gelu(z) = z/2 (1 + erf(z/sqrt2))
 *           MOE_SWIGLU:   W2 (silu(W1 x) * (W3 x))
 *  has_bias GELU experts carry b1, b2 (SwiGLU experts take none)
 *  capacity_factor  > 0: capacity = max(1, floor(cf*T*k/E)) assignments per
 *           expert ("The Capacity Factor"); later assignments, in token order,
 *           are dropped and add nothing.  <= 0: dropless.
 *  scoring  MOE_SCORE_SOFTMAX (default): softmax over all E experts;
 *           MOE_SCORE_SIGMOID: an independent sigmoid per expert
 *           ("Mixture-of-Experts routing", "The knobs": scoring_func)
 *  no_renorm 0 (default): kept scores divided by their sum; 1: kept scores
 *           used as they are (the same page's norm_topk_prob = false)
 *  weight_fp8 0 (default): expert weights in the layer dtype; 1: routed expert
 *           weights W1, W3, W2 are FP8 E4M3 codes (one byte each, same shapes)
 *           with fp32 scales per output row in moe_weights.s1, s3, s2, i.e.
 *           row i of W1 is s1[i] * W1[i,:] ("How Mixture of Experts Works",
 *           "Quantization for MoE").  bf16 layers without a shared expert;
 *           d and F multiples of 16.
 *  weight_fp4 0 (default); 1: routed expert weights are packed 4-bit weights
 *           (not with weight_fp8): each row of K values (K = d for W1, W3; F
 *           for W2; a multiple of 128) is K/128 chunks of 80 bytes -- 64 bytes
 *           of E2M1 codes (value 2i of the chunk in the low nibble of byte i,
 *           value 2i+1 in the high nibble), 8 E4M3 scales (scale b multiplies
 *           values 16b .. 16b+15), 8 zero bytes -- with the fp32 row scales
 *           s1, s3, s2 on top: w = code * block scale * row scale.  bf16
 *           layers without a shared expert; d and F multiples of 128.
 *  gemm_kernel  bf16 expert GEMM kernel: MOE_GEMM_AUTO (default) picks one from
 *           the shape; MOE_GEMM_TC1 (tokens on the MMA's M, 128-row tiles, one
 *           SM per tile), MOE_GEMM_PAIR (tokens on M, 256-row tiles on SM
 *           pairs) or MOE_GEMM_SWAP (weights on M, tokens on N in tiles of up
 *           to 256, SM pairs) forces one.  All give results within the bf16 tolerance of each other;
 *           ignored by fp32 and low-bit layers.
 *  route_path MOE_ROUTE_AUTO (default): decode-sized batches (T <= 256,
 *           T*k <= 512, T*E <= 2048) route and dispatch in one launch;
 *           MOE_ROUTE_SEPARATE: always the separate router and dispatch kernels.
 * A zero-filled moe_cfg with the sizes set gives the pages' default router and
 * the automatic kernel choices.
 *
 * Environment: MOE_PDL=0, read once per process, launches every kernel
 * without programmatic dependent launch (each kernel then starts only after
 * its predecessor has finished); results are the same either way. */
typedef struct moe_cfg {
    int T, d, F, E, k;
    int F_shared;
    int dtype;
    int act;
    int has_bias;
    float capacity_factor;
    int scoring;
    int no_renorm;
    int weight_fp8;
    int weight_fp4;
    int gemm_kernel;
    int route_path;
} moe_cfg;

/* Expert weights (device pointers, dtype of the layer).  W3 only for SwiGLU;
 * b1, b2 only with has_bias; S1, S3, S2 only with F_shared > 0; s1 [E,F],
 * s3 [E,F], s2 [E,d] (fp32 row scales) only with weight_fp8 or weight_fp4. */
typedef struct moe_weights {
    const void *W1, *W3, *W2;
    const void *b1, *b2;
    const void *S1, *S3, *S2;
    const float *s1, *s3, *s2;
} moe_weights;

/* Outputs of moe_layer_forward.  y is required; every other pointer may be
 * NULL, in which case the value is kept in the workspace only.
 *  y           [T, d]  layer output, dtype of the layer
 *  logits      [T, E]  fp32 router logits
 *  topk_idx    [T, k]  int32 selected experts, slot 0 the largest logit
 *  topk_w      [T, k]  fp32 renormalised gate weights
 *  counts_pre  [E]     int32 assignments per expert before capacity
 *  counts_kept [E]     int32 assignments per expert after capacity
 *  drop_mask   [T*k]   uint8 1 = assignment dropped by capacity
 *  stats       [2]     fp32 {aux loss E*sum_e f_e P_e, dropped fraction} */
typedef struct moe_layer_out {
    void *y;
    float *logits;
    int *topk_idx;
    float *topk_w;
    int *counts_pre;
    int *counts_kept;
    unsigned char *drop_mask;
    float *stats;
} moe_layer_out;

/* Human-readable name of a status code (static string). */
const char *moe_status_string(int status);

/* Detail of the last host-side failure on the calling thread (which argument,
 * which CUDA call); empty if none.  Thread-local, static storage. */
const char *moe_last_error(void);

/* Capacity per expert for `cfg` ("The Capacity Factor": max(int(T*k/E*cf), 1)),
 * or -1 when dropless.  Host only. */
long long moe_capacity(const moe_cfg *cfg);

/* Bytes of device workspace that the calls below need for `cfg`.  Host only;
 * validates cfg (returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED). */
int moe_workspace_size(const moe_cfg *cfg, size_t *bytes);

/* Zeroes the workspace's control words and device status.  Call once after
 * allocating a workspace (and after a device error). */
int moe_workspace_init(const moe_cfg *cfg, void *ws, size_t ws_bytes, void *stream);

/* Router ("The Gating Mechanism"; "The router"):
 *   logits[t,e] = sum_i x[t,i] Wr[e,i] (+ logit_bias[e])      fp32 [T,E]
 *   p[t,:] = softmax(logits[t,:]) over all E experts (sigmoid(logits) per
 *            expert with MOE_SCORE_SIGMOID)
 *   topk_idx[t,:] = the k largest logits, descending, ties to the lower index
 *   topk_w[t,s] = p[t,topk_idx[t,s]] / sum_s' p[t,topk_idx[t,s']]
 *            (p[t,topk_idx[t,s]] itself with no_renorm)
 *   prob_mean[e] = mean over t of p[t,e]   (P_e of the aux loss; may be NULL)
 * x [T,d] and Wr [E,d] in the layer dtype; logit_bias [E] fp32 or NULL (a
 * fixed per-expert offset on the logits).  The logits are fp32 sums of exact
 * products; their summation order depends on the batch (decode-sized batches,
 * T <= 256 with T*k <= 512 and T*E <= 2048, take K-sliced sums on CUDA cores;
 * larger bf16 batches tensor-core tiles, larger fp32 ones a tiled CUDA-core
 * GEMM), and moe_layer_forward uses the same order as this call, so both give
 * the same bits.  cfg->route_path = MOE_ROUTE_SEPARATE takes the large-batch
 * path at every size. */
int moe_route(const moe_cfg *cfg, const void *x, const void *Wr, const float *logit_bias,
              float *logits, int *topk_idx, float *topk_w, float *prob_mean,
              void *ws, size_t ws_bytes, void *stream);

/* Dispatch ("The Capacity Factor"; the per-expert grouping of the MoELayer
 * listing; capacity check in token order, "How a sparse MoE layer works"):
 *   counts_pre[e]  = #assignments with topk_idx == e
 *   rank(a)        = #earlier assignments (flattened order) on the same expert
 *   kept(a)        = rank(a) < capacity (always, when dropless)
 *   counts_kept[e] = min(counts_pre[e], capacity)
 *   offsets[e]     = sum_{e'<e} counts_kept[e'];  offsets[E] = R (kept total)
 *   dest[a]        = offsets[e] + rank(a) if kept, else -1
 *   perm_src[r]    = the assignment a with dest[a] = r, for r < R
 *   drop_mask[a]   = 1 if dropped
 *   stats (optional, needs prob_mean): {E * sum_e (counts_pre[e]/T) prob_mean[e],
 *                                        (T*k - R) / (T*k)}
 * Buffers: counts_pre, counts_kept [E]; offsets [E+1]; perm_src, dest,
 * drop_mask [T*k].  topk_idx values outside [0,E) raise MOE_ERR_DEVICE_BOUNDS
 * in the device status and are left out of every count. */
int moe_dispatch(const moe_cfg *cfg, const int *topk_idx, const float *prob_mean,
                 int *counts_pre, int *counts_kept, int *offsets, int *perm_src, int *dest,
                 unsigned char *drop_mask, float *stats, void *ws, size_t ws_bytes, void *stream);

/* Expert FFNs over the expert-grouped rows ("Implementing a complete MoE
 * layer": SwiGLU experts; "How a sparse MoE layer works": GELU experts):
 *   for r < R, a = perm_src[r], t = a / k, e the expert whose segment
 *   [offsets[e], offsets[e+1]) holds r:
 *     Ys[a] = topk_w[a] * FFN_e(x[t])
 *   and, if F_shared > 0, shared_out[t] = FFN_shared(x[t]) for every t.
 * Ys [T*k, d] in the layer dtype; rows of dropped assignments are not written.
 * shared_out [T, d] is required iff F_shared > 0. */
int moe_expert_ffn(const moe_cfg *cfg, const void *x, const int *perm_src, const int *offsets,
                   const float *topk_w, const moe_weights *w, void *Ys, void *shared_out,
                   void *ws, size_t ws_bytes, void *stream);

/* Combine ("The Gating Mechanism": weighted sum of the selected experts;
 * "How a sparse MoE layer works": added through the residual):
 *   y[t] = x[t] + sum over kept slots s of Ys[t*k+s] (+ shared_out[t])
 * accumulated in fp32 in slot order, rounded once to the layer dtype.  A token
 * whose every slot was dropped gets y = x exactly.  shared_out may be NULL. */
int moe_combine(const moe_cfg *cfg, const void *x, const void *Ys, const unsigned char *drop_mask,
                const void *shared_out, void *y, void *stream);

/* The whole layer: moe_route, moe_dispatch, moe_expert_ffn and moe_combine in
 * order on `stream`, intermediates in the workspace. */
int moe_layer_forward(const moe_cfg *cfg, const void *x, const void *Wr, const float *logit_bias,
                      const moe_weights *w, const moe_layer_out *out,
                      void *ws, size_t ws_bytes, void *stream);

/* Backward of the aux loss through the router (training; "How Mixture of
 * Experts Works", "The Load Balancing Problem": the loss adds alpha * aux).
 * f_e = counts_pre[e]/T is piecewise constant and carries no gradient; with
 * g = grad_aux = dLoss/daux and p the router scores of cfg->scoring:
 *   softmax: grad_logits[t,j] = g (E/T) p[t,j] (f_j - sum_e f_e p[t,e])
 *   sigmoid: grad_logits[t,j] = g (E/T) f_j p[t,j] (1 - p[t,j])
 *   grad_Wr[e,i] = sum_t grad_logits[t,e] x[t,i]       (optional, may be NULL)
 *   grad_x[t,i]  = sum_e grad_logits[t,e] Wr[e,i]       (optional, may be NULL)
 * logits [T,E] fp32 and counts_pre [E] are moe_route / moe_dispatch outputs;
 * x [T,d], Wr [E,d] in the layer dtype; all gradients fp32, accumulated in
 * fp32 on CUDA cores. */
int moe_aux_loss_backward(const moe_cfg *cfg, const void *x, const void *Wr, const float *logits,
                          const int *counts_pre, float grad_aux, float *grad_logits,
                          float *grad_Wr, float *grad_x, void *stream);

/* moe_layer_forward that also records seven caller-created CUDA events
 * (cudaEvent_t handles, created with timing enabled) on `stream` at the stage
 * boundaries, so a caller can time each kernel on the stream it runs on:
 *   events[0] before the router      events[4] after the up-projection GEMM
 *   events[1] after the router       events[5] after the down-projection GEMM
 *   events[2] after dispatch         events[6] after the combine
 *   events[3] after the gather
 * The events are only recorded; the caller owns them. */
int moe_layer_forward_profiled(const moe_cfg *cfg, const void *x, const void *Wr,
                               const float *logit_bias, const moe_weights *w,
                               const moe_layer_out *out, void *ws, size_t ws_bytes, void *stream,
                               void *const *events);

/* moe_dispatch for callers that cannot allocate device memory.  (The pages
 * have no counterpart; this is a deployment variant of moe_dispatch.)
 * moe_dispatch needs a caller-allocated workspace for its scratch.  Some
 * callers cannot call cudaMalloc or hand over extra device memory -- e.g. a
 * host framework that owns every allocation and passes an operator only its
 * inputs and outputs.  This variant takes the same inputs and outputs as
 * moe_dispatch (no workspace) and keeps its scratch in a fixed device array
 * inside the library (393,472 bytes per GPU that loads the library, held
 * until the process exits); it allocates nothing.
 *  - T*k must be <= 65536; larger calls return MOE_ERR_INVALID_ARG and launch
 *    nothing.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.  The address is cached per device with the
 *    id of the context it was read in; the first call in a new context on
 *    that device (e.g. after cudaDeviceReset) looks it up again.
 *  - Pointer arguments are checked as moe_dispatch checks them (non-NULL
 *    where required, int / float buffers 4-byte aligned, including stats,
 *    prob_mean and device_status when given); a failed check returns
 *    MOE_ERR_INVALID_ARG and launches nothing.
 *  - Every call clears the scratch's control words, then uses it; all calls
 *    in the process share the one array, so calls that overlap on the GPU
 *    (other streams, other threads) race and must be serialised by the caller.
 *  - device_status (optional, device int): receives the call's device status
 *    (MOE_OK or MOE_ERR_DEVICE_*) on `stream`, in place of moe_get_device_status.
 * Outputs and their meaning are those of moe_dispatch. */
int moe_dispatch_noalloc(const moe_cfg *cfg, const int *topk_idx, const float *prob_mean,
                         int *counts_pre, int *counts_kept, int *offsets, int *perm_src,
                         int *dest, unsigned char *drop_mask, float *stats, int *device_status,
                         void *stream);

/* Reads (and leaves) the device status word of a workspace: MOE_OK, or the
 * first MOE_ERR_DEVICE_* recorded since the last init.  Synchronises `stream`. */
int moe_get_device_status(void *ws, size_t ws_bytes, void *stream, int *status);

/* Test hook for the failure path of dispatch's bounded waits (no
 * counterpart on the pages).  The next moe_dispatch / moe_layer_forward on
 * this workspace runs with look-back block `block` (each block covers 512
 * consecutive assignments) never publishing its counts, so the blocks after
 * it wait about a second, give up, and record MOE_ERR_DEVICE_TIMEOUT in the
 * device status; their outputs are then not meaningful.  The hook clears
 * itself; re-initialise the workspace before further use. */
int moe_test_hold_lookback_block(void *ws, size_t ws_bytes, int block, void *stream);

/* Test hook for the failure path of the expert GEMMs' bounded waits (no
 * counterpart on the pages).  From the next layer call on this workspace, the
 * up-projection GEMM's weight producer in every CTA that reaches shared-memory
 * ring iteration `iteration` (0-based, counted over the CTA's tiles and K
 * blocks) stops there without loading it and without reporting anything, as
 * if the copy had been lost.  The MMA issuer's (or, for FP8 / 4-bit weights,
 * the converters') wait for that stage runs out after about a second; the
 * kernel records MOE_ERR_DEVICE_TIMEOUT, waits for its own copies and MMAs in
 * flight, frees its tensor memory and returns, and the layer's outputs are not
 * meaningful.  The hook stays set until moe_workspace_init, which is needed
 * before further use anyway. */
int moe_test_hold_gemm_stage(void *ws, size_t ws_bytes, int iteration, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
