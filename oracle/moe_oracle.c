/*
 * moe_oracle.c -- plain, slow, obviously correct CPU oracle for the forward pass
 * of a sparse top-k Mixture-of-Experts layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or load
 * this file: it is used by the tests, by the bench's CPU baseline and by the
 * smoke check, to judge the CUDA path.  It shares no code, header, table or
 * helper with the CUDA sources.
 *
 * Arithmetic: every sum, product, exp and erf is taken in double.  Inputs are
 * read in their storage type (fp32, or bf16 given as raw 16-bit patterns) and
 * widened exactly to double.  Loops run in the order the definitions are
 * written; the only parallelism is over independent tokens.
 *
 * Sources (page title, section):
 *  [R]  "How Mixture of Experts Works: Sparse Gating, Expert Routing, ...",
 *       section "The Gating Mechanism": the router is a bias-free linear map to
 *       N logits, softmax over all N, top-k, renormalise the kept k.
 *  [G]  "Mixture of Experts (MoE) -- conditional computation at scale",
 *       section "The router": scores = softmax(h @ W_r).
 *  [D]  "How Mixture of Experts Works ...", MoELayer listing: assignments are
 *       flattened as t*k+s and grouped per expert in flattened (token) order.
 *  [C]  "How Mixture of Experts Works ...", section "The Capacity Factor":
 *       capacity = max(int(T*k/E*cf), 1); excess assignments are dropped and the
 *       token falls through on the residual ("Token Dropping and Overflow
 *       Handling", zero-output strategy).
 *  [P1] "Mixture-of-Experts Routing" (randomcommits), section "How a sparse MoE
 *       layer works": GELU MLP experts, drops in nonzero (token) order, output
 *       + x residual.
 *  [S]  "Mixture of Experts (MoE) -- conditional computation at scale",
 *       section "Implementing a complete MoE layer": SwiGLU expert
 *       w_down(silu(w_gate x) * w_up x); section "The shared expert pattern":
 *       a shared expert sees every token, unweighted.
 *  [A]  "How Mixture of Experts Works ...", section "The Load Balancing
 *       Problem", and "Mixture of Experts (MoE) ...", section "Load balancing
 *       and expert collapse": aux = E * sum_e f_e * P_e, f_e = top-k count / T,
 *       P_e = mean softmax probability (the coefficient alpha is left out).
 *
 * Readings where the pages are silent or disagree (each one is listed in the
 * design notes):
 *  - top-k is taken on the logits (softmax is monotone) and ties go to the
 *    lower expert index;
 *  - drops are decided per expert in token order, whatever the slot;
 *  - a partly dropped token keeps the weight of its surviving slot;
 *  - f_e counts assignments before drops.
 *
 * Pins: tests/test_oracle_pins.py checks this file against brute force,
 * closed forms, library routines and the special cases of the method.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_E4M3 = 2, ORC_E2M1P = 3 };
enum { ORC_GELU_ERF = 0, ORC_SWIGLU = 1 };
enum { ORC_SOFTMAX = 0, ORC_SIGMOID = 1 };

/* E4M3 (FP8, 1 sign, 4 exponent bits with bias 7, 3 mantissa bits): normal
 * codes are (-1)^s 2^(e-7) (1 + m/8); e = 0 gives the subnormals
 * (-1)^s 2^-6 (m/8); e = 15, m = 7 is NaN (the format has no infinities). */
double oracle_e4m3_value(unsigned code)
{
    const int sgn = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sgn ? -v : v;
}

/* E2M1 (FP4: 1 sign, 2 exponent bits with bias 1, 1 mantissa bit): e = 0 gives
 * (-1)^s m/2 (0 and 0.5); otherwise (-1)^s 2^(e-1) (1 + m/2), so the
 * magnitudes are 0, 0.5, 1, 1.5, 2, 3, 4, 6.  The format has no infinity or NaN. */
double oracle_e2m1_value(unsigned code)
{
    const int sgn = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    const double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sgn ? -v : v;
}

/* Packed 4-bit weights (ORC_E2M1P), the 4-bit variant of "Quantization for
 * MoE": each row of K values (K a multiple of 128) is stored as K/128 chunks
 * of 80 bytes -- 64 bytes of E2M1 codes (value 2i of the chunk in the low
 * nibble of byte i, value 2i+1 in the high nibble), then 8 E4M3 block scales
 * (scale b multiplies values 16b .. 16b+15 of the chunk), then 8 zero bytes.
 * The stored value is code * block scale; the row scale applies on top. */
static double orc_load_e2m1p(const unsigned char *row, int col)
{
    const unsigned char *chunk = row + (size_t)(col / 128) * 80;
    const int w = col % 128;
    const unsigned byte = chunk[w / 2];
    const unsigned code = (w & 1) ? (byte >> 4) : (byte & 15);
    return oracle_e2m1_value(code) * oracle_e4m3_value(chunk[64 + w / 16]);
}

/* Bytes of one stored row of K weights. */
static size_t orc_row_bytes(int K, int dtype)
{
    if (dtype == ORC_E2M1P)
        return (size_t)(K / 128) * 80;
    return (size_t)K * (dtype == ORC_F32 ? 4 : dtype == ORC_BF16 ? 2 : 1);
}

/* Exact widening of one stored element to double.  bf16 is the upper half of
 * an IEEE binary32 pattern. */
static double orc_load(const void *base, size_t i, int dtype)
{
    if (dtype == ORC_F32)
        return (double)((const float *)base)[i];
    if (dtype == ORC_E4M3)
        return oracle_e4m3_value(((const unsigned char *)base)[i]);
    uint32_t bits = ((uint32_t)((const uint16_t *)base)[i]) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Element (row, col) of a weight matrix with K values per row. */
static double orc_load_w(const void *base, size_t row, int col, int K, int dtype)
{
    if (dtype == ORC_E2M1P)
        return orc_load_e2m1p((const unsigned char *)base + row * orc_row_bytes(K, dtype), col);
    return orc_load(base, row * (size_t)K + col, dtype);
}

/* ---------------------------------------------------------------- threads */

typedef void (*orc_range_fn)(void *ctx, long lo, long hi);
typedef struct {
    orc_range_fn fn;
    void *ctx;
    long lo, hi;
} orc_job;

static void *orc_thread_main(void *p)
{
    orc_job *j = (orc_job *)p;
    j->fn(j->ctx, j->lo, j->hi);
    return NULL;
}

static int orc_threads = 0;

void oracle_set_threads(int n) { orc_threads = n; }

int oracle_get_threads(void)
{
    if (orc_threads > 0)
        return orc_threads;
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/* Runs fn over [0, n) split into contiguous ranges, one per thread. */
static void orc_parallel(long n, orc_range_fn fn, void *ctx)
{
    int nt = oracle_get_threads();
    if (nt > n)
        nt = (int)n;
    if (nt <= 1) {
        if (n > 0)
            fn(ctx, 0, n);
        return;
    }
    pthread_t th[256];
    orc_job jobs[256];
    if (nt > 256)
        nt = 256;
    for (int i = 0; i < nt; ++i) {
        jobs[i].fn = fn;
        jobs[i].ctx = ctx;
        jobs[i].lo = n * i / nt;
        jobs[i].hi = n * (i + 1) / nt;
        pthread_create(&th[i], NULL, orc_thread_main, &jobs[i]);
    }
    for (int i = 0; i < nt; ++i)
        pthread_join(th[i], NULL);
}

/* ------------------------------------------------------ step 1: router GEMM */
/* logits[t,e] = sum_i x[t,i] * Wr[e,i] (+ bias[e]).  [R], [G].
 * Wr is stored like the router's nn.Linear weight: one row of d per expert.
 * bias is an optional fixed per-expert logit offset (fp32). */
typedef struct {
    int d, E, dtype;
    const void *x, *Wr;
    const float *bias;
    const int *tokens;
    double *logits;
} orc_router_ctx;

static void orc_router_range(void *p, long lo, long hi)
{
    orc_router_ctx *c = (orc_router_ctx *)p;
    for (long r = lo; r < hi; ++r) {
        long t = c->tokens ? c->tokens[r] : r;
        for (int e = 0; e < c->E; ++e) {
            double acc = 0.0;
            for (int i = 0; i < c->d; ++i)
                acc += orc_load(c->x, (size_t)t * c->d + i, c->dtype) *
                       orc_load(c->Wr, (size_t)e * c->d + i, c->dtype);
            if (c->bias)
                acc += (double)c->bias[e];
            c->logits[r * c->E + e] = acc;
        }
    }
}

/* Router logits for ntok tokens (tokens == NULL: tokens 0..ntok-1). */
void oracle_router_logits(int ntok, const int *tokens, int d, int E, int dtype,
                          const void *x, const void *Wr, const float *bias,
                          double *logits)
{
    orc_router_ctx c = {d, E, dtype, x, Wr, bias, tokens, logits};
    orc_parallel(ntok, orc_router_range, &c);
}

/* ------------------------------------- steps 2-4: scores, top-k, renorm */
/* Scores ([R], [G]): softmax over all E experts, or (the variant the
 * "Mixture-of-Experts routing" page names under "The knobs") an independent
 * sigmoid per expert.  top-k: experts ordered by logit descending, ties to the
 * lower index; slot 0 holds the largest (both score functions are monotone in
 * the logit, so the order is the logits').  Weights: the kept scores divided
 * by their sum ([R] "Renormalize so selected weights sum to 1"), or the kept
 * scores as they are when renorm == 0.  probs receives the scores. */
void oracle_topk_ex(int T, int E, int k, int scoring, int renorm, const double *logits,
                    int *topk_idx, double *topk_w, double *probs)
{
    unsigned char *taken = (unsigned char *)malloc((size_t)E);
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    for (int t = 0; t < T; ++t) {
        const double *l = logits + (size_t)t * E;
        if (scoring == ORC_SIGMOID) {
            for (int e = 0; e < E; ++e)
                p[e] = 1.0 / (1.0 + exp(-l[e]));
        } else {
            double m = l[0];
            for (int e = 1; e < E; ++e)
                if (l[e] > m)
                    m = l[e];
            double Z = 0.0;
            for (int e = 0; e < E; ++e)
                Z += exp(l[e] - m);
            for (int e = 0; e < E; ++e)
                p[e] = exp(l[e] - m) / Z;
        }
        if (probs)
            for (int e = 0; e < E; ++e)
                probs[(size_t)t * E + e] = p[e];
        memset(taken, 0, (size_t)E);
        double kept = 0.0;
        for (int s = 0; s < k; ++s) {
            int best = -1;
            for (int e = 0; e < E; ++e)
                if (!taken[e] && (best < 0 || l[e] > l[best]))
                    best = e;
            taken[best] = 1;
            topk_idx[(size_t)t * k + s] = best;
            kept += p[best];
        }
        for (int s = 0; s < k; ++s) {
            double w = p[topk_idx[(size_t)t * k + s]];
            topk_w[(size_t)t * k + s] = renorm ? w / kept : w;
        }
    }
    free(taken);
    free(p);
}

/* The pages' default router: softmax scores, renormalised kept weights. */
void oracle_topk(int T, int E, int k, const double *logits, int *topk_idx,
                 double *topk_w, double *probs)
{
    oracle_topk_ex(T, E, k, ORC_SOFTMAX, 1, logits, topk_idx, topk_w, probs);
}

/* ------------------------------------------------------- step 6: capacity */
/* [C]: capacity = max(int(T*k/E * cf), 1).  cf <= 0 means dropless, returned
 * as -1. */
long long oracle_capacity(long long T, int k, int E, double cf)
{
    if (cf <= 0.0)
        return -1;
    double ideal = ((double)T * (double)k) / (double)E;
    long long cap = (long long)floor(ideal * cf);
    return cap < 1 ? 1 : cap;
}

/* ------------------------------------- steps 5-7: dispatch and permutation */
/* Assignment a = t*k+s picks expert e = topk_idx[a].  Its rank is the number
 * of earlier assignments (in flattened order: token ascending, then slot) that
 * picked e ([D], [P1] nonzero order).  It is dropped iff rank >= cap ([C]).
 * Kept assignments are laid out grouped by expert ascending, then by rank:
 * dest[a] = offsets[e] + rank[a], perm_src[dest[a]] = a.  Returns R, the
 * number of kept assignments. */
int oracle_dispatch(int T, int k, int E, long long cap, const int *topk_idx,
                    int *counts_pre, int *counts_kept, int *offsets, int *rank,
                    int *dest, int *perm_src, unsigned char *drop_mask)
{
    long A = (long)T * k;
    for (int e = 0; e < E; ++e)
        counts_pre[e] = 0;
    for (long a = 0; a < A; ++a) {
        int e = topk_idx[a];
        rank[a] = counts_pre[e];
        counts_pre[e] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) {
        long long kept = counts_pre[e];
        if (cap >= 0 && kept > cap)
            kept = cap;
        counts_kept[e] = (int)kept;
        offsets[e + 1] = offsets[e] + counts_kept[e];
    }
    for (long a = 0; a < A; ++a) {
        int e = topk_idx[a];
        int dropped = (cap >= 0 && rank[a] >= cap);
        drop_mask[a] = (unsigned char)dropped;
        if (dropped) {
            dest[a] = -1;
        } else {
            dest[a] = offsets[e] + rank[a];
            perm_src[dest[a]] = (int)a;
        }
    }
    return offsets[E];
}

/* ----------------------------------------------------- step 8: one expert */
/* GELU MLP ([P1]): out = W2 . gelu(W1 . x + b1) + b2, gelu(z) = z/2 (1+erf(z/sqrt 2))
 * (the exact, erf form that nn.GELU uses by default).
 * SwiGLU ([S]): out = W2 . (silu(W1 . x) * (W3 . x)), silu(z) = z/(1+exp(-z)).
 * W1, W3 hold one row of d per hidden unit ([F, d]); W2 holds one row of F per
 * output ([d, F]) -- the nn.Linear weight layout.  b1 [F], b2 [d] optional.
 * Weights are stored in wdtype, biases in bdtype.  With E4M3 or packed E2M1
 * weights, s1, s3 [F] and s2 [d] are the per-row scales: row f of W1 is
 * s1[f] * W1[f,:] ("How Mixture of Experts Works", "Quantization for MoE");
 * each row's scale multiplies its dot product.  h is caller scratch of F
 * doubles. */
void oracle_expert_ffn_q(int d, int F, int act, int wdtype, int bdtype, const double *xv,
                         const void *W1, const void *W3, const void *W2, const void *b1,
                         const void *b2, const float *s1, const float *s3, const float *s2,
                         double *h, double *out)
{
    for (int f = 0; f < F; ++f) {
        double g = 0.0;
        for (int i = 0; i < d; ++i)
            g += xv[i] * orc_load_w(W1, (size_t)f, i, d, wdtype);
        if (s1)
            g *= (double)s1[f];
        if (act == ORC_SWIGLU) {
            double u = 0.0;
            for (int i = 0; i < d; ++i)
                u += xv[i] * orc_load_w(W3, (size_t)f, i, d, wdtype);
            if (s3)
                u *= (double)s3[f];
            h[f] = g / (1.0 + exp(-g)) * u;
        } else {
            if (b1)
                g += orc_load(b1, (size_t)f, bdtype);
            h[f] = 0.5 * g * (1.0 + erf(g / sqrt(2.0)));
        }
    }
    for (int j = 0; j < d; ++j) {
        double o = 0.0;
        for (int f = 0; f < F; ++f)
            o += h[f] * orc_load_w(W2, (size_t)j, f, F, wdtype);
        if (s2)
            o *= (double)s2[j];
        if (b2)
            o += orc_load(b2, (size_t)j, bdtype);
        out[j] = o;
    }
}

void oracle_expert_ffn(int d, int F, int act, int dtype, const double *xv,
                       const void *W1, const void *W3, const void *W2,
                       const void *b1, const void *b2, double *h, double *out)
{
    oracle_expert_ffn_q(d, F, act, dtype, dtype, xv, W1, W3, W2, b1, b2, NULL, NULL, NULL, h, out);
}

/* ------------------------------------------- step 9: layer output per token */
typedef struct {
    int d, F, E, k, act, dtype, wdtype;
    const void *x;
    const void *W1, *W3, *W2, *b1, *b2; /* [E,F,d], [E,F,d], [E,d,F], [E,F], [E,d] */
    const float *s1, *s3, *s2;          /* low-bit row scales [E,F], [E,F], [E,d] or NULL */
    int F_sh;
    const void *S1, *S3, *S2; /* shared expert [F_sh,d], [F_sh,d], [d,F_sh] */
    const int *topk_idx;
    const double *topk_w;
    const unsigned char *drop_mask;
    const int *tokens;
    double *y, *slots, *shared_out;
} orc_layer_ctx;

static void orc_layer_range(void *p, long lo, long hi)
{
    orc_layer_ctx *c = (orc_layer_ctx *)p;
    int d = c->d, F = c->F, k = c->k;
    int Fmax = F > c->F_sh ? F : c->F_sh;
    double *xv = (double *)malloc(sizeof(double) * (size_t)d);
    double *acc = (double *)malloc(sizeof(double) * (size_t)d);
    double *tmp = (double *)malloc(sizeof(double) * (size_t)d);
    double *h = (double *)malloc(sizeof(double) * (size_t)(Fmax > 0 ? Fmax : 1));
    for (long r = lo; r < hi; ++r) {
        long t = c->tokens[r];
        for (int i = 0; i < d; ++i) {
            xv[i] = orc_load(c->x, (size_t)t * d + i, c->dtype);
            acc[i] = 0.0;
        }
        for (int s = 0; s < k; ++s) {
            long a = t * k + s;
            double *slot = c->slots ? c->slots + ((size_t)r * k + s) * d : NULL;
            if (c->drop_mask[a]) { /* dropped: contributes nothing ([C]) */
                if (slot)
                    for (int i = 0; i < d; ++i)
                        slot[i] = 0.0;
                continue;
            }
            int e = c->topk_idx[a];
            size_t up = (size_t)e * F * orc_row_bytes(d, c->wdtype);   /* W1, W3: F rows of d */
            size_t dn = (size_t)e * d * orc_row_bytes(F, c->wdtype);   /* W2: d rows of F */
            size_t be = c->dtype == ORC_F32 ? 4 : 2;
            oracle_expert_ffn_q(d, F, c->act, c->wdtype, c->dtype, xv,
                                (const char *)c->W1 + up,
                                c->W3 ? (const char *)c->W3 + up : NULL,
                                (const char *)c->W2 + dn,
                                c->b1 ? (const char *)c->b1 + (size_t)e * F * be : NULL,
                                c->b2 ? (const char *)c->b2 + (size_t)e * d * be : NULL,
                                c->s1 ? c->s1 + (size_t)e * F : NULL,
                                c->s3 ? c->s3 + (size_t)e * F : NULL,
                                c->s2 ? c->s2 + (size_t)e * d : NULL, h, tmp);
            double w = c->topk_w[a];
            for (int i = 0; i < d; ++i) {
                acc[i] += w * tmp[i];
                if (slot)
                    slot[i] = w * tmp[i];
            }
        }
        if (c->S1) { /* always-on shared expert, unweighted ([S]) */
            oracle_expert_ffn(d, c->F_sh, ORC_SWIGLU, c->dtype, xv, c->S1, c->S3,
                              c->S2, NULL, NULL, h, tmp);
            for (int i = 0; i < d; ++i) {
                acc[i] += tmp[i];
                if (c->shared_out)
                    c->shared_out[(size_t)r * d + i] = tmp[i];
            }
        }
        for (int i = 0; i < d; ++i) /* residual add ([P1]) */
            c->y[(size_t)r * d + i] = xv[i] + acc[i];
    }
    free(xv);
    free(acc);
    free(tmp);
    free(h);
}

/* Layer output y[r] for the listed tokens, given routing (topk_idx, topk_w)
 * and the drop mask.  slots (optional, [ntok,k,d]) receives w * FFN_e(x) per
 * slot (zero when dropped); shared_out (optional, [ntok,d]) the shared
 * expert's output.  F_sh = 0 means no shared expert. */
void oracle_layer_tokens_q(int ntok, const int *tokens, int d, int F, int E, int k,
                           int act, int dtype, int wdtype, const void *x, const void *W1,
                           const void *W3, const void *W2, const void *b1,
                           const void *b2, const float *s1, const float *s3, const float *s2,
                           int F_sh, const void *S1, const void *S3,
                           const void *S2, const int *topk_idx, const double *topk_w,
                           const unsigned char *drop_mask, double *y, double *slots,
                           double *shared_out)
{
    orc_layer_ctx c;
    c.d = d; c.F = F; c.E = E; c.k = k; c.act = act; c.dtype = dtype; c.wdtype = wdtype;
    c.s1 = s1; c.s3 = s3; c.s2 = s2;
    c.x = x; c.W1 = W1; c.W3 = W3; c.W2 = W2; c.b1 = b1; c.b2 = b2;
    c.F_sh = F_sh; c.S1 = F_sh > 0 ? S1 : NULL; c.S3 = S3; c.S2 = S2;
    c.topk_idx = topk_idx; c.topk_w = topk_w; c.drop_mask = drop_mask;
    c.tokens = tokens; c.y = y; c.slots = slots; c.shared_out = shared_out;
    orc_parallel(ntok, orc_layer_range, &c);
}

void oracle_layer_tokens(int ntok, const int *tokens, int d, int F, int E, int k,
                         int act, int dtype, const void *x, const void *W1,
                         const void *W3, const void *W2, const void *b1,
                         const void *b2, int F_sh, const void *S1, const void *S3,
                         const void *S2, const int *topk_idx, const double *topk_w,
                         const unsigned char *drop_mask, double *y, double *slots,
                         double *shared_out)
{
    oracle_layer_tokens_q(ntok, tokens, d, F, E, k, act, dtype, dtype, x, W1, W3, W2, b1, b2,
                          NULL, NULL, NULL, F_sh, S1, S3, S2, topk_idx, topk_w, drop_mask, y,
                          slots, shared_out);
}

/* ---------------------------------------------------------- step 10: aux */
/* [A]: aux = E * sum_e f_e * P_e with f_e = counts_pre[e] / T (top-k counts,
 * before drops) and P_e = mean over tokens of probs[t,e]. */
double oracle_aux_loss(int T, int E, const int *counts_pre, const double *probs)
{
    double aux = 0.0;
    for (int e = 0; e < E; ++e) {
        double P = 0.0;
        for (int t = 0; t < T; ++t)
            P += probs[(size_t)t * E + e];
        P /= (double)T;
        double f = (double)counts_pre[e] / (double)T;
        aux += f * P;
    }
    return (double)E * aux;
}

/* ------------------------------------------- aux loss backward (router) */
/* The aux term enters the training loss as alpha * aux ("How Mixture of
 * Experts Works", "The Load Balancing Problem").  f_e = counts_pre[e] / T is
 * piecewise constant in the logits and carries no gradient; P_e = mean_t
 * p[t,e] does.  With g = grad_aux (dLoss/daux):
 *   d aux / d p[t,e] = E f_e / T
 *   softmax: d p[t,e] / d l[t,j] = p[t,e] (delta_ej - p[t,j])
 *            => g_l[t,j] = g (E/T) p[t,j] (f_j - sum_e f_e p[t,e])
 *   sigmoid: d p[t,e] / d l[t,e] = p[t,e] (1 - p[t,e])
 *            => g_l[t,j] = g (E/T) f_j p[t,j] (1 - p[t,j])
 * Each term is written out as the chain rule gives it. */
void oracle_aux_grad_logits(int T, int E, int scoring, const double *logits,
                            const int *counts_pre, double grad_aux, double *g_l)
{
    double *p = (double *)malloc(sizeof(double) * (size_t)E);
    double *dp = (double *)malloc(sizeof(double) * (size_t)E);
    for (int t = 0; t < T; ++t) {
        const double *l = logits + (size_t)t * E;
        if (scoring == ORC_SIGMOID) {
            for (int e = 0; e < E; ++e)
                p[e] = 1.0 / (1.0 + exp(-l[e]));
        } else {
            double m = l[0];
            for (int e = 1; e < E; ++e)
                if (l[e] > m)
                    m = l[e];
            double Z = 0.0;
            for (int e = 0; e < E; ++e)
                Z += exp(l[e] - m);
            for (int e = 0; e < E; ++e)
                p[e] = exp(l[e] - m) / Z;
        }
        for (int e = 0; e < E; ++e) /* d aux / d p[t,e] */
            dp[e] = grad_aux * (double)E * ((double)counts_pre[e] / (double)T) / (double)T;
        for (int j = 0; j < E; ++j) {
            double acc = 0.0;
            if (scoring == ORC_SIGMOID) {
                acc = dp[j] * p[j] * (1.0 - p[j]);
            } else {
                for (int e = 0; e < E; ++e)
                    acc += dp[e] * p[e] * ((e == j ? 1.0 : 0.0) - p[j]);
            }
            g_l[(size_t)t * E + j] = acc;
        }
    }
    free(p);
    free(dp);
}
