// front_small.cu -- router GEMM, softmax / top-k / renormalisation and the
// whole dispatch of a decode-sized batch in one launch.
//
// The maths is that of route.cu and dispatch.cu ("How Mixture of Experts
// Works", sections "The Gating Mechanism" and "The Capacity Factor", and the
// MoELayer listing's flattened (token, slot) order; "Mixture-of-Experts
// Routing", section "How a sparse MoE layer works": the first `capacity`
// assignments in token order are kept).  At a few dozen tokens those four
// kernels are each a launch and a few dependent memory round trips with
// almost no work, ~25 us together; here:
//   every CTA  computes fp32 partial logits x[:, K-slice] . Wr[:, K-slice]^T
//              for all T x E outputs (CUDA cores; T*E <= 2048) and writes
//              them to its slot;
//   the last   CTA to finish (an atomic ticket, no waiting) adds the slots in
//              a fixed order (deterministic), adds the logit bias, routes
//              every token (one warp per token), sums P_e in a fixed order,
//              and runs the dispatch in shared memory: per-expert running counts
//              in token order give the ranks, then capacity, offsets, dest /
//              perm_src / drop mask and the aux loss.  It clears the ticket
//              for the next call.
// Measured at T=32 (Mixtral decode, ncu): four launches of 23 us together
// became one of ~11 us.
// Used by the layer call when T*k <= 512 and T*E <= 2048 (T <= 256); the
// router stage call uses the same kernel without the dispatch part, so both
// give the same logits bit for bit.
#include "common.cuh"
#include "kernels.cuh"
#include "launch.cuh"
#include "topk_warp.cuh"

namespace moe {

namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxOut = kFrontMaxTE / kThreads;    // partial outputs per thread
constexpr int kMaxSplits = 32;
constexpr int kRawBytes = 44 * 1024;

// phase 1: [rows][kc + 4] fp32 chunks of x and Wr, kc a multiple of 32 sized
// so that the T + E rows fit (T * E <= 2048 with T, E <= 256 bounds T + E by
// 256 + 2048 / 256: kc >= 32 always; decode shapes take a K-slice in one chunk)
static_assert((kFrontMaxT + kFrontMaxTE / kFrontMaxT) * 36 * 4 <= kRawBytes, "phase-1 shared memory");
// phase 2: logits, P_e partials, slots and ranks
static_assert(2 * kFrontMaxTE * 4 + 2 * kFrontMaxA * 4 + 3 * kMaxExperts * 4 <= kRawBytes,
              "phase-2 shared memory");

template <typename Tin, int VPL>
__global__ void __launch_bounds__(kThreads)
front_small_kernel(const Tin* __restrict__ x, const Tin* __restrict__ Wr,
                   const float* __restrict__ bias, int Ttok, int d, int E, int k, int scoring,
                   int renorm, int dispatch, long long cap, int ks, float* part, int* ticket,
                   float* __restrict__ logits, int* __restrict__ topk_idx,
                   float* __restrict__ topk_w, float* __restrict__ prob_mean,
                   int* __restrict__ counts_pre, int* __restrict__ counts_kept,
                   int* __restrict__ offsets, int* __restrict__ perm_src, int* __restrict__ dest,
                   unsigned char* __restrict__ drop_mask, float* __restrict__ stats) {
    __shared__ __align__(16) unsigned char s_raw[kRawBytes];
    __shared__ int s_last;
    __shared__ int s_wsum[kWarps];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int TE = Ttok * E;
    // x may be the previous kernel's output, and the outputs below may still
    // be read by the previous call's kernels
    pdl_wait();
    pdl_trigger();

    // ---------------------------------------------- phase 1: partial logits
    {
        int kcs = (kRawBytes / 4 / (Ttok + E) - 4) / 32 * 32;   // chunk (K values)
        if (kcs > ks) kcs = ks;
        // rows padded by 4 floats: 16-byte aligned for float4 reads, and
        // consecutive rows start 4 banks apart (conflict-free float4 reads)
        const int ld = kcs + 4;
        float* xs = reinterpret_cast<float*>(s_raw);            // [Ttok][ld]
        float* ws = xs + Ttok * ld;                              // [E][ld]
        const int k0 = blockIdx.x * ks, k1 = min(d, k0 + ks);
        float acc[kMaxOut];
#pragma unroll
        for (int j = 0; j < kMaxOut; ++j) acc[j] = 0.f;
        // rows 0..T-1 of the chunk are x, rows T..T+E-1 are Wr (ws follows xs);
        // 16-byte loads (d % 8 == 0 and 32-aligned slices keep them whole and
        // aligned), all issued before the shared-memory stores
        constexpr int VEC = 16 / (int)sizeof(Tin);
        const int cpr = kcs / VEC;                              // loads per row
        for (int kc = k0; kc < k1; kc += kcs) {
            for (int i = tid; i < (Ttok + E) * cpr; i += kThreads) {
                const int r = i / cpr, cc = (i % cpr) * VEC, kg = kc + cc;
                float* dst = xs + r * ld + cc;
                if (kg < k1) {
                    const Tin* src = r < Ttok ? x + (size_t)r * d + kg
                                              : Wr + (size_t)(r - Ttok) * d + kg;
                    const uint4 v = __ldg(reinterpret_cast<const uint4*>(src));
                    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
                    if constexpr (VEC == 8) {                   // bf16 pairs
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            dst[2 * q] = __uint_as_float(w4[q] << 16);
                            dst[2 * q + 1] = __uint_as_float(w4[q] & 0xffff0000u);
                        }
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q) dst[q] = __uint_as_float(w4[q]);
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < VEC; ++q) dst[q] = 0.f;
                }
            }
            block_sync();
#pragma unroll
            for (int j = 0; j < kMaxOut; ++j) {
                const int o = tid + j * kThreads;
                if (o < TE) {
                    const float* xr = xs + (o / E) * ld;
                    const float* wr = ws + (o % E) * ld;
                    // four independent chains over float4 reads (kcs is a
                    // multiple of 32), added in a fixed order
                    const float4* x4 = reinterpret_cast<const float4*>(xr);
                    const float4* w4 = reinterpret_cast<const float4*>(wr);
                    float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
                    for (int c = 0; c < kcs / 4; ++c) {
                        const float4 a = x4[c], b = w4[c];
                        s4[0] = fmaf(a.x, b.x, s4[0]);
                        s4[1] = fmaf(a.y, b.y, s4[1]);
                        s4[2] = fmaf(a.z, b.z, s4[2]);
                        s4[3] = fmaf(a.w, b.w, s4[3]);
                    }
                    acc[j] += (s4[0] + s4[1]) + (s4[2] + s4[3]);
                }
            }
            block_sync();
        }
        float* mine = part + (size_t)blockIdx.x * TE;
#pragma unroll
        for (int j = 0; j < kMaxOut; ++j) {
            const int o = tid + j * kThreads;
            if (o < TE) mine[o] = acc[j];
        }
    }
    // the block's partials, then one fence and the ticket (the fence of the
    // thread that takes the ticket orders the whole block's writes before it)
    block_sync();
    if (tid == 0) {
        __threadfence();
        s_last = (atomicAdd(ticket, 1) == (int)gridDim.x - 1);
        if (s_last) __threadfence();
    }
    block_sync();
    if (!s_last) return;

    // ---------------------------------------------- phase 2 (last CTA only)
    float* s_logit = reinterpret_cast<float*>(s_raw);               // [TE]
    float* s_prob = s_logit + kFrontMaxTE;                           // [TE] p(t, e)
    int* s_idx = reinterpret_cast<int*>(s_prob + kFrontMaxTE);       // [A]
    int* s_rank = s_idx + kFrontMaxA;                                // [A]
    int* s_cnt = s_rank + kFrontMaxA;                                // [E]
    int* s_off = s_cnt + kMaxExperts;                                // [E]
    float* s_pm = reinterpret_cast<float*>(s_off + kMaxExperts);     // [E]
    const int A = Ttok * k;
    const int S = (int)gridDim.x;

    // logits: every CTA slot loaded at once, then added in a fixed tree order
    for (int o = tid; o < TE; o += kThreads) {
        float v32[kMaxSplits];
#pragma unroll
        for (int a = 0; a < kMaxSplits; ++a)
            v32[a] = a < S ? ld_cg(part + (size_t)a * TE + o) : 0.f;
#pragma unroll
        for (int w = kMaxSplits / 2; w > 0; w >>= 1)
#pragma unroll
            for (int a = 0; a < w; ++a) v32[a] += v32[a + w];
        float v = v32[0];
        if (bias) v += bias[o % E];
        s_logit[o] = v;
        logits[o] = v;
    }
    block_sync();

    // routing: one warp per token
    for (int t = warp; t < Ttok; t += kWarps) {
        float l[VPL];
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            const int e = lane + 32 * j;
            l[j] = e < E ? s_logit[t * E + e] : -INFINITY;
        }
        float ex[VPL], inv;
        int my_idx;
        float my_w;
        route_token_warp<VPL>(l, E, k, scoring, renorm, lane, ex, inv, my_idx, my_w);
#pragma unroll
        for (int j = 0; j < VPL; ++j)
            if (lane + 32 * j < E) s_prob[t * E + lane + 32 * j] = ex[j] * inv;
        if (lane < k) {
            topk_idx[(size_t)t * k + lane] = my_idx;
            topk_w[(size_t)t * k + lane] = my_w;
            s_idx[t * k + lane] = my_idx;
        }
    }
    block_sync();

    // P_e (four token chains, added in a fixed order), then per-expert ranks
    // in flattened order
    if (tid < E) {
        float a4[4] = {0.f, 0.f, 0.f, 0.f};      // four chains, fixed order
        int t = 0;
        for (; t + 4 <= Ttok; t += 4)
#pragma unroll
            for (int q = 0; q < 4; ++q) a4[q] += s_prob[(t + q) * E + tid];
#pragma unroll
        for (int q = 0; q < 3; ++q)
            if (t + q < Ttok) a4[q] += s_prob[(t + q) * E + tid];
        const float acc = (a4[0] + a4[1]) + (a4[2] + a4[3]);
        s_pm[tid] = acc / (float)Ttok;
        if (prob_mean) prob_mean[tid] = s_pm[tid];
    }
    if (!dispatch) {                       // the router stage alone
        if (tid == 0) *ticket = 0;
        return;
    }
    if (tid < E) {
        int c = 0;
        for (int a = 0; a < A; ++a)
            if (s_idx[a] == tid) s_rank[a] = c++;
        s_cnt[tid] = c;
    }
    block_sync();

    // capacity, counts and offsets (exclusive scan of the kept counts)
    int total = 0, kept = 0;
    if (tid < E) {
        total = s_cnt[tid];
        kept = (cap >= 0 && (long long)total > cap) ? (int)cap : total;
        counts_pre[tid] = total;
        counts_kept[tid] = kept;
    }
    int incl = kept;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) s_wsum[warp] = incl;
    block_sync();
    int wbase = 0;
    for (int w = 0; w < warp; ++w) wbase += s_wsum[w];
    if (tid < E) {
        s_off[tid] = wbase + incl - kept;
        offsets[tid] = wbase + incl - kept;
    }
    if (tid == E - 1) offsets[E] = wbase + incl;
    block_sync();

    // dest / perm_src / drop mask
    for (int a = tid; a < A; a += kThreads) {
        const int e = s_idx[a], r = s_rank[a];
        if (cap < 0 || (long long)r < cap) {
            const int dst = s_off[e] + r;
            dest[a] = dst;
            perm_src[dst] = a;
            drop_mask[a] = 0;
        } else {
            dest[a] = -1;
            drop_mask[a] = 1;
        }
    }
    if (tid == 0) {
        int R = 0;
        for (int w = 0; w < kWarps; ++w) R += s_wsum[w];
        float aux = 0.f;
        for (int e = 0; e < E; ++e) aux += ((float)s_cnt[e] / (float)Ttok) * s_pm[e];
        stats[0] = aux * (float)E;
        stats[1] = A > 0 ? (float)(A - R) / (float)A : 0.f;
        *ticket = 0;                       // leave the workspace reusable
    }
}

template <typename Tin>
cudaError_t launch_typed(const FrontSmallArgs& a, int vpl, cudaStream_t st) {
    auto kernel = vpl <= 1 ? front_small_kernel<Tin, 1>
                : vpl <= 2 ? front_small_kernel<Tin, 2>
                : vpl <= 4 ? front_small_kernel<Tin, 4> : front_small_kernel<Tin, 8>;
    return launch_kernel(kernel, dim3(a.splits), dim3(kThreads), 0, st, 1,
                         (const Tin*)a.x, (const Tin*)a.Wr, a.bias, a.T, a.d, a.E, a.k, a.scoring,
                         a.renorm, a.dispatch, a.cap, a.ks, a.part, a.ticket, a.logits, a.topk_idx, a.topk_w,
                         a.prob_mean, a.counts_pre, a.counts_kept, a.offsets, a.perm_src, a.dest,
                         a.drop_mask, a.stats);
}

}  // namespace

FrontSmallPlan front_small_plan(int T, int d, int E, int k) {
    FrontSmallPlan p{};
    p.ok = T >= 1 && T <= kFrontMaxT && E <= kFrontMaxE && (long long)T * k <= kFrontMaxA &&
           (long long)T * E <= kFrontMaxTE;
    // K-slices of at least 128 values, at most 32 of them
    int ks = (d + kMaxSplits - 1) / kMaxSplits;
    ks = (ks + 31) / 32 * 32;
    if (ks < 128) ks = 128;
    p.ks = ks;
    p.splits = (d + ks - 1) / ks;
    return p;
}

cudaError_t launch_front_small(int dtype, const FrontSmallArgs& a, cudaStream_t st) {
    const int vpl = (a.E + 31) / 32;
    return dtype == MOE_F32 ? launch_typed<float>(a, vpl, st)
                            : launch_typed<__nv_bfloat16>(a, vpl, st);
}

}  // namespace moe
