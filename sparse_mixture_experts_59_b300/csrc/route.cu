// route.cu -- router GEMM and the softmax / top-k / renormalisation step.
//
// "How Mixture of Experts Works", section "The Gating Mechanism": a bias-free
// linear router gives one logit per expert, softmax over all experts, top-k,
// and the kept probabilities renormalised to sum to 1.  "Mixture of Experts
// (MoE)", section "The router": scores = softmax(h @ W_r).  Ties in the top-k
// go to the lower expert index; selection is on the fp32 logits (softmax is
// monotone, so this is the same set without the ties that exp rounding can
// create).  P_e (mean probability per expert) feeds the aux loss of "Load
// balancing and expert collapse".
#include "common.cuh"
#include "kernels.cuh"
#include "launch.cuh"
#include "topk_warp.cuh"

namespace moe {

// ----------------------------------------------------------------------------
// logits[T,E] = x[T,d] . Wr[E,d]^T (+ bias[E]) on CUDA cores, fp32 accumulate.
// 64x64 output tile per 256-thread block, 4x4 outputs per thread, K step 16.
// Used for fp32 layers and for routers too narrow for a tensor-core tile.
template <typename T>
__global__ void __launch_bounds__(256)
router_logits_simt(const T* __restrict__ x, const T* __restrict__ Wr,
                   const float* __restrict__ bias, float* __restrict__ logits,
                   int Ttok, int d, int E) {
    constexpr int BM = 64, BN = 64, BK = 16;
    __shared__ __align__(16) float Xs[BK][BM + 4];
    __shared__ __align__(16) float Ws[BK][BN + 4];
    const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    pdl_wait();
    pdl_trigger();
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

    for (int k0 = 0; k0 < d; k0 += BK) {
        for (int i = threadIdx.x; i < BM * BK; i += 256) {
            const int r = i / BK, c = i % BK;
            const int gr = m0 + r, gc = k0 + c;
            Xs[c][r] = (gr < Ttok && gc < d) ? Elem<T>::load(x + (size_t)gr * d + gc) : 0.f;
            const int ge = n0 + r;
            Ws[c][r] = (ge < E && gc < d) ? Elem<T>::load(Wr + (size_t)ge * d + gc) : 0.f;
        }
        block_sync();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            const float4 a = *reinterpret_cast<const float4*>(&Xs[kk][ty * 4]);
            const float4 b = *reinterpret_cast<const float4*>(&Ws[kk][tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w};
            const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        block_sync();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int t = m0 + ty * 4 + i;
        if (t >= Ttok) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int e = n0 + tx * 4 + j;
            if (e < E) logits[(size_t)t * E + e] = acc[i][j] + (bias ? bias[e] : 0.f);
        }
    }
}

// ----------------------------------------------------------------------------
// Softmax / top-k / renormalise: one warp per token, each lane holding the
// logits of experts lane, lane+32, ... (up to 8 per lane, E <= 256).
// Per-block sums of p[t,e] go to prob_part[block][e]; the last block to finish
// adds the partials in block order (deterministic) into prob_mean[e] / T.
template <int VPL>
__global__ void __launch_bounds__(256)
router_topk_kernel(const float* part, int nsplit, const float* __restrict__ bias,
                   float* logits, int Ttok, int E, int k, int scoring, int renorm,
                   int* __restrict__ topk_idx, float* __restrict__ topk_w,
                   float* __restrict__ prob_part, float* __restrict__ prob_mean,
                   int* __restrict__ done_counter) {
    constexpr int WARPS = 8;
    __shared__ float s_psum[WARPS][kMaxExperts];
    __shared__ int s_last;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool want_p = prob_mean != nullptr;
    if (want_p)
        for (int e = lane; e < E; e += 32) s_psum[warp][e] = 0.f;
    pdl_wait();
    pdl_trigger();

    for (int t = blockIdx.x * WARPS + warp; t < Ttok; t += gridDim.x * WARPS) {
        float l[VPL];
        const bool write_logits = (nsplit > 1) || (bias != nullptr) || (part != logits);
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            const int e = lane + 32 * j;
            if (e < E) {
                // the split-K partials, 8 loads in flight: accumulator a takes
                // splits a, a+8, ...; combined in a fixed order (deterministic)
                float acc[8];
#pragma unroll
                for (int a = 0; a < 8; ++a) acc[a] = 0.f;
                const size_t stride = (size_t)Ttok * E;
                const float* src = part + (size_t)t * E + e;
                int sp = 0;
                for (; sp + 8 <= nsplit; sp += 8) {
#pragma unroll
                    for (int a = 0; a < 8; ++a) acc[a] += src[(size_t)(sp + a) * stride];
                }
                for (int a = 0; sp + a < nsplit; ++a) acc[a] += src[(size_t)(sp + a) * stride];
                float v = ((acc[0] + acc[1]) + (acc[2] + acc[3])) +
                          ((acc[4] + acc[5]) + (acc[6] + acc[7]));
                if (bias) v += bias[e];
                if (write_logits) logits[(size_t)t * E + e] = v;
                l[j] = v;
            } else {
                l[j] = -INFINITY;
            }
        }
        float ex[VPL], inv;
        int my_idx;
        float my_w;
        route_token_warp<VPL>(l, E, k, scoring, renorm, lane, ex, inv, my_idx, my_w);
        if (want_p) {
#pragma unroll
            for (int j = 0; j < VPL; ++j)
                if (lane + 32 * j < E) s_psum[warp][lane + 32 * j] += ex[j] * inv;
        }
        if (lane < k) {
            topk_idx[(size_t)t * k + lane] = my_idx;
            topk_w[(size_t)t * k + lane] = my_w;
        }
    }
    if (!want_p) return;
    block_sync();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) s += s_psum[w][e];
        prob_part[(size_t)blockIdx.x * E + e] = s;
    }
    __threadfence();
    block_sync();
    if (threadIdx.x == 0) s_last = (atomicAdd(done_counter, 1) == (int)gridDim.x - 1);
    block_sync();
    if (!s_last) return;
    __threadfence();
    // column sums of prob_part[nblocks][E], in a fixed order so that the
    // result repeats exactly.  One block reads all nblocks x E partials (up to
    // 592 x 256), so the loads go 16 bytes and 8 at a time: with E a multiple
    // of 4, thread t adds rows g, g+G, ... (g = t / C, G = 256 / C groups) of
    // the 4 experts of float4 column t % C (C = E / 4), then the groups are
    // added in order; otherwise one expert per thread the same way.
    float* s_col = &s_psum[0][0];                  // reuse: [G][E] partial columns
    const int nb = (int)gridDim.x;
    int G;
    if ((E & 3) == 0) {
        const int C = E / 4;
        G = (int)blockDim.x / C > 0 ? (int)blockDim.x / C : 1;
        if ((int)threadIdx.x < G * C) {
            const int c = threadIdx.x % C, g = threadIdx.x / C;
            const float4* src = reinterpret_cast<const float4*>(prob_part) + c;
            float4 a[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) a[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            int b = g;
            for (; b + 7 * G < nb; b += 8 * G) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 v = ld_cg(src + (size_t)(b + j * G) * C);
                    a[j].x += v.x; a[j].y += v.y; a[j].z += v.z; a[j].w += v.w;
                }
            }
            for (; b < nb; b += G) {
                const float4 v = ld_cg(src + (size_t)b * C);
                a[0].x += v.x; a[0].y += v.y; a[0].z += v.z; a[0].w += v.w;
            }
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                acc.x += a[j].x; acc.y += a[j].y; acc.z += a[j].z; acc.w += a[j].w;
            }
            float* dst = s_col + g * E + 4 * c;
            dst[0] = acc.x; dst[1] = acc.y; dst[2] = acc.z; dst[3] = acc.w;
        }
    } else {
        G = (int)blockDim.x / E > 0 ? (int)blockDim.x / E : 1;
        if ((int)threadIdx.x < G * E) {
            const int e = threadIdx.x % E, g = threadIdx.x / E;
            float a8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};   // 8 loads in flight
            int b = g;
            for (; b + 7 * G < nb; b += 8 * G)
#pragma unroll
                for (int j = 0; j < 8; ++j) a8[j] += ld_cg(prob_part + (size_t)(b + j * G) * E + e);
            for (; b < nb; b += G) a8[0] += ld_cg(prob_part + (size_t)b * E + e);
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) acc += a8[j];
            s_col[g * E + e] = acc;
        }
    }
    block_sync();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float acc = 0.f;
        for (int g = 0; g < G; ++g) acc += s_col[g * E + e];
        prob_mean[e] = acc / (float)Ttok;
    }
    if (threadIdx.x == 0) *done_counter = 0;   // leave the workspace reusable
}

// ---------------------------------------------------------------- launchers
cudaError_t launch_router_logits_simt(int dtype, const void* x, const void* Wr, const float* bias,
                                      float* logits, int T, int d, int E, cudaStream_t st) {
    dim3 grid((T + 63) / 64, (E + 63) / 64);
    if (dtype == MOE_F32)
        return launch_kernel(router_logits_simt<float>, grid, dim3(256), 0, st, 1,
                             (const float*)x, (const float*)Wr, bias, logits, T, d, E);
    return launch_kernel(router_logits_simt<__nv_bfloat16>, grid, dim3(256), 0, st, 1,
                         (const __nv_bfloat16*)x, (const __nv_bfloat16*)Wr, bias, logits, T, d, E);
}

cudaError_t launch_router_topk(const float* part, int nsplit, const float* bias, float* logits,
                               int T, int E, int k, int scoring, int renorm, int* topk_idx,
                               float* topk_w,
                               float* prob_part, float* prob_mean, int* done, int nblocks,
                               cudaStream_t st) {
    const int vpl = (E + 31) / 32;
    auto kernel = vpl <= 1 ? router_topk_kernel<1>
                : vpl <= 2 ? router_topk_kernel<2>
                : vpl <= 4 ? router_topk_kernel<4> : router_topk_kernel<8>;
    return launch_kernel(kernel, dim3(nblocks), dim3(256), 0, st, 1, part, nsplit, bias, logits, T,
                         E, k, scoring, renorm, topk_idx, topk_w, prob_part, prob_mean, done);
}

}  // namespace moe
