// topk_warp.cuh -- one token's scores, top-k and gate weights, computed by a
// warp ("How Mixture of Experts Works", section "The Gating Mechanism":
// softmax over all experts, top-k, the kept probabilities renormalised to sum
// to 1; "Mixture-of-Experts Routing": ties go to the lower expert index).
// Lane L holds the logits of experts L, L+32, ... (VPL values, E <= 32*VPL).
#pragma once

#include "common.cuh"

namespace moe {

// In: l[j] = logit of expert lane + 32 j (-inf past E).  Out: ex[j] and inv,
// with p(expert) = ex[j] * inv (softmax: ex = exp(l - max), inv = 1 / sum;
// sigmoid: ex = sigmoid(l), inv = 1); on lanes s < k, my_idx / my_w = the
// s-th selected expert (logit descending, index ascending) and its gate
// weight (renormalised over the k kept, or the score itself).
template <int VPL>
__device__ __forceinline__ void route_token_warp(const float (&l)[VPL], int E, int k, int scoring,
                                                 int renorm, int lane, float (&ex)[VPL],
                                                 float& inv, int& my_idx, float& my_w) {
    float m = l[0];
#pragma unroll
    for (int j = 1; j < VPL; ++j) m = fmaxf(m, l[j]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.f;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
        const bool ok = lane + 32 * j < E;
        ex[j] = !ok ? 0.f
              : scoring == MOE_SCORE_SIGMOID ? 1.f / (1.f + expf(-l[j])) : expf(l[j] - m);
        z += ex[j];
    }
    inv = 1.f;
    if (scoring != MOE_SCORE_SIGMOID) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        inv = 1.f / z;
    }
    // top-k by repeated warp arg-max over the logits; (value desc, index asc)
    unsigned taken = 0;       // bit j: lane's value j already selected
    float kept_ex = 0.f, my_ex = 0.f;
    my_idx = -1;
    for (int s = 0; s < k; ++s) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            const int e = lane + 32 * j;
            if (e < E && !(taken & (1u << j)) && (l[j] > bv || bi == 0x7fffffff)) {
                bv = l[j];
                bi = e;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
        }
        // owner marks it; everyone learns the winner's ex
        const int owner = bi & 31, jj = bi >> 5;
        float wex = 0.f;
#pragma unroll
        for (int j = 0; j < VPL; ++j)
            if (j == jj) wex = ex[j];
        wex = __shfl_sync(0xffffffffu, wex, owner);
        if (lane == owner) taken |= 1u << jj;
        kept_ex += wex;
        if (lane == s) { my_idx = bi; my_ex = wex; }
    }
    my_w = renorm ? my_ex / kept_ex : my_ex * inv;
}

}  // namespace moe
