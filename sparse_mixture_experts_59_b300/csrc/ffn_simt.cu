// ffn_simt.cu -- fp32 grouped expert FFN on CUDA cores.
//
// The tensor cores have no fp32-in/fp32-out kind that keeps fp32 products
// (tf32 rounds the operands), so fp32 layers run their expert GEMMs here.
// Same maths and grouping as the tensor-core path: rows r of the expert-
// grouped activations belong to the expert whose segment [offsets[e],
// offsets[e+1]) holds them; an optional shared expert is one more group whose
// rows are the T tokens in order.
//   up   (SwiGLU, "Implementing a complete MoE layer"):  H = silu(A W1^T) * (A W3^T)
//   up   (GELU MLP, "How a sparse MoE layer works"):     H = gelu(A W1^T + b1)
//   down: Ys[perm_src[r]] = topk_w[perm_src[r]] * (H[r] W2^T + b2);  shared: Sh = H_sh S2^T
#include "common.cuh"
#include "kernels.cuh"
#include "launch.cuh"

namespace moe {

constexpr int kSimtBM = 64, kSimtBN = 64, kSimtBK = 16;

template <int MODE>
__global__ void __launch_bounds__(256) ffn_simt_kernel(SimtFfnArgs p) {
    __shared__ int s_start[kMaxExperts + 2];
    __shared__ __align__(16) float As[kSimtBK][kSimtBM + 4];
    __shared__ __align__(16) float Bs[kSimtBK][kSimtBN + 4];
    __shared__ __align__(16) float B2s[kSimtBK][kSimtBN + 4];

    const int nt_r = (p.N + kSimtBN - 1) / kSimtBN;
    const int nt_s = p.rows_sh > 0 ? (p.N_sh + kSimtBN - 1) / kSimtBN : 0;
    pdl_wait();
    pdl_trigger();
    group_tile_prefix(p.offsets, p.E, p.rows_sh, kSimtBM, nt_r, nt_s, s_start);
    const int G = p.E + (p.rows_sh > 0 ? 1 : 0);
    const int tile = blockIdx.x;
    if (tile >= s_start[G]) return;
    const int g = find_group(s_start, G, tile);
    const bool sh = (g == p.E);
    const int seg0 = sh ? 0 : p.offsets[g];
    const int rows = sh ? p.rows_sh : p.offsets[g + 1] - seg0;
    const int mt = (rows + kSimtBM - 1) / kSimtBM;
    const int local = tile - s_start[g];
    const int n0 = (local / mt) * kSimtBN;
    const int r0 = seg0 + (local % mt) * kSimtBM;
    const int r_end = seg0 + rows;
    const int N = sh ? p.N_sh : p.N;
    const int K = sh ? p.K_sh : p.K;
    const float* A = sh ? p.A_sh : p.A;
    const float* B = sh ? p.B_sh : p.B + (size_t)g * N * K;
    const float* B2 = (MODE == kModeSwiglu) ? (sh ? p.B2_sh : p.B2 + (size_t)g * N * K) : nullptr;

    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[4][4], acc2[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = acc2[i][j] = 0.f;

    for (int k0 = 0; k0 < K; k0 += kSimtBK) {
        for (int i = threadIdx.x; i < kSimtBM * kSimtBK; i += 256) {
            const int rr = i / kSimtBK, c = i % kSimtBK;
            const int gr = r0 + rr, gn = n0 + rr, gc = k0 + c;
            As[c][rr] = (gr < r_end && gc < K) ? A[(size_t)gr * K + gc] : 0.f;
            Bs[c][rr] = (gn < N && gc < K) ? B[(size_t)gn * K + gc] : 0.f;
            if (MODE == kModeSwiglu) B2s[c][rr] = (gn < N && gc < K) ? B2[(size_t)gn * K + gc] : 0.f;
        }
        block_sync();
#pragma unroll
        for (int kk = 0; kk < kSimtBK; ++kk) {
            const float4 a = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
            const float4 b = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
            const float av[4] = {a.x, a.y, a.z, a.w};
            const float bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
            if (MODE == kModeSwiglu) {
                const float4 b2 = *reinterpret_cast<const float4*>(&B2s[kk][tx * 4]);
                const float b2v[4] = {b2.x, b2.y, b2.z, b2.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc2[i][j] = fmaf(av[i], b2v[j], acc2[i][j]);
            }
        }
        block_sync();
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = r0 + ty * 4 + i;
        if (r >= r_end) continue;
        float* dst;
        float scale = 1.f;
        if (MODE == kModeDown) {
            if (sh) {
                dst = p.out_sh + (size_t)r * N;
            } else {
                const int a = p.perm_src[r];
                dst = p.out + (size_t)a * N;
                scale = p.gate_w[a];
            }
        } else {
            dst = (sh ? p.out_sh : p.out) + (size_t)r * N;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= N) continue;
            float v = acc[i][j];
            if (MODE == kModeSwiglu) {
                v = silu(v) * acc2[i][j];
            } else if (MODE == kModeGelu) {
                if (p.bias && !sh) v += p.bias[(size_t)g * N + n];
                v = gelu_erf(v);
            } else {
                if (p.bias && !sh) v += p.bias[(size_t)g * N + n];
                v *= scale;
            }
            dst[n] = v;
        }
    }
}

cudaError_t launch_ffn_simt(int mode, const SimtFfnArgs& p, int A_rows, cudaStream_t st) {
    const int nt_r = (p.N + kSimtBN - 1) / kSimtBN;
    const int nt_s = p.rows_sh > 0 ? (p.N_sh + kSimtBN - 1) / kSimtBN : 0;
    const long long blocks = ((long long)(A_rows + kSimtBM - 1) / kSimtBM + p.E) * nt_r +
                             (long long)((p.rows_sh + kSimtBM - 1) / kSimtBM) * nt_s;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    auto kernel = mode == kModeSwiglu ? ffn_simt_kernel<kModeSwiglu>
                : mode == kModeGelu ? ffn_simt_kernel<kModeGelu> : ffn_simt_kernel<kModeDown>;
    return launch_kernel(kernel, dim3((unsigned)blocks), dim3(256), 0, st, 1, p);
}

}  // namespace moe
