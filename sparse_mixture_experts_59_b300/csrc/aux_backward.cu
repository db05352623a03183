// aux_backward.cu -- backward of the aux loss through the router.
//
// "How Mixture of Experts Works", section "The Load Balancing Problem": the
// training loss is task_loss + alpha * aux with aux = E * sum_e f_e P_e.
// f_e = counts_pre[e] / T is piecewise constant in the router logits and
// carries no gradient; P_e = mean_t p[t,e] does.  With g = dLoss/daux:
//   softmax scores: g_l[t,j] = g (E/T) p[t,j] (f_j - sum_e f_e p[t,e])
//   sigmoid scores: g_l[t,j] = g (E/T) f_j p[t,j] (1 - p[t,j])
//   grad_Wr = g_l^T x      [E, d]
//   grad_x  = g_l Wr       [T, d]
// The logit gradient is one warp per token (as the forward top-k); the two
// products run on CUDA cores in fp32, a strided 64x64-tile GEMM.
#include "common.cuh"
#include "kernels.cuh"
#include "launch.cuh"

namespace moe {

template <int VPL>
__global__ void __launch_bounds__(256)
aux_grad_logits_kernel(const float* __restrict__ logits, const int* __restrict__ counts_pre,
                       int Ttok, int E, int scoring, float scale, float* __restrict__ g_l) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    pdl_trigger();
    const float invT = 1.f / (float)Ttok;
    for (int t = blockIdx.x * 8 + warp; t < Ttok; t += gridDim.x * 8) {
        float l[VPL], f[VPL], p[VPL];
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            const int e = lane + 32 * j;
            l[j] = (e < E) ? logits[(size_t)t * E + e] : -INFINITY;
            f[j] = (e < E) ? (float)counts_pre[e] * invT : 0.f;
        }
        if (scoring == MOE_SCORE_SIGMOID) {
#pragma unroll
            for (int j = 0; j < VPL; ++j) {
                const int e = lane + 32 * j;
                if (e < E) {
                    const float s = 1.f / (1.f + expf(-l[j]));
                    g_l[(size_t)t * E + e] = scale * f[j] * s * (1.f - s);
                }
            }
            continue;
        }
        float m = l[0];
#pragma unroll
        for (int j = 1; j < VPL; ++j) m = fmaxf(m, l[j]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float z = 0.f;
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            p[j] = (lane + 32 * j < E) ? expf(l[j] - m) : 0.f;
            z += p[j];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
        const float inv = 1.f / z;
        float c = 0.f;                       // sum_e f_e p[t,e]
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            p[j] *= inv;
            c += f[j] * p[j];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
            const int e = lane + 32 * j;
            if (e < E) g_l[(size_t)t * E + e] = scale * p[j] * (f[j] - c);
        }
    }
}

// C[M,N] = sum_k A(m,k) B(k,n), A(m,k) = A[m*sam + k*sak], B(k,n) = B[k*sbk + n*sbn];
// fp32 accumulate, 64x64 tile per 256-thread block, 4x4 outputs per thread.
template <typename TA, typename TB>
__global__ void __launch_bounds__(256)
gemm_strided_simt(int M, int N, int K, const TA* __restrict__ A, long long sam, long long sak,
                  const TB* __restrict__ B, long long sbk, long long sbn, float* __restrict__ C,
                  long long ldc) {
    constexpr int BM = 64, BN = 64, BK = 16;
    __shared__ __align__(16) float As[BK][BM + 4];
    __shared__ __align__(16) float Bs[BK][BN + 4];
    const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    pdl_wait();
    pdl_trigger();
    float acc[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    for (int k0 = 0; k0 < K; k0 += BK) {
        for (int i = threadIdx.x; i < BM * BK; i += 256) {
            const int r = i / BK, c = i % BK;
            const int gm = m0 + r, gk = k0 + c, gn = n0 + r;
            As[c][r] = (gm < M && gk < K) ? Elem<TA>::load(A + gm * sam + gk * sak) : 0.f;
            Bs[c][r] = (gn < N && gk < K) ? Elem<TB>::load(B + gk * sbk + gn * sbn) : 0.f;
        }
        block_sync();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            const float4 a = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
            const float4 b = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
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
        const int m = m0 + ty * 4 + i;
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n < N) C[m * ldc + n] = acc[i][j];
        }
    }
}

cudaError_t launch_aux_backward(int dtype, int scoring, const void* x, const void* Wr,
                                const float* logits, const int* counts_pre, float grad_aux, int T,
                                int d, int E, float* g_l, float* g_Wr, float* g_x, int num_sms,
                                cudaStream_t st) {
    const int vpl = (E + 31) / 32;
    auto kernel = vpl <= 1 ? aux_grad_logits_kernel<1>
                : vpl <= 2 ? aux_grad_logits_kernel<2>
                : vpl <= 4 ? aux_grad_logits_kernel<4> : aux_grad_logits_kernel<8>;
    int blocks = (T + 7) / 8;
    if (blocks > num_sms * 8) blocks = num_sms * 8;
    if (blocks < 1) blocks = 1;
    const float scale = grad_aux * (float)E / (float)T;
    cudaError_t err = launch_kernel(kernel, dim3(blocks), dim3(256), 0, st, 1, logits, counts_pre,
                                    T, E, scoring, scale, g_l);
    if (err != cudaSuccess) return err;
    if (g_Wr) {     // [E, d] = g_l^T [E, T] x [T, d]
        const dim3 grid((E + 63) / 64, (d + 63) / 64);
        if (dtype == MOE_F32)
            err = launch_kernel(gemm_strided_simt<float, float>, grid, dim3(256), 0, st, 1, E, d, T,
                                (const float*)g_l, 1LL, (long long)E, (const float*)x, (long long)d,
                                1LL, g_Wr, (long long)d);
        else
            err = launch_kernel(gemm_strided_simt<float, __nv_bfloat16>, grid, dim3(256), 0, st, 1,
                                E, d, T, (const float*)g_l, 1LL, (long long)E,
                                (const __nv_bfloat16*)x, (long long)d, 1LL, g_Wr, (long long)d);
        if (err != cudaSuccess) return err;
    }
    if (g_x) {      // [T, d] = g_l [T, E] x Wr [E, d]
        const dim3 grid((T + 63) / 64, (d + 63) / 64);
        if (dtype == MOE_F32)
            err = launch_kernel(gemm_strided_simt<float, float>, grid, dim3(256), 0, st, 1, T, d, E,
                                (const float*)g_l, (long long)E, 1LL, (const float*)Wr,
                                (long long)d, 1LL, g_x, (long long)d);
        else
            err = launch_kernel(gemm_strided_simt<float, __nv_bfloat16>, grid, dim3(256), 0, st, 1,
                                T, d, E, (const float*)g_l, (long long)E, 1LL,
                                (const __nv_bfloat16*)Wr, (long long)d, 1LL, g_x, (long long)d);
    }
    return err;
}

}  // namespace moe
