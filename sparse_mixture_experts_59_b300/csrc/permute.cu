// permute.cu -- gather of token rows into expert-grouped order, and the
// gate-weighted combine back into token order with the residual.
//
// "How Mixture of Experts Works", MoELayer listing: expert_input =
// hidden_states[token_indices] (the gather) and output.index_add_ of the
// weight-scaled expert outputs (the combine); "Mixture-of-Experts Routing",
// "How a sparse MoE layer works": the weighted sum is added through the
// residual.  Both kernels move whole rows with 16-byte vectors; they are
// bandwidth-bound and carry no arithmetic beyond the fp32 sum of the combine.
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.cuh"
#include "launch.cuh"

namespace moe {

// Xp[r] = x[perm_src[r] / k] for r < R = offsets[E] (read on the device).
// One warp per row, 16-byte vectors.
__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint4* __restrict__ x, const int* __restrict__ perm_src,
                   const int* __restrict__ offsets, int E, int k, int Ttok, int vec_per_row,
                   uint4* __restrict__ Xp, int* __restrict__ status) {
    pdl_wait();
    pdl_trigger();
    const int R = offsets[E];
    const int warps = (gridDim.x * blockDim.x) >> 5;
    const int lane = threadIdx.x & 31;
    for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < R; r += warps) {
        const int a = perm_src[r];
        const int t = a / k;
        if (a < 0 || t >= Ttok) {
            if (lane == 0) raise_error(status, MOE_ERR_DEVICE_BOUNDS);
            continue;
        }
        const uint4* src = x + (size_t)t * vec_per_row;
        uint4* dst = Xp + (size_t)r * vec_per_row;
        for (int v = lane; v < vec_per_row; v += 32) dst[v] = __ldg(src + v);
    }
}

// As gather_rows_kernel, converting bf16 x to f16 on the way (the token
// operand of the FP8-weight expert GEMMs, whose MMAs take f16).
__global__ void __launch_bounds__(256)
gather_rows_f16_kernel(const uint4* __restrict__ x, const int* __restrict__ perm_src,
                       const int* __restrict__ offsets, int E, int k, int Ttok, int vec_per_row,
                       uint4* __restrict__ Xp, int* __restrict__ status) {
    pdl_wait();
    pdl_trigger();
    const int R = offsets[E];
    const int warps = (gridDim.x * blockDim.x) >> 5;
    const int lane = threadIdx.x & 31;
    for (int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < R; r += warps) {
        const int a = perm_src[r];
        const int t = a / k;
        if (a < 0 || t >= Ttok) {
            if (lane == 0) raise_error(status, MOE_ERR_DEVICE_BOUNDS);
            continue;
        }
        const uint4* src = x + (size_t)t * vec_per_row;
        uint4* dst = Xp + (size_t)r * vec_per_row;
        for (int v = lane; v < vec_per_row; v += 32) {
            float f[8];
            unpack16(__ldg(src + v), f);
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __half2 h = __floats2half2_rn(f[2 * j], f[2 * j + 1]);
                w[j] = *reinterpret_cast<const uint32_t*>(&h);
            }
            dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// y[t] = x[t] + sum_{s kept} Ys[t*k+s] (+ Sh[t]); fp32 sum in slot order, then
// the shared expert, then the residual, rounded once.
// y[t] = x[t] + sum over kept slots of Ys[t*k+s] (+ Sh[t]), fp32, one rounding.
// USE_MASK = false for dropless layers (nothing is dropped): every load of a
// vector is then independent and issued at once; with a mask, the slot loads
// wait for the mask bytes (a dropped slot's row is never read).
template <typename T, bool USE_MASK>
__global__ void __launch_bounds__(256)
combine_kernel(const T* __restrict__ x, const T* __restrict__ Ys,
               const unsigned char* __restrict__ drop_mask, const T* __restrict__ Sh,
               T* __restrict__ y, int Ttok, int d, int k) {
    constexpr int NV = Vec16<T>::N;
    const int vec_per_row = d / NV;
    pdl_wait();
    pdl_trigger();
    const long long total = (long long)Ttok * vec_per_row;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int t = (int)(i / vec_per_row);
        const int v = (int)(i - (long long)t * vec_per_row);
        const uint4 xv = __ldg(reinterpret_cast<const uint4*>(x + (size_t)t * d) + v);
        float acc[NV];
#pragma unroll
        for (int j = 0; j < NV; ++j) acc[j] = 0.f;
        for (int s = 0; s < k; ++s) {
            const long long a = (long long)t * k + s;
            if (USE_MASK && drop_mask[a]) continue;
            float f[NV];
            unpack16(__ldg(reinterpret_cast<const uint4*>(Ys + a * d) + v), f);
#pragma unroll
            for (int j = 0; j < NV; ++j) acc[j] += f[j];
        }
        if (Sh) {
            float f[NV];
            unpack16(__ldg(reinterpret_cast<const uint4*>(Sh + (size_t)t * d) + v), f);
#pragma unroll
            for (int j = 0; j < NV; ++j) acc[j] += f[j];
        }
        float xf[NV];
        unpack16(xv, xf);
#pragma unroll
        for (int j = 0; j < NV; ++j) acc[j] += xf[j];
        reinterpret_cast<uint4*>(y + (size_t)t * d)[v] = pack16(acc);
    }
}

cudaError_t launch_gather(int dtype, const void* x, const int* perm_src, const int* offsets, int E,
                          int k, int T, int d, void* Xp, int* status, int num_sms,
                          cudaStream_t st) {
    const int esize = dtype == MOE_F32 ? 4 : 2;
    const int vpr = d * esize / 16;
    const int A = T * k;
    long long blocks = ((long long)A * 32 + 255) / 256;
    if (blocks > num_sms * 16) blocks = num_sms * 16;
    if (blocks < 1) blocks = 1;
    return launch_kernel(gather_rows_kernel, dim3((unsigned)blocks), dim3(256), 0, st, 1,
                         (const uint4*)x, perm_src, offsets, E, k, T, vpr, (uint4*)Xp, status);
}

cudaError_t launch_gather_f16(const void* x, const int* perm_src, const int* offsets, int E, int k,
                              int T, int d, void* Xp, int* status, int num_sms, cudaStream_t st) {
    const int vpr = d * 2 / 16;
    const int A = T * k;
    long long blocks = ((long long)A * 32 + 255) / 256;
    if (blocks > num_sms * 16) blocks = num_sms * 16;
    if (blocks < 1) blocks = 1;
    return launch_kernel(gather_rows_f16_kernel, dim3((unsigned)blocks), dim3(256), 0, st, 1,
                         (const uint4*)x, perm_src, offsets, E, k, T, vpr, (uint4*)Xp, status);
}

cudaError_t launch_combine(int dtype, const void* x, const void* Ys, const unsigned char* drop_mask,
                           const void* Sh, void* y, int T, int d, int k, int num_sms,
                           cudaStream_t st, bool use_mask) {
    const int esize = dtype == MOE_F32 ? 4 : 2;
    const long long total = (long long)T * (d * esize / 16);
    long long blocks = (total + 255) / 256;
    if (blocks > num_sms * 16) blocks = num_sms * 16;
    if (blocks < 1) blocks = 1;
    if (dtype == MOE_F32)
        return launch_kernel(use_mask ? combine_kernel<float, true> : combine_kernel<float, false>,
                             dim3((unsigned)blocks), dim3(256), 0, st, 1, (const float*)x,
                             (const float*)Ys, drop_mask, (const float*)Sh, (float*)y, T, d, k);
    return launch_kernel(use_mask ? combine_kernel<__nv_bfloat16, true>
                                  : combine_kernel<__nv_bfloat16, false>,
                         dim3((unsigned)blocks), dim3(256), 0, st, 1, (const __nv_bfloat16*)x,
                         (const __nv_bfloat16*)Ys, drop_mask, (const __nv_bfloat16*)Sh,
                         (__nv_bfloat16*)y, T, d, k);
}

}  // namespace moe
