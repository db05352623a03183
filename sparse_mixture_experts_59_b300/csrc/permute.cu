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

constexpr int kGatherVecs = 4;    // 16-byte vectors a gather thread keeps in flight
constexpr int kCombineVecs = 2;   // vectors per combine thread (x and each slot: 2 loads)

// Xp[r] = x[perm_src[r] / k] for r < R = offsets[E] (read on the device);
// TO_F16 converts bf16 x to f16 on the way (the token operand of the
// low-bit-weight expert GEMMs, whose MMAs take f16).  A row is spread over
// tpr threads (tpr a power of two up to 256, the block holding 256 / tpr
// rows), 16-byte vectors, each thread's loads issued together before its
// stores: at decode sizes (a few dozen rows) every row is a block and the
// gather costs one memory round trip instead of one per 32 vectors.
template <bool TO_F16>
__global__ void __launch_bounds__(256)
gather_rows_kernel(const uint4* __restrict__ x, const int* __restrict__ perm_src,
                   const int* __restrict__ offsets, int E, int k, int Ttok, int vec_per_row,
                   int tpr, uint4* __restrict__ Xp, int* __restrict__ status) {
    constexpr int U = kGatherVecs;           // vectors in flight per thread
    pdl_wait();
    pdl_trigger();
    const int R = offsets[E];
    const int rpb = blockDim.x / tpr;
    const int slot = threadIdx.x / tpr, tl = threadIdx.x % tpr;
    for (int r = blockIdx.x * rpb + slot; r < R; r += gridDim.x * rpb) {
        const int a = perm_src[r];
        const int t = a / k;
        if (a < 0 || t >= Ttok) {
            if (tl == 0) raise_error(status, MOE_ERR_DEVICE_BOUNDS);
            continue;
        }
        const uint4* src = x + (size_t)t * vec_per_row;
        uint4* dst = Xp + (size_t)r * vec_per_row;
        for (int v0 = tl; v0 < vec_per_row; v0 += U * tpr) {
            uint4 q[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = v0 + u * tpr;
                if (v < vec_per_row) q[u] = __ldg(src + v);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int v = v0 + u * tpr;
                if (v >= vec_per_row) continue;
                if constexpr (TO_F16) {
                    float f[8];
                    unpack16(q[u], f);
                    uint32_t w[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const __half2 h = __floats2half2_rn(f[2 * j], f[2 * j + 1]);
                        w[j] = *reinterpret_cast<const uint32_t*>(&h);
                    }
                    dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
                } else {
                    dst[v] = q[u];
                }
            }
        }
    }
}

// y[t] = x[t] + sum over kept slots of Ys[t*k+s] (+ Sh[t]): fp32 sum in slot
// order, then the shared expert, then the residual, rounded once.  A row is
// spread over tpr threads (as in the gather); each thread takes up to U
// vectors of the row and issues each source's U loads together (x first).
// USE_MASK = false for dropless layers: no mask bytes are read; with a mask,
// a dropped slot's row is never read.
template <typename T, bool USE_MASK>
__global__ void __launch_bounds__(256, 4)
combine_kernel(const T* __restrict__ x, const T* __restrict__ Ys,
               const unsigned char* __restrict__ drop_mask, const T* __restrict__ Sh,
               T* __restrict__ y, int Ttok, int d, int k, int tpr) {
    constexpr int NV = Vec16<T>::N;
    constexpr int U = kCombineVecs;
    const int vpr = d / NV;
    pdl_wait();
    pdl_trigger();
    const int rpb = blockDim.x / tpr;
    const int slot = threadIdx.x / tpr, tl = threadIdx.x % tpr;
    for (int t = blockIdx.x * rpb + slot; t < Ttok; t += gridDim.x * rpb) {
        unsigned keep = ~0u;                 // bit s: slot s kept (k <= 8)
        if (USE_MASK) {
            keep = 0u;
            for (int s = 0; s < k; ++s)
                if (!drop_mask[(size_t)t * k + s]) keep |= 1u << s;
        }
        const uint4* xr = reinterpret_cast<const uint4*>(x + (size_t)t * d);
        uint4* yr = reinterpret_cast<uint4*>(y + (size_t)t * d);
        for (int v0 = tl; v0 < vpr; v0 += U * tpr) {
            uint4 xq[U];
#pragma unroll
            for (int u = 0; u < U; ++u)
                if (v0 + u * tpr < vpr) xq[u] = __ldg(xr + v0 + u * tpr);
            float acc[U][NV];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int j = 0; j < NV; ++j) acc[u][j] = 0.f;
            for (int s = 0; s < k; ++s) {
                if (USE_MASK && !((keep >> s) & 1u)) continue;
                const uint4* src = reinterpret_cast<const uint4*>(Ys + ((size_t)t * k + s) * d);
                uint4 q[U];
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (v0 + u * tpr < vpr) q[u] = __ldg(src + v0 + u * tpr);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (v0 + u * tpr >= vpr) continue;
                    float f[NV];
                    unpack16(q[u], f);
#pragma unroll
                    for (int j = 0; j < NV; ++j) acc[u][j] += f[j];
                }
            }
            if (Sh) {
                const uint4* src = reinterpret_cast<const uint4*>(Sh + (size_t)t * d);
                uint4 q[U];
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (v0 + u * tpr < vpr) q[u] = __ldg(src + v0 + u * tpr);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    if (v0 + u * tpr >= vpr) continue;
                    float f[NV];
                    unpack16(q[u], f);
#pragma unroll
                    for (int j = 0; j < NV; ++j) acc[u][j] += f[j];
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (v0 + u * tpr >= vpr) continue;
                float xf[NV];
                unpack16(xq[u], xf);
#pragma unroll
                for (int j = 0; j < NV; ++j) acc[u][j] += xf[j];
                yr[v0 + u * tpr] = pack16(acc[u]);
            }
        }
    }
}

// Threads per row (a power of two, 32..256) for `rows` rows of `vpr` vectors,
// each thread taking up to `u` vectors of its row per pass: with rows enough
// to fill every SM, vpr / u (each thread's loads all in one pass); a
// decode-sized batch spreads each row over up to 256 threads instead.
static int row_threads(int rows, int vpr, int u, int num_sms) {
    const long long full = (long long)num_sms * 2048;     // resident threads
    int t = 32;
    if ((long long)rows * ((vpr + u - 1) / u) >= full) {
        while (t < 256 && t * u < vpr) t <<= 1;
    } else {
        while (t < 256 && t < vpr) t <<= 1;
    }
    return t;
}
// blocks of 256 threads for A rows (at most 16 per SM; the kernel loops)
static unsigned gather_blocks(int A, int tpr, int num_sms) {
    const int rpb = 256 / tpr;
    long long blocks = ((long long)A + rpb - 1) / rpb;
    if (blocks > num_sms * 16) blocks = num_sms * 16;
    if (blocks < 1) blocks = 1;
    return (unsigned)blocks;
}

cudaError_t launch_gather(int dtype, const void* x, const int* perm_src, const int* offsets, int E,
                          int k, int T, int d, void* Xp, int* status, int num_sms,
                          cudaStream_t st) {
    const int esize = dtype == MOE_F32 ? 4 : 2;
    const int vpr = d * esize / 16;
    const int tpr = row_threads(T * k, vpr, kGatherVecs, num_sms);
    return launch_kernel(gather_rows_kernel<false>, dim3(gather_blocks(T * k, tpr, num_sms)),
                         dim3(256), 0, st, 1, (const uint4*)x, perm_src, offsets, E, k, T, vpr,
                         tpr, (uint4*)Xp, status);
}

cudaError_t launch_gather_f16(const void* x, const int* perm_src, const int* offsets, int E, int k,
                              int T, int d, void* Xp, int* status, int num_sms, cudaStream_t st) {
    const int vpr = d * 2 / 16;
    const int tpr = row_threads(T * k, vpr, kGatherVecs, num_sms);
    return launch_kernel(gather_rows_kernel<true>, dim3(gather_blocks(T * k, tpr, num_sms)),
                         dim3(256), 0, st, 1, (const uint4*)x, perm_src, offsets, E, k, T, vpr,
                         tpr, (uint4*)Xp, status);
}

cudaError_t launch_combine(int dtype, const void* x, const void* Ys, const unsigned char* drop_mask,
                           const void* Sh, void* y, int T, int d, int k, int num_sms,
                           cudaStream_t st, bool use_mask) {
    const int esize = dtype == MOE_F32 ? 4 : 2;
    const int tpr = row_threads(T, d * esize / 16, kCombineVecs, num_sms);
    const dim3 grid(gather_blocks(T, tpr, num_sms));
    if (dtype == MOE_F32)
        return launch_kernel(use_mask ? combine_kernel<float, true> : combine_kernel<float, false>,
                             grid, dim3(256), 0, st, 1, (const float*)x, (const float*)Ys,
                             drop_mask, (const float*)Sh, (float*)y, T, d, k, tpr);
    return launch_kernel(use_mask ? combine_kernel<__nv_bfloat16, true>
                                  : combine_kernel<__nv_bfloat16, false>,
                         grid, dim3(256), 0, st, 1, (const __nv_bfloat16*)x,
                         (const __nv_bfloat16*)Ys, drop_mask, (const __nv_bfloat16*)Sh,
                         (__nv_bfloat16*)y, T, d, k, tpr);
}

}  // namespace moe
