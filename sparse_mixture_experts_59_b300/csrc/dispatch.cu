// dispatch.cu -- per-expert histogram, token-order ranks, capacity and the
// stable expert-grouped permutation.
//
// "How Mixture of Experts Works", MoELayer listing: the (token, slot) pairs are
// flattened as a = t*k + s and grouped per expert in that order; section "The
// Capacity Factor": capacity = max(int(T*k/E*cf), 1), excess assignments are
// dropped and fall through on the residual.  "Mixture-of-Experts Routing",
// section "How a sparse MoE layer works": the capacity check keeps the first
// `capacity` pairs in nonzero (token) order.
//
// Kernel 1 (dispatch_rank_kernel): each block takes a chunk of assignments in
// flattened order.  Inside the block the rank of an assignment among the
// chunk's assignments to the same expert comes from __match_any_sync within a
// warp and a per-round scan across warps; across blocks a decoupled look-back
// over an E-wide status vector gives each block the count of earlier
// assignments per expert.  The last block to finish turns the totals into
// counts, capacity-clipped counts, offsets and the aux loss, and clears the
// look-back state for the next call.
// Kernel 2 (dispatch_scatter_kernel): dest / perm_src / drop mask.
#include "common.cuh"
#include "kernels.cuh"
#include "launch.cuh"

namespace moe {

constexpr int kDspThreads = 256;
constexpr int kDspWarps = kDspThreads / 32;
constexpr unsigned kFlagAgg = 1u << 30;       // block aggregate published
constexpr unsigned kFlagPrefix = 2u << 30;    // inclusive prefix published
constexpr unsigned kFlagMask = 3u << 30;
constexpr unsigned kValueMask = (1u << 30) - 1;

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_u32(unsigned* p, unsigned v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__global__ void __launch_bounds__(kDspThreads)
dispatch_rank_kernel(const int* __restrict__ topk_idx, int A, int Ttok, int E,
                     long long cap, unsigned* __restrict__ tile_status, int* __restrict__ ctrl,
                     int* __restrict__ rank, int* __restrict__ counts_pre,
                     int* __restrict__ counts_kept, int* __restrict__ offsets,
                     const float* __restrict__ prob_mean, float* __restrict__ stats) {
    __shared__ int s_cnt[2][kDspWarps][kMaxExperts];
    __shared__ int s_run[kMaxExperts];
    __shared__ int s_excl[kMaxExperts];
    __shared__ int s_bid, s_last;
    int* status = ctrl + kCtrlStatus;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_wait();
    pdl_trigger();
    if (tid == 0) s_bid = atomicAdd(ctrl + kCtrlDispatchTicket, 1);
    if (tid < E) s_run[tid] = 0;
    block_sync();
    const int bid = s_bid;
    const int nblk = gridDim.x;
    const int base = bid * kDspChunk;
    const unsigned lt_mask = (1u << lane) - 1u;

    int my_e[kDspItems], my_rank[kDspItems];
#pragma unroll
    for (int it = 0; it < kDspItems; ++it) {
        const int a = base + it * kDspThreads + tid;
        int e = -1;
        if (a < A) {
            e = topk_idx[a];
            if (e < 0 || e >= E) {
                raise_error(status, MOE_ERR_DEVICE_BOUNDS);
                e = -1;
            }
        }
        const int buf = it & 1;
#pragma unroll
        for (int w = 0; w < kDspWarps; ++w) s_cnt[buf][w][tid] = 0;
        block_sync();
        const unsigned peers = __match_any_sync(0xffffffffu, e);
        const int in_warp = __popc(peers & lt_mask);
        if (e >= 0 && lane == __ffs(peers) - 1) s_cnt[buf][warp][e] = __popc(peers);
        block_sync();
        if (tid < E) {                       // exclusive scan over warps, per expert
            int run = s_run[tid];
#pragma unroll
            for (int w = 0; w < kDspWarps; ++w) {
                const int c = s_cnt[buf][w][tid];
                s_cnt[buf][w][tid] = run;
                run += c;
            }
            s_run[tid] = run;
        }
        block_sync();
        my_e[it] = e;
        my_rank[it] = (e >= 0) ? s_cnt[buf][warp][e] + in_warp : -1;
    }

    // decoupled look-back, one thread per expert.  A block named by the
    // kCtrlHoldBlock test hook publishes nothing, so its successors' bounded
    // waits run out and report MOE_ERR_DEVICE_TIMEOUT.
    const bool hold = ctrl[kCtrlHoldBlock] == bid + 1;
    if (tid < E) {
        const unsigned agg = (unsigned)s_run[tid];
        unsigned* mine = tile_status + (size_t)bid * E + tid;
        if (bid == 0) {
            s_excl[tid] = 0;
            if (!hold) st_release_u32(mine, kFlagPrefix | agg);
        } else {
            if (!hold) st_release_u32(mine, kFlagAgg | agg);
            unsigned excl = 0;
            int j = bid - 1;
            long long t0 = 0;
            bool timed_out = false;
            while (j >= 0) {
                const unsigned v = ld_acquire_u32(tile_status + (size_t)j * E + tid);
                const unsigned flag = v & kFlagMask;
                if (flag == 0) {
                    if (t0 == 0) t0 = clock64();
                    else if (clock64() - t0 > kWaitLimitCycles) { timed_out = true; break; }
                    continue;
                }
                t0 = 0;
                excl += v & kValueMask;
                if (flag == kFlagPrefix) break;
                --j;
            }
            if (timed_out) raise_error(status, MOE_ERR_DEVICE_TIMEOUT);
            s_excl[tid] = (int)excl;
            if (!hold) st_release_u32(mine, kFlagPrefix | ((excl + agg) & kValueMask));
        }
    }
    block_sync();
#pragma unroll
    for (int it = 0; it < kDspItems; ++it) {
        const int a = base + it * kDspThreads + tid;
        if (a < A) rank[a] = (my_e[it] >= 0) ? s_excl[my_e[it]] + my_rank[it] : -1;
    }

    // the last block to finish produces the totals
    __threadfence();
    block_sync();
    if (tid == 0) s_last = (atomicAdd(ctrl + kCtrlDispatchDone, 1) == nblk - 1);
    block_sync();
    if (!s_last) return;
    __threadfence();
    int total = 0, kept = 0;
    if (tid < E) {
        const unsigned v = ld_acquire_u32(tile_status + (size_t)(nblk - 1) * E + tid);
        total = (int)(v & kValueMask);
        kept = (cap >= 0 && (long long)total > cap) ? (int)cap : total;
        counts_pre[tid] = total;
        counts_kept[tid] = kept;
    }
    // exclusive scan of kept over experts (block of 256 = 8 warps)
    int incl = kept;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    __shared__ int s_wsum[kDspWarps];
    if (lane == 31) s_wsum[warp] = incl;
    block_sync();
    int wbase = 0;
    for (int w = 0; w < warp; ++w) wbase += s_wsum[w];
    if (tid < E) offsets[tid] = wbase + incl - kept;
    if (tid == E - 1) offsets[E] = wbase + incl;
    block_sync();
    if (tid == 0) {
        int R = 0;
        for (int w = 0; w < kDspWarps; ++w) R += s_wsum[w];
        if (stats) {
            float aux = 0.f;
            if (prob_mean) {
                for (int e = 0; e < E; ++e)
                    aux += ((float)counts_pre[e] / (float)Ttok) * prob_mean[e];
                aux *= (float)E;
            }
            stats[0] = aux;
            stats[1] = (A > 0) ? (float)(A - R) / (float)A : 0.f;
        }
        ctrl[kCtrlDispatchTicket] = 0;
        ctrl[kCtrlDispatchDone] = 0;
        ctrl[kCtrlHoldBlock] = 0;
    }
    // clear the look-back state for the next call
    for (int i = tid; i < nblk * E; i += kDspThreads) tile_status[i] = 0u;
}

__global__ void __launch_bounds__(256)
dispatch_scatter_kernel(const int* __restrict__ topk_idx, const int* __restrict__ rank, int A,
                        int E, long long cap, const int* __restrict__ offsets,
                        int* __restrict__ dest, int* __restrict__ perm_src,
                        unsigned char* __restrict__ drop_mask, int* __restrict__ status) {
    pdl_wait();
    pdl_trigger();
    for (int a = blockIdx.x * blockDim.x + threadIdx.x; a < A; a += gridDim.x * blockDim.x) {
        const int e = topk_idx[a];
        const int r = rank[a];
        const bool valid = (e >= 0 && e < E && r >= 0);
        const bool kept = valid && (cap < 0 || (long long)r < cap);
        if (kept) {
            const int dst = offsets[e] + r;
            if (dst < offsets[e + 1]) {
                dest[a] = dst;
                perm_src[dst] = a;
                if (drop_mask) drop_mask[a] = 0;
                continue;
            }
            raise_error(status, MOE_ERR_DEVICE_BOUNDS);
        }
        dest[a] = -1;
        if (drop_mask) drop_mask[a] = 1;
    }
}

cudaError_t launch_dispatch(const int* topk_idx, int T, int k, int E, long long cap,
                            unsigned* tile_status, int* ctrl, int* rank, int* counts_pre,
                            int* counts_kept, int* offsets, int* dest, int* perm_src,
                            unsigned char* drop_mask, const float* prob_mean, float* stats,
                            int num_sms, cudaStream_t st) {
    const int A = T * k;
    const int nblk = dispatch_blocks(A);
    cudaError_t err = launch_kernel(dispatch_rank_kernel, dim3(nblk), dim3(kDspThreads), 0, st, 1,
                                    topk_idx, A, T, E, cap, tile_status, ctrl, rank, counts_pre,
                                    counts_kept, offsets, prob_mean, stats);
    if (err != cudaSuccess) return err;
    int sblk = (A + 255) / 256;
    if (sblk > num_sms * 8) sblk = num_sms * 8;
    if (sblk < 1) sblk = 1;
    return launch_kernel(dispatch_scatter_kernel, dim3(sblk), dim3(256), 0, st, 1, topk_idx,
                         (const int*)rank, A, E, cap, (const int*)offsets, dest, perm_src, drop_mask,
                         ctrl + kCtrlStatus);
}

}  // namespace moe
