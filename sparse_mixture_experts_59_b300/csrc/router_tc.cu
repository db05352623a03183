// router_tc.cu -- bf16 router logits on the tensor cores.
//
// "How Mixture of Experts Works", section "The Gating Mechanism": a bias-free
// linear map from the token's hidden state to one logit per expert; "Mixture
// of Experts (MoE)", section "The router": h @ W_r.  The map is a GEMM
// [T, d] x [d, E]; it is read-bound on x, and for many experts (E = 256,
// d = 7168) it is 30 GFLOP, so it runs on tcgen05 like the expert GEMMs.
//
// One CTA per (128-token tile, K split).  N is E rounded up to 16; TMA fills
// the expert rows past E with zeros.  Warp 0 issues TMA into a 4-stage ring,
// warp 1 issues tcgen05.mma (M=128, N=NB, K=16) into one TMEM accumulator,
// then all four warps read it back and store fp32 partial logits
// part[split][t][e].  Splitting K lets enough CTAs stream x at once; the
// partials are added in split order by the top-k kernel, so the result is the
// same on every run.
#include "common.cuh"
#include "kernels.cuh"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int BM = 128, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;

__host__ __device__ constexpr int b_stage_bytes(int nb) { return ((nb * BK * 2) + 1023) / 1024 * 1024; }
__host__ __device__ constexpr int tmem_cols_for(int nb) {
    return nb <= 32 ? 32 : nb <= 64 ? 64 : nb <= 128 ? 128 : 256;
}

__global__ void __launch_bounds__(128)
router_tc_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                 int T, int E, int NB, int nkb, int kb_per_split, float* __restrict__ part,
                 int* __restrict__ status) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int bstage = b_stage_bytes(NB);
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * bstage);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* done = bars + 2 * STAGES;
    uint64_t* endbar = done + 1;              // teardown: every thread
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(endbar + 1);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * BM;
    const int split = blockIdx.y;
    const int kb0 = split * kb_per_split;
    const int kb1 = min(nkb, kb0 + kb_per_split);
    const int ncols = tmem_cols_for(NB);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        ptx::mbar_init(done, 1);
        ptx::mbar_init(endbar, blockDim.x);
        *s_abort = 0;
        ptx::fence_mbarrier_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(s_tmem, ncols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    block_sync();
    ptx::tc_fence_after();
    const uint32_t tmem = *s_tmem;
    pdl_wait();       // x may come from the preceding kernel; part is reused across calls
    pdl_trigger();

    if (warp == 0 && lane == 0) {
        bool ok = true;
        int it = 0;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
            const int s = it % STAGES;
            const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
            if (!ptx::mbar_wait(&empty[s], ph ^ 1u, s_abort)) { ok = false; break; }
            ptx::mbar_arrive_expect_tx(&full[s], A_BYTES + NB * BK * 2);
            ptx::tma_load_2d(sA + s * A_BYTES, &map_x, &full[s], kb * BK, m0);
            ptx::tma_load_2d(sB + s * bstage, &map_w, &full[s], kb * BK, 0);
        }
        if (!ok) {
            *s_abort = 1;
            raise_error(status, MOE_ERR_DEVICE_TIMEOUT);
        }
        for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
            ptx::mbar_wait(&full[j % STAGES], (uint32_t)(j / STAGES) & 1u, nullptr);
    } else if (warp == 1 && lane == 0) {
        bool ok = true;
        const uint32_t idesc = ptx::idesc_bf16_f32(BM, NB);
        int it = 0;
        for (int kb = kb0; kb < kb1; ++kb, ++it) {
            const int s = it % STAGES;
            const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
            if (!ptx::mbar_wait(&full[s], ph, s_abort)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint64_t ad = ptx::sw128_desc(ptx::smem_u32(sA + s * A_BYTES));
            const uint64_t bd = ptx::sw128_desc(ptx::smem_u32(sB + s * bstage));
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
                ptx::mma_bf16(tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc,
                              (it | kk) != 0 ? 1u : 0u);
            ptx::mma_commit(&empty[s]);
        }
        if (!ok) {
            *s_abort = 1;
            raise_error(status, MOE_ERR_DEVICE_TIMEOUT);
        }
        ptx::mma_commit(done);     // arrives once every MMA above has completed
    }
    __syncwarp();

    // epilogue: warp w reads TMEM lanes 32w..32w+31 (token rows)
    int ok = 1;
    if (lane == 0) ok = ptx::mbar_wait(done, 0, nullptr) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (ok && !*s_abort && kb1 > kb0) {
        ptx::tc_fence_after();
        const int t = m0 + warp * 32 + lane;
        float* dst = part + ((size_t)split * T + t) * E;
        for (int c = 0; c < NB; c += 32) {
            __syncwarp();
            float v[32];
            ptx::tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)c, v);
            if (t < T) {
                if ((E & 3) == 0) {          // rows are 16-byte aligned: float4 stores
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        if (c + j < E)
                            *reinterpret_cast<float4*>(dst + c + j) =
                                make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                } else {
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (c + j < E) dst[c + j] = v[j];
                }
            }
        }
    } else if (!ok) {
        if (lane == 0) raise_error(status, MOE_ERR_DEVICE_TIMEOUT);
    }
    ptx::tc_fence_before();
    ptx::mbar_block_sync(endbar);      // every warp's TMEM loads done, then free it
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, ncols);
    }
}

}  // namespace

RouterPlan router_tc_plan(int T, int d, int E) {
    RouterPlan p;
    p.NB = (E + 15) / 16 * 16;
    p.m_tiles = (T + BM - 1) / BM;
    p.nkb = (d + BK - 1) / BK;
    p.smem = STAGES * (A_BYTES + b_stage_bytes(p.NB)) + (2 * STAGES + 2) * 8 + 16 + 1024;
    // about two CTAs per SM stream x at once; few tokens (one or two M tiles)
    // take at most 16 splits, as the top-k kernel adds the partials per token
    const int target = p.m_tiles <= 2 ? 16 * p.m_tiles : 2 * 148;
    int splits = (target + p.m_tiles - 1) / p.m_tiles;
    // A grid larger than the CTAs the 148 SMs hold at once (228 KB of shared
    // memory per SM with 1 KB reserved per CTA, 512 tensor-memory columns)
    // ends in a partial wave that streams x at a fraction of the bandwidth;
    // fewer, longer splits keep it to one wave.
    const int by_smem = (228 * 1024) / (p.smem + 1024);
    const int by_tmem = 512 / tmem_cols_for(p.NB);
    const int per_sm = by_smem < by_tmem ? by_smem : by_tmem;
    const int resident = 148 * (per_sm > 1 ? per_sm : 1);
    if (p.m_tiles * splits > resident) splits = resident / p.m_tiles;
    if (splits > p.nkb) splits = p.nkb;
    if (splits < 1) splits = 1;
    p.kb_per_split = (p.nkb + splits - 1) / splits;
    p.splits = (p.nkb + p.kb_per_split - 1) / p.kb_per_split;
    return p;
}

cudaError_t launch_router_tc(const CUtensorMap& map_x, const CUtensorMap& map_w, int T, int E,
                             const RouterPlan& p, float* part, int* status, cudaStream_t st) {
    cudaError_t err = cudaFuncSetAttribute(router_tc_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem);
    if (err != cudaSuccess) return err;
    return launch_kernel(router_tc_kernel, dim3(p.m_tiles, p.splits), dim3(128), p.smem, st, 1,
                         map_x, map_w, T, E, p.NB, p.nkb, p.kb_per_split, part, status);
}

}  // namespace moe
