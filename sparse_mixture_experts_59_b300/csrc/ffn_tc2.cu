// ffn_tc2.cu -- bf16 grouped expert GEMMs on CTA pairs (tcgen05 cta_group::2).
//
// The same grouped GEMMs and fused epilogues as ffn_tc.cu (see there for the
// pages' basis), with a 256-row tile per cluster of two CTAs on two SMs:
//   - each CTA's TMA producer loads its own 128 rows of A and its own 128-row
//     half of the 256-row B tile (SwiGLU: the leader loads the gate rows, the
//     peer the matching up rows; otherwise the two halves of N) into a 6-deep
//     ring of 32 KB stages, and signals the LEADER's full barrier;
//   - the leader's single MMA thread issues tcgen05.mma.cta_group::2
//     (M = 256, N = 256, K = 16), which reads A and B from both CTAs' shared
//     memory and writes each CTA's 128 accumulator rows into its own TMEM
//     (two 256-column accumulators per CTA), and commits to the empty and
//     accumulator-full barriers of both CTAs at once;
//   - each CTA's four epilogue warps drain their own TMEM rows and arrive on
//     the leader's accumulator-empty barrier.
// Per SM this moves 32 KB per 64-deep K step instead of 48 KB for the same
// FLOPs, and the 192 KB ring holds six steps instead of four.  Used when the
// expert segments are long enough to fill 256-row tiles.
#include "common.cuh"
#include "ffn_tc_common.cuh"
#include "kernels.cuh"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using tcffn::BK;
using tcffn::ModeTraits;
using tcffn::Tile;

constexpr int TILE_M = 256;                  // rows per CTA pair
constexpr int HALF_M = 128;                  // rows per CTA
constexpr int MMA_N = 256;
constexpr int STAGES = 6;
constexpr int A_BYTES = HALF_M * BK * 2;     // 16 KB
constexpr int B_BYTES = 128 * BK * 2;        // 16 KB: this CTA's half of N
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 512;
constexpr int NUM_THREADS = 192;
constexpr uint32_t IDESC = ptx::idesc_bf16_f32(TILE_M, MMA_N);
constexpr uint16_t BOTH = 0x3;               // cluster ranks 0 and 1
constexpr uint16_t LEADER_ONLY = 0x1;

constexpr int OFF_A = 0;
constexpr int OFF_B = STAGES * A_BYTES;
constexpr int OFF_BAR = OFF_B + STAGES * B_BYTES;
constexpr int NUM_BARS = 2 * STAGES + 2 + 2 + 1;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int OFF_START = OFF_MISC + 16;
constexpr int OFF_OFFS = OFF_START + (kMaxExperts + 2) * 4;
constexpr int SMEM_USED = OFF_OFFS + (kMaxExperts + 2) * 4;
constexpr int SMEM_BYTES = SMEM_USED + 1024;

template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
ffn_tc2_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
               const __grid_constant__ CUtensorMap mapB2, const __grid_constant__ CUtensorMap mapA_sh,
               const __grid_constant__ CUtensorMap mapB_sh,
               const __grid_constant__ CUtensorMap mapB2_sh, const TcFfnArgs p) {
    constexpr int BN_OUT = ModeTraits<MODE>::BN_OUT;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem + OFF_A;
    uint8_t* sB = smem + OFF_B;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
    int* s_start = reinterpret_cast<int*>(smem + OFF_START);
    int* s_off = reinterpret_cast<int*>(smem + OFF_OFFS);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const bool leader = (rank == 0);
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&full[s], 1);      // the leader's: one arrive + both CTAs' bytes
            ptx::mbar_init(&empty[s], 1);     // one multicast commit
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&tfull[a], 1);             // one multicast commit
            ptx::mbar_init(&tempty[a], 2 * 128);      // the leader's: both CTAs' epilogue threads
        }
        ptx::mbar_init(drain, 1);
        *s_abort = 0;
        ptx::fence_mbarrier_init();
        ptx::prefetch_tensormap(&mapA);
        ptx::prefetch_tensormap(&mapB);
        ptx::prefetch_tensormap(&mapB2);
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(s_tmem, TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    pdl_wait();       // offsets and the token rows come from the preceding kernels
    pdl_trigger();
    for (int i = threadIdx.x; i <= p.E; i += NUM_THREADS) s_off[i] = p.offsets[i];
    const int nt_r = (p.N + BN_OUT - 1) / BN_OUT;
    const int nt_s = p.rows_sh > 0 ? (p.N_sh + BN_OUT - 1) / BN_OUT : 0;
    group_tile_prefix(p.offsets, p.E, p.rows_sh, TILE_M, nt_r, nt_s, s_start);
    // both CTAs' barriers are initialised before either touches the other's
    ptx::tc_fence_before();
    __syncwarp();
    ptx::cluster_sync();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const int G = p.E + (p.rows_sh > 0 ? 1 : 0);
    const int total = s_start[G];
    const uint32_t full_leader = ptx::mapa_shared(ptx::smem_u32(full), 0);
    const uint32_t tempty_leader = ptx::mapa_shared(ptx::smem_u32(tempty), 0);

    if (warp == 0) {
        // ------------------------------------------- TMA producer (both CTAs)
        if (lane == 0) {
            int it = 0;
            bool ok = true, held = false;
            const int hold_it = p.hold ? *p.hold - 1 : -1;
            for (int tile = cluster; ok && tile < total; tile += nclusters) {
                const Tile t = tcffn::decode_tile<MODE, TILE_M>(p, s_start, s_off, G, tile);
                const CUtensorMap* mA = t.sh ? &mapA_sh : &mapA;
                const CUtensorMap* mB;
                if (MODE == kModeSwiglu)
                    mB = leader ? (t.sh ? &mapB_sh : &mapB) : (t.sh ? &mapB2_sh : &mapB2);
                else
                    mB = t.sh ? &mapB_sh : &mapB;
                const int arow = t.arow + (int)rank * HALF_M;
                const int brow = leader ? t.wrow0 : t.wrow1;
                for (int kb = 0; kb < t.nk; ++kb, ++it) {
                    if (it == hold_it) { ok = false; held = true; break; }   // test hook
                    const int s = it % STAGES;
                    const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
                    if (!ptx::mbar_wait(&empty[s], ph ^ 1u, s_abort)) { ok = false; break; }
                    if (leader) ptx::mbar_arrive_expect_tx(&full[s], 2 * STAGE_BYTES);
                    ptx::tma_load_2d_pair(sA + s * A_BYTES, mA, full_leader + 8u * s, kb * BK, arow);
                    ptx::tma_load_2d_pair(sB + s * B_BYTES, mB, full_leader + 8u * s, kb * BK, brow);
                }
            }
            if (!ok && !held) {
                *s_abort = 1;
                raise_error(p.status, MOE_ERR_DEVICE_TIMEOUT);
            }
            // the leader's full barriers count both CTAs' bytes: let them land
            if (leader)
                for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
                    ptx::mbar_wait(&full[j % STAGES], (uint32_t)(j / STAGES) & 1u, nullptr);
        }
    } else if (warp == 1) {
        // ----------------------------------------- MMA issuer (leader only)
        if (leader && lane == 0) {
            int it = 0, tc = 0;
            bool ok = true;
            for (int tile = cluster; ok && tile < total; tile += nclusters, ++tc) {
                const Tile t = tcffn::decode_tile<MODE, TILE_M>(p, s_start, s_off, G, tile);
                const int acc = tc & 1;
                const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
                if (!ptx::mbar_wait(&tempty[acc], aph ^ 1u, s_abort)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * MMA_N);
                for (int kb = 0; kb < t.nk; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
                    if (!ptx::mbar_wait(&full[s], ph, s_abort)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint64_t ad = ptx::sw128_desc(ptx::smem_u32(sA + s * A_BYTES));
                    const uint64_t bd = ptx::sw128_desc(ptx::smem_u32(sB + s * B_BYTES));
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        ptx::mma_bf16_pair(d_tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2),
                                           IDESC, (kb | kk) != 0 ? 1u : 0u);
                    ptx::mma_commit_pair_mc(&empty[s], BOTH);
                }
                if (!ok) break;
                ptx::mma_commit_pair_mc(&tfull[acc], BOTH);
            }
            if (!ok) {
                *s_abort = 1;
                raise_error(p.status, MOE_ERR_DEVICE_TIMEOUT);
            }
            ptx::mma_commit_pair_mc(drain, LEADER_ONLY);
            ptx::mbar_wait(drain, 0, nullptr);
        }
    } else {
        // ------------------------------------------- epilogue (both CTAs)
        const int q = warp & 3;
        const int row_in_cta = q * 32 + lane;
        int tc = 0;
        for (int tile = cluster; tile < total; tile += nclusters, ++tc) {
            const Tile t = tcffn::decode_tile<MODE, TILE_M>(p, s_start, s_off, G, tile);
            const int acc = tc & 1;
            const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
            int ok = 1;
            if (lane == 0) ok = ptx::mbar_wait(&tfull[acc], aph, s_abort) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) {
                    *s_abort = 1;
                    raise_error(p.status, MOE_ERR_DEVICE_TIMEOUT);
                }
                break;
            }
            ptx::tc_fence_after();
            const uint32_t taddr = tmem_base + (uint32_t)(acc * MMA_N) + ((uint32_t)(q * 32) << 16);
            tcffn::epilogue_tile<MODE>(p, t, taddr, t.arow + (int)rank * HALF_M + row_in_cta);
            ptx::tc_fence_before();
            ptx::mbar_arrive_cluster(tempty_leader + 8u * acc);
        }
    }

    // teardown: both CTAs finished (no remote arrive still targets either),
    // then each frees its half of the pair's TMEM allocation
    ptx::tc_fence_before();
    // The cluster barrier is what holds every warp here: the lanes of a role
    // warp reach this point apart, so the block barrier may count such a warp
    // early; the __syncwarp reconverges it before the (aligned) cluster
    // barrier.  Reconverging before the block barrier instead measured 1-2%
    // slower on the grouped GEMMs of the prefill layer.
    __syncthreads();
    __syncwarp();
    ptx::cluster_sync();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

template <int MODE>
cudaError_t launch_mode(const CUtensorMap* maps, const TcFfnArgs& p, cudaStream_t st) {
    auto kernel = ffn_tc2_kernel<MODE>;
    cudaError_t err =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (err != cudaSuccess) return err;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // persistent: as many pairs as can be resident at once (cached per device)
    static int cached[64] = {};
    int dev = 0;
    if ((err = cudaGetDevice(&dev)) != cudaSuccess) return err;
    int clusters = (dev >= 0 && dev < 64) ? cached[dev] : 0;
    if (clusters == 0) {
        cfg.gridDim = dim3(2);
        if ((err = cudaOccupancyMaxActiveClusters(&clusters, (void*)kernel, &cfg)) != cudaSuccess)
            return err;
        if (clusters < 1) return cudaErrorInvalidConfiguration;
        if (dev >= 0 && dev < 64) cached[dev] = clusters;
    }
    return launch_kernel(kernel, dim3(2 * clusters), dim3(NUM_THREADS), SMEM_BYTES, st, 2, maps[0],
                         maps[1], maps[2], maps[3], maps[4], maps[5], p);
}

}  // namespace

int ffn_tc2_tile_rows() { return TILE_M; }

cudaError_t launch_ffn_tc2(int mode, const CUtensorMap* maps, const TcFfnArgs& p, cudaStream_t st) {
    if (mode == kModeSwiglu) return launch_mode<kModeSwiglu>(maps, p, st);
    if (mode == kModeGelu) return launch_mode<kModeGelu>(maps, p, st);
    return launch_mode<kModeDown>(maps, p, st);
}

}  // namespace moe
