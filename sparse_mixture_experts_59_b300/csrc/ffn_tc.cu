// ffn_tc.cu -- bf16 grouped expert GEMMs on the 5th-generation tensor cores.
//
// "How Mixture of Experts Works": production layers run every expert's rows
// as grouped GEMMs instead of a per-expert loop (remark after the MoELayer
// listing); "Mixture of Experts (MoE)", "Implementing a complete MoE layer":
// SwiGLU experts w_down(silu(w_gate x) * w_up x); "Mixture-of-Experts
// Routing", "How a sparse MoE layer works": GELU MLP experts with biases.
//
// One persistent kernel per projection.  Its tiles cover every (group,
// row-tile, column-tile) of the ragged expert segments -- read on the device
// from `offsets`, so no host sync -- plus, when present, the shared expert as
// one more group whose rows are the T tokens.  Per CTA (one per SM):
//   warp 0      TMA producer: A tile 128x64 and B tile 256x64 (bf16, 128B
//               swizzle) per stage into a 4-deep shared-memory ring;
//   warp 1      allocates 512 TMEM columns and issues tcgen05.mma
//               (M=128, N=256, K=16) from one thread into one of two
//               accumulators (2 x 256 fp32 columns);
//   warps 2-5   epilogue: tcgen05.ld the accumulator (warp w reads TMEM lanes
//               32*(w%4)..+31, i.e. tile rows), apply the fused epilogue and
//               store bf16 rows; the second accumulator lets the next tile's
//               MMAs run meanwhile.
// Epilogues:
//   kModeSwiglu  B = 128 gate rows then 128 up rows of the same hidden units,
//                so one MMA gives [g | u];  H = silu(g) * u        (128 cols/tile)
//   kModeGelu    H = gelu_erf(acc + b1)                             (256 cols/tile)
//   kModeDown    Ys[perm_src[r]] = topk_w[perm_src[r]] * (acc + b2), i.e. the
//                gate scale and the scatter back to the assignment slot;
//                shared group: Sh[t] = acc                          (256 cols/tile)
// Rows past a segment's end and columns past N are computed on whatever the
// tile reads (the next segment, or TMA's zero fill) and never stored.
#include "common.cuh"
#include "kernels.cuh"
#include "launch.cuh"
#include "ffn_tc_common.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

using tcffn::BK;
using tcffn::ModeTraits;
using tcffn::Tile;
constexpr int BM = 128;        // tile rows = MMA M
constexpr int MMA_N = 256;     // B rows per stage
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;        // 16 KB
constexpr int B_BYTES = MMA_N * BK * 2;     // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 512;              // two 256-column accumulators
constexpr int NUM_THREADS = 192;
constexpr uint32_t IDESC = ptx::idesc_bf16_f32(BM, MMA_N);

// shared-memory carve-up (offsets from the 1024-aligned base)
constexpr int OFF_A = 0;
constexpr int OFF_B = STAGES * A_BYTES;
constexpr int OFF_BAR = OFF_B + STAGES * B_BYTES;
constexpr int NUM_BARS = 2 * STAGES + 2 + 2 + 1 + 1;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;          // tmem base, abort flag
constexpr int OFF_START = OFF_MISC + 16;                  // group tile starts
constexpr int OFF_OFFS = OFF_START + (kMaxExperts + 2) * 4;  // cached offsets
constexpr int SMEM_USED = OFF_OFFS + (kMaxExperts + 2) * 4;
constexpr int SMEM_BYTES = SMEM_USED + 1024;              // alignment slack

template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
ffn_tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
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
    uint64_t* endbar = drain + 1;            // teardown: every thread
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
    int* s_start = reinterpret_cast<int*>(smem + OFF_START);
    int* s_off = reinterpret_cast<int*>(smem + OFF_OFFS);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&tfull[a], 1);
            ptx::mbar_init(&tempty[a], 128);
        }
        ptx::mbar_init(drain, 1);
        ptx::mbar_init(endbar, NUM_THREADS);
        *s_abort = 0;
        ptx::fence_mbarrier_init();
        ptx::prefetch_tensormap(&mapA);
        ptx::prefetch_tensormap(&mapB);
        ptx::prefetch_tensormap(&mapB2);
    }
    if (warp == 1) {
        ptx::tmem_alloc(s_tmem, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    pdl_wait();       // offsets and the A rows come from the preceding kernels
    pdl_trigger();
    for (int i = threadIdx.x; i <= p.E; i += NUM_THREADS) s_off[i] = p.offsets[i];
    const int nt_r = (p.N + BN_OUT - 1) / BN_OUT;
    const int nt_s = p.rows_sh > 0 ? (p.N_sh + BN_OUT - 1) / BN_OUT : 0;
    group_tile_prefix(p.offsets, p.E, p.rows_sh, BM, nt_r, nt_s, s_start);
    ptx::tc_fence_before();
    block_sync();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const int G = p.E + (p.rows_sh > 0 ? 1 : 0);
    const int total = s_start[G];

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int it = 0;
            bool ok = true, held = false;
            const int hold_it = p.hold ? *p.hold - 1 : -1;
            for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
                const Tile t = tcffn::decode_tile<MODE, BM>(p, s_start, s_off, G, tile);
                const CUtensorMap* mA = t.sh ? &mapA_sh : &mapA;
                const CUtensorMap* mB0 = t.sh ? &mapB_sh : &mapB;
                const CUtensorMap* mB1 = (MODE == kModeSwiglu) ? (t.sh ? &mapB2_sh : &mapB2) : mB0;
                for (int kb = 0; kb < t.nk; ++kb, ++it) {
                    if (it == hold_it) { ok = false; held = true; break; }   // test hook
                    const int s = it % STAGES;
                    const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
                    if (!ptx::mbar_wait(&empty[s], ph ^ 1u, s_abort)) { ok = false; break; }
                    ptx::mbar_arrive_expect_tx(&full[s], STAGE_BYTES);
                    ptx::tma_load_2d(sA + s * A_BYTES, mA, &full[s], kb * BK, t.arow);
                    ptx::tma_load_2d(sB + s * B_BYTES, mB0, &full[s], kb * BK, t.wrow0);
                    ptx::tma_load_2d(sB + s * B_BYTES + B_BYTES / 2, mB1, &full[s], kb * BK, t.wrow1);
                }
            }
            if (!ok && !held) {
                *s_abort = 1;
                raise_error(p.status, MOE_ERR_DEVICE_TIMEOUT);
            }
            // let this thread's copies land before the CTA can exit
            for (int j = (it > STAGES ? it - STAGES : 0); j < it; ++j)
                ptx::mbar_wait(&full[j % STAGES], (uint32_t)(j / STAGES) & 1u, nullptr);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int it = 0, tc = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x, ++tc) {
                const Tile t = tcffn::decode_tile<MODE, BM>(p, s_start, s_off, G, tile);
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
                    for (int kk = 0; kk < BK / 16; ++kk)   // +32 bytes along K per step
                        ptx::mma_bf16(d_tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2),
                                      IDESC, (kb | kk) != 0 ? 1u : 0u);
                    ptx::mma_commit(&empty[s]);
                }
                if (!ok) break;
                ptx::mma_commit(&tfull[acc]);
            }
            if (!ok) {
                *s_abort = 1;
                raise_error(p.status, MOE_ERR_DEVICE_TIMEOUT);
            }
            // every MMA issued by this thread completes before TMEM is freed
            ptx::mma_commit(drain);
            ptx::mbar_wait(drain, 0, nullptr);
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;                 // TMEM lane quadrant of this warp
        const int row_in_tile = q * 32 + lane;
        int tc = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x, ++tc) {
            const Tile t = tcffn::decode_tile<MODE, BM>(p, s_start, s_off, G, tile);
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
            tcffn::epilogue_tile<MODE>(p, t, taddr, t.arow + row_in_tile);
            ptx::tc_fence_before();
            ptx::mbar_arrive(&tempty[acc]);
        }
    }

    // teardown: all roles done (or aborted); free TMEM
    ptx::tc_fence_before();
    ptx::mbar_block_sync(endbar);
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace

int ffn_tc_smem_bytes() { return SMEM_BYTES; }

cudaError_t launch_ffn_tc(int mode, const CUtensorMap* maps, const TcFfnArgs& p, int num_sms,
                          cudaStream_t st) {
    auto kernel = mode == kModeSwiglu ? ffn_tc_kernel<kModeSwiglu>
                : mode == kModeGelu ? ffn_tc_kernel<kModeGelu> : ffn_tc_kernel<kModeDown>;
    const cudaError_t err =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (err != cudaSuccess) return err;
    return launch_kernel(kernel, dim3(num_sms), dim3(NUM_THREADS), SMEM_BYTES, st, 1, maps[0],
                         maps[1], maps[2], maps[3], maps[4], maps[5], p);
}

}  // namespace moe
