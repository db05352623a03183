// ffn_swap.cu -- bf16 grouped expert GEMMs with the weights as the MMA's M
// operand and the tokens as its N operand, on CTA pairs (tcgen05 cta_group::2).
//
// Same maths and fused epilogues as ffn_tc.cu (see there for the pages'
// basis).  Expert segments are ragged; with tokens on M a segment is padded
// to the M tile (128 or 256 rows).  Here the tokens are the MMA's N, which
// only has to be a multiple of 16, so the last tile of each segment shrinks
// to the next multiple of 32 tokens and the padding is at most 31 rows.
//
// Per tile: 256 weight rows (128 per CTA) x N <= 256 tokens (N/2 per CTA).
//   - SwiGLU up: each CTA's 128 weight rows are 64 gate rows and the 64 up
//     rows of the same hidden units, so TMEM lanes 0-63 hold gate and 64-127
//     hold up; the epilogue warps holding up pass them to the warps holding
//     gate through shared memory.  A pair covers 128 hidden units.
//   - GELU up / down: each CTA's 128 weight rows are 128 consecutive outputs;
//     a pair covers 256.
// Each CTA's TMA producer loads its weight rows and its N/2 tokens into a
// 6-deep ring of 32 KB stages and signals the leader's full barrier; the
// leader's MMA thread issues M=256, N=ntile MMAs and commits to both CTAs'
// barriers; the epilogue reads accumulator columns (tokens) 32 at a time,
// stages them in shared memory as [token][feature] and writes whole output
// rows with 16-byte stores (down: to the assignment's slot, gate-scaled).
#include "common.cuh"
#include "kernels.cuh"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int BK = 64;
constexpr int STAGES = 6;
constexpr int TOK_TILE = 256;                // tokens per pair tile (MMA N max)
constexpr int A_BYTES = 128 * BK * 2;        // this CTA's 128 weight rows
constexpr int B_BYTES = 128 * BK * 2;        // up to 128 token rows (box of 128)
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 512;               // two 256-column accumulators
constexpr int NUM_THREADS = 192;
constexpr int EPI_THREADS = 128;
constexpr uint16_t BOTH = 0x3;
constexpr uint16_t LEADER_ONLY = 0x1;

constexpr int XCH_LD = 33;                   // [64 units][33] fp32: up values, padded
constexpr int OUT_LD = 136;                  // [32 tokens][136] bf16: staged output rows

constexpr int OFF_A = 0;
constexpr int OFF_B = STAGES * A_BYTES;
constexpr int OFF_XCH = OFF_B + STAGES * B_BYTES;
constexpr int OFF_OUT = OFF_XCH + 64 * XCH_LD * 4;
constexpr int OFF_TOKA = OFF_OUT + 32 * OUT_LD * 2;
constexpr int OFF_TOKW = OFF_TOKA + TOK_TILE * 4;
constexpr int OFF_BAR = OFF_TOKW + TOK_TILE * 4;
constexpr int NUM_BARS = 2 * STAGES + 2 + 2 + 1;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int OFF_START = OFF_MISC + 16;
constexpr int OFF_OFFS = OFF_START + (kMaxExperts + 2) * 4;
constexpr int SMEM_USED = OFF_OFFS + (kMaxExperts + 2) * 4;
constexpr int SMEM_BYTES = SMEM_USED + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

// weight units (outputs) per pair tile
template <int MODE> struct SwapTraits { static constexpr int UNITS = 256, UNITS_CTA = 128; };
template <> struct SwapTraits<kModeSwiglu> { static constexpr int UNITS = 128, UNITS_CTA = 64; };

struct STile {
    int g;
    bool sh;
    int tok0;       // first token row of the tile (A-row space of X_p / H, or x / H_sh)
    int ntok;       // valid tokens in the tile
    int nmma;       // MMA N: ntok rounded up to 32
    int u0;         // first output unit of the pair tile
    int N;          // outputs of this group's projection
    int nk;         // K blocks
    int wbase;      // first weight row of the group in its tensor map
};

template <int MODE>
__device__ __forceinline__ STile decode(const TcFfnArgs& p, const int* s_start, const int* s_off,
                                        int G, int tile) {
    STile t;
    t.g = find_group(s_start, G, tile);
    t.sh = (t.g == p.E);
    const int seg0 = t.sh ? 0 : s_off[t.g];
    const int rows = t.sh ? p.rows_sh : s_off[t.g + 1] - seg0;
    const int nt = (rows + TOK_TILE - 1) / TOK_TILE;
    const int local = tile - s_start[t.g];
    const int w = local / nt, tt = local - w * nt;
    t.tok0 = seg0 + tt * TOK_TILE;
    t.ntok = min(TOK_TILE, rows - tt * TOK_TILE);
    t.nmma = (t.ntok + 31) & ~31;
    t.N = t.sh ? p.N_sh : p.N;
    t.nk = ((t.sh ? p.K_sh : p.K) + BK - 1) / BK;
    t.u0 = w * SwapTraits<MODE>::UNITS;
    t.wbase = t.sh ? 0 : t.g * p.N;
    return t;
}

// Named barrier of the four epilogue warps.  bar.sync counts a warp's
// arrival as the whole warp, so every call below sits where the warp has
// reconverged: the only lane-divergent code before one is a single-lane `if`
// that closes before the call.
__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
ffn_swap_kernel(const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapW3,
                const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapW_sh,
                const __grid_constant__ CUtensorMap mapW3_sh,
                const __grid_constant__ CUtensorMap mapX_sh, const TcFfnArgs p) {
    constexpr int UNITS_CTA = SwapTraits<MODE>::UNITS_CTA;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem + OFF_A;
    uint8_t* sB = smem + OFF_B;
    float* s_xch = reinterpret_cast<float*>(smem + OFF_XCH);
    __nv_bfloat16* s_out = reinterpret_cast<__nv_bfloat16*>(smem + OFF_OUT);
    int* s_tok_a = reinterpret_cast<int*>(smem + OFF_TOKA);
    float* s_tok_w = reinterpret_cast<float*>(smem + OFF_TOKW);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);
    volatile int* s_go = reinterpret_cast<volatile int*>(smem + OFF_MISC + 8);
    int* s_start = reinterpret_cast<int*>(smem + OFF_START);
    int* s_off = reinterpret_cast<int*>(smem + OFF_OFFS);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const bool leader = (rank == 0);
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&tfull[a], 1);
            ptx::mbar_init(&tempty[a], 2 * EPI_THREADS);
        }
        ptx::mbar_init(drain, 1);
        *s_abort = 0;
        ptx::fence_mbarrier_init();
        ptx::prefetch_tensormap(&mapW);
        ptx::prefetch_tensormap(&mapW3);
        ptx::prefetch_tensormap(&mapX);
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(s_tmem, TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    pdl_wait();       // offsets and the token rows come from the preceding kernels
    pdl_trigger();
    for (int i = threadIdx.x; i <= p.E; i += NUM_THREADS) s_off[i] = p.offsets[i];
    constexpr int UNITS = SwapTraits<MODE>::UNITS;
    const int nw_r = (p.N + UNITS - 1) / UNITS;
    const int nw_s = p.rows_sh > 0 ? (p.N_sh + UNITS - 1) / UNITS : 0;
    group_tile_prefix(p.offsets, p.E, p.rows_sh, TOK_TILE, nw_r, nw_s, s_start);
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
                const STile t = decode<MODE>(p, s_start, s_off, G, tile);
                const CUtensorMap* mW = t.sh ? &mapW_sh : &mapW;
                const CUtensorMap* mW3 = t.sh ? &mapW3_sh : &mapW3;
                const CUtensorMap* mX = t.sh ? &mapX_sh : &mapX;
                const int wrow = t.wbase + t.u0 + (int)rank * UNITS_CTA;
                const int trow = t.tok0 + (int)rank * (t.nmma >> 1);
                for (int kb = 0; kb < t.nk; ++kb, ++it) {
                    if (it == hold_it) { ok = false; held = true; break; }   // test hook
                    const int s = it % STAGES;
                    const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
                    if (!ptx::mbar_wait(&empty[s], ph ^ 1u, s_abort)) { ok = false; break; }
                    if (leader) ptx::mbar_arrive_expect_tx(&full[s], 2 * STAGE_BYTES);
                    const uint32_t fb = full_leader + 8u * s;
                    if (MODE == kModeSwiglu) {   // 64 gate rows, then the 64 matching up rows
                        ptx::tma_load_2d_pair(sA + s * A_BYTES, mW, fb, kb * BK, wrow);
                        ptx::tma_load_2d_pair(sA + s * A_BYTES + A_BYTES / 2, mW3, fb, kb * BK, wrow);
                    } else {
                        ptx::tma_load_2d_pair(sA + s * A_BYTES, mW, fb, kb * BK, wrow);
                    }
                    ptx::tma_load_2d_pair(sB + s * B_BYTES, mX, fb, kb * BK, trow);
                }
            }
            if (!ok && !held) {
                *s_abort = 1;
                raise_error(p.status, MOE_ERR_DEVICE_TIMEOUT);
            }
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
                const STile t = decode<MODE>(p, s_start, s_off, G, tile);
                const int acc = tc & 1;
                const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
                if (!ptx::mbar_wait(&tempty[acc], aph ^ 1u, s_abort)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * TOK_TILE);
                const uint32_t idesc = ptx::idesc_bf16_f32(256, t.nmma);
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
                                           idesc, (kb | kk) != 0 ? 1u : 0u);
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
        const int q = warp & 3;                  // TMEM lane quadrant = weight rows q*32..
        const int et = threadIdx.x - 64;         // 0..127 among the epilogue threads
        int tc = 0;
        for (int tile = cluster; tile < total; tile += nclusters, ++tc) {
            const STile t = decode<MODE>(p, s_start, s_off, G, tile);
            const int acc = tc & 1;
            const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
            int ok = 1;
            if (lane == 0) ok = ptx::mbar_wait(&tfull[acc], aph, s_abort) ? 1 : 0;
            ok = __shfl_sync(0xffffffffu, ok, 0);
            // the four epilogue warps share named barriers below, so they take
            // one decision: a snapshot of the abort flag between two barriers
            if (lane == 0 && !ok) *s_abort = 1;
            epi_bar();
            if (et == 0) *s_go = *s_abort ? 0 : 1;
            epi_bar();
            if (!*s_go) {
                if (et == 0) raise_error(p.status, MOE_ERR_DEVICE_TIMEOUT);
                break;
            }
            ptx::tc_fence_after();
            const uint32_t tq = tmem_base + (uint32_t)(acc * TOK_TILE) + ((uint32_t)(q * 32) << 16);
            const int ubase = t.u0 + (int)rank * UNITS_CTA;     // first output unit of this CTA
            if (MODE == kModeDown) {                            // per-token slot and gate weight
                for (int j = et; j < t.ntok; j += EPI_THREADS) {
                    const int r = t.tok0 + j;
                    if (t.sh) {
                        s_tok_a[j] = r;
                        s_tok_w[j] = 1.f;
                    } else {
                        const int a = p.perm_src[r];
                        s_tok_a[j] = a;
                        s_tok_w[j] = p.gate_w[a];
                    }
                }
            }
            __nv_bfloat16* out_base = reinterpret_cast<__nv_bfloat16*>(t.sh ? p.out_sh : p.out);
            const __nv_bfloat16* bias = (p.bias && !t.sh) ? p.bias + (size_t)t.g * t.N : nullptr;
            for (int c = 0; c < t.nmma; c += 32) {
                __syncwarp();
                float v[32];
                if (MODE == kModeSwiglu) {
                    if (q >= 2) {       // up values of units (q-2)*32 + lane
                        ptx::tmem_ld32(tq + (uint32_t)c, v);
                        float* xr = s_xch + ((q - 2) * 32 + lane) * XCH_LD;
#pragma unroll
                        for (int j = 0; j < 32; ++j) xr[j] = v[j];
                    }
                    epi_bar();
                    if (q < 2) {        // gate values of units q*32 + lane
                        ptx::tmem_ld32(tq + (uint32_t)c, v);
                        const float* xr = s_xch + (q * 32 + lane) * XCH_LD;
                        const int u = q * 32 + lane;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            s_out[j * OUT_LD + u] = __float2bfloat16_rn(silu(v[j]) * xr[j]);
                    }
                } else {
                    ptx::tmem_ld32(tq + (uint32_t)c, v);
                    const int u = q * 32 + lane;
                    const int ug = ubase + u;
                    const float b = (bias && ug < t.N) ? __bfloat162float(bias[ug]) : 0.f;
                    if (MODE == kModeGelu) {
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            s_out[j * OUT_LD + u] = __float2bfloat16_rn(gelu_erf(v[j] + b));
                    } else {
                        epi_bar();      // token metadata is in place
#pragma unroll
                        for (int j = 0; j < 32; ++j) {
                            const float w = (c + j < t.ntok) ? s_tok_w[c + j] : 0.f;
                            s_out[j * OUT_LD + u] = __float2bfloat16_rn(w * (v[j] + b));
                        }
                    }
                }
                epi_bar();
                // 32 staged rows of UNITS_CTA outputs -> global, 16 bytes per store
                constexpr int VPR = UNITS_CTA / 8;              // 16-byte vectors per row
                for (int i = et; i < 32 * VPR; i += EPI_THREADS) {
                    const int j = i / VPR, vv = i - j * VPR;
                    const int col = ubase + vv * 8;
                    if (c + j < t.ntok && col < t.N) {
                        const int row = (MODE == kModeDown) ? s_tok_a[c + j] : t.tok0 + c + j;
                        const uint4 val = *reinterpret_cast<const uint4*>(s_out + j * OUT_LD + vv * 8);
                        *reinterpret_cast<uint4*>(out_base + (size_t)row * t.N + col) = val;
                    }
                }
                epi_bar();
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive_cluster(tempty_leader + 8u * acc);
        }
    }

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
    auto kernel = ffn_swap_kernel<MODE>;
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

int ffn_swap_weight_box_rows(int mode) { return mode == kModeSwiglu ? 64 : 128; }

cudaError_t launch_ffn_swap(int mode, const CUtensorMap* maps, const TcFfnArgs& p, cudaStream_t st) {
    if (mode == kModeSwiglu) return launch_mode<kModeSwiglu>(maps, p, st);
    if (mode == kModeGelu) return launch_mode<kModeGelu>(maps, p, st);
    return launch_mode<kModeDown>(maps, p, st);
}

}  // namespace moe
