// ffn_fp8.cu -- grouped expert GEMMs with FP8 (E4M3) expert weights.
//
// The low-bit-weights variant of the expert FFNs: expert weights are stored
// as E4M3 codes q with one fp32 scale per output row, w = q * s, which halves
// the bytes that cross HBM -- the bound of decode-sized batches ("How Mixture
// of Experts Works", "Quantization for MoE": quantised expert weights).  The
// maths is that of ffn_tc.cu on the dequantised weights:
//   SwiGLU  H = silu(s1 (A q1^T)) * (s3 (A q3^T))
//   GELU    H = gelu(s1 (A q1^T) + b1)
//   down    Ys[perm_src[r]] = topk_w * (s2 (H q2^T) + b2)
// Tokens on M (128-row tiles), one CTA per SM, 320 threads:
//   warp 0      TMA: f16 token tile 128x64 and the FP8 weight tile 256x64
//               (no swizzle, 64-byte rows) into a 4-stage ring;
//   warps 6-9   converters: E4M3 -> f16 (exact) straight into the 128-byte
//               swizzled operand layout of one of two f16 weight buffers,
//               then a proxy fence so the tensor core sees the writes;
//   warp 1      TMEM + tcgen05.mma kind::f16 (M=128, N=256, K=16);
//   warps 2-5   epilogue: scale the fp32 accumulator by the row scales, fused
//               activation / gate scale, f16 H (A operand of the down GEMM)
//               or bf16 slot outputs.
#include <cuda_fp16.h>

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

constexpr int BM = 128;
constexpr int MMA_N = 256;
constexpr int STAGES = 4;
constexpr int NB16 = 2;
constexpr int A_BYTES = BM * BK * 2;          // f16 tokens
constexpr int BQ_BYTES = MMA_N * BK;           // FP8 weights, 64-byte rows
constexpr int B16_BYTES = MMA_N * BK * 2;      // converted f16 weights, swizzled
constexpr int TMEM_COLS = 512;
constexpr int NUM_THREADS = 320;
constexpr int CVT_THREADS = 128;
constexpr uint32_t IDESC = ptx::idesc_f16_f32(BM, MMA_N);

constexpr int OFF_A = 0;
constexpr int OFF_BQ = STAGES * A_BYTES;
constexpr int OFF_B16 = OFF_BQ + STAGES * BQ_BYTES;
constexpr int OFF_BAR = OFF_B16 + NB16 * B16_BYTES;
constexpr int NUM_BARS = 2 * STAGES + 2 * NB16 + 2 + 2 + 1;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int OFF_START = OFF_MISC + 16;
constexpr int OFF_OFFS = OFF_START + (kMaxExperts + 2) * 4;
constexpr int SMEM_USED = OFF_OFFS + (kMaxExperts + 2) * 4;
constexpr int SMEM_BYTES = SMEM_USED + 1024;
static_assert(OFF_B16 % 1024 == 0, "swizzled f16 operand buffers need 1024-byte alignment");
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");

__device__ __forceinline__ void store_row32_f16(__half* dst, const float (&v)[32], int ncols) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if (q * 8 < ncols) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const __half2 h = __floats2half2_rn(v[q * 8 + 2 * j], v[q * 8 + 2 * j + 1]);
                w[j] = *reinterpret_cast<const uint32_t*>(&h);
            }
            reinterpret_cast<uint4*>(dst)[q] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// Epilogue of one accumulator for the thread's row r (a global A row).
template <int MODE>
__device__ __forceinline__ void epilogue_fp8(const TcFfnArgs& p, const Tile& t, uint32_t taddr,
                                             int r) {
    constexpr int BN_OUT = ModeTraits<MODE>::BN_OUT;
    const bool row_ok = r < t.row_end;
    const size_t srow = (size_t)t.g * t.N;          // this group's first scale
    if (MODE == kModeSwiglu) {
        __half* dst = reinterpret_cast<__half*>(p.out) + (size_t)r * t.N + t.n0;
#pragma unroll 1
        for (int c = 0; c < BN_OUT; c += 32) {
            __syncwarp();
            float g[32], u[32];
            ptx::tmem_ld32(taddr + c, g);
            ptx::tmem_ld32(taddr + 128 + c, u);
            const int ncols = t.N - (t.n0 + c);
            if (row_ok && ncols > 0) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int n = t.n0 + c + j;
                    const float sg = n < t.N ? p.wscale[srow + n] : 0.f;
                    const float su = n < t.N ? p.wscale2[srow + n] : 0.f;
                    g[j] = silu(g[j] * sg) * (u[j] * su);
                }
                store_row32_f16(dst + c, g, ncols);
            }
        }
    } else if (MODE == kModeGelu) {
        __half* dst = reinterpret_cast<__half*>(p.out) + (size_t)r * t.N + t.n0;
        const __nv_bfloat16* bias = p.bias ? p.bias + srow : nullptr;
#pragma unroll 1
        for (int c = 0; c < BN_OUT; c += 32) {
            __syncwarp();
            float v[32];
            ptx::tmem_ld32(taddr + c, v);
            const int ncols = t.N - (t.n0 + c);
            if (row_ok && ncols > 0) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int n = t.n0 + c + j;
                    const float sc = n < t.N ? p.wscale[srow + n] : 0.f;
                    const float b = (bias && n < t.N) ? __bfloat162float(bias[n]) : 0.f;
                    v[j] = gelu_erf(v[j] * sc + b);
                }
                store_row32_f16(dst + c, v, ncols);
            }
        }
    } else {
        __nv_bfloat16* dst = nullptr;
        float gate = 1.f;
        if (row_ok) {
            const int a = p.perm_src[r];
            gate = p.gate_w[a];
            dst = reinterpret_cast<__nv_bfloat16*>(p.out) + (size_t)a * t.N + t.n0;
        }
        const __nv_bfloat16* bias = p.bias ? p.bias + srow : nullptr;
#pragma unroll 1
        for (int c = 0; c < BN_OUT; c += 32) {
            __syncwarp();
            float v[32];
            ptx::tmem_ld32(taddr + c, v);
            const int ncols = t.N - (t.n0 + c);
            if (row_ok && ncols > 0) {
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int n = t.n0 + c + j;
                    const float sc = n < t.N ? p.wscale[srow + n] : 0.f;
                    const float b = (bias && n < t.N) ? __bfloat162float(bias[n]) : 0.f;
                    v[j] = gate * (v[j] * sc + b);
                }
                tcffn::store_row32(dst + c, v, ncols);
            }
        }
    }
}

template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
ffn_fp8_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
               const __grid_constant__ CUtensorMap mapB2, const TcFfnArgs p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem + OFF_A;
    uint8_t* sBq = smem + OFF_BQ;
    uint8_t* sB16 = smem + OFF_B16;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* full = bars;                       // TMA landed (tokens + FP8 weights)
    uint64_t* empty = full + STAGES;             // MMA done with the stage
    uint64_t* cfull = empty + STAGES;            // converted f16 weights ready
    uint64_t* cempty = cfull + NB16;             // MMA done with the f16 buffer
    uint64_t* tfull = cempty + NB16;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
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
        for (int b = 0; b < NB16; ++b) {
            ptx::mbar_init(&cfull[b], CVT_THREADS);
            ptx::mbar_init(&cempty[b], 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&tfull[a], 1);
            ptx::mbar_init(&tempty[a], 128);
        }
        ptx::mbar_init(drain, 1);
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
    pdl_wait();
    pdl_trigger();
    for (int i = threadIdx.x; i <= p.E; i += NUM_THREADS) s_off[i] = p.offsets[i];
    constexpr int BN_OUT = ModeTraits<MODE>::BN_OUT;
    const int nt_r = (p.N + BN_OUT - 1) / BN_OUT;
    group_tile_prefix(p.offsets, p.E, 0, BM, nt_r, 0, s_start);
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const int G = p.E;
    const int total = s_start[G];

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
                const Tile t = tcffn::decode_tile<MODE, BM>(p, s_start, s_off, G, tile);
                const CUtensorMap* mB1 = (MODE == kModeSwiglu) ? &mapB2 : &mapB;
                for (int kb = 0; kb < t.nk; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
                    if (!ptx::mbar_wait(&empty[s], ph ^ 1u, s_abort)) { ok = false; break; }
                    ptx::mbar_arrive_expect_tx(&full[s], A_BYTES + BQ_BYTES);
                    ptx::tma_load_2d(sA + s * A_BYTES, &mapA, &full[s], kb * BK, t.arow);
                    ptx::tma_load_2d(sBq + s * BQ_BYTES, &mapB, &full[s], kb * BK, t.wrow0);
                    ptx::tma_load_2d(sBq + s * BQ_BYTES + BQ_BYTES / 2, mB1, &full[s], kb * BK,
                                     t.wrow1);
                }
            }
            if (!ok) {
                *s_abort = 1;
                raise_error(p.status, MOE_ERR_DEVICE_TIMEOUT);
            }
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
                    const int s = it % STAGES, b = it % NB16;
                    const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
                    const uint32_t bph = (uint32_t)(it / NB16) & 1u;
                    if (!ptx::mbar_wait(&full[s], ph, s_abort)) { ok = false; break; }
                    if (!ptx::mbar_wait(&cfull[b], bph, s_abort)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint64_t ad = ptx::sw128_desc(ptx::smem_u32(sA + s * A_BYTES));
                    const uint64_t bd = ptx::sw128_desc(ptx::smem_u32(sB16 + b * B16_BYTES));
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        ptx::mma_bf16(d_tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2),
                                      IDESC, (kb | kk) != 0 ? 1u : 0u);
                    ptx::mma_commit(&empty[s]);
                    ptx::mma_commit(&cempty[b]);
                }
                if (!ok) break;
                ptx::mma_commit(&tfull[acc]);
            }
            if (!ok) {
                *s_abort = 1;
                raise_error(p.status, MOE_ERR_DEVICE_TIMEOUT);
            }
            ptx::mma_commit(drain);
            ptx::mbar_wait(drain, 0, nullptr);
        }
    } else if (warp >= 6) {
        // -------------------------------------------------------- converters
        // 256 weight rows x 8 chunks of 8 E4M3 bytes per stage; chunk c of row
        // r becomes 16 f16 bytes at r*128 + ((c ^ (r & 7)) * 16), the 128-byte
        // swizzle the MMA's operand descriptor expects.
        const int ct = threadIdx.x - 6 * 32;
        int it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
            const Tile t = tcffn::decode_tile<MODE, BM>(p, s_start, s_off, G, tile);
            for (int kb = 0; kb < t.nk; ++kb, ++it) {
                const int s = it % STAGES, b = it % NB16;
                const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
                const uint32_t bph = (uint32_t)(it / NB16) & 1u;
                int w = 1;
                if (lane == 0)
                    w = ptx::mbar_wait(&full[s], ph, s_abort) &&
                        ptx::mbar_wait(&cempty[b], bph ^ 1u, s_abort);
                w = __shfl_sync(0xffffffffu, w, 0);
                if (!w) { ok = false; break; }
                const uint8_t* src = sBq + s * BQ_BYTES;
                uint8_t* dst = sB16 + b * B16_BYTES;
#pragma unroll 4
                for (int i = 0; i < (MMA_N * 8) / CVT_THREADS; ++i) {
                    const int j = ct + CVT_THREADS * i;
                    const int r = j >> 3, c = j & 7;
                    const uint2 q = *reinterpret_cast<const uint2*>(src + r * 64 + c * 8);
                    const uint4 h = make_uint4(ptx::cvt_e4m3x2_f16x2((uint16_t)(q.x & 0xffffu)),
                                               ptx::cvt_e4m3x2_f16x2((uint16_t)(q.x >> 16)),
                                               ptx::cvt_e4m3x2_f16x2((uint16_t)(q.y & 0xffffu)),
                                               ptx::cvt_e4m3x2_f16x2((uint16_t)(q.y >> 16)));
                    *reinterpret_cast<uint4*>(dst + r * 128 + ((c ^ (r & 7)) << 4)) = h;
                }
                ptx::fence_proxy_async_smem();
                ptx::mbar_arrive(&cfull[b]);
            }
        }
        if (!ok && lane == 0) {
            *s_abort = 1;
            raise_error(p.status, MOE_ERR_DEVICE_TIMEOUT);
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;
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
            epilogue_fp8<MODE>(p, t, taddr, t.arow + row_in_tile);
            ptx::tc_fence_before();
            ptx::mbar_arrive(&tempty[acc]);
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace

cudaError_t launch_ffn_fp8(int mode, const CUtensorMap* maps, const TcFfnArgs& p, int num_sms,
                           cudaStream_t st) {
    auto kernel = mode == kModeSwiglu ? ffn_fp8_kernel<kModeSwiglu>
                : mode == kModeGelu ? ffn_fp8_kernel<kModeGelu> : ffn_fp8_kernel<kModeDown>;
    const cudaError_t err =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (err != cudaSuccess) return err;
    return launch_kernel(kernel, dim3(num_sms), dim3(NUM_THREADS), SMEM_BYTES, st, 1, maps[0],
                         maps[1], maps[2], p);
}

}  // namespace moe
