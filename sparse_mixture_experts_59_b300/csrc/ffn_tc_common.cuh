// ffn_tc_common.cuh -- tile decoding and fused epilogues shared by the 1-SM
// (ffn_tc.cu) and 2-SM (ffn_tc2.cu) tcgen05 grouped-GEMM kernels.
#pragma once

#include "common.cuh"
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace tcffn {

constexpr int BK = 64;   // bf16 elements per 128-byte swizzled row (one K block)

template <int MODE> struct ModeTraits;
template <> struct ModeTraits<kModeSwiglu> { static constexpr int BN_OUT = 128; };
template <> struct ModeTraits<kModeGelu> { static constexpr int BN_OUT = 256; };
template <> struct ModeTraits<kModeDown> { static constexpr int BN_OUT = 256; };

struct Tile {
    int g;             // group (E = shared expert)
    bool sh;
    int arow;          // first A row of the tile in its tensor map
    int row_end;       // one past the segment's last A row
    int n0;            // first output column
    int wrow0, wrow1;  // weight rows of the two 128-row B boxes
    int N, nk;
};

// Tile `tile` of the (group, N-tile, M-tile) enumeration, M-tiles of TILE_M
// rows, M fastest so that consecutive tiles share a weight tile in L2.
template <int MODE, int TILE_M>
__device__ __forceinline__ Tile decode_tile(const TcFfnArgs& p, const int* s_start,
                                            const int* s_off, int G, int tile) {
    constexpr int BN_OUT = ModeTraits<MODE>::BN_OUT;
    Tile t;
    t.g = find_group(s_start, G, tile);
    t.sh = (t.g == p.E);
    const int seg0 = t.sh ? 0 : s_off[t.g];
    const int rows = t.sh ? p.rows_sh : s_off[t.g + 1] - seg0;
    const int mt = (rows + TILE_M - 1) / TILE_M;
    const int local = tile - s_start[t.g];
    const int n = local / mt, m = local - n * mt;
    t.arow = seg0 + m * TILE_M;
    t.row_end = seg0 + rows;
    t.N = t.sh ? p.N_sh : p.N;
    const int K = t.sh ? p.K_sh : p.K;
    t.nk = (K + BK - 1) / BK;
    t.n0 = n * BN_OUT;
    const int wbase = t.sh ? 0 : t.g * p.N;
    if (MODE == kModeSwiglu) {
        t.wrow0 = wbase + t.n0;      // gate rows (map B)
        t.wrow1 = wbase + t.n0;      // up rows   (map B2)
    } else {
        t.wrow0 = wbase + t.n0;
        t.wrow1 = wbase + t.n0 + 128;
    }
    return t;
}

__device__ __forceinline__ void store_row32(__nv_bfloat16* dst, const float (&v)[32], int ncols) {
    // ncols = valid columns from dst on (a multiple of 8, possibly > 32)
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        if (q * 8 < ncols) {
            const uint4 pk = make_uint4(pack_bf16x2(v[q * 8 + 0], v[q * 8 + 1]),
                                        pack_bf16x2(v[q * 8 + 2], v[q * 8 + 3]),
                                        pack_bf16x2(v[q * 8 + 4], v[q * 8 + 5]),
                                        pack_bf16x2(v[q * 8 + 6], v[q * 8 + 7]));
            reinterpret_cast<uint4*>(dst)[q] = pk;
        }
    }
}

// Epilogue of one accumulator for the calling thread's row r (a global A row
// of tile t): taddr is the TMEM address of the warp's lane quadrant at the
// accumulator's first column.  Called by whole warps (tcgen05.ld is aligned);
// rows past the segment end load but do not store.
//   Swiglu: cols [0,128) = gate, [128,256) = up;  H[r] = silu(g) * u
//   Gelu:   H[r] = gelu_erf(acc + b1)
//   Down:   Ys[perm_src[r]] = topk_w * (acc + b2); shared group: Sh[r] = acc
template <int MODE>
__device__ __forceinline__ void epilogue_tile(const TcFfnArgs& p, const Tile& t, uint32_t taddr,
                                              int r) {
    constexpr int BN_OUT = ModeTraits<MODE>::BN_OUT;
    const bool row_ok = r < t.row_end;
    if (MODE == kModeSwiglu) {
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(t.sh ? p.out_sh : p.out) +
                             (size_t)r * t.N + t.n0;
#pragma unroll 1
        for (int c = 0; c < BN_OUT; c += 32) {
            __syncwarp();
            float g[32], u[32];
            ptx::tmem_ld32(taddr + c, g);
            ptx::tmem_ld32(taddr + 128 + c, u);
            const int ncols = t.N - (t.n0 + c);
            if (row_ok && ncols > 0) {
#pragma unroll
                for (int j = 0; j < 32; ++j) g[j] = silu(g[j]) * u[j];
                store_row32(dst + c, g, ncols);
            }
        }
    } else if (MODE == kModeGelu) {
        __nv_bfloat16* dst = reinterpret_cast<__nv_bfloat16*>(t.sh ? p.out_sh : p.out) +
                             (size_t)r * t.N + t.n0;
        const __nv_bfloat16* bias = (p.bias && !t.sh) ? p.bias + (size_t)t.g * t.N : nullptr;
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
                    const float b = (bias && n < t.N) ? __bfloat162float(bias[n]) : 0.f;
                    v[j] = gelu_erf(v[j] + b);
                }
                store_row32(dst + c, v, ncols);
            }
        }
    } else {   // kModeDown
        __nv_bfloat16* dst = nullptr;
        float scale = 1.f;
        if (row_ok) {
            if (t.sh) {
                dst = reinterpret_cast<__nv_bfloat16*>(p.out_sh) + (size_t)r * t.N + t.n0;
            } else {
                const int a = p.perm_src[r];
                scale = p.gate_w[a];
                dst = reinterpret_cast<__nv_bfloat16*>(p.out) + (size_t)a * t.N + t.n0;
            }
        }
        const __nv_bfloat16* bias = (p.bias && !t.sh) ? p.bias + (size_t)t.g * t.N : nullptr;
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
                    const float b = (bias && n < t.N) ? __bfloat162float(bias[n]) : 0.f;
                    v[j] = scale * (v[j] + b);
                }
                store_row32(dst + c, v, ncols);
            }
        }
    }
}

}  // namespace tcffn
}  // namespace moe
