// ffn_fp8.cu -- grouped expert GEMMs with low-bit expert weights: FP8 (E4M3)
// codes, or packed 4-bit (E2M1) codes with E4M3 block scales.
//
// The low-bit-weights variant of the expert FFNs: expert weights are stored
// as codes q with one fp32 scale per output row, w = q * s (for 4-bit codes
// q = code * block scale, one block scale per 16 values), which halves (E4M3)
// or cuts to 0.31 (packed E2M1) the bytes that cross HBM -- the bound of
// decode-sized batches ("How Mixture of Experts Works", "Quantization for
// MoE": quantised expert weights).  The maths is that of ffn_tc.cu on the
// dequantised weights:
//   SwiGLU  H = silu(s1 (A q1^T)) * (s3 (A q3^T))
//   GELU    H = gelu(s1 (A q1^T) + b1)
//   down    Ys[perm_src[r]] = topk_w * (s2 (H q2^T) + b2)
//
// Decode batches give each expert a handful of tokens, so the weights are the
// MMA's M operand and the tokens its N operand (at most 32 per tile, rounded
// up to 16).  A weight block is 128 rows: 64 gate + 64 up rows of the same
// hidden units for SwiGLU, else 128 consecutive outputs.  A tile is G = 4
// weight blocks of one expert against one token tile, so that each k-block of
// tokens is loaded once for 4 blocks.  (While the weight stream saturates HBM
// every load of an SM waits several microseconds -- its in-flight bytes over
// its share of the bandwidth -- L2 hits included; token loads of 4 KB per 16 KB
// weight stage would both slow the weight stream and arrive late for the
// MMAs.)
//
// The converted f16 weights go to tensor memory, which the MMA reads as its A
// operand: staging them in shared memory instead would move about 6.5
// shared-memory bytes per weight byte (TMA write, converter read and write,
// MMA read), which at 128 B/clock caps the weight stream near the HBM rate;
// through TMEM it is 2 bytes.
//
// One CTA per SM, 384 threads for E4M3 and 512 for E2M1; the warps that issue TMA or MMA instructions
// sit on different schedulers (warp % 4), as issuing them slows the other
// warps of the scheduler (measured: a converter warp sharing its scheduler
// with two MMA issuers ran ~2400 clocks behind one sharing with none, and the
// slowest converter gates both the weight ring and the MMAs):
//   warp 0      TMA: weight rows (E4M3: 128 bytes of K, 128-byte swizzle;
//               E2M1: 80 bytes) into rings of stages (one ring per converter
//               set, 160 KB in all; a stage is one E4M3 block or two E2M1
//               blocks) that the converters release as soon as they hold a
//               stage's codes in registers;
//   warp 1      TMEM owner; TMA: the tile's f16 token rows (128-byte swizzle)
//               in chunks of up to 24 KB into two buffers, a chunk ahead;
//   warps 6..   converters, one set (E4M3) or two (E2M1) of one warp per
//               TMEM lane quadrant; set z takes the stages of its blocks from
//               a ring of its own, thread = weight row: codes -> f16 pairs in
//               registers, tcgen05.st into the TMEM A buffer of each block;
//   last two    MMA issuers, issuer i for blocks 2i and 2i + 1:
//               tcgen05.mma kind::f16 (M=128, N=tokens, K=16), A from the
//               block's TMEM buffer, B (tokens) from shared memory, into the
//               block's accumulator.  A thread issues a small MMA only every
//               ~50-100 clocks and a block needs 8 per k-block, so one issuer
//               could not keep up with the weight stream;
//   warps 2-5   epilogue: row scales, fused activation / gate scale, f16 H
//               (A operand of the down GEMM) or bf16 slot outputs.  The
//               scales, biases and token slots of a tile are copied to shared
//               memory before its accumulators are ready: a global load waits
//               several microseconds while the weight stream runs.
//
// The waits of the warps off the critical path (producers, issuers, epilogue)
// sleep between polls: the converters that share their schedulers are the
// bound, and polling takes issue slots from them (measured: 4% on the 4-bit
// up-projection of a decode batch).
//
// Every E4M3 value (subnormals included, |v| <= 448) is an f16 value, so the
// conversion (cvt.rn.f16x2.e4m3x2, two codes per instruction) is exact and the
// products with the f16 tokens are exact in the fp32 accumulator.  (Measured:
// the conversion instruction beats a bit re-layout on the integer pipe, which
// needs 7 operations per 4 codes and leaves the converters ALU-bound.)
//
// Work balance (stream-K): the W = tiles x k-blocks units of work are cut into
// one contiguous range per CTA.  A tile that lies in one range is finished
// from TMEM; a tile that straddles ranges is accumulated in parts, each part
// writes fp32 partial sums to its CTA's slot, and the CTA that finishes the
// tile's last part (a ticket counter) adds the parts in CTA order and runs the
// epilogue -- deterministic whatever the finishing order.  A CTA takes its
// shared tiles first (the one its range starts inside, the one it ends inside)
// and its whole tiles after, so that the partial sums and their reductions
// overlap the work that follows instead of trailing it.
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.cuh"
#include "launch.cuh"
#include "tc_lowbit.cuh"

namespace moe {

namespace {

constexpr int BK = 128;                        // K values per stage
constexpr int WROWS = 128;                     // weight rows per block (MMA M, TMEM lanes)
constexpr int G = 4;                           // weight blocks per tile
constexpr int NISS = 2;                        // MMA issuers
constexpr int TOK = 32;                        // tokens per tile at most (MMA N)
constexpr int TOK_BOX = 16;                    // token rows per TMA box
constexpr int TB_BYTES = 24 * 1024;            // token chunk buffer (two of them)
constexpr int A_COLS = BK / 2;                 // TMEM columns of one A buffer (f16 pairs)
constexpr int ACC_SET = G * TOK;               // TMEM columns of a tile's accumulators
constexpr int A_COL0 = 2 * ACC_SET;            // two accumulator sets, then the A buffers
constexpr int TMEM_COLS = 512;
static_assert(A_COL0 + G * A_COLS <= TMEM_COLS, "tensor memory budget (an A buffer per block)");
constexpr int TOKP_WARP = 1;                   // token producer (and TMEM owner)
constexpr int XCH_LD = 33;

// Weight formats.  Both give a block 128 values of each weight row (one MMA K
// range of 128): E4M3 rows of 128 bytes (128-byte swizzle), or packed E2M1
// rows of 80 bytes (64 code bytes, 8 E4M3 block scales, 8 zero bytes; 80-byte
// rows put the 16-byte pieces of 8 consecutive rows in 8 different bank
// groups without a swizzle).
//
// A ring stage holds SB blocks of one k-block in two boxes of SB * 64 rows
// (packed E2M1: SB = 2, 20 KB stages).  Each stage costs the producer, the
// converters and the barriers a fixed number of clocks whatever its size, and
// with one 10 KB block of E2M1 per stage that cost, not HBM, set the weight
// stream's pace (measured: a bare TMA ring of 10 KB stages streams 5.2 TB/s,
// of 20 KB stages 6.6 TB/s, at the same 160 KB in flight).
//
// The converters are SETS sets of four warps; set z converts blocks BPS z ..
// BPS z + BPS - 1 of every k-block.  Each set has a ring of its own (RS
// slots): a slot shared by two consumers that run at their own pace could see
// its barrier two phases ahead of one of them, where a parity wait cannot
// tell the phases apart.  Packed E2M1 has two sets (a block's conversion
// costs twice E4M3's: a cvt and a block-scale multiply per code pair); E4M3
// has one (measured: a second set made its stream-bound up-projection ~5%
// slower).
enum { kFmtE4M3 = 0, kFmtE2M1 = 1 };
constexpr int BPI = G / NISS;                  // blocks per MMA issuer
static_assert(G % NISS == 0, "whole blocks per issuer");
template <int FMT>
struct WF {
    static constexpr int ROW_BYTES = FMT == kFmtE4M3 ? 128 : 80;
    static constexpr int SB = FMT == kFmtE4M3 ? 1 : 2;          // blocks per ring stage
    static constexpr int BLK_BYTES = WROWS * ROW_BYTES;         // one block of a k-block
    static constexpr int WQ_BYTES = SB * BLK_BYTES;             // one ring stage
    static constexpr int SETS = FMT == kFmtE4M3 ? 1 : 2;        // converter sets
    static constexpr int BPS = G / SETS;                        // blocks per converter set
    static constexpr int RS = FMT == kFmtE4M3 ? 10 : 4;         // slots per set: 160 KB in flight
    static constexpr int WSTAGES = SETS * RS;
    static constexpr int CVT_WARPS = 4 * SETS;                  // one warp per lane quadrant and set
    static_assert(G % SETS == 0 && BPS % SB == 0, "a set's blocks are whole stages");
    static constexpr int MMA_WARP0 = 6 + CVT_WARPS;             // first MMA issuer
    static constexpr int NUM_THREADS = (MMA_WARP0 + NISS) * 32;
    static constexpr int OFF_TOK = 0;
    static constexpr int OFF_WQ = OFF_TOK + 2 * TB_BYTES;
    static constexpr int OFF_XCH = OFF_WQ + WSTAGES * WQ_BYTES;
    static constexpr int OFF_PRE = OFF_XCH + 64 * XCH_LD * 4;   // [2][G][128] row scales, biases
    static constexpr int OFF_TOKA = OFF_PRE + 2 * G * WROWS * 4;
    static constexpr int OFF_TOKW = OFF_TOKA + 2 * TOK * 4;     // token slots and weights, 2 buffers
    static constexpr int OFF_BAR = OFF_TOKW + 2 * TOK * 4;
    static constexpr int NUM_BARS = 2 * WSTAGES + 2 + 2 + 2 * G + 2 + 2 + NISS + 1;
    static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
    static constexpr int OFF_START = OFF_MISC + 32;
    static constexpr int OFF_OFFS = OFF_START + (kMaxExperts + 2) * 4;
    static constexpr int SMEM_USED = OFF_OFFS + (kMaxExperts + 2) * 4;
    static constexpr int SMEM_BYTES = SMEM_USED + 1024;
    static_assert(MMA_WARP0 % 4 == 2 && NISS <= 4, "issuers on different schedulers");
    static_assert(OFF_TOK % 1024 == 0 && TB_BYTES % 1024 == 0, "swizzled token atoms");
    static_assert(OFF_WQ % 1024 == 0 && (FMT != kFmtE4M3 || WQ_BYTES % 1024 == 0),
                  "swizzled weight stages");
    static_assert(BLK_BYTES % 1024 == 0 || FMT != kFmtE4M3, "swizzled second box");
    static_assert(BLK_BYTES % 256 == 0, "128-byte aligned weight boxes");
    static_assert(SETS <= 2, "ring bookkeeping for up to two sets");
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};
template struct WF<kFmtE4M3>;
template struct WF<kFmtE2M1>;

template <int MODE>
struct Fp8Traits {
    // output units (hidden units for SwiGLU, output columns otherwise) per block
    static constexpr int UNITS = MODE == kModeSwiglu ? 64 : 128;
};

// Four E4M3 codes (byte i = code i) -> four f16 of the same values, in two
// words (codes 0,1 in lo; 2,3 in hi; lower code in the lower half).
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t x, uint32_t& lo, uint32_t& hi) {
    lo = ptx::cvt_e4m3x2_f16x2((uint16_t)(x & 0xffffu));
    hi = ptx::cvt_e4m3x2_f16x2((uint16_t)(x >> 16));
}

// Stream-K ranges: CTA c owns work units [cta_start(c), cta_start(c + 1)).
__device__ __forceinline__ long long cta_start(long long W, int grid, int c) {
    return (long long)c * W / grid;
}
// The CTA that owns unit x: the largest c with cta_start(c) <= x.
__device__ __forceinline__ int cta_of(long long x, long long W, int grid) {
    return (int)(((x + 1) * grid + W - 1) / W) - 1;
}

// One CTA's part of one tile: k-blocks [kb0, kb1).
struct Seg {
    int tile;
    int g;             // expert
    int tok0, ntok;    // first gathered row, valid tokens
    int nmma;          // MMA N: ntok rounded up to 16
    int blk0, nblk;    // first weight block (within the expert), blocks in the tile
    int kb0, kb1;
    int c_first, c_last;  // CTAs whose ranges meet the tile
};

// Tiles enumerate (expert, block group, token tile), token tile fastest.
__device__ __forceinline__ Seg decode_seg(const TcFfnArgs& p, const int* s_start, const int* s_off,
                                          int nwb, int nk, long long W, int tile, int kb0,
                                          int kb1) {
    Seg t;
    t.tile = tile;
    t.g = find_group(s_start, p.E, tile);
    const int seg0 = s_off[t.g];
    const int rows = s_off[t.g + 1] - seg0;
    const int ntt = (rows + TOK - 1) / TOK;
    const int local = tile - s_start[t.g];
    const int wbg = local / ntt, tt = local - wbg * ntt;
    t.tok0 = seg0 + tt * TOK;
    t.ntok = min(TOK, rows - tt * TOK);
    t.nmma = (t.ntok + 15) & ~15;
    t.blk0 = wbg * G;
    t.nblk = min(G, nwb - t.blk0);
    t.kb0 = kb0;
    t.kb1 = kb1;
    const int grid = (int)gridDim.x;
    t.c_first = cta_of((long long)tile * nk, W, grid);
    t.c_last = cta_of((long long)tile * nk + nk - 1, W, grid);
    return t;
}

// First weight rows of the two boxes of stage st of a tile (blocks SB st ..):
// SwiGLU: the gate rows (W1) and the up rows (W3) of the stage's 128 hidden
// units; otherwise the stage's blocks one after the other, a box each.
template <int MODE, int SB>
__device__ __forceinline__ int2 stage_rows(const TcFfnArgs& p, const Seg& t, int st) {
    const int u0 = (t.blk0 + st * SB) * Fp8Traits<MODE>::UNITS;
    const int r0 = t.g * p.N + u0;
    return make_int2(r0, MODE == kModeSwiglu ? r0 : r0 + SB * 64);
}
// Shared-memory row, within its stage, of row r of the stage's block jl.
template <int MODE, int SB>
__device__ __forceinline__ int stage_row(int jl, int r) {
    if (MODE == kModeSwiglu) return r < 64 ? jl * 64 + r : SB * 64 + jl * 64 + (r - 64);
    return jl * WROWS + r;
}

// Named barrier of the four epilogue warps.  Each warp reconverges first:
// bar.sync counts a warp's arrival as the whole warp, and one lane may still
// be in a branch of its own (the ticket of a shared tile): arriving without
// it would release the barrier early and pair the warps' later barriers up
// out of step.
__device__ __forceinline__ void epi_bar() {
    __syncwarp();
    asm volatile("bar.sync 1, 128;" ::: "memory");
}

// Epilogue of one block's accumulator (tokens 0..31) for the calling thread's
// weight row `row`; v holds the sums over the unscaled codes.
// Row scales and biases of the tile's blocks for the calling thread's weight
// row, into its own slots of the prefetch area.
template <int MODE>
__device__ __forceinline__ void prefetch_rows(const TcFfnArgs& p, const Seg& t, int row,
                                              float* s_pre) {
    const size_t sbase = (size_t)t.g * p.N;
    for (int j = 0; j < t.nblk; ++j) {
        const int u0 = (t.blk0 + j) * Fp8Traits<MODE>::UNITS;
        float sc = 0.f, b = 0.f;
        if (MODE == kModeSwiglu) {
            const int u = u0 + (row & 63);
            if (u < p.N) sc = (row < 64 ? p.wscale : p.wscale2)[sbase + u];
        } else {
            const int n = u0 + row;
            if (n < p.N) {
                sc = p.wscale[sbase + n];
                if (p.bias) b = __bfloat162float(p.bias[sbase + n]);
            }
        }
        s_pre[j * WROWS + row] = sc;
        s_pre[G * WROWS + j * WROWS + row] = b;
    }
}

template <int MODE>
__device__ __forceinline__ void finish_block(const TcFfnArgs& p, const Seg& t, int j, int row,
                                             float (&v)[32], float* s_xch, const float* s_pre,
                                             const int* s_tok_a, const float* s_tok_w) {
    const int u0 = (t.blk0 + j) * Fp8Traits<MODE>::UNITS;
    const float sc = s_pre[j * WROWS + row];
    if (MODE == kModeSwiglu) {
        const int u = u0 + (row & 63);
        const bool u_ok = u < p.N;
        if (row >= 64) {
            float* xr = s_xch + (row - 64) * XCH_LD;
#pragma unroll
            for (int c = 0; c < 32; ++c) xr[c] = v[c] * sc;
        }
        epi_bar();
        if (row < 64 && u_ok) {
            const float sg = sc;
            const float* xr = s_xch + row * XCH_LD;
            __half* H = reinterpret_cast<__half*>(p.out);
#pragma unroll
            for (int c = 0; c < 32; ++c)
                if (c < t.ntok)
                    H[(size_t)(t.tok0 + c) * p.N + u] = __float2half_rn(silu(v[c] * sg) * xr[c]);
        }
        epi_bar();
    } else {
        const int n = u0 + row;
        if (n >= p.N) return;
        const float b = s_pre[G * WROWS + j * WROWS + row];
        if (MODE == kModeGelu) {
            __half* H = reinterpret_cast<__half*>(p.out);
#pragma unroll
            for (int c = 0; c < 32; ++c)
                if (c < t.ntok)
                    H[(size_t)(t.tok0 + c) * p.N + n] = __float2half_rn(gelu_erf(v[c] * sc + b));
        } else {
            __nv_bfloat16* Ys = reinterpret_cast<__nv_bfloat16*>(p.out);
#pragma unroll
            for (int c = 0; c < 32; ++c)
                if (c < t.ntok)
                    Ys[(size_t)s_tok_a[c] * p.N + n] = __float2bfloat16_rn(s_tok_w[c] * (v[c] * sc + b));
        }
    }
}

template <int MODE, int FMT>
__global__ void __launch_bounds__(WF<FMT>::NUM_THREADS, 1)
ffn_fp8_kernel(const __grid_constant__ CUtensorMap mapX, const __grid_constant__ CUtensorMap mapW,
               const __grid_constant__ CUtensorMap mapW3, const TcFfnArgs p) {
    using F = WF<FMT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sTok = smem + F::OFF_TOK;
    uint8_t* sWq = smem + F::OFF_WQ;
    float* s_xch = reinterpret_cast<float*>(smem + F::OFF_XCH);
    float* s_pre = reinterpret_cast<float*>(smem + F::OFF_PRE);
    int* s_tok_a = reinterpret_cast<int*>(smem + F::OFF_TOKA);
    float* s_tok_w = reinterpret_cast<float*>(smem + F::OFF_TOKW);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + F::OFF_BAR);
    uint64_t* wfull = bars;                      // E4M3 codes landed
    uint64_t* wempty = wfull + F::WSTAGES;          // converters hold the codes
    uint64_t* kfull = wempty + F::WSTAGES;          // a token chunk landed
    uint64_t* kempty = kfull + 2;                // the issuers done with the chunk
    uint64_t* cfull = kempty + 2;                // converted weights in block j's A buffer
    uint64_t* cempty = cfull + G;                // block j's MMAs done with it
    uint64_t* tfull = cempty + G;                // the issuers' accumulators complete
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;                // per issuer
    uint64_t* endbar = drain + NISS;             // teardown: every thread
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + F::OFF_MISC);
    volatile int* s_abort = reinterpret_cast<volatile int*>(smem + F::OFF_MISC + 4);
    volatile int* s_go = reinterpret_cast<volatile int*>(smem + F::OFF_MISC + 8);
    volatile int* s_last = reinterpret_cast<volatile int*>(smem + F::OFF_MISC + 12);
    int* s_maxrows = reinterpret_cast<int*>(smem + F::OFF_MISC + 16);
    int* s_start = reinterpret_cast<int*>(smem + F::OFF_START);
    int* s_off = reinterpret_cast<int*>(smem + F::OFF_OFFS);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < F::WSTAGES; ++s) {
            ptx::mbar_init(&wfull[s], 1);
            ptx::mbar_init(&wempty[s], 4);     // the four warps of one converter set
        }
        for (int s = 0; s < 2; ++s) {
            ptx::mbar_init(&kfull[s], 1);
            ptx::mbar_init(&kempty[s], NISS);
        }
        for (int b = 0; b < G; ++b) {
            ptx::mbar_init(&cfull[b], 4);
            ptx::mbar_init(&cempty[b], 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(&tfull[a], NISS);
            ptx::mbar_init(&tempty[a], 128);
        }
        for (int j = 0; j < NISS; ++j) ptx::mbar_init(&drain[j], 1);
        ptx::mbar_init(endbar, F::NUM_THREADS);
        *s_abort = 0;
        ptx::fence_mbarrier_init();
        ptx::prefetch_tensormap(&mapX);
        ptx::prefetch_tensormap(&mapW);
        ptx::prefetch_tensormap(&mapW3);
    }
    if (warp == 1) {
        ptx::tmem_alloc(s_tmem, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    // Only the token rows come from the kernel just before this one (the
    // gather, or the up projection for the down projection): the offsets,
    // slots and gate weights are older and the weights and scales are inputs.
    // So the weight stream starts now, over the previous kernel's tail, and
    // only the token producer waits for that kernel (pdl_wait below).  The
    // partial-sum scratch, which the two projections share, is first touched
    // by the epilogue, after MMAs that consumed waited-for tokens.
    pdl_trigger();
    for (int i = threadIdx.x; i <= p.E; i += F::NUM_THREADS) s_off[i] = p.offsets[i];
    block_sync();
    const int nwb = (p.N + Fp8Traits<MODE>::UNITS - 1) / Fp8Traits<MODE>::UNITS;
    if (warp == 0) {            // longest segment: sizes the token chunks
        int m = 0;
        for (int g = lane; g < p.E; g += 32) m = max(m, s_off[g + 1] - s_off[g]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) *s_maxrows = m;
    }
    group_tile_prefix(s_off, p.E, 0, TOK, (nwb + G - 1) / G, 0, s_start);
    ptx::tc_fence_before();
    block_sync();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const int grid = (int)gridDim.x;
    const int nk = (p.K + BK - 1) / BK;
    const long long W = (long long)s_start[p.E] * nk;
    const long long my0 = cta_start(W, grid, blockIdx.x);
    const long long my1 = cta_start(W, grid, blockIdx.x + 1);
    const long long slot_floats = (long long)WROWS * TOK;              // one block's partials
    // k-blocks per token chunk: the widest token tile fills a buffer
    const int CH = TB_BYTES / (min(TOK, max(16, (*s_maxrows + 15) & ~15)) * 256);
    // room for two slots of G blocks per CTA and a ticket per CTA
    const bool room = p.split_ticket && grid <= p.split_tickets &&
                      2LL * grid * G * slot_floats * 4 <= p.split_bytes;
    long long end = my1;
    if (!room && W > 0) {
        if (threadIdx.x == 0) raise_error(p.status, MOE_ERR_INVALID_ARG);
        end = my0;                                                    // no work
    }
    // The segments of this CTA; every role walks the same list: the shared
    // head tile (the range starts inside it), the shared tail tile (the range
    // ends inside it), then the whole tiles in order.
    const int t_first = (int)(my0 / nk);
    const int t_last = end > my0 ? (int)((end - 1) / nk) : t_first - 1;
    const int head_kb0 = (int)(my0 - (long long)t_first * nk);
    const int tail_kb1 = (int)(end - (long long)t_last * nk);
    const bool single = t_first == t_last;
    const int head_part = !single && head_kb0 > 0;
    const int tail_part = !single && tail_kb1 < nk;
    const int nseg = t_last < t_first ? 0 : single ? 1 : t_last - t_first + 1;
    auto seg_of = [&](int i, int& tile, int& kb0, int& kb1) {
        if (single) { tile = t_first; kb0 = head_kb0; kb1 = tail_kb1; return; }
        if (head_part) {
            if (i == 0) { tile = t_first; kb0 = head_kb0; kb1 = nk; return; }
            --i;
        }
        if (tail_part) {
            if (i == 0) { tile = t_last; kb0 = 0; kb1 = tail_kb1; return; }
            --i;
        }
        tile = t_first + head_part + i;
        kb0 = 0;
        kb1 = nk;
    };
#define FOR_EACH_SEG(t)                                                                    \
    for (int si_ = 0; si_ < nseg; ++si_) {                                                 \
        int tile_, kb0_, kb1_;                                                             \
        seg_of(si_, tile_, kb0_, kb1_);                                                    \
        const Seg t = decode_seg(p, s_start, s_off, nwb, nk, W, tile_, kb0_, kb1_);

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (weights)
        if (lane == 0) {
            int it = 0;
            bool ok = true, held = false;
            const int hold_it = p.hold ? *p.hold - 1 : -1;
            int used0 = 0, used1 = 0;            // stages issued into each set's ring
            FOR_EACH_SEG(t)
                const int nst = (t.nblk + F::SB - 1) / F::SB;
                for (int kb = t.kb0; ok && kb < t.kb1; ++kb)
                    for (int st = 0; st < nst; ++st, ++it) {
                        if (it == hold_it) { ok = false; held = true; break; }   // test hook
                        const int z = st * F::SB / F::BPS, u = z ? used1++ : used0++;
                        const int s = z * F::RS + u % F::RS;
                        const uint32_t ph = (uint32_t)(u / F::RS) & 1u;
                        if (!ptx::mbar_wait_nap(&wempty[s], ph ^ 1u, s_abort, 64)) { ok = false; break; }
                        ptx::mbar_arrive_expect_tx(&wfull[s], F::WQ_BYTES);
                        const int2 wr = stage_rows<MODE, F::SB>(p, t, st);
                        uint8_t* wq = sWq + s * F::WQ_BYTES;
                        ptx::tma_load_2d(wq, &mapW, &wfull[s], kb * F::ROW_BYTES, wr.x);
                        ptx::tma_load_2d(wq + F::WQ_BYTES / 2, &mapW3, &wfull[s], kb * F::ROW_BYTES, wr.y);
                    }
                if (!ok) break;
            }
            if (!ok && !held) {
                *s_abort = 1;
                raise_error(p.status, MOE_ERR_DEVICE_TIMEOUT);
            }
            for (int z = 0; z < F::SETS; ++z) {  // the copies still in flight
                const int n = z ? used1 : used0;
                for (int j = (n > F::RS ? n - F::RS : 0); j < n; ++j)
                    ptx::mbar_wait(&wfull[z * F::RS + j % F::RS], (uint32_t)(j / F::RS) & 1u, nullptr);
            }
        }
    } else if (warp == TOKP_WARP) {
        // ----------------------------------- TMA producer (token chunks)
        // Chunk = nmma rows x up to CH k-blocks of a segment; atom i = 2(kb -
        // first kb of the chunk) + a (64 k each) at i * nmma * 128, 16-row
        // boxes inside.
        if (lane == 0) {
            pdl_wait();                          // the token rows are the previous kernel's
            int cc = 0;
            bool ok = true;
            FOR_EACH_SEG(t)
                const int atom = t.nmma * 128;
                for (int kc = t.kb0; kc < t.kb1; kc += CH, ++cc) {
                    const int kend = min(kc + CH, t.kb1);
                    const int ub = cc & 1;
                    if (!ptx::mbar_wait_nap(&kempty[ub], ((uint32_t)(cc >> 1) & 1u) ^ 1u, s_abort, 256)) {
                        ok = false;
                        break;
                    }
                    ptx::mbar_arrive_expect_tx(&kfull[ub], (uint32_t)((kend - kc) * 2 * atom));
                    uint8_t* tb = sTok + ub * TB_BYTES;
                    for (int kb = kc; kb < kend; ++kb)
                        for (int a = 0; a < 2; ++a)
                            for (int r = 0; r < t.nmma; r += TOK_BOX)
                                ptx::tma_load_2d(tb + (2 * (kb - kc) + a) * atom + r * 128, &mapX,
                                                 &kfull[ub], kb * BK + a * 64, t.tok0 + r);
                }
                if (!ok) break;
            }
            if (!ok) {
                *s_abort = 1;
                raise_error(p.status, MOE_ERR_DEVICE_TIMEOUT);
            }
            for (int j = (cc > 2 ? cc - 2 : 0); j < cc; ++j)
                ptx::mbar_wait(&kfull[j & 1], (uint32_t)(j >> 1) & 1u, nullptr);
        }
    } else if (warp >= F::MMA_WARP0) {
        // ------------------------------------------------------- MMA issuers
        // Issuer mi takes blocks BPI mi .. BPI mi + BPI - 1 of every k-block
        // (their A buffers and accumulators), the blocks converter set mi
        // fills.  (Four issuers, one per block, measured slower: 18 warps
        // leave 96 registers a thread, and the up-projections spill.)  An issuer without a block in a tile still
        // arrives on the tile's shared barriers (token chunks, accumulators).
        const int mi = warp - F::MMA_WARP0;
        if (lane == 0) {
            uint32_t nfill = 0;                 // bit j: parity of block j's fills so far
            int tc = 0, cc = 0;                 // tiles, token chunks
            bool ok = true;
            FOR_EACH_SEG(t)
                const int acc = tc & 1;
                const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
                ++tc;
                const bool mine = mi * BPI < t.nblk;
                if (!ptx::mbar_wait_nap(&tempty[acc], aph ^ 1u, s_abort, 64)) { ok = false; break; }
                ptx::tc_fence_after();
                const uint32_t idesc = ptx::idesc_f16_f32(WROWS, t.nmma);
                // The issuing thread runs a serial chain on a scheduler shared with
                // two converter warps, so the k-block loop keeps its scalar work
                // small: a counter within the token chunk instead of a division
                // by the chunk length, and B descriptors advanced by a constant
                // (atoms are 1024-byte aligned; the descriptor's address field
                // counts 16-byte units).
                const uint64_t atom_d = (uint64_t)(t.nmma * 128 / 16);
                uint64_t bd0 = 0;
                int kk = 0;                                       // k-blocks into the chunk
                for (int kb = t.kb0; ok && kb < t.kb1; ++kb) {
                    if (kk == 0) {                                // next token chunk
                        if (!ptx::mbar_wait_nap(&kfull[cc & 1], (uint32_t)(cc >> 1) & 1u, s_abort, 64)) {
                            ok = false;
                            break;
                        }
                        bd0 = ptx::sw128_desc(ptx::smem_u32(sTok + (cc & 1) * TB_BYTES));
                    }
                    const uint64_t bd1 = bd0 + atom_d;
                    const uint32_t first = kb > t.kb0 ? 1u : 0u;
                    for (int j = mi * BPI; j < min(mi * BPI + BPI, t.nblk); ++j) {
                        if (!ptx::mbar_wait_nap(&cfull[j], (nfill >> j) & 1u, s_abort, 64)) {
                            ok = false;
                            break;
                        }
                        nfill ^= 1u << j;
                        ptx::tc_fence_after();
                        const uint32_t d_tmem =
                            tmem_base + (uint32_t)(acc * ACC_SET + j * TOK);
                        const uint32_t a_tmem = tmem_base + (uint32_t)(A_COL0 + j * A_COLS);
                        ptx::mma_f16_tmem_a(d_tmem, a_tmem + 0, bd0 + 0, idesc, first);
                        ptx::mma_f16_tmem_a(d_tmem, a_tmem + 8, bd0 + 2, idesc, 1u);
                        ptx::mma_f16_tmem_a(d_tmem, a_tmem + 16, bd0 + 4, idesc, 1u);
                        ptx::mma_f16_tmem_a(d_tmem, a_tmem + 24, bd0 + 6, idesc, 1u);
                        ptx::mma_f16_tmem_a(d_tmem, a_tmem + 32, bd1 + 0, idesc, 1u);
                        ptx::mma_f16_tmem_a(d_tmem, a_tmem + 40, bd1 + 2, idesc, 1u);
                        ptx::mma_f16_tmem_a(d_tmem, a_tmem + 48, bd1 + 4, idesc, 1u);
                        ptx::mma_f16_tmem_a(d_tmem, a_tmem + 56, bd1 + 6, idesc, 1u);
                        ptx::mma_commit(&cempty[j]);
                    }
                    bd0 += 2 * atom_d;
                    if (ok && (++kk == CH || kb + 1 == t.kb1)) {       // chunk done
                        if (mine) ptx::mma_commit(&kempty[cc & 1]);
                        else ptx::mbar_arrive(&kempty[cc & 1]);
                        ++cc;
                        kk = 0;
                    }
                }
                if (!ok) break;
                if (mine) ptx::mma_commit(&tfull[acc]);
                else ptx::mbar_arrive(&tfull[acc]);
            }
            if (!ok) {
                *s_abort = 1;
                raise_error(p.status, MOE_ERR_DEVICE_TIMEOUT);
            }
            ptx::mma_commit(&drain[mi]);
            ptx::mbar_wait(&drain[mi], 0, nullptr);
        }
    } else if (warp >= 6) {
        // -------------------------------------------------------- converters
        // Thread = weight row r of the warp's TMEM lane quadrant q; the warp
        // converts all 128 values of its 32 rows of each block of a stage
        // into that block's A buffer (64 TMEM columns of f16 pairs).  Set z
        // (four warps) takes the stages of its blocks from its own ring, so
        // the two sets convert two stages at once.
        //   E4M3: chunk c (16 codes) of the row sits at c ^ (r & 7) (128-byte
        //   swizzle: 8 consecutive rows hit 8 different bank groups); a code
        //   pair -> an f16 pair (exact).
        //   E2M1: the row's 80 bytes hold 64 code bytes (values 2i, 2i+1 in the
        //   low, high nibble of byte i) and 8 E4M3 scales, one per 16 values;
        //   a code byte -> an f16 pair, times its block scale as an f16 pair
        //   (exact: every E2M1 value times an E4M3 value is an f16 value).
        constexpr int SB = F::SB;
        const int q = warp & 3, z = (warp - 6) >> 2;
        const int r = q * 32 + lane;
        const uint32_t a_lane = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)A_COL0;
        int u = 0;                               // stages taken from this set's ring
        uint32_t nfill = 0;                      // bit j: parity of A buffer j's fills so far
        bool ok = true;
        FOR_EACH_SEG(t)
            const int nst = (t.nblk + SB - 1) / SB;
            for (int kb = t.kb0; ok && kb < t.kb1; ++kb)
                for (int st = z * F::BPS / SB; ok && st < min(nst, (z + 1) * F::BPS / SB); ++st, ++u) {
                    const int s = z * F::RS + u % F::RS;
                    const uint32_t ph = (uint32_t)(u / F::RS) & 1u;
                    if (!__all_sync(0xffffffffu, ptx::mbar_wait(&wfull[s], ph, s_abort))) {
                        ok = false;
                        break;
                    }
                    const int jn = min(SB, t.nblk - st * SB);    // blocks of the stage
                    for (int jl = 0; jl < jn; ++jl) {
                        const int b = st * SB + jl;
                        const uint32_t bph = (nfill >> b) & 1u;
                        nfill ^= 1u << b;
                        const uint8_t* src =
                            sWq + s * F::WQ_BYTES + stage_row<MODE, SB>(jl, r) * F::ROW_BYTES;
                        constexpr int NQ = FMT == kFmtE4M3 ? 8 : 4;   // 16-byte code chunks
                        uint4 qv[NQ];
                        uint2 sc = make_uint2(0u, 0u);                // E2M1: the 8 block scales
                        if constexpr (FMT == kFmtE4M3) {
#pragma unroll
                            for (int i = 0; i < NQ; ++i)
                                qv[i] = *reinterpret_cast<const uint4*>(src + ((i ^ (r & 7)) << 4));
                        } else {
#pragma unroll
                            for (int i = 0; i < NQ; ++i)
                                qv[i] = *reinterpret_cast<const uint4*>(src + i * 16);
                            sc = *reinterpret_cast<const uint2*>(src + 64);
                        }
                        if (jl == jn - 1) {                      // the stage's codes are in registers
                            __syncwarp();
                            if (lane == 0) ptx::mbar_arrive(&wempty[s]);
                        }
                        if (!__all_sync(0xffffffffu, ptx::mbar_wait(&cempty[b], bph ^ 1u, s_abort))) {
                            ok = false;
                            break;
                        }
                        ptx::tc_fence_after();
                        if constexpr (FMT == kFmtE4M3) {
#pragma unroll
                            for (int hh = 0; hh < NQ / 2; ++hh) {     // 16 columns at a time
                                uint32_t wv[16];
#pragma unroll
                                for (int i = 0; i < 2; ++i) {
                                    const uint4 c = qv[2 * hh + i];
                                    e4m3x4_to_f16x4(c.x, wv[8 * i + 0], wv[8 * i + 1]);
                                    e4m3x4_to_f16x4(c.y, wv[8 * i + 2], wv[8 * i + 3]);
                                    e4m3x4_to_f16x4(c.z, wv[8 * i + 4], wv[8 * i + 5]);
                                    e4m3x4_to_f16x4(c.w, wv[8 * i + 6], wv[8 * i + 7]);
                                }
                                ptx::tmem_st16(a_lane + (uint32_t)(b * A_COLS + hh * 16), wv);
                            }
                        } else {
                            // 16 bytes = 32 values = two blocks of 16 per piece
#pragma unroll
                            for (int i = 0; i < NQ; ++i) {              // 16 columns per piece
                                const uint32_t sw = i < 2 ? sc.x : sc.y;
                                const uint32_t pair = ptx::cvt_e4m3x2_f16x2(
                                    (uint16_t)((i & 1) ? (sw >> 16) : (sw & 0xffffu)));
                                const uint32_t b0 = __byte_perm(pair, 0, 0x1010);   // low half, twice
                                const uint32_t b1 = __byte_perm(pair, 0, 0x3232);   // high half, twice
                                const uint32_t words[4] = {qv[i].x, qv[i].y, qv[i].z, qv[i].w};
                                uint32_t wv[16];
#pragma unroll
                                for (int w = 0; w < 4; ++w) {
                                    const uint32_t bs = w < 2 ? b0 : b1;
                                    uint32_t c[4];
                                    ptx::cvt_e2m1x8_f16x8(words[w], c);
#pragma unroll
                                    for (int by = 0; by < 4; ++by)
                                        wv[4 * w + by] = ptx::mul_f16x2(c[by], bs);
                                }
                                ptx::tmem_st16(a_lane + (uint32_t)(b * A_COLS + i * 16), wv);
                            }
                        }
                        ptx::tmem_wait_st();                  // the block's stores, then signal
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(&cfull[b]);
                    }
                }
            if (!ok) break;
        }
        if (!ok && lane == 0) {
            *s_abort = 1;
            raise_error(p.status, MOE_ERR_DEVICE_TIMEOUT);
        }
    } else if (warp >= 2 && warp < 6) {
        // ---------------------------------------------------------- epilogue
        const int q = warp & 3;                  // TMEM lane quadrant
        const int row = q * 32 + lane;           // weight row of the block
        const int et = threadIdx.x - 64;
        int tc = 0;
        FOR_EACH_SEG(t)
            const int acc = tc & 1;
            const uint32_t aph = (uint32_t)(tc >> 1) & 1u;
            ++tc;
            // inputs of the epilogue, while the tile's MMAs run: own row slots,
            // and the token slots into the buffer of this tile's parity
            prefetch_rows<MODE>(p, t, row, s_pre);
            int* tok_a = s_tok_a + acc * TOK;
            float* tok_w = s_tok_w + acc * TOK;
            if (MODE == kModeDown) {
                for (int c = et; c < t.ntok; c += 128) {
                    const int a = p.perm_src[t.tok0 + c];
                    tok_a[c] = a;
                    tok_w[c] = p.gate_w[a];
                }
            }
            int ok = 1;
            if (lane == 0) ok = ptx::mbar_wait_nap(&tfull[acc], aph, s_abort, 512) ? 1 : 0;
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
            const uint32_t tq = tmem_base + (uint32_t)(acc * ACC_SET) + ((uint32_t)(q * 32) << 16);
            if (t.c_first == t.c_last) {                     // the whole tile is ours
                for (int j = 0; j < t.nblk; ++j) {
                    __syncwarp();
                    float v[32];
                    ptx::tmem_ld32(tq + (uint32_t)(j * TOK), v);
                    finish_block<MODE>(p, t, j, row, v, s_xch, s_pre, tok_a, tok_w);
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(&tempty[acc]);
                continue;
            }
            // part of a shared tile: partial sums -> this CTA's slot
            // (0 = the tile of its first segment, 1 = of its last), [block][column][row]
            const int slot = (t.tile == t_first) ? 0 : 1;
            float* mine = p.split_part + ((size_t)blockIdx.x * 2 + slot) * G * slot_floats;
            for (int j = 0; j < t.nblk; ++j) {
                __syncwarp();
                float v[32];
                ptx::tmem_ld32(tq + (uint32_t)(j * TOK), v);
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    if (c < t.ntok) mine[j * slot_floats + (size_t)c * WROWS + row] = v[c];
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(&tempty[acc]);
            __threadfence();
            epi_bar();
            if (et == 0) {
                int parts = 0;                               // CTAs with work in the tile
                for (int c = t.c_first; c <= t.c_last; ++c)
                    parts += cta_start(W, grid, c) < cta_start(W, grid, c + 1);
                const int prev = atomicAdd(p.split_ticket + t.c_last, 1);
                const int last = prev == parts - 1;
                if (last) p.split_ticket[t.c_last] = 0;      // ready for the next launch
                *s_last = last;
            }
            epi_bar();
            if (!*s_last) continue;
            __threadfence();
            // The parts are added in CTA order (the result repeats exactly).
            // The loads of up to four parts and eight columns are issued
            // together: these L2 round trips trail the kernel, and one at a
            // time per part made the last tiles of a decode-sized down
            // projection finish 15-25 us after the others.
            for (int j = 0; j < t.nblk; ++j) {
                float v[32];
#pragma unroll
                for (int c = 0; c < 32; ++c) v[c] = 0.f;
                for (int cta0 = t.c_first; cta0 <= t.c_last; cta0 += 4) {
                    const float* src[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int cta = cta0 + q;
                        src[q] = nullptr;
                        if (cta > t.c_last) continue;
                        const long long s0 = cta_start(W, grid, cta);
                        if (s0 == cta_start(W, grid, cta + 1)) continue;    // no work there
                        const int sl = (t.tile == (int)(s0 / nk)) ? 0 : 1;
                        src[q] = p.split_part + ((size_t)cta * 2 + sl) * G * slot_floats +
                                 j * slot_floats + row;
                    }
#pragma unroll
                    for (int c0 = 0; c0 < 32; c0 += 8) {
                        if (c0 >= t.ntok) break;
                        float x[4][8];
#pragma unroll
                        for (int q = 0; q < 4; ++q)
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                x[q][i] = (src[q] && c0 + i < t.ntok)
                                              ? ld_cg(src[q] + (size_t)(c0 + i) * WROWS) : 0.f;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            if (!src[q]) continue;
#pragma unroll
                            for (int i = 0; i < 8; ++i) v[c0 + i] += x[q][i];
                        }
                    }
                }
                finish_block<MODE>(p, t, j, row, v, s_xch, s_pre, tok_a, tok_w);
            }
        }
    }
#undef FOR_EACH_SEG

    // every role done, then free TMEM
    ptx::tc_fence_before();
    ptx::mbar_block_sync(endbar);
    if (warp == 1) {
        __syncwarp();
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

}  // namespace

template <int MODE, int FMT>
cudaError_t launch_one(const CUtensorMap* maps, const TcFfnArgs& p, int num_sms, cudaStream_t st) {
    auto kernel = ffn_fp8_kernel<MODE, FMT>;
    const cudaError_t err = cudaFuncSetAttribute(
        kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, WF<FMT>::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    const int grid = num_sms < kFp8MaxGrid ? num_sms : kFp8MaxGrid;
    return launch_kernel(kernel, dim3(grid), dim3(WF<FMT>::NUM_THREADS), WF<FMT>::SMEM_BYTES, st,
                         1, maps[0], maps[1], maps[2], p);
}

template <int FMT>
cudaError_t launch_fmt(int mode, const CUtensorMap* maps, const TcFfnArgs& p, int num_sms,
                       cudaStream_t st) {
    if (mode == kModeSwiglu) return launch_one<kModeSwiglu, FMT>(maps, p, num_sms, st);
    if (mode == kModeGelu) return launch_one<kModeGelu, FMT>(maps, p, num_sms, st);
    return launch_one<kModeDown, FMT>(maps, p, num_sms, st);
}

int lowbit_box_rows(bool fp4) {
    return fp4 ? WF<kFmtE2M1>::SB * 64 : WF<kFmtE4M3>::SB * 64;
}

cudaError_t launch_ffn_fp8(int mode, const CUtensorMap* maps, const TcFfnArgs& p, int num_sms,
                           cudaStream_t st, bool fp4) {
    return fp4 ? launch_fmt<kFmtE2M1>(mode, maps, p, num_sms, st)
               : launch_fmt<kFmtE4M3>(mode, maps, p, num_sms, st);
}

}  // namespace moe
