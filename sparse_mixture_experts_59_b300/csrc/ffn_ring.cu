// ffn_ring.cu -- bf16 grouped expert GEMMs for layers with many short expert
// segments (a few hundred rows each, e.g. 256 routed experts with top-8):
// weights on the MMA's M, tokens on N, on CTA pairs (tcgen05 cta_group::2),
// one token tile for a whole segment of up to 288 rows, accumulators taken
// from a ring of tensor-memory columns.
//
// Same maths and fused epilogues as ffn_swap.cu (see ffn_tc.cu for the pages'
// basis: "How Mixture of Experts Works", the grouped-GEMM remark after the
// MoELayer listing; "Mixture of Experts (MoE)", "Implementing a complete MoE
// layer" and "The shared expert pattern").  What differs is the token tile.
// A tcgen05 MMA takes time in proportion to N, and the weight tile of a pair
// (256 rows x K) costs the same to stream whatever N is.  So a segment is best
// covered by a single token tile: every weight byte then feeds all of the
// segment's tokens.  With ~256 +- 16 rows per segment that needs N up to ~288,
// above one MMA's 256: a tile is issued as up to three MMAs of <= 256 columns
// over the same weight stage.  Two 288-column accumulators do not fit in the
// 512 columns of TMEM, so instead of two fixed accumulators the columns form a
// ring of 16 chunks of 32: tile i takes the next ceil(n_i / 32) chunks (its
// MMAs split where the ring wraps), the epilogue frees each chunk as soon as it
// has read it, and the MMAs of tile i+1 start once the chunks they need are
// free -- usually while the epilogue is still draining tile i.
//
// Per pair tile: 256 weight rows (128 per CTA; SwiGLU: 64 gate + the 64
// matching up rows per CTA) x up to 288 tokens.  Segments longer than 288
// rows are cut into ceil(rows / 288) tiles of equal size (+-1).  Token counts
// are rounded up to a multiple of 32; the extra rows are computed on whatever
// the tile reads (next segment, or TMA's zero fill) and never stored.
//
// Roles (224 threads per CTA):
//   warp 0      weight producer (both CTAs): this CTA's 128 weight rows of each
//               K block into an 8-deep ring of 16 KB stages
//   warp 6      token producer (both CTAs): this CTA's half of each MMA's token
//               rows (boxes of 128/64/32/16 rows) into a 4-deep ring
//   warp 1      TMEM allocation (512 columns, pair); MMA issuer (leader only)
//   warps 2-5   epilogue (both CTAs): 32 tokens at a time from TMEM, staged as
//               [token][unit] in shared memory, written with 16-byte stores
// Barriers: full (the leader's: both CTAs' bytes) and empty per stage of each
// ring; tfull/slot_free per tile slot (at most NSLOT
// tiles between issuer and epilogue); chunk_free per TMEM chunk (8 arrivals:
// the four epilogue warps of both CTAs).  Every wait is bounded.
#include "common.cuh"
#include "kernels.cuh"
#include "launch.cuh"
#include "tc_ptx.cuh"

namespace moe {

namespace {

constexpr int BK = 64;
// Weight and token rows sit in two rings of their own depth.  Every weight
// byte is read by one SM only and comes from DRAM (~3 us away under load), so
// each SM needs ~128 KB of weight loads in flight to keep HBM busy; the token
// rows are shared by the tiles of a segment and mostly hit L2.
constexpr int WSTAGES = 8;                   // 16 KB weight stages
constexpr int KSTAGES = 4;                   // up to 18 KB token stages
constexpr int TOK_MAX = 288;                 // tokens per tile
constexpr int HALF_MAX = TOK_MAX / 2;        // token rows per CTA
constexpr int CHUNK = 32;                    // TMEM columns per ring chunk
constexpr int NCHUNK = 16;                   // 512 columns
constexpr int PIECE_MAX = 8;                 // chunks per MMA (N <= 256)
constexpr int NSLOT = 4;                     // tiles in flight between issuer and epilogue
constexpr int TOK_BOX = 16;                  // smallest token box (rows)
constexpr int A_BYTES = 128 * BK * 2;        // this CTA's 128 weight rows
constexpr int B_BYTES = HALF_MAX * BK * 2;   // up to 144 token rows
constexpr int TMEM_COLS = 512;
constexpr int NUM_THREADS = 224;             // 7 warps: weight producer, issuer, 4 epilogue, token producer
constexpr int EPI_THREADS = 128;
constexpr int TOKP_WARP = 6;
constexpr uint16_t BOTH = 0x3;
constexpr uint16_t LEADER_ONLY = 0x1;
constexpr uint32_t CHUNK_ARRIVALS = 8;       // 4 epilogue warps x 2 CTAs

constexpr int XCH_LD = 33;                   // [64 units][33] fp32: up values, padded
constexpr int OUT_LD = 136;                  // [32 tokens][136] bf16: staged output rows

constexpr int OFF_A = 0;
constexpr int OFF_B = WSTAGES * A_BYTES;
constexpr int OFF_XCH = OFF_B + KSTAGES * B_BYTES;
constexpr int OFF_OUT = OFF_XCH + 64 * XCH_LD * 4;
constexpr int OFF_TOKA = OFF_OUT + 32 * OUT_LD * 2;
constexpr int OFF_TOKW = OFF_TOKA + TOK_MAX * 4;
constexpr int OFF_BAR = OFF_TOKW + TOK_MAX * 4;
constexpr int NUM_BARS = 2 * WSTAGES + 2 * KSTAGES + 2 * NSLOT + NCHUNK + 1;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int OFF_START = OFF_MISC + 16;
constexpr int OFF_OFFS = OFF_START + (kMaxExperts + 2) * 4;
constexpr int SMEM_USED = OFF_OFFS + (kMaxExperts + 2) * 4;
constexpr int SMEM_BYTES = SMEM_USED + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "128-byte swizzle atoms stay aligned");
static_assert(HALF_MAX % TOK_BOX == 0 && (CHUNK / 2) % TOK_BOX == 0, "token boxes tile a piece");
// a tile of at most 10 chunks splits into at most 3 pieces: the first piece
// ends at the ring's end or after 8 chunks, and so can the second
static_assert(TOK_MAX / CHUNK <= 10, "ring_pieces returns at most three pieces");

// weight units (outputs) per pair tile
template <int MODE> struct RingTraits { static constexpr int UNITS = 256, UNITS_CTA = 128; };
template <> struct RingTraits<kModeSwiglu> { static constexpr int UNITS = 128, UNITS_CTA = 64; };

struct RTile {
    int g;
    bool sh;
    int tok0;       // first token row of the tile (A-row space of X_p / H, or x / H_sh)
    int ntok;       // valid tokens in the tile
    int nch;        // TMEM chunks = MMA columns / 32
    int u0;         // first output unit of the pair tile
    int N;          // outputs of this group's projection
    int nk;         // K blocks
    int wbase;      // first weight row of the group in its tensor map
};

// Tile `tile`: group g, weight-unit tile w, token tile tt of ceil(rows/TOK_MAX)
// equal parts (token tiles fastest, so tiles that run at the same time share
// the segment's token rows in L2).
template <int MODE>
__device__ __forceinline__ RTile decode(const TcFfnArgs& p, const int* s_start, const int* s_off,
                                        int G, int tile) {
    RTile t;
    t.g = find_group(s_start, G, tile);
    t.sh = (t.g == p.E);
    const int seg0 = t.sh ? 0 : s_off[t.g];
    const int rows = t.sh ? p.rows_sh : s_off[t.g + 1] - seg0;
    const int nt = (rows + TOK_MAX - 1) / TOK_MAX;
    const int local = tile - s_start[t.g];
    const int w = local / nt, tt = local - w * nt;
    const int base = rows / nt, rem = rows - base * nt;
    t.tok0 = seg0 + tt * base + min(tt, rem);
    t.ntok = base + (tt < rem ? 1 : 0);
    t.nch = (t.ntok + CHUNK - 1) / CHUNK;
    t.N = t.sh ? p.N_sh : p.N;
    t.nk = ((t.sh ? p.K_sh : p.K) + BK - 1) / BK;
    t.u0 = w * RingTraits<MODE>::UNITS;
    t.wbase = t.sh ? 0 : t.g * p.N;
    return t;
}

// The MMAs of a tile whose accumulator starts at ring chunk `pos` and spans
// `nch` chunks: contiguous runs of at most PIECE_MAX chunks, split where the
// ring wraps.  Piece j covers tile tokens [32*off_j, 32*(off_j + len_j)).
struct Pieces {
    int n;
    int c[3];       // first ring chunk
    int len[3];     // chunks
};
__device__ __forceinline__ Pieces ring_pieces(int pos, int nch) {
    Pieces pc;
    pc.n = 0;
    int c = pos, left = nch;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const int run = min(min(left, NCHUNK - c), PIECE_MAX);
        pc.c[j] = c;
        pc.len[j] = run;
        pc.n += run > 0 ? 1 : 0;
        c = (c + run) % NCHUNK;
        left -= run;
    }
    return pc;
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Tensor maps of one launch: weights (boxes of ffn_ring_weight_box_rows rows)
// and token rows with boxes of 128, 64, 32 and 16 rows, so that any piece
// half (a multiple of 16 rows up to 128) loads in at most three copies.
struct RingMaps {
    CUtensorMap w, w3, w_sh, w3_sh;
    CUtensorMap x[4], x_sh[4];
};

template <int MODE>
__global__ void __launch_bounds__(NUM_THREADS, 1)
ffn_ring_kernel(const __grid_constant__ RingMaps maps, const TcFfnArgs p) {
    const CUtensorMap& mapW = maps.w;
    const CUtensorMap& mapW3 = maps.w3;
    const CUtensorMap& mapW_sh = maps.w_sh;
    const CUtensorMap& mapW3_sh = maps.w3_sh;
    constexpr int UNITS_CTA = RingTraits<MODE>::UNITS_CTA;
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
    uint64_t* wfull = bars;                  // weight stage landed
    uint64_t* wempty = wfull + WSTAGES;      // weight stage consumed by the MMAs
    uint64_t* kfull = wempty + WSTAGES;      // token stage landed
    uint64_t* kempty = kfull + KSTAGES;      // token stage consumed
    uint64_t* tfull = kempty + KSTAGES;
    uint64_t* slot_free = tfull + NSLOT;
    uint64_t* chunk_free = slot_free + NSLOT;
    uint64_t* drain = chunk_free + NCHUNK;
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
        for (int s = 0; s < WSTAGES; ++s) {
            ptx::mbar_init(&wfull[s], 1);
            ptx::mbar_init(&wempty[s], 1);
        }
        for (int s = 0; s < KSTAGES; ++s) {
            ptx::mbar_init(&kfull[s], 1);
            ptx::mbar_init(&kempty[s], 1);
        }
        for (int a = 0; a < NSLOT; ++a) {
            ptx::mbar_init(&tfull[a], 1);
            ptx::mbar_init(&slot_free[a], CHUNK_ARRIVALS);
        }
        for (int c = 0; c < NCHUNK; ++c) ptx::mbar_init(&chunk_free[c], CHUNK_ARRIVALS);
        ptx::mbar_init(drain, 1);
        *s_abort = 0;
        ptx::fence_mbarrier_init();
        ptx::prefetch_tensormap(&mapW);
        ptx::prefetch_tensormap(&mapW3);
        for (int i = 0; i < 4; ++i) ptx::prefetch_tensormap(&maps.x[i]);
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(s_tmem, TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    pdl_wait();       // offsets and the token rows come from the preceding kernels
    pdl_trigger();
    for (int i = threadIdx.x; i <= p.E; i += NUM_THREADS) s_off[i] = p.offsets[i];
    constexpr int UNITS = RingTraits<MODE>::UNITS;
    const int nw_r = (p.N + UNITS - 1) / UNITS;
    const int nw_s = p.rows_sh > 0 ? (p.N_sh + UNITS - 1) / UNITS : 0;
    group_tile_prefix(p.offsets, p.E, p.rows_sh, TOK_MAX, nw_r, nw_s, s_start);
    ptx::tc_fence_before();
    __syncwarp();
    ptx::cluster_sync();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *s_tmem;
    const int G = p.E + (p.rows_sh > 0 ? 1 : 0);
    const int total = s_start[G];
    const uint32_t wfull_leader = ptx::mapa_shared(ptx::smem_u32(wfull), 0);
    const uint32_t kfull_leader = ptx::mapa_shared(ptx::smem_u32(kfull), 0);
    const uint32_t slot_free_leader = ptx::mapa_shared(ptx::smem_u32(slot_free), 0);
    const uint32_t chunk_free_leader = ptx::mapa_shared(ptx::smem_u32(chunk_free), 0);

    if (warp == 0 || warp == TOKP_WARP) {
        // ---------------------- TMA producers (both CTAs): weights / tokens
        // Issuing a bulk-tensor copy keeps its thread busy ~150 cycles here,
        // and a stage takes two weight copies plus one to three token copies,
        // more than one thread can issue in the ~600 cycles of MMA work per
        // stage.  So warp 0 loads the weight rows and warp 6 the token rows,
        // each on its own full barrier of the stage (both CTAs' bytes land on
        // the leader's barriers).
        const bool wprod = (warp == 0);
        const int NST = wprod ? WSTAGES : KSTAGES;
        if (lane == 0) {
            int it = 0, pos = 0;
            bool ok = true, held = false;
            const int hold_it = (wprod && p.hold) ? *p.hold - 1 : -1;
            const uint32_t fbase = wprod ? wfull_leader : kfull_leader;
            for (int tile = cluster; ok && tile < total; tile += nclusters) {
                const RTile t = decode<MODE>(p, s_start, s_off, G, tile);
                const Pieces pc = ring_pieces(pos, t.nch);
                pos = (pos + t.nch) % NCHUNK;
                const CUtensorMap* mW = t.sh ? &mapW_sh : &mapW;
                const CUtensorMap* mW3 = t.sh ? &mapW3_sh : &mapW3;
                const CUtensorMap* mX = t.sh ? maps.x_sh : maps.x;   // boxes of 128, 64, 32, 16 rows
                const int wrow = t.wbase + t.u0 + (int)rank * UNITS_CTA;
                const uint32_t tx = wprod ? 2u * (uint32_t)A_BYTES
                                          : 2u * (uint32_t)(t.nch * (CHUNK / 2) * BK * 2);
                for (int kb = 0; kb < t.nk; ++kb, ++it) {
                    if (it == hold_it) { ok = false; held = true; break; }   // test hook
                    const int s = it % NST;
                    const uint32_t ph = (uint32_t)(it / NST) & 1u;
                    if (!ptx::mbar_wait(wprod ? &wempty[s] : &kempty[s], ph ^ 1u, s_abort)) {
                        ok = false;
                        break;
                    }
                    if (leader) ptx::mbar_arrive_expect_tx(wprod ? &wfull[s] : &kfull[s], tx);
                    const uint32_t fb = fbase + 8u * s;
                    if (wprod) {
                        if (MODE == kModeSwiglu) {   // 64 gate rows, then the 64 matching up rows
                            ptx::tma_load_2d_pair(sA + s * A_BYTES, mW, fb, kb * BK, wrow);
                            ptx::tma_load_2d_pair(sA + s * A_BYTES + A_BYTES / 2, mW3, fb, kb * BK, wrow);
                        } else {
                            ptx::tma_load_2d_pair(sA + s * A_BYTES, mW, fb, kb * BK, wrow);
                        }
                        continue;
                    }
                    // piece j: this CTA holds its half of the piece's tokens, at
                    // shared-memory row (first token of the piece) / 2
                    int tp = 0;
#pragma unroll
                    for (int j = 0; j < 3; ++j) {
                        if (j < pc.n) {
                            const int h = pc.len[j] * (CHUNK / 2);   // 16..128 rows
                            const int src = t.tok0 + tp + (int)rank * h;
                            uint8_t* dst = sB + s * B_BYTES + (tp / 2) * (BK * 2);
                            int r = 0;
#pragma unroll
                            for (int b = 0; b < 4; ++b) {
                                const int rows = 128 >> b;
                                if (h == 128 ? b == 0 : (b > 0 && (h & rows))) {
                                    ptx::tma_load_2d_pair(dst + r * (BK * 2), &mX[b], fb, kb * BK, src + r);
                                    r += rows;
                                }
                            }
                            tp += pc.len[j] * CHUNK;
                        }
                    }
                }
            }
            if (!ok && !held) {
                *s_abort = 1;
                raise_error(p.status, MOE_ERR_DEVICE_TIMEOUT);
            }
            // the leader's barriers count both CTAs' bytes: let them land
            if (leader)
                for (int j = (it > NST ? it - NST : 0); j < it; ++j)
                    ptx::mbar_wait(wprod ? &wfull[j % NST] : &kfull[j % NST],
                                   (uint32_t)(j / NST) & 1u, nullptr);
        }
    } else if (warp == 1) {
        // ----------------------------------------- MMA issuer (leader only)
        if (leader && lane == 0) {
            int it = 0, tc = 0, pos = 0;
            uint32_t cpar = 0;            // bit c: parity of the next use of chunk c
            bool ok = true;
            for (int tile = cluster; ok && tile < total; tile += nclusters, ++tc) {
                const RTile t = decode<MODE>(p, s_start, s_off, G, tile);
                const Pieces pc = ring_pieces(pos, t.nch);
                const int slot = tc % NSLOT;
                if (!ptx::mbar_wait(&slot_free[slot], ((uint32_t)(tc / NSLOT) & 1u) ^ 1u, s_abort)) {
                    ok = false;
                    break;
                }
                for (int j = 0; ok && j < t.nch; ++j) {     // the tile's chunks are drained
                    const int c = (pos + j) % NCHUNK;
                    if (!ptx::mbar_wait(&chunk_free[c], ((cpar >> c) & 1u) ^ 1u, s_abort)) ok = false;
                    cpar ^= 1u << c;
                }
                if (!ok) break;
                pos = (pos + t.nch) % NCHUNK;
                ptx::tc_fence_after();
                uint32_t idesc[3], dcol[3], boff[3];   // per piece: instruction, TMEM column, B row offset
#pragma unroll
                for (int j = 0, tp = 0; j < 3; ++j) {
                    const int len = j < pc.n ? pc.len[j] : 1;
                    idesc[j] = ptx::idesc_bf16_f32(256, len * CHUNK);
                    dcol[j] = (uint32_t)((j < pc.n ? pc.c[j] : 0) * CHUNK);
                    boff[j] = (uint32_t)((tp / 2) * BK * 2);
                    tp += len * CHUNK;
                }
                for (int kb = 0; kb < t.nk; ++kb, ++it) {
                    const int ws = it % WSTAGES, ks = it % KSTAGES;
                    if (!ptx::mbar_wait(&wfull[ws], (uint32_t)(it / WSTAGES) & 1u, s_abort) ||
                        !ptx::mbar_wait(&kfull[ks], (uint32_t)(it / KSTAGES) & 1u, s_abort)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
                    const uint64_t ad = ptx::sw128_desc(ptx::smem_u32(sA + ws * A_BYTES));
                    const uint32_t b0 = ptx::smem_u32(sB + ks * B_BYTES);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
#pragma unroll
                        for (int j = 0; j < 3; ++j) {
                            if (j < pc.n) {
                                const uint64_t bd = ptx::sw128_desc(b0 + boff[j]);
                                ptx::mma_bf16_pair(tmem_base + dcol[j], ad + (uint64_t)(kk * 2),
                                                   bd + (uint64_t)(kk * 2), idesc[j],
                                                   (kb | kk) != 0 ? 1u : 0u);
                            }
                        }
                    }
                    ptx::mma_commit_pair_mc(&wempty[ws], BOTH);
                    ptx::mma_commit_pair_mc(&kempty[ks], BOTH);
                }
                if (!ok) break;
                ptx::mma_commit_pair_mc(&tfull[slot], BOTH);
            }
            if (!ok) {
                *s_abort = 1;
                raise_error(p.status, MOE_ERR_DEVICE_TIMEOUT);
            }
            ptx::mma_commit_pair_mc(drain, LEADER_ONLY);
            ptx::mbar_wait(drain, 0, nullptr);
        }
    } else if (warp >= 2 && warp < 6) {
        // ------------------------------------------- epilogue (both CTAs)
        const int q = warp & 3;                  // TMEM lane quadrant = weight rows q*32..
        const int et = threadIdx.x - 64;         // 0..127 among the epilogue threads
        int tc = 0, pos = 0;
        for (int tile = cluster; tile < total; tile += nclusters, ++tc) {
            const RTile t = decode<MODE>(p, s_start, s_off, G, tile);
            const int slot = tc % NSLOT;
            int ok = 1;
            if (lane == 0) ok = ptx::mbar_wait(&tfull[slot], (uint32_t)(tc / NSLOT) & 1u, s_abort) ? 1 : 0;
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
            const uint32_t tq = tmem_base + ((uint32_t)(q * 32) << 16);
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
            for (int ci = 0; ci < t.nch; ++ci) {
                const int chunk = (pos + ci) % NCHUNK;
                const uint32_t col = (uint32_t)(chunk * CHUNK);
                const uint32_t free_bar = chunk_free_leader + 8u * (uint32_t)chunk;
                const int c = ci * CHUNK;                      // first token of the chunk
                __syncwarp();
                float v[32];
                if (MODE == kModeSwiglu) {
                    if (q >= 2) {       // up values of units (q-2)*32 + lane
                        ptx::tmem_ld32(tq + col, v);
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive_cluster(free_bar);
                        float* xr = s_xch + ((q - 2) * 32 + lane) * XCH_LD;
#pragma unroll
                        for (int j = 0; j < 32; ++j) xr[j] = v[j];
                    }
                    epi_bar();
                    if (q < 2) {        // gate values of units q*32 + lane
                        ptx::tmem_ld32(tq + col, v);
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive_cluster(free_bar);
                        const float* xr = s_xch + (q * 32 + lane) * XCH_LD;
                        const int u = q * 32 + lane;
#pragma unroll
                        for (int j = 0; j < 32; ++j)
                            s_out[j * OUT_LD + u] = __float2bfloat16_rn(silu(v[j]) * xr[j]);
                    }
                } else {
                    ptx::tmem_ld32(tq + col, v);
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive_cluster(free_bar);
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
                    const int col_out = ubase + vv * 8;
                    if (c + j < t.ntok && col_out < t.N) {
                        const int row = (MODE == kModeDown) ? s_tok_a[c + j] : t.tok0 + c + j;
                        const uint4 val = *reinterpret_cast<const uint4*>(s_out + j * OUT_LD + vv * 8);
                        *reinterpret_cast<uint4*>(out_base + (size_t)row * t.N + col_out) = val;
                    }
                }
                epi_bar();
            }
            pos = (pos + t.nch) % NCHUNK;
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive_cluster(slot_free_leader + 8u * (uint32_t)slot);
        }
    }

    ptx::tc_fence_before();
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
cudaError_t launch_mode(const CUtensorMap* m, const TcFfnArgs& p, cudaStream_t st) {
    auto kernel = ffn_ring_kernel<MODE>;
    RingMaps maps;
    maps.w = m[0]; maps.w3 = m[1]; maps.w_sh = m[2]; maps.w3_sh = m[3];
    for (int i = 0; i < 4; ++i) {
        maps.x[i] = m[4 + i];
        maps.x_sh[i] = m[8 + i];
    }
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
    return launch_kernel(kernel, dim3(2 * clusters), dim3(NUM_THREADS), SMEM_BYTES, st, 2, maps, p);
}

}  // namespace

int ffn_ring_weight_box_rows(int mode) { return mode == kModeSwiglu ? 64 : 128; }

cudaError_t launch_ffn_ring(int mode, const CUtensorMap* maps, const TcFfnArgs& p, cudaStream_t st) {
    if (mode == kModeSwiglu) return launch_mode<kModeSwiglu>(maps, p, st);
    if (mode == kModeGelu) return launch_mode<kModeGelu>(maps, p, st);
    return launch_mode<kModeDown>(maps, p, st);
}

}  // namespace moe
