// kernels.cuh -- launchers of the MoE kernels, called by the C ABI in capi.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace moe {

// epilogue / activation modes of the grouped FFN kernels
enum FfnMode { kModeSwiglu = 0, kModeGelu = 1, kModeDown = 2 };

// dispatch geometry: assignments per block
constexpr int kDspItems = 2;
constexpr int kDspChunk = 256 * kDspItems;
inline int dispatch_blocks(int A) { return A > 0 ? (A + kDspChunk - 1) / kDspChunk : 1; }

// capi.cu: record a host-side failure for moe_last_error and return `code`
int set_last_error(int code, const char* msg);
int set_cuda_error(cudaError_t e, const char* where);   // returns MOE_ERR_CUDA
// MOE_OK if p is non-NULL and 4-byte aligned, else MOE_ERR_INVALID_ARG naming `name`
int check_aligned4(const void* p, const char* name);

// route.cu
cudaError_t launch_router_logits_simt(int dtype, const void* x, const void* Wr, const float* bias,
                                      float* logits, int T, int d, int E, cudaStream_t st);
// top-k reads nsplit partial-logit slabs part[s][T][E], adds them in order
// and the bias, writes logits, then softmax / top-k / renormalise.
// Decode-sized route + dispatch in one launch (front_small.cu): router GEMM
// partials over K-slices, then the last CTA routes and dispatches.
constexpr int kFrontMaxT = 256;       // tokens
constexpr int kFrontMaxE = 256;       // experts
constexpr int kFrontMaxA = 512;       // assignments T*k
constexpr int kFrontMaxTE = 2048;     // router outputs T*E
struct FrontSmallPlan {
    bool ok;       // the shape fits the one-launch path
    int ks;        // K values per CTA slice (a multiple of 32)
    int splits;    // CTAs = K-slices (<= 32)
};
FrontSmallPlan front_small_plan(int T, int d, int E, int k);
struct FrontSmallArgs {
    const void* x;            // [T, d] (dtype of the layer)
    const void* Wr;           // [E, d]
    const float* bias;        // [E] logit bias or nullptr
    int T, d, E, k, scoring, renorm;
    int dispatch;             // 0: route only (the dispatch outputs untouched)
    long long cap;            // capacity, < 0 = dropless
    int ks, splits;
    float* part;              // [splits][T][E] scratch
    int* ticket;              // zero between calls
    float* logits;            // [T, E]
    int* topk_idx;            // [T, k]
    float* topk_w;            // [T, k]
    float* prob_mean;         // [E] or nullptr (route only)
    int* counts_pre;          // [E]
    int* counts_kept;         // [E]
    int* offsets;             // [E + 1]
    int* perm_src;            // [T*k] (first R entries written)
    int* dest;                // [T*k]
    unsigned char* drop_mask; // [T*k]
    float* stats;             // [2]: aux loss, dropped fraction
};
cudaError_t launch_front_small(int dtype, const FrontSmallArgs& a, cudaStream_t st);

cudaError_t launch_router_topk(const float* part, int nsplit, const float* bias, float* logits,
                               int T, int E, int k, int scoring, int renorm, int* topk_idx,
                               float* topk_w,
                               float* prob_part, float* prob_mean, int* done, int nblocks,
                               cudaStream_t st);

// router_tc.cu (bf16 router logits on tcgen05, split over K)
struct RouterPlan {
    int NB;             // E rounded up to 16 (MMA N)
    int m_tiles, nkb;   // 128-token tiles, 64-wide K blocks
    int splits, kb_per_split;
    int smem;           // dynamic shared memory bytes
};
RouterPlan router_tc_plan(int T, int d, int E);
cudaError_t launch_router_tc(const CUtensorMap& map_x, const CUtensorMap& map_w, int T, int E,
                             const RouterPlan& p, float* part, int* status, cudaStream_t st);

// aux_backward.cu (router gradients of the aux loss)
cudaError_t launch_aux_backward(int dtype, int scoring, const void* x, const void* Wr,
                                const float* logits, const int* counts_pre, float grad_aux, int T,
                                int d, int E, float* g_l, float* g_Wr, float* g_x, int num_sms,
                                cudaStream_t st);

// dispatch.cu
cudaError_t launch_dispatch(const int* topk_idx, int T, int k, int E, long long cap,
                            unsigned* tile_status, int* ctrl, int* rank, int* counts_pre,
                            int* counts_kept, int* offsets, int* dest, int* perm_src,
                            unsigned char* drop_mask, const float* prob_mean, float* stats,
                            int num_sms, cudaStream_t st);

// permute.cu
cudaError_t launch_gather(int dtype, const void* x, const int* perm_src, const int* offsets, int E,
                          int k, int T, int d, void* Xp, int* status, int num_sms,
                          cudaStream_t st);
// bf16 x -> f16 gathered rows (the FP8-weight path's token operand)
cudaError_t launch_gather_f16(const void* x, const int* perm_src, const int* offsets, int E, int k,
                              int T, int d, void* Xp, int* status, int num_sms, cudaStream_t st);
// use_mask = false: nothing was dropped (dropless layer), drop_mask is not read
cudaError_t launch_combine(int dtype, const void* x, const void* Ys, const unsigned char* drop_mask,
                           const void* Sh, void* y, int T, int d, int k, int num_sms,
                           cudaStream_t st, bool use_mask = true);

// ffn_simt.cu (fp32)
struct SimtFfnArgs {
    const float* A;           // routed rows [*, K]
    const float* B;           // [E, N, K]
    const float* B2;          // [E, N, K] (SwiGLU up) or null
    const float* bias;        // [E, N] or null
    const int* offsets;       // [E+1]
    int E, N, K;
    const float* A_sh;        // shared-expert rows [rows_sh, K_sh]
    const float* B_sh;
    const float* B2_sh;
    int rows_sh, N_sh, K_sh;
    float* out;               // up: H [*, N]; down: Ys [T*k, N]
    float* out_sh;            // up: H_sh; down: Sh
    const int* perm_src;      // down
    const float* gate_w;      // down
};
cudaError_t launch_ffn_simt(int mode, const SimtFfnArgs& p, int A_rows, cudaStream_t st);

// ffn_tc.cu (bf16, tcgen05)
struct TcFfnArgs {
    const int* offsets;       // [E+1] segment starts (routed groups)
    int E;
    int rows_sh;              // shared-expert rows (0 = no shared group)
    int N, K;                 // routed output columns / reduction length
    int N_sh, K_sh;           // shared group
    void* out;                // bf16: up H [*, N]; down Ys [T*k, N]
    void* out_sh;             // bf16: up H_sh [T, N_sh]; down Sh [T, N_sh]
    const __nv_bfloat16* bias;  // [E, N] (GELU b1 / down b2) or null
    const int* perm_src;      // down
    const float* gate_w;      // down
    int* status;
    const float* wscale;      // FP8 weights: per-row scales [E, N] (gate / fc1 / down)
    const float* wscale2;     // FP8 SwiGLU: up-projection scales [E, N]
    int* split_ticket;        // FP8 split-K: per-tile counters, zero between launches
    int split_tickets;        //   their number
    float* split_part;        //   fp32 partial sums
    long long split_bytes;    //   their capacity
    const int* hold;          // test hook (up-projection launches): if *hold = n > 0, each
                              //   CTA's weight producer stops before ring iteration n - 1
};
int ffn_tc_smem_bytes();
// maps: A, B, B2, A_sh, B_sh, B2_sh (see ffn_tc.cu)
cudaError_t launch_ffn_tc(int mode, const CUtensorMap* maps, const TcFfnArgs& p, int num_sms,
                          cudaStream_t st);
// ffn_fp8.cu: FP8 (E4M3) weights with per-row scales, weights on the MMA's M;
// at most kFp8MaxGrid CTAs (its partial-sum slots: 2 per CTA of 4 weight blocks
// x 128 rows x 32 tokens fp32, and one ticket per CTA)
// maps: X (f16 token rows, box 64 x 16), W and W3 (E4M3 rows, box 128 bytes x
// lowbit_box_rows(false) rows; W3 = W for GELU / down), all with the 128-byte swizzle
constexpr int kFp8MaxGrid = 160;
constexpr size_t kFp8SplitBytes = (size_t)2 * kFp8MaxGrid * 4 * 128 * 32 * 4;
// fp4: packed E2M1 weights (rows of 80-byte chunks: 64 code bytes, 8 E4M3 block
// scales, 8 zero bytes per 128 values; weight maps with box 80 bytes x
// lowbit_box_rows(true) rows, no swizzle) instead of E4M3
// rows of one TMA box of low-bit weight rows (a ring stage is two boxes)
int lowbit_box_rows(bool fp4);
cudaError_t launch_ffn_fp8(int mode, const CUtensorMap* maps, const TcFfnArgs& p, int num_sms,
                           cudaStream_t st, bool fp4 = false);
// ffn_tc2.cu: the same on CTA pairs (cta_group::2), 256-row tiles; same maps
int ffn_tc2_tile_rows();
cudaError_t launch_ffn_tc2(int mode, const CUtensorMap* maps, const TcFfnArgs& p, cudaStream_t st);
// ffn_swap.cu: weights as the MMA's M, tokens as N, on CTA pairs.
// maps: W, W3 (SwiGLU up; else unused), X (token rows), and the shared
// expert's W_sh, W3_sh, X_sh; weight maps with ffn_swap_weight_box_rows rows
int ffn_swap_weight_box_rows(int mode);
cudaError_t launch_ffn_swap(int mode, const CUtensorMap* maps, const TcFfnArgs& p, cudaStream_t st);

}  // namespace moe
