// capi.cu -- the C ABI of include/moe.h: argument checks, workspace layout,
// TMA descriptors, and the launch sequence of each stage.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

using namespace moe;

namespace {

thread_local char g_last_error[256] = "";

int fail(int code, const char* fmt, const char* detail = "") {
    snprintf(g_last_error, sizeof g_last_error, fmt, detail);
    return code;
}
int fail_cuda(cudaError_t e, const char* where) {
    snprintf(g_last_error, sizeof g_last_error, "%s: %s", where, cudaGetErrorString(e));
    return MOE_ERR_CUDA;
}

size_t esize(const moe_cfg& c) { return c.dtype == MOE_F32 ? 4 : 2; }
size_t align_up(size_t v) { return (v + 255) & ~(size_t)255; }
bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// The top-k kernel's 256-thread blocks take 64 registers a thread, so an SM
// holds 4: 592 blocks are one wave.  More would only add a partial wave and
// rows to the P partials that the last block adds up alone.
constexpr int kRouterTopkMaxBlocks = 4 * 148;
int router_blocks(int T) {
    const int b = (T + 7) / 8;
    return b < 1 ? 1 : (b > kRouterTopkMaxBlocks ? kRouterTopkMaxBlocks : b);
}

struct Layout {
    size_t ctrl, tile_status, split_ticket, rank, prob_part, prob_mean, router_part, logits, topk_idx, topk_w,
        counts_pre, counts_kept, offsets, perm_src, dest, drop_mask, stats, xp, h, hsh, ys, sh,
        split_part, front_part, total;
};

// FP8 expert GEMMs: tickets and fp32 partial sums of the tiles that straddle
// two CTAs' stream-K ranges (ffn_fp8.cu).
constexpr int kFp8SplitTickets = kFp8MaxGrid;
size_t fp8_split_bytes(const moe_cfg&) { return kFp8SplitBytes; }

Layout layout_of(const moe_cfg& c) {
    Layout L;
    const size_t A = (size_t)c.T * c.k, E = c.E, T = c.T, es = esize(c);
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes); return at; };
    L.ctrl = take(kCtrlWords * 4);
    L.tile_status = take((size_t)dispatch_blocks((int)A) * E * 4);
    L.split_ticket = take(c.weight_fp8 || c.weight_fp4 ? (size_t)kFp8SplitTickets * 4 : 0);
    L.rank = take(A * 4);
    L.prob_part = take((size_t)router_blocks(c.T) * E * 4);
    L.prob_mean = take(E * 4);
    L.router_part = take(c.dtype == MOE_BF16
                             ? (size_t)router_tc_plan(c.T > 0 ? c.T : 1, c.d, c.E).splits * T * E * 4
                             : 0);
    L.logits = take(T * E * 4);
    L.topk_idx = take(A * 4);
    L.topk_w = take(A * 4);
    L.counts_pre = take(E * 4);
    L.counts_kept = take(E * 4);
    L.offsets = take((E + 1) * 4);
    L.perm_src = take(A * 4);
    L.dest = take(A * 4);
    L.drop_mask = take(A);
    L.stats = take(2 * 4);
    L.xp = take(A * c.d * es);
    L.h = take(A * c.F * es);
    L.hsh = take(T * (size_t)c.F_shared * es);
    L.ys = take(A * c.d * es);
    L.sh = take(c.F_shared > 0 ? T * c.d * es : 0);
    L.split_part = take(c.weight_fp8 || c.weight_fp4 ? fp8_split_bytes(c) : 0);
    const FrontSmallPlan fp = front_small_plan(c.T, c.d, c.E, c.k);
    L.front_part = take(fp.ok ? (size_t)fp.splits * T * E * 4 : 0);
    L.total = o;
    return L;
}

int check_cfg(const moe_cfg* c) {
    if (!c) return fail(MOE_ERR_INVALID_ARG, "cfg is NULL%s");
    if (c->T < 0 || c->T > (1 << 24)) return fail(MOE_ERR_INVALID_ARG, "T out of range [0, 2^24]%s");
    if (c->d < 8 || c->d % 8) return fail(MOE_ERR_INVALID_ARG, "d must be a positive multiple of 8%s");
    if (c->F < 8 || c->F % 8) return fail(MOE_ERR_INVALID_ARG, "F must be a positive multiple of 8%s");
    if (c->E < 1 || c->E > kMaxExperts) return fail(MOE_ERR_INVALID_ARG, "E must be in [1, 256]%s");
    if (c->k < 1 || c->k > c->E || c->k > kMaxTopK)
        return fail(MOE_ERR_INVALID_ARG, "k must be in [1, min(E, 8)]%s");
    if ((long long)c->T * c->k > (1LL << 26)) return fail(MOE_ERR_INVALID_ARG, "T*k above 2^26%s");
    if (c->F_shared < 0 || c->F_shared % 8)
        return fail(MOE_ERR_INVALID_ARG, "F_shared must be 0 or a multiple of 8%s");
    // the expert GEMMs address weight rows (expert x outputs) with 32-bit
    // coordinates, in the kernels and in the TMA maps
    if ((long long)c->E * (c->F > c->d ? c->F : c->d) >= (1LL << 31))
        return fail(MOE_ERR_INVALID_ARG, "E*max(d, F) must stay below 2^31%s");
    if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return fail(MOE_ERR_INVALID_ARG, "unknown dtype%s");
    if (c->act != MOE_GELU_ERF && c->act != MOE_SWIGLU) return fail(MOE_ERR_INVALID_ARG, "unknown act%s");
    if (c->has_bias && c->act == MOE_SWIGLU)
        return fail(MOE_ERR_UNSUPPORTED, "SwiGLU experts take no biases%s");
    if (c->F_shared > 0 && c->act != MOE_SWIGLU)
        return fail(MOE_ERR_UNSUPPORTED, "the shared expert is a SwiGLU expert; needs act = SwiGLU%s");
    if (!(c->capacity_factor == c->capacity_factor)) return fail(MOE_ERR_INVALID_ARG, "capacity_factor is NaN%s");
    if (c->scoring != MOE_SCORE_SOFTMAX && c->scoring != MOE_SCORE_SIGMOID)
        return fail(MOE_ERR_INVALID_ARG, "unknown scoring%s");
    if (c->no_renorm != 0 && c->no_renorm != 1) return fail(MOE_ERR_INVALID_ARG, "no_renorm must be 0 or 1%s");
    if (c->weight_fp8 != 0 && c->weight_fp8 != 1) return fail(MOE_ERR_INVALID_ARG, "weight_fp8 must be 0 or 1%s");
    if (c->weight_fp8 && (c->dtype != MOE_BF16 || c->F_shared > 0))
        return fail(MOE_ERR_UNSUPPORTED, "FP8 expert weights need a bf16 layer without a shared expert%s");
    if (c->weight_fp4 != 0 && c->weight_fp4 != 1) return fail(MOE_ERR_INVALID_ARG, "weight_fp4 must be 0 or 1%s");
    if (c->weight_fp4 && c->weight_fp8) return fail(MOE_ERR_INVALID_ARG, "weight_fp4 and weight_fp8 exclude each other%s");
    if (c->weight_fp4 && (c->dtype != MOE_BF16 || c->F_shared > 0))
        return fail(MOE_ERR_UNSUPPORTED, "4-bit expert weights need a bf16 layer without a shared expert%s");
    if (c->weight_fp4 && (c->d % 128 || c->F % 128))
        return fail(MOE_ERR_INVALID_ARG, "4-bit expert weights need d and F multiples of 128 (80-byte chunks)%s");
    if (c->weight_fp8 && (c->d % 16 || c->F % 16))
        return fail(MOE_ERR_INVALID_ARG, "FP8 expert weights need d and F multiples of 16 (16-byte rows)%s");
    if (c->gemm_kernel < MOE_GEMM_AUTO || c->gemm_kernel > MOE_GEMM_SWAP)
        return fail(MOE_ERR_INVALID_ARG, "unknown gemm_kernel%s");
    if (c->route_path != MOE_ROUTE_AUTO && c->route_path != MOE_ROUTE_SEPARATE)
        return fail(MOE_ERR_INVALID_ARG, "unknown route_path%s");
    return MOE_OK;
}

int check_ws(const moe_cfg& c, const void* ws, size_t ws_bytes) {
    if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL%s");
    if (!aligned16(ws)) return fail(MOE_ERR_INVALID_ARG, "workspace must be 16-byte aligned%s");
    if (ws_bytes < layout_of(c).total) return fail(MOE_ERR_WORKSPACE, "workspace too small%s");
    return MOE_OK;
}

// data pointer checks: non-null; bf16 row buffers 16-byte aligned (TMA and
// 16-byte vector access); fp32 buffers too (16-byte vectors).
int check_ptr(const void* p, const char* name) {
    if (!p) return fail(MOE_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned16(p)) return fail(MOE_ERR_INVALID_ARG, "%s must be 16-byte aligned", name);
    return MOE_OK;
}
int check_ptr4(const void* p, const char* name) {
    if (!p) return fail(MOE_ERR_INVALID_ARG, "%s is NULL", name);
    if (((uintptr_t)p & 3u) != 0) return fail(MOE_ERR_INVALID_ARG, "%s must be 4-byte aligned", name);
    return MOE_OK;
}

#define MOE_TRY(x)                  \
    do {                            \
        const int _rc = (x);        \
        if (_rc != MOE_OK) return _rc; \
    } while (0)
#define MOE_CUDA(x, where)                           \
    do {                                             \
        const cudaError_t _e = (x);                  \
        if (_e != cudaSuccess) return fail_cuda(_e, where); \
    } while (0)

int check_weights(const moe_cfg& c, const moe_weights* w) {
    if (!w) return fail(MOE_ERR_INVALID_ARG, "weights is NULL%s");
    MOE_TRY(check_ptr(w->W1, "W1"));
    MOE_TRY(check_ptr(w->W2, "W2"));
    if (c.act == MOE_SWIGLU) MOE_TRY(check_ptr(w->W3, "W3"));
    if (c.has_bias) {
        MOE_TRY(check_ptr(w->b1, "b1"));
        MOE_TRY(check_ptr(w->b2, "b2"));
    }
    if (c.F_shared > 0) {
        MOE_TRY(check_ptr(w->S1, "S1"));
        MOE_TRY(check_ptr(w->S3, "S3"));
        MOE_TRY(check_ptr(w->S2, "S2"));
    }
    if (c.weight_fp8 || c.weight_fp4) {
        MOE_TRY(check_ptr4(w->s1, "s1"));
        MOE_TRY(check_ptr4(w->s2, "s2"));
        if (c.act == MOE_SWIGLU) MOE_TRY(check_ptr4(w->s3, "s3"));
    }
    return MOE_OK;
}

// ---------------------------------------------------------------- devices
struct DevInfo {
    int num_sms = 0;
    int cc = 0;
};

int device_info(DevInfo* out) {
    static std::mutex mu;
    static DevInfo cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= 64) return fail(MOE_ERR_NO_DEVICE, "device ordinal out of range%s");
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev].num_sms == 0) {
        int sms = 0, maj = 0, mnr = 0;
        MOE_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev), "attr SMs");
        MOE_CUDA(cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev), "attr cc");
        MOE_CUDA(cudaDeviceGetAttribute(&mnr, cudaDevAttrComputeCapabilityMinor, dev), "attr cc");
        cache[dev].num_sms = sms;
        cache[dev].cc = maj * 10 + mnr;
    }
    *out = cache[dev];
    return MOE_OK;
}

// ------------------------------------------------------------- TMA maps
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// Row-major [rows, cols] matrix of 2-byte elements (bf16, or f16 with
// dt = CU_TENSOR_MAP_DATA_TYPE_FLOAT16); box = box_rows rows x 64 columns
// (128 bytes), 128-byte swizzle, out-of-range elements read as zero.
// 1-byte elements (low-bit weights, dt = UINT8): box_cols bytes per box row;
// swizzle = false leaves the box rows packed (packed 4-bit weights).
int encode_rows(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, const char* what,
                uint32_t box_rows = 128,
                CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                uint32_t box_cols = 64, bool swizzle = true) {
    auto fn = encode_fn();
    if (!fn) return fail(MOE_ERR_CUDA, "cuTensorMapEncodeTiled unavailable%s");
    if (rows == 0) rows = 1;
    const bool byte_elems = (dt == CU_TENSOR_MAP_DATA_TYPE_UINT8);
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * (byte_elems ? 1 : 2)};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(MOE_ERR_CUDA, "tensor map encode failed for %s", what);
    return MOE_OK;
}

// Decode-sized batches route and dispatch in one launch (front_small.cu)
// unless the config asks for the separate router and dispatch kernels.
bool small_front_enabled(const moe_cfg& c) { return c.route_path == MOE_ROUTE_AUTO; }

// Kernel for the bf16 expert GEMMs:
//   kGemmTc1   1-SM kernel, tokens on M in 128-row tiles (ffn_tc.cu)
//   kGemmPair  2-SM kernel, tokens on M in 256-row tiles (ffn_tc2.cu)
//   kGemmSwap  2-SM kernel, weights on M and tokens on N (ffn_swap.cu): a
//              segment's last tile shrinks to a multiple of 32 tokens
// Automatic choice (from B300 measurements: the five workloads and a sweep of
// the token count on Mixtral-shaped weights): capacity-limited segments that
// fit one token tile -> swap; long segments (>= 512 rows on average) -> swap;
// at most one row per expert (a few tokens) -> swap; 128+ rows per expert on
// few (<= 16) experts -> swap; otherwise tc1 (decode-sized segments of a few
// rows, and many experts with ~256-row segments, where swap's second, ragged
// token tile costs more than tc1's ragged 128-row tile).  cfg.gemm_kernel
// forces one.
enum GemmKernel { kGemmTc1, kGemmPair, kGemmSwap };
GemmKernel choose_gemm(const moe_cfg& c) {
    if (c.gemm_kernel == MOE_GEMM_TC1) return kGemmTc1;
    if (c.gemm_kernel == MOE_GEMM_PAIR) return kGemmPair;
    if (c.gemm_kernel == MOE_GEMM_SWAP) return kGemmSwap;
    const long long rows = (long long)c.T * c.k;
    const long long cap = moe_capacity(&c);
    if (cap >= 0 && cap <= 256 && rows >= 32LL * c.E) return kGemmSwap;   // one tile each
    if (rows >= 512LL * c.E) return kGemmSwap;
    if (rows <= c.E) return kGemmSwap;
    if (c.E <= 16 && rows >= 128LL * c.E) return kGemmSwap;
    return kGemmTc1;
}

template <typename T>
T* at(void* ws, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(ws) + off); }

// --------------------------------------------------------------- stages
int run_route(const moe_cfg& c, const DevInfo& di, const void* x, const void* Wr,
              const float* bias, float* logits, int* topk_idx, float* topk_w, float* prob_mean,
              void* ws, cudaStream_t st) {
    const Layout L = layout_of(c);
    const FrontSmallPlan fp = front_small_plan(c.T, c.d, c.E, c.k);
    if (fp.ok && small_front_enabled(c)) {
        // decode-sized batch: the route part of the one-launch front, so that
        // this call and the layer call give the same logits
        FrontSmallArgs a{};
        a.x = x; a.Wr = Wr; a.bias = bias;
        a.T = c.T; a.d = c.d; a.E = c.E; a.k = c.k;
        a.scoring = c.scoring; a.renorm = !c.no_renorm;
        a.dispatch = 0;
        a.cap = moe_capacity(&c);
        a.ks = fp.ks; a.splits = fp.splits;
        a.part = at<float>(ws, L.front_part);
        a.ticket = at<int>(ws, L.ctrl) + kCtrlFrontDone;
        a.logits = logits; a.topk_idx = topk_idx; a.topk_w = topk_w; a.prob_mean = prob_mean;
        MOE_CUDA(launch_front_small(c.dtype, a, st), "router launch");
        return MOE_OK;
    }
    const float* part = logits;
    int nsplit = 1;
    const float* topk_bias = nullptr;
    if (c.dtype == MOE_BF16) {
        if (di.cc != 103)
            return fail(MOE_ERR_UNSUPPORTED, "the bf16 router needs an sm_103a (B300) device%s");
        const RouterPlan plan = router_tc_plan(c.T, c.d, c.E);
        CUtensorMap mx, mw;
        MOE_TRY(encode_rows(&mx, x, (uint64_t)c.T, c.d, "x", 128));
        MOE_TRY(encode_rows(&mw, Wr, (uint64_t)c.E, c.d, "Wr", (uint32_t)plan.NB));
        float* rp = at<float>(ws, L.router_part);
        MOE_CUDA(launch_router_tc(mx, mw, c.T, c.E, plan, rp, at<int>(ws, L.ctrl) + kCtrlStatus, st),
                 "router GEMM launch");
        part = rp;
        nsplit = plan.splits;
        topk_bias = bias;
    } else {
        MOE_CUDA(launch_router_logits_simt(c.dtype, x, Wr, bias, logits, c.T, c.d, c.E, st),
                 "router logits launch");
    }
    MOE_CUDA(launch_router_topk(part, nsplit, topk_bias, logits, c.T, c.E, c.k, c.scoring,
                                !c.no_renorm, topk_idx, topk_w,
                                at<float>(ws, L.prob_part), prob_mean,
                                at<int>(ws, L.ctrl) + kCtrlRouterDone, router_blocks(c.T), st),
             "router top-k launch");
    return MOE_OK;
}

int run_dispatch(const moe_cfg& c, const DevInfo& di, const int* topk_idx, const float* prob_mean,
                 int* counts_pre, int* counts_kept, int* offsets, int* perm_src, int* dest,
                 unsigned char* drop_mask, float* stats, void* ws, cudaStream_t st) {
    const Layout L = layout_of(c);
    MOE_CUDA(launch_dispatch(topk_idx, c.T, c.k, c.E, moe_capacity(&c),
                             at<unsigned>(ws, L.tile_status), at<int>(ws, L.ctrl),
                             at<int>(ws, L.rank), counts_pre, counts_kept, offsets, dest, perm_src,
                             drop_mask, prob_mean, stats, di.num_sms, st),
             "dispatch launch");
    return MOE_OK;
}

// ev (optional): events recorded after the gather, the up- and the
// down-projection.
int run_expert_ffn(const moe_cfg& c, const DevInfo& di, const void* x, const int* perm_src,
                   const int* offsets, const float* topk_w, const moe_weights& w, void* Ys,
                   void* Sh, void* ws, cudaStream_t st, cudaEvent_t const* ev = nullptr) {
    const Layout L = layout_of(c);
    int* status = at<int>(ws, L.ctrl) + kCtrlStatus;
    const int A = c.T * c.k;
    void* Xp = at<char>(ws, L.xp);
    void* H = at<char>(ws, L.h);
    void* Hsh = at<char>(ws, L.hsh);
    const int rows_sh = c.F_shared > 0 ? c.T : 0;
    if (c.weight_fp8 || c.weight_fp4) {
        if (di.cc != 103)
            return fail(MOE_ERR_UNSUPPORTED, "low-bit expert GEMMs need an sm_103a (B300) device%s");
        const bool fp4 = c.weight_fp4 != 0;
        // E4M3: rows of K bytes, 128-byte boxes, swizzled; packed E2M1: rows of
        // K/128 * 80 bytes, 80-byte boxes, not swizzled
        auto wmap = [&](CUtensorMap* m, const void* base, uint64_t rows, int K, const char* what) {
            return fp4 ? encode_rows(m, base, rows, (uint64_t)(K / 128) * 80, what, lowbit_box_rows(true),
                                     CU_TENSOR_MAP_DATA_TYPE_UINT8, 80, false)
                       : encode_rows(m, base, rows, (uint64_t)K, what, lowbit_box_rows(false),
                                     CU_TENSOR_MAP_DATA_TYPE_UINT8, 128);
        };
        const int up_mode = c.act == MOE_SWIGLU ? kModeSwiglu : kModeGelu;
        MOE_CUDA(launch_gather_f16(x, perm_src, offsets, c.E, c.k, c.T, c.d, Xp, status,
                                   di.num_sms, st),
                 "gather launch");
        if (ev) MOE_CUDA(cudaEventRecord(ev[0], st), "event record");
        CUtensorMap maps[3];
        MOE_TRY(encode_rows(&maps[0], Xp, (uint64_t)A, c.d, "gathered rows", 16,
                            CU_TENSOR_MAP_DATA_TYPE_FLOAT16));
        MOE_TRY(wmap(&maps[1], w.W1, (uint64_t)c.E * c.F, c.d, "W1"));
        MOE_TRY(wmap(&maps[2], c.act == MOE_SWIGLU ? w.W3 : w.W1, (uint64_t)c.E * c.F, c.d, "W3"));
        int* tickets = at<int>(ws, L.split_ticket);
        float* part = at<float>(ws, L.split_part);
        const long long part_bytes = (long long)fp8_split_bytes(c);
        TcFfnArgs up{};
        up.split_ticket = tickets; up.split_tickets = kFp8SplitTickets;
        up.split_part = part; up.split_bytes = part_bytes;
        up.offsets = offsets; up.E = c.E; up.N = c.F; up.K = c.d;
        up.out = H;
        up.bias = c.has_bias ? (const __nv_bfloat16*)w.b1 : nullptr;
        up.status = status;
        up.wscale = w.s1;
        up.wscale2 = c.act == MOE_SWIGLU ? w.s3 : nullptr;
        up.hold = at<int>(ws, L.ctrl) + kCtrlHoldGemm;
        MOE_CUDA(launch_ffn_fp8(up_mode, maps, up, di.num_sms, st, fp4), "up-projection launch");
        if (ev) MOE_CUDA(cudaEventRecord(ev[1], st), "event record");
        MOE_TRY(encode_rows(&maps[0], H, (uint64_t)A, c.F, "hidden rows", 16,
                            CU_TENSOR_MAP_DATA_TYPE_FLOAT16));
        MOE_TRY(wmap(&maps[1], w.W2, (uint64_t)c.E * c.d, c.F, "W2"));
        maps[2] = maps[1];
        TcFfnArgs dn{};
        dn.split_ticket = tickets; dn.split_tickets = kFp8SplitTickets;
        dn.split_part = part; dn.split_bytes = part_bytes;
        dn.offsets = offsets; dn.E = c.E; dn.N = c.d; dn.K = c.F;
        dn.out = Ys;
        dn.bias = c.has_bias ? (const __nv_bfloat16*)w.b2 : nullptr;
        dn.perm_src = perm_src; dn.gate_w = topk_w;
        dn.status = status;
        dn.wscale = w.s2;
        MOE_CUDA(launch_ffn_fp8(kModeDown, maps, dn, di.num_sms, st, fp4),
                 "down-projection launch");
        if (ev) MOE_CUDA(cudaEventRecord(ev[2], st), "event record");
        return MOE_OK;
    }
    MOE_CUDA(launch_gather(c.dtype, x, perm_src, offsets, c.E, c.k, c.T, c.d, Xp, status,
                           di.num_sms, st),
             "gather launch");
    if (ev) MOE_CUDA(cudaEventRecord(ev[0], st), "event record");
    if (c.dtype == MOE_F32) {
        SimtFfnArgs up{};
        up.A = (const float*)Xp; up.B = (const float*)w.W1; up.B2 = (const float*)w.W3;
        up.bias = c.has_bias ? (const float*)w.b1 : nullptr;
        up.offsets = offsets; up.E = c.E; up.N = c.F; up.K = c.d;
        up.A_sh = (const float*)x; up.B_sh = (const float*)w.S1; up.B2_sh = (const float*)w.S3;
        up.rows_sh = rows_sh; up.N_sh = c.F_shared; up.K_sh = c.d;
        up.out = (float*)H; up.out_sh = (float*)Hsh;
        MOE_CUDA(launch_ffn_simt(c.act == MOE_SWIGLU ? kModeSwiglu : kModeGelu, up, A, st),
                 "fp32 up-projection launch");
        if (ev) MOE_CUDA(cudaEventRecord(ev[1], st), "event record");
        SimtFfnArgs dn{};
        dn.A = (const float*)H; dn.B = (const float*)w.W2; dn.B2 = nullptr;
        dn.bias = c.has_bias ? (const float*)w.b2 : nullptr;
        dn.offsets = offsets; dn.E = c.E; dn.N = c.d; dn.K = c.F;
        dn.A_sh = (const float*)Hsh; dn.B_sh = (const float*)w.S2; dn.B2_sh = nullptr;
        dn.rows_sh = rows_sh; dn.N_sh = c.d; dn.K_sh = c.F_shared;
        dn.out = (float*)Ys; dn.out_sh = (float*)Sh;
        dn.perm_src = perm_src; dn.gate_w = topk_w;
        MOE_CUDA(launch_ffn_simt(kModeDown, dn, A, st), "fp32 down-projection launch");
        if (ev) MOE_CUDA(cudaEventRecord(ev[2], st), "event record");
        return MOE_OK;
    }
    if (di.cc != 103)
        return fail(MOE_ERR_UNSUPPORTED, "bf16 expert GEMMs need an sm_103a (B300) device%s");
    const GemmKernel gk = choose_gemm(c);
    const int up_mode = c.act == MOE_SWIGLU ? kModeSwiglu : kModeGelu;
    TcFfnArgs up{};
    up.offsets = offsets; up.E = c.E; up.rows_sh = rows_sh;
    up.N = c.F; up.K = c.d; up.N_sh = c.F_shared; up.K_sh = c.d;
    up.out = H; up.out_sh = Hsh;
    up.bias = c.has_bias ? (const __nv_bfloat16*)w.b1 : nullptr;
    up.status = status;
    up.hold = at<int>(ws, L.ctrl) + kCtrlHoldGemm;
    TcFfnArgs dn{};
    dn.offsets = offsets; dn.E = c.E; dn.rows_sh = rows_sh;
    dn.N = c.d; dn.K = c.F; dn.N_sh = c.d; dn.K_sh = c.F_shared;
    dn.out = Ys; dn.out_sh = Sh;
    dn.bias = c.has_bias ? (const __nv_bfloat16*)w.b2 : nullptr;
    dn.perm_src = perm_src; dn.gate_w = topk_w;
    dn.status = status;
    CUtensorMap maps[6];
    if (gk == kGemmSwap) {
        // maps: W, W3, X (token rows), W_sh, W3_sh, X_sh
        const uint32_t wb_up = (uint32_t)ffn_swap_weight_box_rows(up_mode);
        MOE_TRY(encode_rows(&maps[0], w.W1, (uint64_t)c.E * c.F, c.d, "W1", wb_up));
        MOE_TRY(encode_rows(&maps[1], c.act == MOE_SWIGLU ? w.W3 : w.W1, (uint64_t)c.E * c.F, c.d,
                            "W3", wb_up));
        MOE_TRY(encode_rows(&maps[2], Xp, (uint64_t)A, c.d, "gathered rows"));
        if (rows_sh) {
            MOE_TRY(encode_rows(&maps[3], w.S1, (uint64_t)c.F_shared, c.d, "S1", wb_up));
            MOE_TRY(encode_rows(&maps[4], w.S3, (uint64_t)c.F_shared, c.d, "S3", wb_up));
            MOE_TRY(encode_rows(&maps[5], x, (uint64_t)c.T, c.d, "x"));
        } else {
            maps[3] = maps[0]; maps[4] = maps[1]; maps[5] = maps[2];
        }
        MOE_CUDA(launch_ffn_swap(up_mode, maps, up, st), "up-projection launch");
        if (ev) MOE_CUDA(cudaEventRecord(ev[1], st), "event record");
        const uint32_t wb_dn = (uint32_t)ffn_swap_weight_box_rows(kModeDown);
        MOE_TRY(encode_rows(&maps[0], w.W2, (uint64_t)c.E * c.d, c.F, "W2", wb_dn));
        maps[1] = maps[0];
        MOE_TRY(encode_rows(&maps[2], H, (uint64_t)A, c.F, "hidden rows"));
        if (rows_sh) {
            MOE_TRY(encode_rows(&maps[3], w.S2, (uint64_t)c.d, c.F_shared, "S2", wb_dn));
            maps[4] = maps[3];
            MOE_TRY(encode_rows(&maps[5], Hsh, (uint64_t)c.T, c.F_shared, "shared hidden rows"));
        } else {
            maps[3] = maps[0]; maps[4] = maps[1]; maps[5] = maps[2];
        }
        MOE_CUDA(launch_ffn_swap(kModeDown, maps, dn, st), "down-projection launch");
        if (ev) MOE_CUDA(cudaEventRecord(ev[2], st), "event record");
        return MOE_OK;
    }
    // tokens on M: maps A, B, B2, A_sh, B_sh, B2_sh
    MOE_TRY(encode_rows(&maps[0], Xp, (uint64_t)A, c.d, "gathered rows"));
    MOE_TRY(encode_rows(&maps[1], w.W1, (uint64_t)c.E * c.F, c.d, "W1"));
    MOE_TRY(encode_rows(&maps[2], c.act == MOE_SWIGLU ? w.W3 : w.W1, (uint64_t)c.E * c.F, c.d, "W3"));
    if (rows_sh) {
        MOE_TRY(encode_rows(&maps[3], x, (uint64_t)c.T, c.d, "x"));
        MOE_TRY(encode_rows(&maps[4], w.S1, (uint64_t)c.F_shared, c.d, "S1"));
        MOE_TRY(encode_rows(&maps[5], w.S3, (uint64_t)c.F_shared, c.d, "S3"));
    } else {
        maps[3] = maps[0]; maps[4] = maps[1]; maps[5] = maps[2];
    }
    const bool pair = (gk == kGemmPair);
    MOE_CUDA(pair ? launch_ffn_tc2(up_mode, maps, up, st)
                  : launch_ffn_tc(up_mode, maps, up, di.num_sms, st),
             "up-projection launch");
    if (ev) MOE_CUDA(cudaEventRecord(ev[1], st), "event record");
    MOE_TRY(encode_rows(&maps[0], H, (uint64_t)A, c.F, "hidden rows"));
    MOE_TRY(encode_rows(&maps[1], w.W2, (uint64_t)c.E * c.d, c.F, "W2"));
    maps[2] = maps[1];
    if (rows_sh) {
        MOE_TRY(encode_rows(&maps[3], Hsh, (uint64_t)c.T, c.F_shared, "shared hidden rows"));
        MOE_TRY(encode_rows(&maps[4], w.S2, (uint64_t)c.d, c.F_shared, "S2"));
        maps[5] = maps[4];
    } else {
        maps[3] = maps[0]; maps[4] = maps[1]; maps[5] = maps[2];
    }
    MOE_CUDA(pair ? launch_ffn_tc2(kModeDown, maps, dn, st)
                  : launch_ffn_tc(kModeDown, maps, dn, di.num_sms, st),
             "down-projection launch");
    if (ev) MOE_CUDA(cudaEventRecord(ev[2], st), "event record");
    return MOE_OK;
}

}  // namespace

// Error reporting for the other host translation units of the library.
namespace moe {
int set_last_error(int code, const char* msg) { return fail(code, "%s", msg); }
int set_cuda_error(cudaError_t e, const char* where) { return fail_cuda(e, where); }
int check_aligned4(const void* p, const char* name) { return check_ptr4(p, name); }
}  // namespace moe

// ====================================================================== ABI
extern "C" {

const char* moe_status_string(int status) {
    switch (status) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT";
        case MOE_ERR_DEVICE_BOUNDS: return "MOE_ERR_DEVICE_BOUNDS";
        case MOE_ERR_NO_DEVICE: return "MOE_ERR_NO_DEVICE";
        default: return "MOE_ERR_UNKNOWN";
    }
}

const char* moe_last_error(void) { return g_last_error; }

long long moe_capacity(const moe_cfg* cfg) {
    if (!cfg || cfg->E < 1) return -1;
    if (!(cfg->capacity_factor > 0.f)) return -1;
    const double ideal = (double)cfg->T * (double)cfg->k / (double)cfg->E;
    const long long cap = (long long)floor(ideal * (double)cfg->capacity_factor);
    return cap < 1 ? 1 : cap;
}

int moe_workspace_size(const moe_cfg* cfg, size_t* bytes) {
    MOE_TRY(check_cfg(cfg));
    if (!bytes) return fail(MOE_ERR_INVALID_ARG, "bytes is NULL%s");
    *bytes = layout_of(*cfg).total;
    return MOE_OK;
}

int moe_workspace_init(const moe_cfg* cfg, void* ws, size_t ws_bytes, void* stream) {
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_ws(*cfg, ws, ws_bytes));
    const Layout L = layout_of(*cfg);
    MOE_CUDA(cudaMemsetAsync(ws, 0, L.rank, (cudaStream_t)stream), "workspace init");
    return MOE_OK;
}

int moe_route(const moe_cfg* cfg, const void* x, const void* Wr, const float* logit_bias,
              float* logits, int* topk_idx, float* topk_w, float* prob_mean, void* ws,
              size_t ws_bytes, void* stream) {
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_ws(*cfg, ws, ws_bytes));
    if (cfg->T == 0) return MOE_OK;
    MOE_TRY(check_ptr(x, "x"));
    MOE_TRY(check_ptr(Wr, "Wr"));
    if (logit_bias) MOE_TRY(check_ptr4(logit_bias, "logit_bias"));
    MOE_TRY(check_ptr4(logits, "logits"));
    MOE_TRY(check_ptr4(topk_idx, "topk_idx"));
    MOE_TRY(check_ptr4(topk_w, "topk_w"));
    if (prob_mean) MOE_TRY(check_ptr4(prob_mean, "prob_mean"));
    DevInfo di;
    MOE_TRY(device_info(&di));
    return run_route(*cfg, di, x, Wr, logit_bias, logits, topk_idx, topk_w, prob_mean, ws,
                     (cudaStream_t)stream);
}

int moe_dispatch(const moe_cfg* cfg, const int* topk_idx, const float* prob_mean, int* counts_pre,
                 int* counts_kept, int* offsets, int* perm_src, int* dest,
                 unsigned char* drop_mask, float* stats, void* ws, size_t ws_bytes, void* stream) {
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_ws(*cfg, ws, ws_bytes));
    MOE_TRY(check_ptr4(counts_pre, "counts_pre"));
    MOE_TRY(check_ptr4(counts_kept, "counts_kept"));
    MOE_TRY(check_ptr4(offsets, "offsets"));
    if (cfg->T == 0) return MOE_OK;
    MOE_TRY(check_ptr4(topk_idx, "topk_idx"));
    MOE_TRY(check_ptr4(perm_src, "perm_src"));
    MOE_TRY(check_ptr4(dest, "dest"));
    if (!drop_mask) return fail(MOE_ERR_INVALID_ARG, "drop_mask is NULL%s");
    if (stats) MOE_TRY(check_ptr4(stats, "stats"));
    if (prob_mean) MOE_TRY(check_ptr4(prob_mean, "prob_mean"));
    DevInfo di;
    MOE_TRY(device_info(&di));
    return run_dispatch(*cfg, di, topk_idx, prob_mean, counts_pre, counts_kept, offsets, perm_src,
                        dest, drop_mask, stats, ws, (cudaStream_t)stream);
}

int moe_expert_ffn(const moe_cfg* cfg, const void* x, const int* perm_src, const int* offsets,
                   const float* topk_w, const moe_weights* w, void* Ys, void* shared_out, void* ws,
                   size_t ws_bytes, void* stream) {
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_ws(*cfg, ws, ws_bytes));
    if (cfg->T == 0) return MOE_OK;
    MOE_TRY(check_ptr(x, "x"));
    MOE_TRY(check_ptr4(perm_src, "perm_src"));
    MOE_TRY(check_ptr4(offsets, "offsets"));
    MOE_TRY(check_ptr4(topk_w, "topk_w"));
    MOE_TRY(check_weights(*cfg, w));
    MOE_TRY(check_ptr(Ys, "Ys"));
    if (cfg->F_shared > 0) MOE_TRY(check_ptr(shared_out, "shared_out"));
    DevInfo di;
    MOE_TRY(device_info(&di));
    return run_expert_ffn(*cfg, di, x, perm_src, offsets, topk_w, *w, Ys,
                          cfg->F_shared > 0 ? shared_out : nullptr, ws, (cudaStream_t)stream);
}

int moe_combine(const moe_cfg* cfg, const void* x, const void* Ys, const unsigned char* drop_mask,
                const void* shared_out, void* y, void* stream) {
    MOE_TRY(check_cfg(cfg));
    if (cfg->T == 0) return MOE_OK;
    MOE_TRY(check_ptr(x, "x"));
    MOE_TRY(check_ptr(Ys, "Ys"));
    MOE_TRY(check_ptr(y, "y"));
    if (!drop_mask) return fail(MOE_ERR_INVALID_ARG, "drop_mask is NULL%s");
    if (shared_out) MOE_TRY(check_ptr(shared_out, "shared_out"));
    DevInfo di;
    MOE_TRY(device_info(&di));
    MOE_CUDA(launch_combine(cfg->dtype, x, Ys, drop_mask, shared_out, y, cfg->T, cfg->d, cfg->k,
                            di.num_sms, (cudaStream_t)stream),
             "combine launch");
    return MOE_OK;
}

static int layer_forward_impl(const moe_cfg* cfg, const void* x, const void* Wr,
                              const float* logit_bias, const moe_weights* w,
                              const moe_layer_out* out, void* ws, size_t ws_bytes, void* stream,
                              void* const* events) {
    MOE_TRY(check_cfg(cfg));
    MOE_TRY(check_ws(*cfg, ws, ws_bytes));
    if (!out) return fail(MOE_ERR_INVALID_ARG, "out is NULL%s");
    if (cfg->T == 0) return MOE_OK;
    const moe_cfg& c = *cfg;
    MOE_TRY(check_ptr(x, "x"));
    MOE_TRY(check_ptr(Wr, "Wr"));
    if (logit_bias) MOE_TRY(check_ptr4(logit_bias, "logit_bias"));
    MOE_TRY(check_weights(c, w));
    MOE_TRY(check_ptr(out->y, "y"));
    if (out->logits) MOE_TRY(check_ptr4(out->logits, "logits"));
    if (out->topk_idx) MOE_TRY(check_ptr4(out->topk_idx, "topk_idx"));
    if (out->topk_w) MOE_TRY(check_ptr4(out->topk_w, "topk_w"));
    if (out->counts_pre) MOE_TRY(check_ptr4(out->counts_pre, "counts_pre"));
    if (out->counts_kept) MOE_TRY(check_ptr4(out->counts_kept, "counts_kept"));
    if (out->stats) MOE_TRY(check_ptr4(out->stats, "stats"));
    DevInfo di;
    MOE_TRY(device_info(&di));
    const Layout L = layout_of(c);
    cudaStream_t st = (cudaStream_t)stream;
    float* logits = out->logits ? out->logits : at<float>(ws, L.logits);
    int* topk_idx = out->topk_idx ? out->topk_idx : at<int>(ws, L.topk_idx);
    float* topk_w = out->topk_w ? out->topk_w : at<float>(ws, L.topk_w);
    int* counts_pre = out->counts_pre ? out->counts_pre : at<int>(ws, L.counts_pre);
    int* counts_kept = out->counts_kept ? out->counts_kept : at<int>(ws, L.counts_kept);
    unsigned char* drop = out->drop_mask ? out->drop_mask : at<unsigned char>(ws, L.drop_mask);
    float* stats = out->stats ? out->stats : at<float>(ws, L.stats);
    float* prob_mean = at<float>(ws, L.prob_mean);
    int* offsets = at<int>(ws, L.offsets);
    int* perm_src = at<int>(ws, L.perm_src);
    int* dest = at<int>(ws, L.dest);
    void* Ys = at<char>(ws, L.ys);
    void* Sh = c.F_shared > 0 ? at<char>(ws, L.sh) : nullptr;
    cudaEvent_t const* ev = reinterpret_cast<cudaEvent_t const*>(events);
    if (ev) MOE_CUDA(cudaEventRecord(ev[0], st), "event record");
    const FrontSmallPlan fp = front_small_plan(c.T, c.d, c.E, c.k);
    if (fp.ok && small_front_enabled(c)) {
        // decode-sized batch: route + dispatch in one launch (the stage
        // events after it coincide: the dispatch stage reads as zero)
        FrontSmallArgs a{};
        a.x = x; a.Wr = Wr; a.bias = logit_bias;
        a.T = c.T; a.d = c.d; a.E = c.E; a.k = c.k;
        a.scoring = c.scoring; a.renorm = !c.no_renorm;
        a.dispatch = 1;
        a.cap = moe_capacity(&c);
        a.ks = fp.ks; a.splits = fp.splits;
        a.part = at<float>(ws, L.front_part);
        a.ticket = at<int>(ws, L.ctrl) + kCtrlFrontDone;
        a.logits = logits; a.topk_idx = topk_idx; a.topk_w = topk_w; a.prob_mean = prob_mean;
        a.counts_pre = counts_pre; a.counts_kept = counts_kept; a.offsets = offsets;
        a.perm_src = perm_src; a.dest = dest; a.drop_mask = drop; a.stats = stats;
        MOE_CUDA(launch_front_small(c.dtype, a, st), "route + dispatch launch");
        if (ev) MOE_CUDA(cudaEventRecord(ev[1], st), "event record");
    } else {
        MOE_TRY(run_route(c, di, x, Wr, logit_bias, logits, topk_idx, topk_w, prob_mean, ws, st));
        if (ev) MOE_CUDA(cudaEventRecord(ev[1], st), "event record");
        MOE_TRY(run_dispatch(c, di, topk_idx, prob_mean, counts_pre, counts_kept, offsets,
                             perm_src, dest, drop, stats, ws, st));
    }
    if (ev) MOE_CUDA(cudaEventRecord(ev[2], st), "event record");
    MOE_TRY(run_expert_ffn(c, di, x, perm_src, offsets, topk_w, *w, Ys, Sh, ws, st,
                           ev ? ev + 3 : nullptr));
    MOE_CUDA(launch_combine(c.dtype, x, Ys, drop, Sh, out->y, c.T, c.d, c.k, di.num_sms, st,
                            c.capacity_factor > 0.f),
             "combine launch");
    if (ev) MOE_CUDA(cudaEventRecord(ev[6], st), "event record");
    return MOE_OK;
}

int moe_layer_forward(const moe_cfg* cfg, const void* x, const void* Wr, const float* logit_bias,
                      const moe_weights* w, const moe_layer_out* out, void* ws, size_t ws_bytes,
                      void* stream) {
    return layer_forward_impl(cfg, x, Wr, logit_bias, w, out, ws, ws_bytes, stream, nullptr);
}

int moe_layer_forward_profiled(const moe_cfg* cfg, const void* x, const void* Wr,
                               const float* logit_bias, const moe_weights* w,
                               const moe_layer_out* out, void* ws, size_t ws_bytes, void* stream,
                               void* const* events) {
    if (!events) return fail(MOE_ERR_INVALID_ARG, "events is NULL%s");
    for (int i = 0; i < 7; ++i)
        if (!events[i]) return fail(MOE_ERR_INVALID_ARG, "events[i] is NULL%s");
    return layer_forward_impl(cfg, x, Wr, logit_bias, w, out, ws, ws_bytes, stream, events);
}

int moe_aux_loss_backward(const moe_cfg* cfg, const void* x, const void* Wr, const float* logits,
                          const int* counts_pre, float grad_aux, float* grad_logits,
                          float* grad_Wr, float* grad_x, void* stream) {
    MOE_TRY(check_cfg(cfg));
    if (cfg->T == 0) return MOE_OK;
    MOE_TRY(check_ptr4(logits, "logits"));
    MOE_TRY(check_ptr4(counts_pre, "counts_pre"));
    MOE_TRY(check_ptr4(grad_logits, "grad_logits"));
    if (grad_Wr) {
        MOE_TRY(check_ptr(x, "x"));
        MOE_TRY(check_ptr4(grad_Wr, "grad_Wr"));
    }
    if (grad_x) {
        MOE_TRY(check_ptr(Wr, "Wr"));
        MOE_TRY(check_ptr4(grad_x, "grad_x"));
    }
    DevInfo di;
    MOE_TRY(device_info(&di));
    MOE_CUDA(launch_aux_backward(cfg->dtype, cfg->scoring, x, Wr, logits, counts_pre, grad_aux,
                                 cfg->T, cfg->d, cfg->E, grad_logits, grad_Wr, grad_x, di.num_sms,
                                 (cudaStream_t)stream),
             "aux backward launch");
    return MOE_OK;
}

int moe_test_hold_lookback_block(void* ws, size_t ws_bytes, int block, void* stream) {
    if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL%s");
    if (ws_bytes < kCtrlWords * 4) return fail(MOE_ERR_WORKSPACE, "workspace too small%s");
    if (block < 0) return fail(MOE_ERR_INVALID_ARG, "block must be >= 0%s");
    static thread_local int value;      // pageable source; the copy is staged at enqueue
    value = block + 1;
    MOE_CUDA(cudaMemcpyAsync(at<int>(ws, 0) + kCtrlHoldBlock, &value, sizeof(int),
                             cudaMemcpyHostToDevice, (cudaStream_t)stream),
             "hold-block write");
    return MOE_OK;
}

int moe_test_hold_gemm_stage(void* ws, size_t ws_bytes, int iteration, void* stream) {
    if (!ws) return fail(MOE_ERR_INVALID_ARG, "workspace is NULL%s");
    if (ws_bytes < kCtrlWords * 4) return fail(MOE_ERR_WORKSPACE, "workspace too small%s");
    if (iteration < 0) return fail(MOE_ERR_INVALID_ARG, "iteration must be >= 0%s");
    static thread_local int value;      // pageable source; the copy is staged at enqueue
    value = iteration + 1;
    MOE_CUDA(cudaMemcpyAsync(at<int>(ws, 0) + kCtrlHoldGemm, &value, sizeof(int),
                             cudaMemcpyHostToDevice, (cudaStream_t)stream),
             "hold-stage write");
    return MOE_OK;
}

int moe_get_device_status(void* ws, size_t ws_bytes, void* stream, int* status) {
    if (!ws || !status) return fail(MOE_ERR_INVALID_ARG, "ws/status is NULL%s");
    if (ws_bytes < kCtrlWords * 4) return fail(MOE_ERR_WORKSPACE, "workspace too small%s");
    int v = 0;
    MOE_CUDA(cudaMemcpyAsync(&v, at<int>(ws, 0) + kCtrlStatus, sizeof v, cudaMemcpyDeviceToHost,
                             (cudaStream_t)stream),
             "status read");
    MOE_CUDA(cudaStreamSynchronize((cudaStream_t)stream), "status sync");
    *status = v;
    return MOE_OK;
}

}  // extern "C"
