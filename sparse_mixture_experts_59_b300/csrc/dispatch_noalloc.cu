// dispatch_noalloc.cu -- moe_dispatch without a caller-supplied workspace.
//
// moe_dispatch needs scratch memory (the decoupled look-back's status words,
// the per-assignment ranks and a few control words), which normally lives in
// a workspace the caller allocates.  Some callers cannot call cudaMalloc or
// hand over extra device memory -- for example a host framework that owns
// every device allocation and gives an operator only its input and output
// buffers.  moe_dispatch_noalloc serves them: its scratch is the file-scope
// device array below, of a fixed maximum size, which every GPU that loads
// this library holds until the process exits.  It allocates nothing.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "kernels.cuh"

namespace {

// Largest T*k the static scratch covers, and its layout:
//   [control words][look-back status: blocks x 256 experts][rank: T*k]
constexpr int kNoAllocMaxAssignments = 65536;
constexpr size_t kCtrlBytes = (size_t)moe::kCtrlWords * 4;
constexpr size_t kMaxBlocks =
    (size_t)(kNoAllocMaxAssignments + moe::kDspChunk - 1) / moe::kDspChunk;
constexpr size_t kStatusBytes = kMaxBlocks * moe::kMaxExperts * 4;
constexpr size_t kRankBytes = (size_t)kNoAllocMaxAssignments * 4;
constexpr size_t kScratchBytes = kCtrlBytes + kStatusBytes + kRankBytes;   // 393,472 bytes
static_assert(kCtrlBytes % 256 == 0 && kStatusBytes % 256 == 0, "scratch regions stay aligned");
static_assert(kScratchBytes == 393472, "the size stated in include/moe.h");

// Shared by every call on a device; keeps the last call's contents.
static __device__ __align__(256) unsigned char g_dispatch_scratch[kScratchBytes];

// Driver calls that identify the calling thread's current context.  A
// context's id is never reused within a process, so an address cached under
// it cannot outlive the module it was read from (cudaDeviceReset destroys the
// primary context; the runtime then loads the module again into a new one,
// where the array may sit at another address).
struct CtxApi {
    CUresult (*get_current)(CUcontext*) = nullptr;
    CUresult (*get_id)(CUcontext, unsigned long long*) = nullptr;
};
const CtxApi& ctx_api() {
    static const CtxApi api = [] {
        CtxApi a;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
            a.get_current = reinterpret_cast<CUresult (*)(CUcontext*)>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            a.get_id = reinterpret_cast<CUresult (*)(CUcontext, unsigned long long*)>(p);
        return a;
    }();
    return api;
}
// Id of the current context (0 if there is none yet or it cannot be read).
unsigned long long current_ctx_id() {
    const CtxApi& a = ctx_api();
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!a.get_current || !a.get_id || a.get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (a.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of g_dispatch_scratch in the current context.  Looked up
// with the device current the first time a context calls this, and cached
// per device together with that context's id; a different context on the
// same device (after cudaDeviceReset) looks it up again.  In host code the
// array's name is only a host-side stand-in, so kernels must be given this
// address.
cudaError_t scratch_address(void** out) {
    static std::mutex mu;
    static void* cache[64] = {};
    static unsigned long long cache_ctx[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    const unsigned long long id = current_ctx_id();
    if (!cache[dev] || id == 0 || id != cache_ctx[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_dispatch_scratch);   // creates the context if needed
        if (e != cudaSuccess) return e;
        cache[dev] = p;
        cache_ctx[dev] = current_ctx_id();
    }
    *out = cache[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" int moe_dispatch_noalloc(const moe_cfg* cfg, const int* topk_idx,
                                    const float* prob_mean, int* counts_pre, int* counts_kept,
                                    int* offsets, int* perm_src, int* dest,
                                    unsigned char* drop_mask, float* stats, int* device_status,
                                    void* stream) {
    size_t unused = 0;
    const int rc = moe_workspace_size(cfg, &unused);   // validates cfg
    if (rc != MOE_OK) return rc;
    const long long A = (long long)cfg->T * cfg->k;
    if (A > kNoAllocMaxAssignments)
        return moe::set_last_error(MOE_ERR_INVALID_ARG,
                                   "moe_dispatch_noalloc: T*k exceeds its static scratch maximum "
                                   "of 65536 assignments; use moe_dispatch with a workspace");
    // the pointer checks of moe_dispatch: every int / float buffer non-NULL
    // (where required) and 4-byte aligned, so no misaligned access reaches
    // the kernels
    int pc = MOE_OK;
    if ((pc = moe::check_aligned4(counts_pre, "counts_pre")) != MOE_OK ||
        (pc = moe::check_aligned4(counts_kept, "counts_kept")) != MOE_OK ||
        (pc = moe::check_aligned4(offsets, "offsets")) != MOE_OK)
        return pc;
    if (A == 0) return MOE_OK;
    if ((pc = moe::check_aligned4(topk_idx, "topk_idx")) != MOE_OK ||
        (pc = moe::check_aligned4(perm_src, "perm_src")) != MOE_OK ||
        (pc = moe::check_aligned4(dest, "dest")) != MOE_OK ||
        (stats && (pc = moe::check_aligned4(stats, "stats")) != MOE_OK) ||
        (prob_mean && (pc = moe::check_aligned4(prob_mean, "prob_mean")) != MOE_OK) ||
        (device_status && (pc = moe::check_aligned4(device_status, "device_status")) != MOE_OK))
        return pc;
    if (!drop_mask)
        return moe::set_last_error(MOE_ERR_INVALID_ARG, "moe_dispatch_noalloc: drop_mask is NULL");

    cudaStream_t st = (cudaStream_t)stream;
    void* base = nullptr;
    cudaError_t e = scratch_address(&base);
    if (e != cudaSuccess) return moe::set_cuda_error(e, "moe_dispatch_noalloc: scratch address");
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
        return moe::set_cuda_error(e, "moe_dispatch_noalloc: device attributes");

    unsigned char* scratch = static_cast<unsigned char*>(base);
    int* ctrl = reinterpret_cast<int*>(scratch);
    unsigned* tile_status = reinterpret_cast<unsigned*>(scratch + kCtrlBytes);
    int* rank = reinterpret_cast<int*>(scratch + kCtrlBytes + kStatusBytes);
    // The control words and the look-back status must start at zero; an
    // earlier call that stopped on a device error may have left them set.
    const size_t clear = kCtrlBytes + (size_t)moe::dispatch_blocks((int)A) * cfg->E * 4;
    if ((e = cudaMemsetAsync(scratch, 0, clear, st)) != cudaSuccess)
        return moe::set_cuda_error(e, "moe_dispatch_noalloc: clear scratch");
    e = moe::launch_dispatch(topk_idx, cfg->T, cfg->k, cfg->E, moe_capacity(cfg), tile_status,
                             ctrl, rank, counts_pre, counts_kept, offsets, dest, perm_src,
                             drop_mask, prob_mean, stats, sms, st);
    if (e != cudaSuccess) return moe::set_cuda_error(e, "moe_dispatch_noalloc: launch");
    if (device_status) {
        e = cudaMemcpyAsync(device_status, ctrl + moe::kCtrlStatus, sizeof(int),
                            cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) return moe::set_cuda_error(e, "moe_dispatch_noalloc: status copy");
    }
    return MOE_OK;
}
