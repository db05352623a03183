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

// Device address of g_dispatch_scratch on the current device.  Looked up once
// per device (with that device current) and cached.  In host code the array's
// name is only a host-side stand-in, so kernels must be given this address.
cudaError_t scratch_address(void** out) {
    static std::mutex mu;
    static void* cache[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_dispatch_scratch);
        if (e != cudaSuccess) return e;
        cache[dev] = p;
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
    if (!counts_pre || !counts_kept || !offsets)
        return moe::set_last_error(MOE_ERR_INVALID_ARG, "moe_dispatch_noalloc: NULL count output");
    if (A == 0) return MOE_OK;
    if (!topk_idx || !perm_src || !dest || !drop_mask)
        return moe::set_last_error(MOE_ERR_INVALID_ARG, "moe_dispatch_noalloc: NULL argument");

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
