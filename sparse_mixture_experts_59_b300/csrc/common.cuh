// common.cuh -- small shared pieces of the MoE CUDA path (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Block-wide barrier.  Each warp reconverges first: bar.sync counts a warp's
// arrival as the whole warp, so in code where the lanes of a warp can reach
// the barrier apart (a role loop run by lane 0, per-lane spin waits) the
// lanes that arrive first would count the warp as arrived, and the barrier
// could pass while other warps still work.
__device__ __forceinline__ void block_sync() {
    __syncwarp();
    __syncthreads();
}

// Loads, at L2, of values that other CTAs published before a ticket or flag
// this thread has already observed.  Volatile with a memory clobber: __ldcg's
// asm is neither, and nothing would then stop the compiler from moving it
// above the synchronisation that makes the values valid.
__device__ __forceinline__ float ld_cg(const float* p) {
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ float4 ld_cg(const float4* p) {
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}


// ---------------------------------------------------------------- limits
constexpr int kMaxExperts = 256;   // one dispatch thread per expert
constexpr int kMaxTopK = 8;

// Workspace control words (int32 each, at the start of the workspace).
enum CtrlWord {
    kCtrlStatus = 0,        // first device error (MOE_ERR_DEVICE_*), 0 = none
    kCtrlDispatchTicket = 1,
    kCtrlDispatchDone = 2,
    kCtrlRouterDone = 3,
    kCtrlHoldBlock = 4,     // test hook: look-back block (id + 1) that never publishes
    kCtrlFrontDone = 5,     // decode-sized route + dispatch: CTAs done with phase 1
    kCtrlHoldGemm = 6,      // test hook: up-projection ring iteration (+ 1) never loaded
    kCtrlWords = 64
};

// Bounded waits: about a second at the B300's clocks.  Legitimate waits in
// these kernels last microseconds.
constexpr long long kWaitLimitCycles = 2000000000LL;

// Programmatic dependent launch.  Every kernel of the layer is launched so
// that it may start while its stream predecessor finishes: it does its
// on-chip set-up, then pdl_wait() before its first global-memory access (that
// returns once the predecessor grid has completed and its writes are
// visible), then pdl_trigger() so that its own successor may be scheduled.
// Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void raise_error(int* status, int code) {
    if (status) atomicCAS(status, 0, code);
}

// --------------------------------------------------------- element access
template <typename T> struct Elem;
template <> struct Elem<float> {
    __device__ __forceinline__ static float load(const float* p) { return *p; }
    __device__ __forceinline__ static float to_f(float v) { return v; }
    __device__ __forceinline__ static float from_f(float v) { return v; }
};
template <> struct Elem<__nv_bfloat16> {
    __device__ __forceinline__ static float load(const __nv_bfloat16* p) { return __bfloat162float(*p); }
    __device__ __forceinline__ static float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
    __device__ __forceinline__ static __nv_bfloat16 from_f(float v) { return __float2bfloat16_rn(v); }
};

// 16-byte vector of T: 4 floats or 8 bf16.
template <typename T> struct Vec16 { static constexpr int N = 16 / sizeof(T); };

__device__ __forceinline__ void unpack16(const uint4& v, float (&f)[4]) {
    f[0] = __uint_as_float(v.x); f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z); f[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void unpack16(const uint4& v, float (&f)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float2 p = __bfloat1622float2(h[i]);
        f[2 * i] = p.x; f[2 * i + 1] = p.y;
    }
}
__device__ __forceinline__ uint4 pack16(const float (&f)[4]) {
    return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]),
                      __float_as_uint(f[2]), __float_as_uint(f[3]));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint4 pack16(const float (&f)[8]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]),
                      pack_bf16x2(f[4], f[5]), pack_bf16x2(f[6], f[7]));
}

// ------------------------------------------------------------ activations
// GELU, exact erf form (nn.GELU default): z/2 * (1 + erf(z/sqrt(2))).
__device__ __forceinline__ float gelu_erf(float z) {
    return 0.5f * z * (1.0f + erff(z * 0.70710678118654752f));
}
// SiLU z * sigmoid(z).
__device__ __forceinline__ float silu(float z) {
    return z / (1.0f + __expf(-z));
}

// ------------------------------------------------------ group tile prefix
// Fills s_start[0..G] with the exclusive prefix of per-group tile counts,
// tiles(g) = ceil(rows(g) / tile_rows) * ntiles_n(g), where rows(g) comes from
// offsets for routed groups g < E and is `shared_rows` for g == E (when
// shared_rows > 0).  Must be called by all threads of the block; ends with a
// block barrier.  Uses warp 0 for the scan.
__device__ __forceinline__ void group_tile_prefix(const int* __restrict__ offsets, int E,
                                                  int shared_rows, int tile_rows, int nt_routed,
                                                  int nt_shared, int* s_start) {
    const int G = E + (shared_rows > 0 ? 1 : 0);
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int carry = 0;
        for (int base = 0; base < G; base += 32) {
            const int g = base + lane;
            int v = 0;
            if (g < E) {
                const int rows = offsets[g + 1] - offsets[g];
                v = (rows + tile_rows - 1) / tile_rows * nt_routed;
            } else if (g < G) {
                v = (shared_rows + tile_rows - 1) / tile_rows * nt_shared;
            }
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            if (g < G) s_start[g] = carry + incl - v;
            carry += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) s_start[G] = carry;
    }
    block_sync();
}

// Group g holding linear tile index `tile` (s_start ascending, G groups).
__device__ __forceinline__ int find_group(const int* s_start, int G, int tile) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_start[mid] <= tile) lo = mid; else hi = mid - 1;
    }
    return lo;
}

}  // namespace moe
