// tc_lowbit.cuh -- PTX wrappers used by the FP8-weight expert GEMMs only
// (ffn_fp8.cu): E4M3 -> f16 conversion, kind::f16 MMAs with A in tensor
// memory, TMEM stores, and the proxy fence for shared-memory reuse.
#pragma once

#include "tc_ptx.cuh"

namespace moe {
namespace ptx {

// Orders this thread's generic-proxy shared-memory accesses before the async
// proxy (TMA, tcgen05.mma) accesses that follow.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// mbar_wait for a warp whose wait is off the critical path: it sleeps `ns`
// between polls, so that its polling takes no issue slots from the warps that
// share its scheduler.  Same bounds as mbar_wait (abort flag, cycle limit).
__device__ __forceinline__ bool mbar_wait_nap(uint64_t* bar, uint32_t parity,
                                              const volatile int* abort_flag, unsigned ns) {
    const uint32_t addr = smem_u32(bar);
    if (mbar_try_wait(addr, parity)) return true;
    const long long t0 = clock64();
    while (true) {
        __nanosleep(ns);
        if (mbar_try_wait(addr, parity)) return true;
        if (abort_flag && *abort_flag) return false;
        if (clock64() - t0 > kWaitLimitCycles) return false;
    }
}

// Two E4M3 floats (low byte first) -> two f16 packed in 32 bits; exact, as
// every E4M3 value is an f16 value.
__device__ __forceinline__ uint32_t cvt_e4m3x2_f16x2(uint16_t v) {
    uint32_t out;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"(v));
    return out;
}

// Eight E2M1 floats (four bytes of a word; in each byte the low nibble first)
// -> four f16 pairs, c[i] from byte i.  The word is unpacked into byte
// registers inside one asm block: extracting each byte with shifts and masks
// in C++ cost ~3 more ALU instructions per byte, and the 4-bit converters are
// ALU-bound (measured: 16% of the 4-bit decode layer).
__device__ __forceinline__ void cvt_e2m1x8_f16x8(uint32_t w, uint32_t (&c)[4]) {
    asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
        "mov.b32 {q0, q1, q2, q3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, q0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, q1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, q2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, q3;\n\t}"
        : "=r"(c[0]), "=r"(c[1]), "=r"(c[2]), "=r"(c[3])
        : "r"(w));
}

// a * b for two f16 pairs (round to nearest even).
__device__ __forceinline__ uint32_t mul_f16x2(uint32_t a, uint32_t b) {
    uint32_t out;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(out) : "r"(a), "r"(b));
    return out;
}

// Instruction descriptor, kind::f16 with f16 A/B (format 0), fp32 accumulator.
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[tmem] * B[smem]^T, issued by one thread.  a_tmem addresses
// the tile's first column at lane 0; row m of A sits in lane m, two 16-bit
// elements per 32-bit column (lower k in the lower half), K/2 columns.
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                               uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 16 consecutive 32-bit columns of the warp's 32 lanes <- v (one lane per
// thread), then waits until the stores are done.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
        "r"(v[15])
        : "memory");
}
// Wait until this thread's earlier tcgen05.st have completed.
__device__ __forceinline__ void tmem_wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace ptx
}  // namespace moe
