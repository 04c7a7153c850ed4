// tc_common.cuh -- device helpers shared by the tensor-core kernels (forward and
// backward): instruction and shared-memory descriptors of tcgen05.mma, bounded mbarrier
// waits that end in a status word instead of a hang, and 16-bit packing.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "ptx.cuh"

namespace fa {
namespace tc {
namespace {

constexpr int kPanelCols = 64;          // 16-bit elements per 128-byte swizzled row
constexpr int kPanelBytes = 128 * 128;  // one 128-row x 64-column panel
constexpr float kLn2 = 0.6931471805599453f;

// Roles recorded in the status word when a wait gives up.
constexpr uint32_t kRoleSoftmax = 1, kRoleMma = 2, kRoleLoad = 3;

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator, A and B both bf16
// (or both fp16), A K-major, B K-major or MN-major, shape M x N.
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, bool b_mn_major, bool f16) {
    return (1u << 4)                                   // D format: f32
           | ((f16 ? 0u : 1u) << 7)                    // A format: f16 = 0, bf16 = 1
           | ((f16 ? 0u : 1u) << 10)                   // B format
           | ((b_mn_major ? 1u : 0u) << 16)            // B major-ness
           | ((uint32_t)(N >> 3) << 17)                // N / 8
           | ((uint32_t)(M >> 4) << 24);               // M / 16
}

// Shared-memory matrix descriptor, 128-byte swizzle (the layout TMA writes with
// CU_TENSOR_MAP_SWIZZLE_128B; tiles start on 1024-byte boundaries).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// ----------------------------------------------------------------- bounded waits
struct Ctl {
    uint32_t bars;                 // smem address of barrier 0
    volatile int* abort;           // CTA-wide abort flag (shared memory)
    unsigned long long limit;      // cycles
    unsigned int* status;          // device status word of the kernel's library unit
};

__device__ __forceinline__ uint32_t bar_addr(const Ctl& c, int i) { return c.bars + 8u * (uint32_t)i; }

__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int* abort,
                                       unsigned long long limit, uint32_t role, uint32_t id,
                                       unsigned int* status) {
    const long long t0 = clock64();
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if ((unsigned long long)(clock64() - t0) > limit) {
            *abort = 1;
            if (atomicCAS(&status[0], 0u, 1u) == 0u) {
                status[1] = role;
                status[2] = blockIdx.x;
                status[3] = id;
            }
            __threadfence();
            return false;
        }
    }
}

// Wait for the phase with `parity` of barrier `i`; false if the CTA is aborting.
__device__ __forceinline__ bool wait(const Ctl& c, int i, uint32_t parity, uint32_t role) {
    const uint32_t bar = bar_addr(c, i);
    if (ptx::mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, c.abort, c.limit, role, (uint32_t)i, c.status);
}

// Warp-wide wait: every lane waits, and the outcome is made uniform across the warp so
// that no lane reaches a .sync.aligned tcgen05 instruction without the others.
__device__ __forceinline__ bool wait_warp(const Ctl& c, int i, uint32_t parity, uint32_t role) {
    const bool ok = wait(c, i, parity, role);
    return __all_sync(0xFFFFFFFFu, ok);
}

// Teardown wait: bounded by time only (ignores the abort flag).
__device__ __noinline__ bool wait_drain(uint32_t bar, uint32_t parity, unsigned long long limit) {
    const long long t0 = clock64();
    while (!ptx::mbar_try_wait(bar, parity)) {
        if ((unsigned long long)(clock64() - t0) > limit) return false;
    }
    return true;
}

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    if constexpr (F16) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
}

// The low / high 16-bit value of a packed pair, as fp32.
template <bool F16>
__device__ __forceinline__ float unpack_lo(uint32_t w) {
    if constexpr (F16) return __half2float(__ushort_as_half((unsigned short)(w & 0xFFFFu)));
    else return __uint_as_float(w << 16);
}
template <bool F16>
__device__ __forceinline__ float unpack_hi(uint32_t w) {
    if constexpr (F16) return __half2float(__ushort_as_half((unsigned short)(w >> 16)));
    else return __uint_as_float(w & 0xFFFF0000u);
}

// Four fp32 values rounded to fp8 e4m3 (saturating at +-448) in one 32-bit word, the
// first value in the lowest byte.  cvt...e4m3x2 puts its first source in the upper byte.
__device__ __forceinline__ uint32_t pack4_e4m3(float a, float b, float c, float d) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

}  // namespace
}  // namespace tc
}  // namespace fa
