// bwd_common.cuh -- pieces shared by the backward tensor-core kernels (fa_bwd.cu for head
// dimensions 32 to 128, fa_bwd256.cu for 256): where the rows of a slice live, the
// staged 16-bit store of an fp32 TMEM accumulator, and the predicate barrier of the
// elementwise warps.
#pragma once

#include <cstdint>

#include "fa_internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace fa {
namespace bwdc {
namespace {

using namespace tc;

// Where the rows of one (b, h) slice live.  MODE 0, [B, H, N, D]: N rows of D elements
// from element bh*N*D; LSE and delta at bh*N.  MODE 1, token-major [tokens, H, D]: rows H*D
// elements apart from token tok0 (fixed length N: tok0 = b*N; packed sequences: the
// clamped offsets of cu_seqlens), LSE and delta at [B, H, N] index bh*N, or [H, total]
// index h*total + tok0 for packed sequences.  A malformed offset can only give wrong
// values, never an access outside the tensors.
struct Slice {
    int len;          // rows of the slice
    int h, tok0;      // token-major: TMA coordinates of row 0 (head, token)
    size_t row0;      // element offset of row 0 in q, k, v, o, dout, dq, dk, dv
    size_t stride;    // elements from one row to the next
    size_t vec0;      // index of row 0 in lse and delta
};

template <int MODE, int D>
__device__ __forceinline__ Slice slice_at(const BwdParams& p, int bh) {
    Slice sl;
    if (MODE == 0) {
        sl.len = p.n;
        sl.h = 0;
        sl.tok0 = 0;
        sl.row0 = (size_t)bh * (size_t)p.n * D;
        sl.stride = D;
        sl.vec0 = (size_t)bh * (size_t)p.n;
        return sl;
    }
    const int b = bh / p.heads;
    sl.h = bh % p.heads;
    if (p.cu_seqlens != nullptr) {
        int s0 = __ldg(p.cu_seqlens + b), s1 = __ldg(p.cu_seqlens + b + 1);
        s0 = min(max(s0, 0), p.total);
        s1 = min(max(s1, s0), p.total);
        sl.len = min(s1 - s0, p.n);
        sl.tok0 = s0;
        sl.vec0 = (size_t)sl.h * (size_t)p.total + (size_t)s0;
    } else {
        sl.len = p.n;
        sl.tok0 = b * p.n;
        sl.vec0 = (size_t)bh * (size_t)p.n;
    }
    sl.row0 = ((size_t)sl.tok0 * p.heads + sl.h) * D;
    sl.stride = (size_t)p.heads * D;
    return sl;
}

// This warp's 32 TMEM lanes x 64 fp32 columns at t_acc, times mul, rounded to 16 bits, to
// global rows base + (row0 + r) * stride (r < 32, only rows with row0 + r < nrows; base
// points at the panel's first column), through a 4 KB staging slot so every store
// instruction writes whole 128-byte lines.
template <bool F16>
__device__ __forceinline__ void store_rows(uint32_t t_acc, float mul, uint32_t stage,
                                           uint16_t* base, size_t stride, int row0, int nrows,
                                           int lane) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t o[32];
        ptx::tmem_ld32_wait(t_acc + (uint32_t)(h * 32), o);
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = pack2<F16>(u2f(o[2 * i]) * mul, u2f(o[2 * i + 1]) * mul);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t chunk = (uint32_t)(h * 4 + i) ^ (uint32_t)(lane & 7);
            ptx::st_shared_v4(stage + (uint32_t)lane * 128u + chunk * 16u, w[4 * i],
                              w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        }
    }
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int r = 4 * k + (lane >> 3);
        const int ch = lane & 7;
        const uint4 v = ptx::ld_shared_v4(stage + (uint32_t)r * 128u + (uint32_t)((ch ^ (r & 7)) * 16));
        if (row0 + r < nrows)
            *reinterpret_cast<uint4*>(base + (size_t)(row0 + r) * stride + ch * 8) = v;
    }
    __syncwarp();
}

// Named barrier 1 over the 256 elementwise threads (warps 0-7) that also ANDs a predicate:
// a stop decision taken here is common to all eight warps, so no warp is ever left at a
// barrier that a warp which gave up will not reach.
__device__ __forceinline__ bool ew_barrier_and(bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 256, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok)
        : "memory");
    return r != 0;
}

}  // namespace
}  // namespace bwdc
}  // namespace fa
