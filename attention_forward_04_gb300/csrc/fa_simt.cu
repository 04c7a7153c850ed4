// fa_simt.cu -- fp32 attention forward on the CUDA cores (fp32 storage, fp32 arithmetic).
//
// The same tiled online-softmax forward as the tensor-core path, in plain fp32 FFMA:
// tensor-core TF32 would not hold fp32 accuracy.  The pages' fp32 kernel ("KingOfEgg:
// Flash Attention v1" §5.2) is the functional model; the structure here is the
// query-outer form instead ("08 · FlashAttention" §二; "第 13 课：GPU 内核与
// FlashAttention" Figure 13-2): each CTA owns 32 query rows of one (b, h) slice, keeps
// (m, l, O) on chip for the whole key loop, and writes O and LSE once.
//
// Layouts: [B, H, N, D] slices, or token-major [tokens, H, D] (fixed length N, or packed
// sequences with token offsets cu_seqlens), as in the tensor-core path.
//
// CTA = 128 threads = 32 rows x 4 threads.  Thread q of a row owns head-dim columns
// q, q+4, q+8, ... (interleaved, so the 4 threads of a row hit 4 different banks when
// reading a shared K/V row).  Per key tile (32 keys; 16 at D = 256, which keeps the K and V
// tiles at 32 KB of static shared memory): partial dot products are summed
// across the 4 threads with two shuffles, then the running max / sum update, exp with
// the new max, and the O update.  O is divided by l once at the end.
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kRows = 32;     // query rows per CTA
constexpr int kThreads = 128;

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads) fa_simt_kernel(const float* __restrict__ q,
                                                           const float* __restrict__ k,
                                                           const float* __restrict__ v,
                                                           float* __restrict__ o,
                                                           float* __restrict__ lse,
                                                           const SliceLayout g, float scale) {
    constexpr int DQ = D / 4;  // columns per thread
    constexpr int kKeys = D == 256 ? 16 : 32;   // keys per shared-memory tile
    __shared__ __align__(16) float Ks[kKeys][D];
    __shared__ __align__(16) float Vs[kKeys][D];

    const int tid = threadIdx.x;
    const int r = tid / 4;         // row within the CTA
    const int qd = tid % 4;        // column phase: columns qd + 4*i
    const int nblk = (g.n + kRows - 1) / kRows;
    const int bh = (int)(blockIdx.x / (unsigned)nblk);     // slice b*H + h
    const int blk = (int)(blockIdx.x % (unsigned)nblk);    // row block within the slice
    const int b = bh / g.heads, h = bh % g.heads;
    // Length and first token of the slice; packed offsets are clamped to [0, total] and
    // lengths to the declared maximum, so malformed offsets cannot move an access out of bounds.
    int n = g.n, tok0 = b * g.n;
    if (g.cu_seqlens != nullptr) {
        int s0 = g.cu_seqlens[b], s1 = g.cu_seqlens[b + 1];
        s0 = min(max(s0, 0), g.total);
        s1 = min(max(s1, s0), g.total);
        n = min(s1 - s0, g.n);
        tok0 = s0;
    }
    if (blk * kRows >= n) return;   // the whole block lies past the end of the sequence
    // row j of the slice starts at element slice + j * rs
    const size_t rs = g.layout == 0 ? (size_t)D : (size_t)g.heads * D;
    const size_t slice = g.layout == 0 ? (size_t)bh * (size_t)g.n * D : ((size_t)tok0 * g.heads + h) * D;
    const size_t lse0 = g.cu_seqlens != nullptr ? (size_t)h * g.total + tok0 : (size_t)bh * g.n;
    const int row = blk * kRows + r;
    const bool live = row < n;

    float qv[DQ], acc[DQ];
#pragma unroll
    for (int i = 0; i < DQ; ++i) {
        qv[i] = live ? q[slice + (size_t)row * rs + qd + 4 * i] : 0.0f;
        acc[i] = 0.0f;
    }
    float m = -INFINITY, l = 0.0f;

    // Keys beyond the last row of the CTA are never visible under the causal mask.
    const int kend = CAUSAL ? min(n, (blk + 1) * kRows) : n;
    const int limit = CAUSAL ? min(row + 1, n) : n;   // visible keys: j < limit

    for (int k0 = 0; k0 < kend; k0 += kKeys) {
        __syncthreads();
        // Cooperative float4 loads of K and V rows k0..k0+kKeys-1 (rows >= n read as zero).
        for (int idx = tid; idx < kKeys * D / 4; idx += kThreads) {
            const int kr = idx / (D / 4);
            const int kc = (idx % (D / 4)) * 4;
            float4 kx = make_float4(0.f, 0.f, 0.f, 0.f), vx = kx;
            if (k0 + kr < n) {
                kx = *reinterpret_cast<const float4*>(k + slice + (size_t)(k0 + kr) * rs + kc);
                vx = *reinterpret_cast<const float4*>(v + slice + (size_t)(k0 + kr) * rs + kc);
            }
            *reinterpret_cast<float4*>(&Ks[kr][kc]) = kx;
            *reinterpret_cast<float4*>(&Vs[kr][kc]) = vx;
        }
        __syncthreads();

        float s[kKeys];
        float tmax = -INFINITY;
#pragma unroll
        for (int c = 0; c < kKeys; ++c) {
            float part = 0.0f;
#pragma unroll
            for (int i = 0; i < DQ; ++i) part = fmaf(qv[i], Ks[c][qd + 4 * i], part);
            part += __shfl_xor_sync(0xFFFFFFFFu, part, 1);
            part += __shfl_xor_sync(0xFFFFFFFFu, part, 2);
            const bool vis = k0 + c < limit;
            s[c] = vis ? part * scale : -INFINITY;
            tmax = fmaxf(tmax, s[c]);
        }
        // Key 0 lies in the first tile and is visible to every row, so m is finite after
        // it; a later tile with no visible key for a row leaves that row as it was
        // (alpha = 1, p = 0).  Rows past the end keep finite values and are never stored.
        const float m_new = fmaxf(m, tmax);
        const float base = (m_new == -INFINITY) ? 0.0f : m_new;
        const float alpha = expf(m - base);   // m = -inf on the first tile -> 0
        float psum = 0.0f;
#pragma unroll
        for (int c = 0; c < kKeys; ++c) {
            s[c] = (s[c] == -INFINITY) ? 0.0f : expf(s[c] - base);
            psum += s[c];
        }
        l = l * alpha + psum;
#pragma unroll
        for (int i = 0; i < DQ; ++i) {
            float a = acc[i] * alpha;
#pragma unroll
            for (int c = 0; c < kKeys; ++c) a = fmaf(s[c], Vs[c][qd + 4 * i], a);
            acc[i] = a;
        }
        m = m_new;
    }

    if (live) {
        const float inv_l = 1.0f / l;
#pragma unroll
        for (int i = 0; i < DQ; ++i) o[slice + (size_t)row * rs + qd + 4 * i] = acc[i] * inv_l;
        if (qd == 0) lse[lse0 + row] = m + logf(l);
    }
}

template <int D, bool CAUSAL>
cudaError_t launch(const float* q, const float* k, const float* v, float* o, float* lse, int bh,
                   const SliceLayout& g, float scale, cudaStream_t stream) {
    const long long blocks = (long long)((g.n + kRows - 1) / kRows) * bh;
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
    fa_simt_kernel<D, CAUSAL><<<(unsigned)blocks, kThreads, 0, stream>>>(q, k, v, o, lse, g, scale);
    return cudaGetLastError();
}

}  // namespace

cudaError_t simt_launch(int D, bool causal, const float* q, const float* k, const float* v,
                        float* o, float* lse, int bh, const SliceLayout& g, float scale,
                        cudaStream_t stream) {
    if (D == 32)
        return causal ? launch<32, true>(q, k, v, o, lse, bh, g, scale, stream)
                      : launch<32, false>(q, k, v, o, lse, bh, g, scale, stream);
    if (D == 64)
        return causal ? launch<64, true>(q, k, v, o, lse, bh, g, scale, stream)
                      : launch<64, false>(q, k, v, o, lse, bh, g, scale, stream);
    if (D == 256)
        return causal ? launch<256, true>(q, k, v, o, lse, bh, g, scale, stream)
                      : launch<256, false>(q, k, v, o, lse, bh, g, scale, stream);
    return causal ? launch<128, true>(q, k, v, o, lse, bh, g, scale, stream)
                  : launch<128, false>(q, k, v, o, lse, bh, g, scale, stream);
}

}  // namespace fa
