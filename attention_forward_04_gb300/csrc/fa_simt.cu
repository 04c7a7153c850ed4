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
// CTA = 128 threads = 32 rows x 4 threads, or, when that grid would leave SMs idle (a
// small problem), 8 rows x 16 threads: four times the CTAs and a quarter of the dependent
// work per thread and key.  Thread q of a row owns head-dim columns q, q+T, q+2T, ... (T
// threads per row; interleaved, so the threads of a row hit different banks when reading
// a shared K/V row).  Per key tile (32 keys; 16 at D = 256, which keeps the K and V tiles
// at 32 KB of static shared memory): partial dot products are summed across the T threads
// with shuffles, then the running max / sum update, exp with the new max, and the O
// update.  O is divided by l once at the end.
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kThreads = 128;

template <int D, int TPR, bool CAUSAL>
__global__ void __launch_bounds__(kThreads) fa_simt_kernel(const float* __restrict__ q,
                                                           const float* __restrict__ k,
                                                           const float* __restrict__ v,
                                                           float* __restrict__ o,
                                                           float* __restrict__ lse,
                                                           const SliceLayout g, float scale) {
    constexpr int kRows = kThreads / TPR;   // query rows per CTA
    constexpr int DQ = D / TPR;             // columns per thread
    constexpr int kKeys = D == 256 ? 16 : 32;   // keys per shared-memory tile
    __shared__ __align__(16) float Ks[kKeys][D];
    __shared__ __align__(16) float Vs[kKeys][D];

    const int tid = threadIdx.x;
    const int r = tid / TPR;       // row within the CTA
    const int qd = tid % TPR;      // column phase: columns qd + TPR*i
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
        qv[i] = live ? q[slice + (size_t)row * rs + qd + TPR * i] : 0.0f;
        acc[i] = 0.0f;
    }
    float m = -INFINITY, l = 0.0f;

    // Keys beyond the last row of the CTA are never visible under the causal mask.
    const int kend = CAUSAL ? min(n, (blk + 1) * kRows) : n;
    const int limit = CAUSAL ? min(row + 1, n) : n;   // visible keys: j < limit

    // Cooperative float4 loads of K and V rows k0..k0+kKeys-1 (rows >= n read as zero): each
    // thread moves kLoads float4 of each.  With 16 threads per row (few, short CTAs) the next
    // tile's loads are issued before the current tile's arithmetic, so their latency hides
    // behind it; with 4 threads per row the registers go to the longer rows instead.
    constexpr int kLoads = kKeys * D / 4 / kThreads;
    constexpr bool kPrefetch = TPR == 16;
    float4 kx[kLoads], vx[kLoads];
    auto fetch = [&](int k0) {
#pragma unroll
        for (int e = 0; e < kLoads; ++e) {
            const int idx = tid + e * kThreads;
            const int kr = idx / (D / 4);
            const int kc = (idx % (D / 4)) * 4;
            kx[e] = make_float4(0.f, 0.f, 0.f, 0.f);
            vx[e] = kx[e];
            if (k0 + kr < n) {
                kx[e] = *reinterpret_cast<const float4*>(k + slice + (size_t)(k0 + kr) * rs + kc);
                vx[e] = *reinterpret_cast<const float4*>(v + slice + (size_t)(k0 + kr) * rs + kc);
            }
        }
    };
    auto stash = [&]() {
#pragma unroll
        for (int e = 0; e < kLoads; ++e) {
            const int idx = tid + e * kThreads;
            const int kr = idx / (D / 4);
            const int kc = (idx % (D / 4)) * 4;
            *reinterpret_cast<float4*>(&Ks[kr][kc]) = kx[e];
            *reinterpret_cast<float4*>(&Vs[kr][kc]) = vx[e];
        }
    };
    if (kPrefetch && kend > 0) fetch(0);

    for (int k0 = 0; k0 < kend; k0 += kKeys) {
        __syncthreads();
        if (!kPrefetch) fetch(k0);
        stash();
        __syncthreads();
        if (kPrefetch && k0 + kKeys < kend) fetch(k0 + kKeys);

        float s[kKeys];
        float tmax = -INFINITY;
#pragma unroll
        for (int c = 0; c < kKeys; ++c) {
            float part = 0.0f;
#pragma unroll
            for (int i = 0; i < DQ; ++i) part = fmaf(qv[i], Ks[c][qd + TPR * i], part);
#pragma unroll
            for (int m = 1; m < TPR; m <<= 1) part += __shfl_xor_sync(0xFFFFFFFFu, part, m);
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
            for (int c = 0; c < kKeys; ++c) a = fmaf(s[c], Vs[c][qd + TPR * i], a);
            acc[i] = a;
        }
        m = m_new;
    }

    if (live) {
        const float inv_l = 1.0f / l;
#pragma unroll
        for (int i = 0; i < DQ; ++i) o[slice + (size_t)row * rs + qd + TPR * i] = acc[i] * inv_l;
        if (qd == 0) lse[lse0 + row] = m + logf(l);
    }
}

template <int D, int TPR, bool CAUSAL>
cudaError_t launch(const float* q, const float* k, const float* v, float* o, float* lse, int bh,
                   const SliceLayout& g, float scale, cudaStream_t stream) {
    constexpr int kRows = kThreads / TPR;
    const long long blocks = (long long)((g.n + kRows - 1) / kRows) * bh;
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
    fa_simt_kernel<D, TPR, CAUSAL><<<(unsigned)blocks, kThreads, 0, stream>>>(q, k, v, o, lse, g, scale);
    return cudaGetLastError();
}

template <int D, int TPR>
cudaError_t launch_c(bool causal, const float* q, const float* k, const float* v, float* o,
                     float* lse, int bh, const SliceLayout& g, float scale, cudaStream_t stream) {
    return causal ? launch<D, TPR, true>(q, k, v, o, lse, bh, g, scale, stream)
                  : launch<D, TPR, false>(q, k, v, o, lse, bh, g, scale, stream);
}

template <int D>
cudaError_t launch_d(bool wide, bool causal, const float* q, const float* k, const float* v,
                     float* o, float* lse, int bh, const SliceLayout& g, float scale,
                     cudaStream_t stream) {
    return wide ? launch_c<D, 16>(causal, q, k, v, o, lse, bh, g, scale, stream)
                : launch_c<D, 4>(causal, q, k, v, o, lse, bh, g, scale, stream);
}

}  // namespace

cudaError_t simt_launch(int D, bool causal, const float* q, const float* k, const float* v,
                        float* o, float* lse, int bh, const SliceLayout& g, float scale,
                        int sm_count, cudaStream_t stream) {
    // 16 threads per row when 32-row CTAs would not give every SM one
    const bool wide = (long long)((g.n + 31) / 32) * bh < (long long)sm_count;
    if (D == 32) return launch_d<32>(wide, causal, q, k, v, o, lse, bh, g, scale, stream);
    if (D == 64) return launch_d<64>(wide, causal, q, k, v, o, lse, bh, g, scale, stream);
    if (D == 256) return launch_d<256>(wide, causal, q, k, v, o, lse, bh, g, scale, stream);
    return launch_d<128>(wide, causal, q, k, v, o, lse, bh, g, scale, stream);
}

}  // namespace fa
