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

#include <atomic>
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

// Tiny problems (all query rows fit in about two waves of CTAs): each CTA owns kRowsR = 2
// rows and its 256 threads work across keys instead of across the head dimension, so no
// per-key shuffle sits on the critical path.  Per chunk of keys, K and V are first copied
// into shared memory with coalesced loads that are all issued before any is used (one
// memory latency per chunk); then thread j (or, at D = 128, a pair of threads) forms the
// scores of key j for both rows, block-wide max and sum give the running (m, l) update, P
// goes to shared memory, and thread (part, r, d) accumulates O[r][d] over its share of the
// chunk's keys.  The partial O of the key shares are added through shared memory at the end.
constexpr int kRowsR = 2;
constexpr int kThreadsR = 256;

template <int D>
struct RowsGeo {
    static constexpr int kTpk = D >= 128 ? D / 64 : 1;       // threads per key (scores)
    static constexpr int kKeys = kThreadsR / kTpk;            // keys per chunk
    static constexpr int kKStride = D + 1;                    // padded K row (bank-conflict free)
    static constexpr int kParts = kThreadsR / (kRowsR * D);   // key shares of the O accumulation
    static constexpr int kSmemFloats = kKeys * kKStride + kKeys * D + kRowsR * kKeys;
    static constexpr int kSmemBytes = kSmemFloats * 4;
    static_assert(kRowsR * D <= kThreadsR && kThreadsR % (kRowsR * D) == 0, "threads per (row, column)");
};

__device__ __forceinline__ float block_reduce(float x, float* red, bool is_max) {
    // 8 warps: shuffle within the warp, then one value per warp through shared memory
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) {
        const float y = __shfl_xor_sync(0xFFFFFFFFu, x, m);
        x = is_max ? fmaxf(x, y) : x + y;
    }
    __syncthreads();   // red[] free to reuse
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = x;
    __syncthreads();
    float t = red[0];
#pragma unroll
    for (int w = 1; w < kThreadsR / 32; ++w) t = is_max ? fmaxf(t, red[w]) : t + red[w];
    return t;
}

// x[r] for a run-time r, without indexing a register array (which would go to local memory)
__device__ __forceinline__ float pick(const float (&x)[kRowsR], int r) {
    float y = x[0];
#pragma unroll
    for (int i = 1; i < kRowsR; ++i) y = r == i ? x[i] : y;
    return y;
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreadsR) fa_simt_rows_kernel(const float* __restrict__ q,
                                                                 const float* __restrict__ k,
                                                                 const float* __restrict__ v,
                                                                 float* __restrict__ o,
                                                                 float* __restrict__ lse,
                                                                 const SliceLayout g, float scale) {
    using G = RowsGeo<D>;
    constexpr int kKeys = G::kKeys, kTpk = G::kTpk, kParts = G::kParts;
    extern __shared__ __align__(16) float dyn[];
    float* ks = dyn;                              // [kKeys][D + 1]
    float* vs = ks + kKeys * G::kKStride;         // [kKeys][D]
    float* ps = vs + kKeys * D;                   // [kRowsR][kKeys]
    __shared__ __align__(16) float qs[kRowsR][D];
    __shared__ float red[kThreadsR / 32];
    __shared__ float os[kParts][kRowsR][D];

    const int tid = threadIdx.x;
    const int nblk = (g.n + kRowsR - 1) / kRowsR;
    const int bh = (int)(blockIdx.x / (unsigned)nblk);
    const int blk = (int)(blockIdx.x % (unsigned)nblk);
    const int b = bh / g.heads, h = bh % g.heads;
    int n = g.n, tok0 = b * g.n;
    if (g.cu_seqlens != nullptr) {   // clamped as in fa_simt_kernel
        int s0 = g.cu_seqlens[b], s1 = g.cu_seqlens[b + 1];
        s0 = min(max(s0, 0), g.total);
        s1 = min(max(s1, s0), g.total);
        n = min(s1 - s0, g.n);
        tok0 = s0;
    }
    const int row0 = blk * kRowsR;
    if (row0 >= n) return;   // the whole block lies past the end of the sequence
    const size_t rs = g.layout == 0 ? (size_t)D : (size_t)g.heads * D;
    const size_t slice = g.layout == 0 ? (size_t)bh * (size_t)g.n * D : ((size_t)tok0 * g.heads + h) * D;
    const size_t lse0 = g.cu_seqlens != nullptr ? (size_t)h * g.total + tok0 : (size_t)bh * g.n;

    for (int e = tid; e < kRowsR * D; e += kThreadsR) {   // the rows' Q (zeros past the end)
        const int r = e / D, c = e % D;
        qs[r][c] = row0 + r < n ? q[slice + (size_t)(row0 + r) * rs + c] : 0.0f;
    }
    // score role: key kj of the chunk, head-dim quarter kq of kTpk
    const int kj = tid / kTpk, kq = tid % kTpk;
    // accumulation role: row ar, column ad, key share part
    const int ar = (tid / D) % kRowsR, ad = tid % D, part = tid / (kRowsR * D);
    float acc = 0.0f;
    float m[kRowsR], l[kRowsR];
#pragma unroll
    for (int r = 0; r < kRowsR; ++r) { m[r] = -INFINITY; l[r] = 0.0f; }

    // under the causal mask no key after the block's last row is visible
    const int kend = CAUSAL ? min(n, row0 + kRowsR) : n;
    for (int k0 = 0; k0 < kend; k0 += kKeys) {
        const int jn = min(kKeys, kend - k0);   // keys of this chunk
        // K and V rows k0.. into shared memory: every float4 load issued before any store
        constexpr int kVec = kKeys * D / 4 / kThreadsR;   // float4 of K (and of V) per thread
        float4 kx[kVec], vx[kVec];
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
            const int idx = tid + e * kThreadsR;
            const int kr = idx / (D / 4), kc = (idx % (D / 4)) * 4;
            kx[e] = make_float4(0.f, 0.f, 0.f, 0.f);
            vx[e] = kx[e];
            if (kr < jn) {
                kx[e] = *reinterpret_cast<const float4*>(k + slice + (size_t)(k0 + kr) * rs + kc);
                vx[e] = *reinterpret_cast<const float4*>(v + slice + (size_t)(k0 + kr) * rs + kc);
            }
        }
        __syncthreads();   // the previous chunk's readers of ks, vs, ps are done (and qs is stored)
#pragma unroll
        for (int e = 0; e < kVec; ++e) {
            const int idx = tid + e * kThreadsR;
            const int kr = idx / (D / 4), kc = (idx % (D / 4)) * 4;
            float* kd = ks + kr * G::kKStride + kc;
            kd[0] = kx[e].x; kd[1] = kx[e].y; kd[2] = kx[e].z; kd[3] = kx[e].w;
            *reinterpret_cast<float4*>(vs + kr * D + kc) = vx[e];
        }
        __syncthreads();
        float sc[kRowsR];
#pragma unroll
        for (int r = 0; r < kRowsR; ++r) sc[r] = 0.0f;
        {
            const float* kr = ks + kj * G::kKStride + kq * (D / kTpk);
#pragma unroll 16
            for (int c = 0; c < D / kTpk; ++c) {
                const float kvv = kr[c];
#pragma unroll
                for (int r = 0; r < kRowsR; ++r) sc[r] = fmaf(qs[r][kq * (D / kTpk) + c], kvv, sc[r]);
            }
#pragma unroll
            for (int r = 0; r < kRowsR; ++r)
#pragma unroll
                for (int w = 1; w < kTpk; w <<= 1) sc[r] += __shfl_xor_sync(0xFFFFFFFFu, sc[r], w);
        }
        const int j = k0 + kj;   // this thread's key (shared by the kTpk threads of a key)
        float alpha[kRowsR];
#pragma unroll
        for (int r = 0; r < kRowsR; ++r) {
            const int row = row0 + r;
            const int limit = CAUSAL ? min(row + 1, n) : n;   // visible keys: j < limit
            const float s = (kj < jn && j < limit) ? sc[r] * scale : -INFINITY;
            const float m_new = fmaxf(m[r], block_reduce(s, red, true));
            // a row past the end (or with no visible key yet) keeps m = -inf: nothing added
            const float base = m_new == -INFINITY ? 0.0f : m_new;
            const float p = s == -INFINITY ? 0.0f : expf(s - base);
            alpha[r] = expf(m[r] - base);   // m = -inf on the first chunk: 0
            // the kTpk threads of a key hold the same p: count it once
            l[r] = l[r] * alpha[r] + block_reduce(kq == 0 ? p : 0.0f, red, false);
            m[r] = m_new;
            if (kq == 0) ps[r * kKeys + kj] = p;
        }
        __syncthreads();   // P of the chunk is complete
        // four independent sums keep the dependent FMA chain a quarter as long
        float a4[4] = {acc * pick(alpha, ar), 0.0f, 0.0f, 0.0f};
        int jj = part;
        for (; jj + 3 * kParts < jn; jj += 4 * kParts) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
                a4[u] = fmaf(ps[ar * kKeys + jj + u * kParts], vs[(jj + u * kParts) * D + ad], a4[u]);
        }
        for (; jj < jn; jj += kParts) a4[0] = fmaf(ps[ar * kKeys + jj], vs[jj * D + ad], a4[0]);
        acc = (a4[0] + a4[1]) + (a4[2] + a4[3]);
    }
    os[part][ar][ad] = acc;
    __syncthreads();
    if (part == 0 && row0 + ar < n) {
        float t = 0.0f;
#pragma unroll
        for (int pp = 0; pp < kParts; ++pp) t += os[pp][ar][ad];
        const float l_r = pick(l, ar);
        o[slice + (size_t)(row0 + ar) * rs + ad] = t / l_r;
        if (ad == 0) lse[lse0 + row0 + ar] = pick(m, ar) + logf(l_r);
    }
}

template <int D, bool CAUSAL>
cudaError_t launch_rows(const float* q, const float* k, const float* v, float* o, float* lse,
                        int bh, const SliceLayout& g, float scale, cudaStream_t stream) {
    // the dynamic shared-memory limit is raised once per device
    static std::atomic<uint32_t> raised{0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint32_t bit = 1u << (dev & 31);
    if (!(raised.load() & bit)) {
        e = cudaFuncSetAttribute(fa_simt_rows_kernel<D, CAUSAL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 RowsGeo<D>::kSmemBytes);
        if (e != cudaSuccess) return e;
        raised.fetch_or(bit);
    }
    const long long blocks = (long long)((g.n + kRowsR - 1) / kRowsR) * bh;
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
    fa_simt_rows_kernel<D, CAUSAL><<<(unsigned)blocks, kThreadsR, RowsGeo<D>::kSmemBytes, stream>>>(
        q, k, v, o, lse, g, scale);
    return cudaGetLastError();
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
    // two rows per CTA, threads across keys, when all of them fit in about two waves
    // (D <= 128); else 16 threads per row when 32-row CTAs would not give every SM one
    if (D <= 128 && (long long)((g.n + kRowsR - 1) / kRowsR) * bh <= 2LL * sm_count) {
        if (D == 32) return causal ? launch_rows<32, true>(q, k, v, o, lse, bh, g, scale, stream)
                                   : launch_rows<32, false>(q, k, v, o, lse, bh, g, scale, stream);
        if (D == 64) return causal ? launch_rows<64, true>(q, k, v, o, lse, bh, g, scale, stream)
                                   : launch_rows<64, false>(q, k, v, o, lse, bh, g, scale, stream);
        return causal ? launch_rows<128, true>(q, k, v, o, lse, bh, g, scale, stream)
                      : launch_rows<128, false>(q, k, v, o, lse, bh, g, scale, stream);
    }
    const bool wide = (long long)((g.n + 31) / 32) * bh < (long long)sm_count;
    if (D == 32) return launch_d<32>(wide, causal, q, k, v, o, lse, bh, g, scale, stream);
    if (D == 64) return launch_d<64>(wide, causal, q, k, v, o, lse, bh, g, scale, stream);
    if (D == 256) return launch_d<256>(wide, causal, q, k, v, o, lse, bh, g, scale, stream);
    return launch_d<128>(wide, causal, q, k, v, o, lse, bh, g, scale, stream);
}

}  // namespace fa
