// fa_simt_bwd.cu -- fp32 attention backward on the CUDA cores (fp32 storage and arithmetic).
//
// The gradients of the forward in fa_simt.cu, with P rebuilt from the forward's LSE
// ("08 · FlashAttention" §三; "第 13 课：GPU 内核与 FlashAttention" §4B):
//     P = exp(scale * Q K^T - LSE),  dP = dO V^T,  delta = rowsum(dO * O),
//     dS = P * (dP - delta),  dV = P^T dO,  dQ = scale * dS K,  dK = scale * dS^T Q.
// Two kernels, as on the tensor cores, and no atomics:
//   * dQ: one CTA per 32 query rows (16 at D = 256); it forms delta for its rows (written
//     to the workspace for the next kernel), then walks the key tiles with K and V in
//     shared memory;
//   * dK, dV: one CTA per 32 key rows (16 at D = 256); it walks the query tiles with Q,
//     dO, LSE and delta in shared memory.
// CTA = 128 threads = 32 rows x 4 threads (16 rows x 8 threads at D = 256, which keeps 32
// columns per thread and the shared tiles at 32 KB), or 8 rows x 16 threads when those
// CTAs would not give every SM one; thread t of a row owns head-dim columns t, t+T, t+2T,
// ... (T threads per row); a dot product over D is the T partial sums added with shuffles.  Layouts as the forward: [B, H, N, D], token-major [tokens, H, D],
// packed sequences.
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_internal.h"

namespace fa {
namespace {

constexpr int kThreads = 128;

// Threads per row, rows per CTA, columns per thread, and rows per streamed tile (the key
// tiles of the dQ kernel, the query tiles of the dK/dV kernel; 16 at D = 256 so the two
// shared tiles stay at 32 KB).  WIDE: 16 threads on 8 rows, for problems whose 32-row
// (16 at D = 256) CTAs would not give every SM one; the next streamed tile is then fetched
// into registers during the current tile's arithmetic.
template <int D, bool WIDE> struct Shape {
    static constexpr int kTpr = WIDE ? 16 : (D == 256 ? 8 : 4);
    static constexpr int kRows = kThreads / kTpr;
    static constexpr int kCols = D / kTpr;
    static constexpr int kTile = D == 256 ? 16 : 32;
    static constexpr int kLoads = kTile * D / 4 / kThreads;   // float4 per thread per tensor
};

// Length, element offset of row 0, row stride (elements) and LSE / delta index of row 0 of
// slice bh; packed offsets are clamped to [0, total] and lengths to the declared maximum.
struct SimtSlice {
    int len;
    size_t base, rs, vec0;
};

template <int D>
__device__ __forceinline__ SimtSlice simt_slice(const SliceLayout& g, int bh) {
    const int b = bh / g.heads, h = bh % g.heads;
    int n = g.n, tok0 = b * g.n;
    if (g.cu_seqlens != nullptr) {
        int s0 = g.cu_seqlens[b], s1 = g.cu_seqlens[b + 1];
        s0 = min(max(s0, 0), g.total);
        s1 = min(max(s1, s0), g.total);
        n = min(s1 - s0, g.n);
        tok0 = s0;
    }
    SimtSlice s;
    s.len = n;
    s.rs = g.layout == 0 ? (size_t)D : (size_t)g.heads * D;
    s.base = g.layout == 0 ? (size_t)bh * (size_t)g.n * D : ((size_t)tok0 * g.heads + h) * D;
    s.vec0 = g.cu_seqlens != nullptr ? (size_t)h * g.total + tok0 : (size_t)bh * g.n;
    return s;
}

// Sum over the TPR consecutive lanes that share a row.
template <int TPR>
__device__ __forceinline__ float row_sum(float x) {
#pragma unroll
    for (int m = 1; m < TPR; m <<= 1) x += __shfl_xor_sync(0xFFFFFFFFu, x, m);
    return x;
}

// Two streamed [kTile][D] tiles of one slice (K and V, or Q and dO) through registers:
// fetch() issues the float4 loads of rows r0.. (rows at or past len read as zero), stash()
// writes them to shared memory.
template <int D, bool WIDE>
struct TilePair {
    static constexpr int kTile = Shape<D, WIDE>::kTile, kLoads = Shape<D, WIDE>::kLoads;
    float4 a[kLoads], b[kLoads];
    __device__ __forceinline__ void fetch(const float* __restrict__ sa, const float* __restrict__ sb,
                                          const SimtSlice& s, int r0) {
#pragma unroll
        for (int e = 0; e < kLoads; ++e) {
            const int idx = (int)threadIdx.x + e * kThreads;
            const int r = idx / (D / 4), c = (idx % (D / 4)) * 4;
            a[e] = make_float4(0.f, 0.f, 0.f, 0.f);
            b[e] = a[e];
            if (r0 + r < s.len) {
                const size_t off = s.base + (size_t)(r0 + r) * s.rs + c;
                a[e] = *reinterpret_cast<const float4*>(sa + off);
                b[e] = *reinterpret_cast<const float4*>(sb + off);
            }
        }
    }
    __device__ __forceinline__ void stash(float (*da)[D], float (*db)[D]) const {
#pragma unroll
        for (int e = 0; e < kLoads; ++e) {
            const int idx = (int)threadIdx.x + e * kThreads;
            const int r = idx / (D / 4), c = (idx % (D / 4)) * 4;
            *reinterpret_cast<float4*>(&da[r][c]) = a[e];
            *reinterpret_cast<float4*>(&db[r][c]) = b[e];
        }
    }
};

template <int D, bool WIDE, bool CAUSAL>
__global__ void __launch_bounds__(kThreads) simt_bwd_dq_kernel(
    const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
    const float* __restrict__ o, const float* __restrict__ dout, const float* __restrict__ lse,
    float* __restrict__ delta, float* __restrict__ dq, const SliceLayout g, float scale) {
    using S = Shape<D, WIDE>;
    constexpr int kRows = S::kRows, TPR = S::kTpr, DQ = S::kCols, kTile = S::kTile;
    __shared__ __align__(16) float Ks[kTile][D];
    __shared__ __align__(16) float Vs[kTile][D];
    const int nblk = (g.n + kRows - 1) / kRows;
    const int bh = (int)(blockIdx.x / (unsigned)nblk), blk = (int)(blockIdx.x % (unsigned)nblk);
    const SimtSlice s = simt_slice<D>(g, bh);
    if (blk * kRows >= s.len) return;   // the whole block lies past the end of the sequence
    const int r = threadIdx.x / TPR, qd = threadIdx.x % TPR;
    const int i = blk * kRows + r;
    const bool live = i < s.len;
    const size_t row = s.base + (size_t)(live ? i : 0) * s.rs;

    float qv[DQ], dov[DQ], acc[DQ];
    float dl = 0.0f;
#pragma unroll
    for (int c = 0; c < DQ; ++c) {
        qv[c] = live ? q[row + qd + TPR * c] : 0.0f;
        dov[c] = live ? dout[row + qd + TPR * c] : 0.0f;
        dl = fmaf(dov[c], live ? o[row + qd + TPR * c] : 0.0f, dl);
        acc[c] = 0.0f;
    }
    dl = row_sum<TPR>(dl);   // delta_i = sum_d dO_id O_id
    const float li = live ? lse[s.vec0 + i] : 0.0f;
    if (live && qd == 0) delta[s.vec0 + i] = dl;
    const int kend = CAUSAL ? min(s.len, (blk + 1) * kRows) : s.len;
    const int limit = CAUSAL ? min(i + 1, s.len) : s.len;   // visible keys: j < limit

    TilePair<D, WIDE> kvt;
    if (WIDE) kvt.fetch(k, v, s, 0);
    for (int k0 = 0; k0 < kend; k0 += kTile) {
        __syncthreads();
        if (!WIDE) kvt.fetch(k, v, s, k0);
        kvt.stash(Ks, Vs);
        __syncthreads();
        if (WIDE && k0 + kTile < kend) kvt.fetch(k, v, s, k0 + kTile);
#pragma unroll 4
        for (int c = 0; c < kTile; ++c) {
            float sp = 0.0f, dp = 0.0f;
#pragma unroll
            for (int e = 0; e < DQ; ++e) {
                sp = fmaf(qv[e], Ks[c][qd + TPR * e], sp);
                dp = fmaf(dov[e], Vs[c][qd + TPR * e], dp);
            }
            sp = row_sum<TPR>(sp);
            dp = row_sum<TPR>(dp);
            const float pij = (k0 + c < limit) ? expf(sp * scale - li) : 0.0f;
            const float ds = pij * (dp - dl);
#pragma unroll
            for (int e = 0; e < DQ; ++e) acc[e] = fmaf(ds, Ks[c][qd + TPR * e], acc[e]);
        }
    }
    if (live) {
#pragma unroll
        for (int c = 0; c < DQ; ++c) dq[row + qd + TPR * c] = acc[c] * scale;
    }
}

template <int D, bool WIDE, bool CAUSAL>
__global__ void __launch_bounds__(kThreads) simt_bwd_dkdv_kernel(
    const float* __restrict__ q, const float* __restrict__ k, const float* __restrict__ v,
    const float* __restrict__ dout, const float* __restrict__ lse,
    const float* __restrict__ delta, float* __restrict__ dk, float* __restrict__ dv,
    const SliceLayout g, float scale) {
    using S = Shape<D, WIDE>;
    constexpr int kRows = S::kRows, TPR = S::kTpr, DQ = S::kCols, kTile = S::kTile;
    __shared__ __align__(16) float Qs[kTile][D];
    __shared__ __align__(16) float DOs[kTile][D];
    __shared__ float Ls[kTile], Dl[kTile];
    const int nblk = (g.n + kRows - 1) / kRows;
    const int bh = (int)(blockIdx.x / (unsigned)nblk), blk = (int)(blockIdx.x % (unsigned)nblk);
    const SimtSlice s = simt_slice<D>(g, bh);
    if (blk * kRows >= s.len) return;
    const int r = threadIdx.x / TPR, qd = threadIdx.x % TPR;
    const int j = blk * kRows + r;   // key row
    const bool live = j < s.len;
    const size_t row = s.base + (size_t)(live ? j : 0) * s.rs;

    float kv[DQ], vv[DQ], ak[DQ], av[DQ];
#pragma unroll
    for (int c = 0; c < DQ; ++c) {
        kv[c] = live ? k[row + qd + TPR * c] : 0.0f;
        vv[c] = live ? v[row + qd + TPR * c] : 0.0f;
        ak[c] = 0.0f;
        av[c] = 0.0f;
    }
    // queries before this block never see its keys under the causal mask
    const int qstart = CAUSAL ? blk * kRows : 0;
    TilePair<D, WIDE> qt;
    float lsv = 0.0f, dlv = 0.0f;   // LSE and delta of query q0 + threadIdx.x (threads < kTile)
    auto fetch_vec = [&](int q0) {
        const int qi = q0 + (int)threadIdx.x;
        const bool ok = threadIdx.x < (unsigned)kTile && qi < s.len;
        lsv = ok ? lse[s.vec0 + qi] : 0.0f;
        dlv = ok ? delta[s.vec0 + qi] : 0.0f;
    };
    if (WIDE && qstart < s.len) {
        qt.fetch(q, dout, s, qstart);
        fetch_vec(qstart);
    }
    for (int q0 = qstart; q0 < s.len; q0 += kTile) {
        __syncthreads();
        if (!WIDE) {
            qt.fetch(q, dout, s, q0);
            fetch_vec(q0);
        }
        qt.stash(Qs, DOs);
        if (threadIdx.x < kTile) {
            Ls[threadIdx.x] = lsv;
            Dl[threadIdx.x] = dlv;
        }
        __syncthreads();
        if (WIDE && q0 + kTile < s.len) {
            qt.fetch(q, dout, s, q0 + kTile);
            fetch_vec(q0 + kTile);
        }
#pragma unroll 4
        for (int c = 0; c < kTile; ++c) {
            float sp = 0.0f, dp = 0.0f;
#pragma unroll
            for (int e = 0; e < DQ; ++e) {
                sp = fmaf(kv[e], Qs[c][qd + TPR * e], sp);
                dp = fmaf(vv[e], DOs[c][qd + TPR * e], dp);
            }
            sp = row_sum<TPR>(sp);
            dp = row_sum<TPR>(dp);
            const int qi = q0 + c;
            const bool vis = qi < s.len && (!CAUSAL || qi >= j);
            const float pij = vis ? expf(sp * scale - Ls[c]) : 0.0f;
            const float ds = pij * (dp - Dl[c]);
#pragma unroll
            for (int e = 0; e < DQ; ++e) {
                av[e] = fmaf(pij, DOs[c][qd + TPR * e], av[e]);
                ak[e] = fmaf(ds, Qs[c][qd + TPR * e], ak[e]);
            }
        }
    }
    if (live) {
#pragma unroll
        for (int c = 0; c < DQ; ++c) {
            dk[row + qd + TPR * c] = ak[c] * scale;
            dv[row + qd + TPR * c] = av[c];
        }
    }
}

template <int D, bool WIDE, bool CAUSAL>
cudaError_t launch(const float* q, const float* k, const float* v, const float* o,
                   const float* dout, const float* lse, float* delta, float* dq, float* dk,
                   float* dv, int bh, const SliceLayout& g, float scale, cudaStream_t stream) {
    constexpr int kRows = Shape<D, WIDE>::kRows;
    const long long blocks = (long long)((g.n + kRows - 1) / kRows) * bh;
    if (blocks > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
    simt_bwd_dq_kernel<D, WIDE, CAUSAL><<<(unsigned)blocks, kThreads, 0, stream>>>(
        q, k, v, o, dout, lse, delta, dq, g, scale);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    simt_bwd_dkdv_kernel<D, WIDE, CAUSAL><<<(unsigned)blocks, kThreads, 0, stream>>>(
        q, k, v, dout, lse, delta, dk, dv, g, scale);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_d(bool causal, int sm_count, const float* q, const float* k, const float* v,
                     const float* o, const float* dout, const float* lse, float* delta, float* dq,
                     float* dk, float* dv, int bh, const SliceLayout& g, float scale,
                     cudaStream_t stream) {
    // 16 threads per row when the narrow CTAs would not give every SM one
    constexpr int kNarrow = Shape<D, false>::kRows;
    const bool wide = (long long)((g.n + kNarrow - 1) / kNarrow) * bh < (long long)sm_count;
    if (wide)
        return causal ? launch<D, true, true>(q, k, v, o, dout, lse, delta, dq, dk, dv, bh, g, scale, stream)
                      : launch<D, true, false>(q, k, v, o, dout, lse, delta, dq, dk, dv, bh, g, scale, stream);
    return causal ? launch<D, false, true>(q, k, v, o, dout, lse, delta, dq, dk, dv, bh, g, scale, stream)
                  : launch<D, false, false>(q, k, v, o, dout, lse, delta, dq, dk, dv, bh, g, scale, stream);
}

}  // namespace

cudaError_t simt_bwd_launch(int D, bool causal, const float* q, const float* k, const float* v,
                            const float* o, const float* dout, const float* lse, float* delta,
                            float* dq, float* dk, float* dv, int bh, const SliceLayout& g,
                            float scale, int sm_count, cudaStream_t stream) {
    if (D == 32) return launch_d<32>(causal, sm_count, q, k, v, o, dout, lse, delta, dq, dk, dv, bh, g, scale, stream);
    if (D == 64) return launch_d<64>(causal, sm_count, q, k, v, o, dout, lse, delta, dq, dk, dv, bh, g, scale, stream);
    if (D == 256) return launch_d<256>(causal, sm_count, q, k, v, o, dout, lse, delta, dq, dk, dv, bh, g, scale, stream);
    return launch_d<128>(causal, sm_count, q, k, v, o, dout, lse, delta, dq, dk, dv, bh, g, scale, stream);
}

}  // namespace fa
