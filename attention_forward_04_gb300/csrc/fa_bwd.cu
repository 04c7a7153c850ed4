// fa_bwd.cu -- attention backward on the GB300 tensor cores (tcgen05 + TMEM + TMA).
//
// Gradients of a loss through O = softmax(scale * Q K^T) V, recomputing the probabilities
// from the forward's LSE instead of storing them ("08 · FlashAttention" §三: the backward
// recomputes P from the saved statistics; "第 13 课" §4B):
//     P = exp(scale * Q K^T - LSE),  dP = dO V^T,  delta = rowsum(dO * O),
//     dS = P * (dP - delta),  dV = P^T dO,  dQ = scale * dS K,  dK = scale * dS^T Q.
//
// Three kernels, no atomics (results do not depend on scheduling):
//   * delta: one warp per row, rowsum(dO * O) in fp32;
//   * dQ: one CTA per 128-query tile; per 128-key tile the MMA warp computes S = Q K^T and
//     dP = dO V^T into TMEM, the four elementwise warps (TMEM lane = query row) form
//     P and dS = P (dP - delta) and write dS (16-bit) back over dP, and the MMA warp
//     accumulates dQ += dS K with K read as the MN-major operand;
//   * dK, dV: one CTA per 128-key tile; per 128-query tile S^T = K Q^T and dP^T = V dO^T
//     (TMEM lane = key row), the elementwise warps write P^T and dS^T (16-bit) over them,
//     and the MMA warp accumulates dV += P^T dO and dK += dS^T Q.
// Warps: 0-3 elementwise, 4 MMA issuer (converged, one elected lane issues), 5 TMA loader.
// Every wait is bounded as in the forward kernel.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fa_internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace fa {
namespace {

using namespace tc;

// Device status word: [0] flags (1 = a wait ran out), [1] role, [2] CTA, [3] wait id.
__device__ unsigned int g_status[4];

constexpr int kT = 128;          // tile rows (TMEM lanes) and tile columns
constexpr int kThreads = 192;
constexpr int kMmaWarp = 4;
constexpr int kLoadWarp = 5;
constexpr int kSlots = 4;        // ring of streamed tiles (two per step)
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BGeo {
    static constexpr int kPanels = D / kPanelCols;
    static constexpr int kTile = kPanels * kPanelBytes;        // one 128 x D tile
    static constexpr int kRingOff = 2 * kTile;                 // after the two fixed tiles
    static constexpr int kStageOff = kRingOff + kSlots * kTile;
    static constexpr int kVecOff = kStageOff + 4 * 4096;       // per-column LSE/delta (dK/dV)
    static constexpr int kBarOff = kVecOff + 2 * 2 * kT * 4;
    // barriers: fixed_full, ring_full[S], ring_empty[S], s_full, ew_full, done, drain
    static constexpr int kNumBars = 1 + 2 * kSlots + 4;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
    // TMEM columns: S (or S^T), dP (or dP^T), accumulator 0 (dQ or dV), accumulator 1 (dK)
    static constexpr uint32_t kColS = 0, kColDP = 128, kColAcc0 = 256, kColAcc1 = 256 + D;
};

constexpr int b_fixed_full() { return 0; }
constexpr int b_ring_full(uint32_t i) { return 1 + (int)(i % kSlots); }
constexpr int b_ring_empty(uint32_t i) { return 1 + kSlots + (int)(i % kSlots); }
constexpr int b_s_full() { return 1 + 2 * kSlots; }
constexpr int b_ew_full() { return 2 + 2 * kSlots; }
constexpr int b_done() { return 3 + 2 * kSlots; }
constexpr int b_drain() { return 4 + 2 * kSlots; }
__device__ __forceinline__ uint32_t ring_par(uint32_t i) { return (i / kSlots) & 1u; }

// ----------------------------------------------------------------- MMA helpers
// D_tmem (+)= A[128 x D] * B[128 x D]^T with both operands K-major in shared memory.
template <int D>
__device__ __forceinline__ void mma_nt(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc) {
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const uint64_t off = ((uint64_t)(kk / 4) * kPanelBytes + (uint64_t)(kk % 4) * 32u) >> 4;
        ptx::mma_ss_elect(d_tmem, a_desc + off, b_desc + off, idesc, kk > 0 ? 1u : 0u);
    }
}

// acc_tmem (+)= A_tmem[128 x 128] * B, B a 128 x D shared tile read as the MN-major operand.
__device__ __forceinline__ void mma_tn(uint32_t acc_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, bool accumulate) {
#pragma unroll
    for (int kk = 0; kk < kT / 16; ++kk)
        ptx::mma_ts_elect(acc_tmem, a_tmem + (uint32_t)kk * 8u,
                          b_desc + (uint64_t)((kk * 2048) >> 4), idesc,
                          (accumulate || kk > 0) ? 1u : 0u);
}

// ----------------------------------------------------------------- epilogue
// This warp's 32 TMEM lanes x D fp32 columns at t_acc, times mul, rounded to 16 bits, to
// global rows base + r * D (r < 32, only rows with row0 + r < nrows), through a 4 KB
// staging slot so every store instruction writes whole 128-byte lines.
template <int D, bool F16>
__device__ __forceinline__ void store_rows(uint32_t t_acc, float mul, uint32_t stage,
                                           uint16_t* base, int row0, int nrows, int lane) {
#pragma unroll 1
    for (int pc = 0; pc < D / 64; ++pc) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint32_t o[32];
            ptx::tmem_ld32_wait(t_acc + (uint32_t)(pc * 64 + h * 32), o);
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
                *reinterpret_cast<uint4*>(base + (size_t)(row0 + r) * D + pc * 64 + ch * 8) = v;
        }
        __syncwarp();
    }
}

// Named barrier 1 over the 128 elementwise threads (warps 0-3) that also ANDs a predicate.
__device__ __forceinline__ bool ew_barrier_and(bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok)
        : "memory");
    return r != 0;
}

// ----------------------------------------------------------------- common prologue
struct Setup {
    Ctl c;
    uint32_t sbase, tmem;
};

template <int D>
__device__ __forceinline__ Setup setup_cta(uint8_t* smem_raw, const BwdParams& p, int ew_count) {
    using G = BGeo<D>;
    Setup su;
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    su.sbase = ptx::smem_addr(smem);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::kMiscOff);
    su.c.bars = su.sbase + (uint32_t)G::kBarOff;
    su.c.abort = reinterpret_cast<volatile int*>(smem + G::kMiscOff + 4);
    su.c.limit = p.wait_limit;
    su.c.status = g_status;
    const int warp = threadIdx.x / 32;
    if (threadIdx.x == 0) {
        ptx::mbar_init(bar_addr(su.c, b_fixed_full()), 1);
        for (int s = 0; s < kSlots; ++s) {
            ptx::mbar_init(bar_addr(su.c, b_ring_full(s)), 1);
            ptx::mbar_init(bar_addr(su.c, b_ring_empty(s)), 1);
        }
        ptx::mbar_init(bar_addr(su.c, b_s_full()), 1);
        ptx::mbar_init(bar_addr(su.c, b_ew_full()), ew_count);
        ptx::mbar_init(bar_addr(su.c, b_done()), 1);
        ptx::mbar_init(bar_addr(su.c, b_drain()), 1);
        *su.c.abort = 0;
        ptx::fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    su.tmem = *tmem_slot;
    return su;
}

__device__ __forceinline__ void teardown_cta(const Setup& su) {
    ptx::tc_fence_before();
    __syncthreads();
    if (threadIdx.x / 32 == kMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(su.tmem, kTmemCols);
    }
}

// Loader: two fixed tiles (rows fixed_row of maps f0, f1), then per step two streamed tiles
// (rows 128 * (first + s) of maps r0, r1) through the ring.  Waits for its own copies before
// returning, so no copy is in flight when the CTA leaves.
template <int D>
__device__ void load_tiles(const Ctl& c, uint32_t sbase, const CUtensorMap* f0,
                           const CUtensorMap* f1, int fixed_row, const CUtensorMap* r0,
                           const CUtensorMap* r1, int first, int steps, int bh) {
    using G = BGeo<D>;
    uint32_t pos = 0;
    const uint32_t fb = bar_addr(c, b_fixed_full());
    ptx::mbar_arrive_expect_tx(fb, 2u * G::kTile);
#pragma unroll
    for (int pc = 0; pc < G::kPanels; ++pc) {
        ptx::tma_load_3d(sbase + (uint32_t)pc * kPanelBytes, f0, fb, pc * kPanelCols, fixed_row, bh);
        ptx::tma_load_3d(sbase + (uint32_t)G::kTile + (uint32_t)pc * kPanelBytes, f1, fb,
                         pc * kPanelCols, fixed_row, bh);
    }
    for (int s = 0; s < steps; ++s) {
        for (int w = 0; w < 2; ++w) {
            if (!wait(c, b_ring_empty(pos), ring_par(pos) ^ 1u, kRoleLoad)) goto out;
            const uint32_t bar = bar_addr(c, b_ring_full(pos));
            const uint32_t dst = sbase + (uint32_t)G::kRingOff + (pos % kSlots) * (uint32_t)G::kTile;
            ptx::mbar_arrive_expect_tx(bar, (uint32_t)G::kTile);
#pragma unroll
            for (int pc = 0; pc < G::kPanels; ++pc)
                ptx::tma_load_3d(dst + (uint32_t)pc * kPanelBytes, w == 0 ? r0 : r1, bar,
                                 pc * kPanelCols, (first + s) * kT, bh);
            ++pos;
        }
    }
out:
    wait_drain(fb, 0, c.limit);
    for (uint32_t i = (pos > (uint32_t)kSlots ? pos - kSlots : 0u); i < pos; ++i)
        wait_drain(bar_addr(c, b_ring_full(i)), ring_par(i), c.limit);
}

// ----------------------------------------------------------------- dQ kernel
template <int D, bool CAUSAL, bool F16>
__global__ void __launch_bounds__(kThreads, 1) bwd_dq_kernel(const __grid_constant__ BwdParams p) {
    using G = BGeo<D>;
    extern __shared__ uint8_t smem_raw[];
    const Setup su = setup_cta<D>(smem_raw, p, 128);
    const Ctl& c = su.c;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bh = blockIdx.x / p.ntiles, qt = blockIdx.x % p.ntiles;
    const int nkv = CAUSAL ? min(qt + 1, p.ntiles) : p.ntiles;
    const uint32_t tm = su.tmem;

    if (warp == kLoadWarp) {
        if (lane == 0)
            load_tiles<D>(c, su.sbase, &p.tmap_q, &p.tmap_do, qt * kT, &p.tmap_k, &p.tmap_v, 0,
                          nkv, bh);
        __syncwarp();
    } else if (warp == kMmaWarp) {
        constexpr uint32_t id_nt = make_idesc(kT, kT, false, F16);
        constexpr uint32_t id_tn = make_idesc(kT, D, true, F16);
        const uint64_t dQ = sw128_desc(su.sbase, 16, 1024);
        const uint64_t dDO = sw128_desc(su.sbase + (uint32_t)G::kTile, 16, 1024);
        const uint64_t dRing = sw128_desc(su.sbase + (uint32_t)G::kRingOff, 16, 1024);
        const uint64_t dRingMN = sw128_desc(su.sbase + (uint32_t)G::kRingOff, kPanelBytes, 1024);
        auto slot_off = [](uint32_t i) { return (uint64_t)((i % kSlots) * (uint32_t)G::kTile) >> 4; };
        if (!wait_warp(c, b_fixed_full(), 0, kRoleMma)) goto mma_out;
        for (int j = 0; j < nkv; ++j) {
            const uint32_t kpos = 2u * j, vpos = 2u * j + 1u;
            if (!wait_warp(c, b_ring_full(kpos), ring_par(kpos), kRoleMma)) goto mma_out;
            ptx::tc_fence_after();
            mma_nt<D>(tm + G::kColS, dQ, dRing + slot_off(kpos), id_nt);          // S = Q K^T
            if (!wait_warp(c, b_ring_full(vpos), ring_par(vpos), kRoleMma)) goto mma_out;
            ptx::tc_fence_after();
            mma_nt<D>(tm + G::kColDP, dDO, dRing + slot_off(vpos), id_nt);        // dP = dO V^T
            ptx::mma_commit_elect(bar_addr(c, b_s_full()));
            ptx::mma_commit_elect(bar_addr(c, b_ring_empty(vpos)));
            if (!wait_warp(c, b_ew_full(), (uint32_t)j & 1u, kRoleMma)) goto mma_out;
            ptx::tc_fence_after();
            mma_tn(tm + G::kColAcc0, tm + G::kColDP, dRingMN + slot_off(kpos), id_tn, j > 0);  // dQ += dS K
            ptx::mma_commit_elect(bar_addr(c, b_ring_empty(kpos)));
        }
        ptx::mma_commit_elect(bar_addr(c, b_done()));
    mma_out:
        ptx::mma_commit_elect(bar_addr(c, b_drain()));
        wait_drain(bar_addr(c, b_drain()), 0, c.limit);
        __syncwarp();
    } else {
        // elementwise: thread = query row
        const int r = warp * 32 + lane;
        const int i = qt * kT + r;
        const bool live = i < p.n;
        const size_t row = (size_t)bh * p.n + (live ? i : 0);
        const float lse2 = live ? p.lse[row] * kLog2e : 0.0f;
        const float dlt = live ? p.delta[row] : 0.0f;
        const int limit = CAUSAL ? min(i + 1, p.n) : p.n;    // visible keys: key < limit
        const uint32_t tl = (uint32_t)(warp * 32) << 16;
        for (int j = 0; j < nkv; ++j) {
            if (!wait_warp(c, b_s_full(), (uint32_t)j & 1u, kRoleSoftmax)) goto ew_out;
            ptx::tc_fence_after();
            const bool mask = __any_sync(0xFFFFFFFFu, j * kT + kT > limit);
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t sv[32], dp[32];
                ptx::tmem_ld32x2_wait(tm + tl + G::kColS + 32u * ch, tm + tl + G::kColDP + 32u * ch, sv, dp);
                uint32_t pk[16];
#pragma unroll
                for (int cc = 0; cc < 32; cc += 2) {
                    const int key = j * kT + ch * 32 + cc;
                    float p0 = ptx::ex2(fmaf(u2f(sv[cc]), p.scale_log2, -lse2));
                    float p1 = ptx::ex2(fmaf(u2f(sv[cc + 1]), p.scale_log2, -lse2));
                    if (mask) {
                        if (key >= limit) p0 = 0.0f;
                        if (key + 1 >= limit) p1 = 0.0f;
                    }
                    pk[cc >> 1] = pack2<F16>(p0 * (u2f(dp[cc]) - dlt), p1 * (u2f(dp[cc + 1]) - dlt));
                }
                __syncwarp();
                // dS over dP columns 16ch.. (dP columns already loaded)
                ptx::tmem_st16(tm + tl + G::kColDP + 16u * ch, pk);
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar_addr(c, b_ew_full()));
        }
        if (!wait_warp(c, b_done(), 0, kRoleSoftmax)) goto ew_out;
        ptx::tc_fence_after();
        store_rows<D, F16>(tm + tl + G::kColAcc0, p.scale,
                           su.sbase + (uint32_t)G::kStageOff + (uint32_t)warp * 4096u,
                           reinterpret_cast<uint16_t*>(p.dq) + (size_t)bh * p.n * D, qt * kT + warp * 32,
                           p.n, lane);
    ew_out:;
    }
    teardown_cta(su);
}

// ----------------------------------------------------------------- dK, dV kernel
template <int D, bool CAUSAL, bool F16>
__global__ void __launch_bounds__(kThreads, 1) bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
    using G = BGeo<D>;
    extern __shared__ uint8_t smem_raw[];
    const Setup su = setup_cta<D>(smem_raw, p, 128);
    const Ctl& c = su.c;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int bh = blockIdx.x / p.ntiles, kt = blockIdx.x % p.ntiles;
    const int i0 = CAUSAL ? kt : 0;                 // first query tile that sees this key tile
    const int nq = p.ntiles - i0;
    const uint32_t tm = su.tmem;

    if (warp == kLoadWarp) {
        if (lane == 0)
            load_tiles<D>(c, su.sbase, &p.tmap_k, &p.tmap_v, kt * kT, &p.tmap_q, &p.tmap_do, i0, nq,
                          bh);
        __syncwarp();
    } else if (warp == kMmaWarp) {
        constexpr uint32_t id_nt = make_idesc(kT, kT, false, F16);
        constexpr uint32_t id_tn = make_idesc(kT, D, true, F16);
        const uint64_t dK = sw128_desc(su.sbase, 16, 1024);
        const uint64_t dV = sw128_desc(su.sbase + (uint32_t)G::kTile, 16, 1024);
        const uint64_t dRing = sw128_desc(su.sbase + (uint32_t)G::kRingOff, 16, 1024);
        const uint64_t dRingMN = sw128_desc(su.sbase + (uint32_t)G::kRingOff, kPanelBytes, 1024);
        auto slot_off = [](uint32_t i) { return (uint64_t)((i % kSlots) * (uint32_t)G::kTile) >> 4; };
        if (!wait_warp(c, b_fixed_full(), 0, kRoleMma)) goto mma_out;
        for (int s = 0; s < nq; ++s) {
            const uint32_t qpos = 2u * s, dopos = 2u * s + 1u;
            if (!wait_warp(c, b_ring_full(qpos), ring_par(qpos), kRoleMma)) goto mma_out;
            ptx::tc_fence_after();
            mma_nt<D>(tm + G::kColS, dK, dRing + slot_off(qpos), id_nt);         // S^T = K Q^T
            if (!wait_warp(c, b_ring_full(dopos), ring_par(dopos), kRoleMma)) goto mma_out;
            ptx::tc_fence_after();
            mma_nt<D>(tm + G::kColDP, dV, dRing + slot_off(dopos), id_nt);       // dP^T = V dO^T
            ptx::mma_commit_elect(bar_addr(c, b_s_full()));
            if (!wait_warp(c, b_ew_full(), (uint32_t)s & 1u, kRoleMma)) goto mma_out;
            ptx::tc_fence_after();
            mma_tn(tm + G::kColAcc0, tm + G::kColS, dRingMN + slot_off(dopos), id_tn, s > 0);   // dV += P^T dO
            ptx::mma_commit_elect(bar_addr(c, b_ring_empty(dopos)));
            mma_tn(tm + G::kColAcc1, tm + G::kColDP, dRingMN + slot_off(qpos), id_tn, s > 0);   // dK += dS^T Q
            ptx::mma_commit_elect(bar_addr(c, b_ring_empty(qpos)));
        }
        ptx::mma_commit_elect(bar_addr(c, b_done()));
    mma_out:
        ptx::mma_commit_elect(bar_addr(c, b_drain()));
        wait_drain(bar_addr(c, b_drain()), 0, c.limit);
        __syncwarp();
    } else {
        // elementwise: thread = key row; columns = the 128 queries of the current tile
        const int r = warp * 32 + lane;
        const int key = kt * kT + r;
        const uint32_t tl = (uint32_t)(warp * 32) << 16;
        float* vec = reinterpret_cast<float*>(smem_raw + (su.sbase - ptx::smem_addr(smem_raw)) + G::kVecOff);
        // per-column LSE (log2 units) and delta of query tile i0 + s, staged in shared memory;
        // the next tile's pair is fetched one step ahead into registers
        auto fetch = [&](int s, float& l2, float& d) {
            const int q = (i0 + s) * kT + r;
            const bool ok = s < nq && q < p.n;
            l2 = ok ? p.lse[(size_t)bh * p.n + q] * kLog2e : INFINITY;   // p = 0 past N
            d = ok ? p.delta[(size_t)bh * p.n + q] : 0.0f;
        };
        float l2_next, d_next;
        fetch(0, l2_next, d_next);
        for (int s = 0; s < nq; ++s) {
            float* vl = vec + (s & 1) * 2 * kT;   // [0, 128): LSE * log2 e, [128, 256): delta
            vl[r] = l2_next;
            vl[kT + r] = d_next;
            // One barrier over the four elementwise warps publishes the staged vectors and
            // makes the stop decision common to all four, so no warp is left at a barrier
            // that a warp which gave up will never reach.
            const bool ok = wait_warp(c, b_s_full(), (uint32_t)s & 1u, kRoleSoftmax);
            if (!ew_barrier_and(ok)) goto ew_out;
            ptx::tc_fence_after();
            fetch(s + 1, l2_next, d_next);
            const int qbase = (i0 + s) * kT;
            const bool diag = CAUSAL && (i0 + s == kt);   // queries before this key are masked
#pragma unroll 1
            for (int ch = 0; ch < 4; ++ch) {
                uint32_t sv[32], dp[32];
                ptx::tmem_ld32x2_wait(tm + tl + G::kColS + 32u * ch, tm + tl + G::kColDP + 32u * ch, sv, dp);
                uint32_t pp[16], pd[16];
#pragma unroll
                for (int cc = 0; cc < 32; cc += 2) {
                    const int col = ch * 32 + cc;
                    float p0 = ptx::ex2(fmaf(u2f(sv[cc]), p.scale_log2, -vl[col]));
                    float p1 = ptx::ex2(fmaf(u2f(sv[cc + 1]), p.scale_log2, -vl[col + 1]));
                    if (diag) {
                        if (qbase + col < key) p0 = 0.0f;
                        if (qbase + col + 1 < key) p1 = 0.0f;
                    }
                    pp[cc >> 1] = pack2<F16>(p0, p1);
                    pd[cc >> 1] = pack2<F16>(p0 * (u2f(dp[cc]) - vl[kT + col]),
                                             p1 * (u2f(dp[cc + 1]) - vl[kT + col + 1]));
                }
                __syncwarp();
                ptx::tmem_st16(tm + tl + G::kColS + 16u * ch, pp);    // P^T over S^T columns
                ptx::tmem_st16(tm + tl + G::kColDP + 16u * ch, pd);   // dS^T over dP^T columns
            }
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar_addr(c, b_ew_full()));
        }
        if (!wait_warp(c, b_done(), 0, kRoleSoftmax)) goto ew_out;
        ptx::tc_fence_after();
        {
            const uint32_t stage = su.sbase + (uint32_t)G::kStageOff + (uint32_t)warp * 4096u;
            const int row0 = kt * kT + warp * 32;
            store_rows<D, F16>(tm + tl + G::kColAcc0, 1.0f, stage,
                               reinterpret_cast<uint16_t*>(p.dv) + (size_t)bh * p.n * D, row0, p.n, lane);
            store_rows<D, F16>(tm + tl + G::kColAcc1, p.scale, stage,
                               reinterpret_cast<uint16_t*>(p.dk) + (size_t)bh * p.n * D, row0, p.n, lane);
        }
    ew_out:;
    }
    teardown_cta(su);
}

// ----------------------------------------------------------------- delta kernel
template <int D, bool F16>
__global__ void __launch_bounds__(256) bwd_delta_kernel(const uint16_t* __restrict__ o,
                                                       const uint16_t* __restrict__ dout,
                                                       float* __restrict__ delta, long long rows) {
    constexpr int E = D / 32;   // elements per lane
    const int lane = threadIdx.x % 32;
    const long long warps = (long long)gridDim.x * (blockDim.x / 32);
    for (long long r = (long long)blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; r < rows; r += warps) {
        const uint16_t* a = o + r * D + lane * E;
        const uint16_t* b = dout + r * D + lane * E;
        float acc = 0.0f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
            float x, y;
            if constexpr (F16) {
                x = __half2float(__ushort_as_half(a[e]));
                y = __half2float(__ushort_as_half(b[e]));
            } else {
                x = __bfloat162float(__ushort_as_bfloat16(a[e]));
                y = __bfloat162float(__ushort_as_bfloat16(b[e]));
            }
            acc = fmaf(x, y, acc);
        }
#pragma unroll
        for (int m = 16; m > 0; m >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, m);
        if (lane == 0) delta[r] = acc;
    }
}

template <int D, bool CAUSAL, bool F16>
cudaError_t prepare3() {
    cudaError_t e = cudaFuncSetAttribute(bwd_dq_kernel<D, CAUSAL, F16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, BGeo<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(bwd_dkdv_kernel<D, CAUSAL, F16>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, BGeo<D>::kSmemBytes);
}

template <int D, bool CAUSAL, bool F16>
cudaError_t launch3(const BwdParams& p, int bh, cudaStream_t stream) {
    const long long ctas = (long long)bh * p.ntiles;
    if (ctas > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
    bwd_dq_kernel<D, CAUSAL, F16><<<(unsigned)ctas, kThreads, BGeo<D>::kSmemBytes, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_dkdv_kernel<D, CAUSAL, F16><<<(unsigned)ctas, kThreads, BGeo<D>::kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

template <int D>
cudaError_t dispatch(bool causal, bool f16, bool prepare, const BwdParams* p, int bh, cudaStream_t s) {
    if (prepare) {
        if (causal) return f16 ? prepare3<D, true, true>() : prepare3<D, true, false>();
        return f16 ? prepare3<D, false, true>() : prepare3<D, false, false>();
    }
    if (causal) return f16 ? launch3<D, true, true>(*p, bh, s) : launch3<D, true, false>(*p, bh, s);
    return f16 ? launch3<D, false, true>(*p, bh, s) : launch3<D, false, false>(*p, bh, s);
}

}  // namespace

cudaError_t bwd_delta_launch(int D, bool f16, const void* o, const void* dout, float* delta,
                             long long rows, cudaStream_t stream) {
    const long long blocks = (rows + 7) / 8;
    const unsigned grid = (unsigned)(blocks < 65536 ? blocks : 65536);
    const uint16_t* a = static_cast<const uint16_t*>(o);
    const uint16_t* b = static_cast<const uint16_t*>(dout);
    if (D == 64) {
        if (f16) bwd_delta_kernel<64, true><<<grid, 256, 0, stream>>>(a, b, delta, rows);
        else bwd_delta_kernel<64, false><<<grid, 256, 0, stream>>>(a, b, delta, rows);
    } else {
        if (f16) bwd_delta_kernel<128, true><<<grid, 256, 0, stream>>>(a, b, delta, rows);
        else bwd_delta_kernel<128, false><<<grid, 256, 0, stream>>>(a, b, delta, rows);
    }
    return cudaGetLastError();
}

cudaError_t bwd_prepare(int D, bool causal, bool f16) {
    return D == 64 ? dispatch<64>(causal, f16, true, nullptr, 0, nullptr)
                   : dispatch<128>(causal, f16, true, nullptr, 0, nullptr);
}

cudaError_t bwd_launch(int D, bool causal, bool f16, const BwdParams& p, int bh, cudaStream_t stream) {
    return D == 64 ? dispatch<64>(causal, f16, false, &p, bh, stream)
                   : dispatch<128>(causal, f16, false, &p, bh, stream);
}

cudaError_t bwd_status_read_reset(uint32_t out[4]) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_status, sizeof(unsigned int) * 4);
    if (e != cudaSuccess) return e;
    const unsigned int zero[4] = {0, 0, 0, 0};
    return cudaMemcpyToSymbol(g_status, zero, sizeof(zero));
}

}  // namespace fa
