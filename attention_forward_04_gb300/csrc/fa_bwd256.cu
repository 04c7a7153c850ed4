// fa_bwd256.cu -- attention backward at head dimension 256 on the GB300 tensor cores
// (tcgen05 + TMEM + TMA), for bf16 and fp16 storage.
//
// The same gradients as the narrower head dimensions ("08 · FlashAttention" §三, the
// backward recomputes P from the saved statistics; "第 13 课" §4B):
//     P = exp(scale * Q K^T - LSE),  dP = dO V^T,  delta = rowsum(dO * O),
//     dS = P * (dP - delta),  dV = P^T dO,  dQ = scale * dS K,  dK = scale * dS^T Q.
//
// At D = 256 one 128 x 256 fp32 accumulator fills half of the 512 TMEM columns and one
// 128 x 256 16-bit tile takes 64 KB of shared memory, so a CTA holding both dK and dV (as
// the narrower kernels do) does not fit.  Three kernels, one accumulator each, no atomics:
//   * dQ (ROLE 0): one CTA per 128-query tile.  Q in TMEM (16-bit pairs, 128 columns), dO
//     fixed in shared memory; keys stream in 64-row sub-tiles: S = Q K_j^T and dP = dO V_j^T
//     (64 columns each), dS = P (dP - delta) written 16-bit over dP, dQ += dS K_j.  It also
//     forms delta for its rows and writes it for the dK kernel;
//   * dK (ROLE 1): one CTA per 128-key tile.  K in TMEM, V fixed in shared memory; queries
//     stream in 64-row sub-tiles: S^T = K Q_s^T, dP^T = V dO_s^T, dS^T = P^T (dP^T - delta)
//     over dP^T, dK += dS^T Q_s;
//   * dV (ROLE 2): one CTA per 128-key tile.  K in TMEM; S^T = K Q_s^T into one of two
//     64-column buffers (the next one is computed while the current one is turned into
//     P^T), P^T written over it, dV += P^T dO_s.
// The dQ and dK kernels are one template: the row side (Q or K) sits in TMEM, the fixed
// tile (dO or V) is the A operand of the second product, and the streamed sub-tile X (K_j
// or Q_s) serves twice, as the K-major B operand of S and as the MN-major B operand of the
// accumulation, so its ring slot is released only after the accumulation.
// Products: M = 128; S, dP: N = 64, K = 256 (16 steps); accumulation: N = 256, K = 64 (4
// steps).  dS and P^T are stored by the elementwise warp that read the fp32 values, in the
// first half of its own 32 columns, so no warp overwrites columns another is reading.
// Warps: 0-7 elementwise (warp w: TMEM lanes 32 (w % 4).., the 32 columns 32 (w / 4).. of
// each 64-column product), 8 MMA issuer, 9 TMA loader.  Every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "bwd_common.cuh"
#include "fa_internal.h"
#include "ptx.cuh"
#include "tc_common.cuh"

namespace fa {
namespace {

using namespace tc;
using namespace bwdc;

// Device status word: [0] flags (1 = a wait ran out), [1] role, [2] CTA, [3] wait id.
__device__ unsigned int g_status256[4];

constexpr int kD = 256;
constexpr int kT = 128;                  // CTA tile rows (TMEM lanes)
constexpr int kSub = 64;                 // streamed sub-tile rows
constexpr int kThreads = 320;
constexpr int kEwThreads = 256;          // warps 0-7
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kSubPanel = kSub * 128;    // 8 KB: 64 rows x 64 columns (128-byte swizzle)
constexpr int kSubBytes = 4 * kSubPanel; // 32 KB: a 64 x 256 sub-tile, four panels
constexpr int kFixPanel = kT * 128;      // 16 KB
constexpr int kFixBytes = 4 * kFixPanel; // 64 KB: a 128 x 256 tile

constexpr int kRoleDQ = 0, kRoleDK = 1, kRoleDV = 2;

// TMEM columns.  Row tile (Q or K) as 16-bit pairs [0, 128); dQ, dK: S [128, 192), dP
// [192, 256); dV: S^T buffers [128, 192) and [192, 256); accumulator [256, 512).
constexpr uint32_t kColRow = 0, kColS = 128, kColDP = 192, kColAcc = 256;

template <int ROLE>
struct G256 {
    static constexpr bool kFixed = ROLE != kRoleDV;   // dO (dQ) or V (dK) in shared memory
    static constexpr int kSlots = ROLE == kRoleDV ? 6 : 5;
    static constexpr int kRingOff = kFixed ? kFixBytes : 0;
    // epilogue staging (4 KB per elementwise warp) reuses the ring: it starts only after
    // the last product, hence the last read of the ring, has completed
    static constexpr int kStageOff = kRingOff;
    // dQ: 2 x 128 partial row sums of delta; dK: per query column of the sub-tile LSE and
    // delta, double-buffered (2 x 128 floats); dV: per elementwise warp, the LSE of its 32
    // query columns, double-buffered (8 x 2 x 32 floats)
    static constexpr int kVecOff = kRingOff + kSlots * kSubBytes;
    static constexpr int kBarOff = kVecOff + (ROLE == kRoleDV ? 8 * 2 * 32 * 4 : 2 * 128 * 4);
    static constexpr int kNumBars = 1 + 2 * kSlots + 9;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory");
    static_assert(8 * 4096 <= kSlots * kSubBytes, "staging fits the ring");

    static constexpr int fixed_full() { return 0; }
    static constexpr int ring_full(uint32_t slot) { return 1 + (int)slot; }
    static constexpr int ring_empty(uint32_t slot) { return 1 + kSlots + (int)slot; }
    static constexpr int s_ready(int b) { return 1 + 2 * kSlots + b; }    // S (buffer b) in TMEM
    static constexpr int x_ready(int b) { return 3 + 2 * kSlots + b; }    // S read (dV: P^T stored)
    static constexpr int dp_ready() { return 5 + 2 * kSlots; }
    static constexpr int ds_ready() { return 6 + 2 * kSlots; }
    static constexpr int row_ready() { return 7 + 2 * kSlots; }           // row tile in TMEM
    static constexpr int done() { return 8 + 2 * kSlots; }
    static constexpr int drain() { return 9 + 2 * kSlots; }
    // streamed sub-tile `pos` (0, 1: the row tile's halves) in slot pos % kSlots
    static __device__ __forceinline__ uint32_t slot(uint32_t pos) { return pos % (uint32_t)kSlots; }
    static __device__ __forceinline__ uint32_t par(uint32_t pos) { return (pos / (uint32_t)kSlots) & 1u; }
};

// ----------------------------------------------------------------- descriptors, products
// K-major operand with 128-byte rows in panels of `panel` bytes: K step kk (16 values) is
// 32 bytes of a row of panel kk / 4.
__device__ __forceinline__ uint64_t kmaj(uint32_t base, int kk, uint32_t panel) {
    return sw128_desc(base + (uint32_t)(kk >> 2) * panel + (uint32_t)(kk & 3) * 32u, 16u, 1024u);
}

// D_tmem[128 x 64] = A[128 x 256] * B^T, B a 64 x 256 sub-tile (K-major) at b_smem; A from
// TMEM (16-bit pairs at a, A_TMEM) or the fixed 128 x 256 tile in shared memory (at a).
template <bool A_TMEM>
__device__ __forceinline__ void mma_rows_x_sub(uint32_t d_tmem, uint32_t a, uint32_t b_smem,
                                               uint32_t idesc) {
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
        const uint64_t b = kmaj(b_smem, kk, kSubPanel);
        if constexpr (A_TMEM)
            ptx::mma_ts_elect(d_tmem, a + (uint32_t)kk * 8u, b, idesc, kk > 0 ? 1u : 0u);
        else
            ptx::mma_ss_elect(d_tmem, kmaj(a, kk, kFixPanel), b, idesc, kk > 0 ? 1u : 0u);
    }
}

// acc[128 x 256] (+)= A[128 x 64] * B, A 16-bit pairs in TMEM (keys or queries 32 w..32 w + 31
// of the 64 in the first 16 columns of the 32-column block w at a_tmem + 32 w), B the 64 x 256
// sub-tile read as the MN-major operand (16 rows per K step, panels 8 KB apart).
__device__ __forceinline__ void mma_acc(uint32_t acc_tmem, uint32_t a_tmem, uint32_t b_smem,
                                        uint32_t idesc, bool accumulate) {
#pragma unroll
    for (int kk = 0; kk < kSub / 16; ++kk)
        ptx::mma_ts_elect(acc_tmem, a_tmem + (uint32_t)(kk >> 1) * 32u + (uint32_t)(kk & 1) * 8u,
                          sw128_desc(b_smem + (uint32_t)kk * 2048u, (uint32_t)kSubPanel, 1024u),
                          idesc, (accumulate || kk > 0) ? 1u : 0u);
}

// ----------------------------------------------------------------- loads
// Rows row.. row + 63 of the slice (all 256 columns) into shared memory at dst as four
// 8 KB panels (a 64-row box per panel), or, with `step` = 8 KB and dst panels 16 KB apart,
// one half of a 128-row tile.
template <int MODE>
__device__ __forceinline__ void load_rows64(uint32_t dst, uint32_t panel, const CUtensorMap* map,
                                            uint32_t bar, int row, int bh, const Slice& sl) {
#pragma unroll
    for (int pc = 0; pc < 4; ++pc) {
        if (MODE == 0)
            ptx::tma_load_3d(dst + (uint32_t)pc * panel, map, bar, pc * 64, row, bh);
        else
            ptx::tma_load_3d(dst + (uint32_t)pc * panel, map, bar, pc * 64, sl.h, sl.tok0 + row);
    }
}

// The loader: the fixed tile (dQ: dO, dK: V; rows fix_row..), the row tile's two halves
// (pos 0, 1; rows row0..), then the streamed sub-tiles in the order the MMA warp takes
// them: dQ, dK: X_0, Y_0, X_1, Y_1, ...; dV: X_0, X_1, Y_0, X_2, Y_1, X_3, ... (sub-tile
// t covers rows (s0 + t) * 64..).  Waits for its own copies before returning.  Position
// `skipped` (failure-detection test hook) is never loaded, so the waits for it run out.
template <int ROLE, int MODE>
__device__ void load_role(const Ctl& c, uint32_t sbase, const CUtensorMap* fixed,
                          const CUtensorMap* rowmap, int row0, const CUtensorMap* xmap,
                          const CUtensorMap* ymap, int s0, int n, int bh, const Slice& sl,
                          uint32_t skipped) {
    using G = G256<ROLE>;
    const uint32_t ring = sbase + (uint32_t)G::kRingOff;
    if constexpr (G::kFixed) {
        const uint32_t fb = bar_addr(c, G::fixed_full());
        ptx::mbar_arrive_expect_tx(fb, (uint32_t)kFixBytes);
        load_rows64<MODE>(sbase, kFixPanel, fixed, fb, row0, bh, sl);
        load_rows64<MODE>(sbase + (uint32_t)kSubPanel, kFixPanel, fixed, fb, row0 + kSub, bh, sl);
    }
    const uint32_t count = 2u + 2u * (uint32_t)n;
    uint32_t pos = 0;
    for (; pos < count; ++pos) {
        const uint32_t slot = G::slot(pos);
        if (!wait(c, G::ring_empty(slot), G::par(pos) ^ 1u, kRoleLoad)) break;
        if (pos == skipped) continue;
        const uint32_t bar = bar_addr(c, G::ring_full(slot));
        const CUtensorMap* map;
        int row;
        if (pos < 2) {
            map = rowmap;
            row = row0 + (int)pos * kSub;
        } else {
            const int k = (int)pos - 2;
            int t;
            bool is_x;
            if (ROLE != kRoleDV) {
                t = k >> 1;
                is_x = (k & 1) == 0;
            } else if (k < 2 || n < 2) {   // X_0, X_1 (or X_0, Y_0 when n = 1)
                is_x = n >= 2 || k == 0;
                t = (n >= 2) ? k : 0;
            } else {
                // after X_0, X_1: Y_s then X_{s+2} while s + 2 < n, then the last Y's
                const int m = k - 2;
                const int pairs = n - 2;           // (Y_s, X_{s+2}) for s < n - 2
                if (m < 2 * pairs) {
                    is_x = (m & 1) == 1;
                    t = is_x ? (m >> 1) + 2 : (m >> 1);
                } else {
                    is_x = false;
                    t = pairs + (m - 2 * pairs);
                }
            }
            map = is_x ? xmap : ymap;
            row = (s0 + t) * kSub;
        }
        ptx::mbar_arrive_expect_tx(bar, (uint32_t)kSubBytes);
        load_rows64<MODE>(ring + slot * (uint32_t)kSubBytes, kSubPanel, map, bar, row, bh, sl);
    }
    if constexpr (G::kFixed) wait_drain(bar_addr(c, G::fixed_full()), 0, c.limit);
    for (uint32_t i = (pos > (uint32_t)G::kSlots ? pos - G::kSlots : 0u); i < pos; ++i)
        if (i != skipped) wait_drain(bar_addr(c, G::ring_full(G::slot(i))), G::par(i), c.limit);
}

// ----------------------------------------------------------------- prologue
struct Setup {
    Ctl c;
    uint32_t sbase, tmem;
    uint8_t* smem;
};

template <int ROLE>
__device__ __forceinline__ Setup setup_cta(uint8_t* smem_raw, const BwdParams& p) {
    using G = G256<ROLE>;
    Setup su;
    su.smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    su.sbase = ptx::smem_addr(su.smem);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(su.smem + G::kMiscOff);
    su.c.bars = su.sbase + (uint32_t)G::kBarOff;
    su.c.abort = reinterpret_cast<volatile int*>(su.smem + G::kMiscOff + 4);
    su.c.limit = p.wait_limit;
    su.c.status = g_status256;
    if (threadIdx.x == 0) {
        ptx::mbar_init(bar_addr(su.c, G::fixed_full()), 1);
        for (int s = 0; s < G::kSlots; ++s) {
            ptx::mbar_init(bar_addr(su.c, G::ring_full(s)), 1);
            ptx::mbar_init(bar_addr(su.c, G::ring_empty(s)), 1);
        }
        for (int b = 0; b < 2; ++b) {
            ptx::mbar_init(bar_addr(su.c, G::s_ready(b)), 1);
            ptx::mbar_init(bar_addr(su.c, G::x_ready(b)), kEwThreads);
        }
        ptx::mbar_init(bar_addr(su.c, G::dp_ready()), 1);
        ptx::mbar_init(bar_addr(su.c, G::ds_ready()), kEwThreads);
        ptx::mbar_init(bar_addr(su.c, G::row_ready()), 1);
        ptx::mbar_init(bar_addr(su.c, G::done()), 1);
        ptx::mbar_init(bar_addr(su.c, G::drain()), 1);
        *su.c.abort = 0;
        ptx::fence_barrier_init();
    }
    if (threadIdx.x / 32 == kMmaWarp) {
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

// Elementwise warps: the row tile (ring positions 0 and 1, rows 0-63 and 64-127) into TMEM
// as 16-bit pairs, this warp's rows and panels 2 ch, 2 ch + 1; then the two slots are
// released and the MMA warp told.  False if the CTA is aborting.
template <int ROLE>
__device__ __forceinline__ bool row_tile_to_tmem(const Ctl& c, uint32_t sbase, uint32_t tm,
                                                 int quarter, int ch, int lane) {
    using G = G256<ROLE>;
    const int r = quarter * 32 + lane;
    const uint32_t half = (uint32_t)(quarter >> 1);
    const bool ok = wait_warp(c, G::ring_full(G::slot(half)), 0, kRoleSoftmax);
    if (ok) {
        const int rr = r & (kSub - 1);
        const uint32_t tl = (uint32_t)(quarter * 32) << 16;
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
            const int pc = 2 * ch + pp;
            const uint32_t src = sbase + (uint32_t)G::kRingOff + G::slot(half) * (uint32_t)kSubBytes +
                                 (uint32_t)pc * kSubPanel + (uint32_t)rr * 128u;
            uint32_t w[32];
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                const uint4 v = ptx::ld_shared_v4(src + (uint32_t)((cc ^ (rr & 7)) * 16));
                w[4 * cc] = v.x; w[4 * cc + 1] = v.y; w[4 * cc + 2] = v.z; w[4 * cc + 3] = v.w;
            }
            ptx::tmem_st32(tm + tl + kColRow + 32u * (uint32_t)pc, w);
        }
        ptx::tmem_wait_st();
    }
    ptx::tc_fence_before();
    if (!ew_barrier_and(ok)) return false;
    if (threadIdx.x == 0) {
        ptx::mbar_arrive(bar_addr(c, G::ring_empty(G::slot(0))));
        ptx::mbar_arrive(bar_addr(c, G::ring_empty(G::slot(1))));
        ptx::mbar_arrive(bar_addr(c, G::row_ready()));
    }
    return true;
}

// Epilogue: this warp's rows, panels 2 ch and 2 ch + 1 of the accumulator, times mul.
template <int ROLE, bool F16>
__device__ __forceinline__ void store_acc(uint32_t sbase, uint32_t tm, int warp, int quarter,
                                          int ch, int lane, float mul, void* out,
                                          const Slice& sl, int tile) {
    using G = G256<ROLE>;
    const uint32_t tl = (uint32_t)(quarter * 32) << 16;
    const uint32_t stage = sbase + (uint32_t)G::kStageOff + (uint32_t)warp * 4096u;
#pragma unroll 1
    for (int pp = 0; pp < 2; ++pp) {
        const int pc = 2 * ch + pp;
        store_rows<F16>(tm + tl + kColAcc + 64u * (uint32_t)pc, mul, stage,
                        reinterpret_cast<uint16_t*>(out) + sl.row0 + 64 * pc, sl.stride,
                        tile * kT + quarter * 32, sl.len, lane);
    }
}

// CTA -> (slice, tile): slice-major, so the CTAs in flight share their slices' streamed
// tiles through L2; under the causal mask the heaviest tile of a slice comes first.
__device__ __forceinline__ void cta_tile(const BwdParams& p, bool heavy_last, int& bh, int& tile) {
    bh = blockIdx.x / p.ntiles;
    const int t = blockIdx.x % p.ntiles;
    tile = heavy_last ? p.ntiles - 1 - t : t;
}

// ----------------------------------------------------------------- dQ and dK kernels
template <int ROLE, bool CAUSAL, bool F16, int MODE>
__global__ void __launch_bounds__(kThreads, 1) bwd256_kernel(const __grid_constant__ BwdParams p) {
    static_assert(ROLE == kRoleDQ || ROLE == kRoleDK, "dQ or dK");
    constexpr bool kDQ = ROLE == kRoleDQ;
    using G = G256<ROLE>;
    int bh, tile;
    cta_tile(p, CAUSAL && kDQ, bh, tile);   // dQ: the last query tile sees the most keys
    const Slice sl = slice_at<MODE, kD>(p, bh);
    if (tile * kT >= sl.len) return;   // past a (shorter packed) sequence: nothing to do
    const int nsub_all = (sl.len + kSub - 1) / kSub;
    // streamed sub-tiles: dQ: keys 0.. (causal: up to the tile's last query); dK: queries
    // from the first that sees this key tile (causal) to the end
    const int s0 = (CAUSAL && !kDQ) ? 2 * tile : 0;
    const int n = kDQ ? (CAUSAL ? min(2 * (tile + 1), nsub_all) : nsub_all) : nsub_all - s0;
    extern __shared__ uint8_t smem_raw[];
    const Setup su = setup_cta<ROLE>(smem_raw, p);
    const Ctl& c = su.c;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t tm = su.tmem;

    if (warp == kLoadWarp) {
        if (lane == 0) {
            const uint32_t skipped = (p.inject_stall == 1 && blockIdx.x == 0) ? 0u : 0xFFFFFFFFu;
            if (kDQ)
                load_role<ROLE, MODE>(c, su.sbase, &p.tmap_do, &p.tmap_q, tile * kT, &p.tmap_k,
                                      &p.tmap_v, s0, n, bh, sl, skipped);
            else
                load_role<ROLE, MODE>(c, su.sbase, &p.tmap_v, &p.tmap_k, tile * kT, &p.tmap_q,
                                      &p.tmap_do, s0, n, bh, sl, skipped);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        constexpr uint32_t id_s = make_idesc(kT, kSub, false, F16);
        constexpr uint32_t id_acc = make_idesc(kT, kD, true, F16);
        const uint32_t ring = su.sbase + (uint32_t)G::kRingOff;
        auto sub = [&](uint32_t pos) { return ring + G::slot(pos) * (uint32_t)kSubBytes; };
        auto issue_s = [&](int j) -> bool {    // S = R X_j^T, R the row tile in TMEM
            const uint32_t pos = 2u + 2u * (uint32_t)j;
            if (!wait_warp(c, G::ring_full(G::slot(pos)), G::par(pos), kRoleMma)) return false;
            ptx::tc_fence_after();
            mma_rows_x_sub<true>(tm + kColS, tm + kColRow, sub(pos), id_s);
            ptx::mma_commit_elect(bar_addr(c, G::s_ready(0)));
            return true;
        };
        auto issue_dp = [&](int j) -> bool {   // dP = F Y_j^T, F the fixed tile; Y_j is then done
            const uint32_t pos = 3u + 2u * (uint32_t)j;
            if (!wait_warp(c, G::ring_full(G::slot(pos)), G::par(pos), kRoleMma)) return false;
            ptx::tc_fence_after();
            mma_rows_x_sub<false>(tm + kColDP, su.sbase, sub(pos), id_s);
            ptx::mma_commit_elect(bar_addr(c, G::dp_ready()));
            ptx::mma_commit_elect(bar_addr(c, G::ring_empty(G::slot(pos))));
            return true;
        };
        if (!wait_warp(c, G::fixed_full(), 0, kRoleMma)) goto mma_out;
        if (!wait_warp(c, G::row_ready(), 0, kRoleMma)) goto mma_out;
        ptx::tc_fence_after();
        if (!issue_s(0) || !issue_dp(0)) goto mma_out;
        for (int j = 0; j < n; ++j) {
            const uint32_t par = (uint32_t)j & 1u;
            if (!wait_warp(c, G::x_ready(0), par, kRoleMma)) goto mma_out;   // S(j) read
            if (j + 1 < n && !issue_s(j + 1)) goto mma_out;
            if (!wait_warp(c, G::ds_ready(), par, kRoleMma)) goto mma_out;   // dS(j) over dP
            ptx::tc_fence_after();
            const uint32_t xpos = 2u + 2u * (uint32_t)j;
            mma_acc(tm + kColAcc, tm + kColDP, sub(xpos), id_acc, j > 0);    // acc += dS X_j
            ptx::mma_commit_elect(bar_addr(c, G::ring_empty(G::slot(xpos))));
            // dP(j + 1) overwrites dS(j): products run in issue order
            if (j + 1 < n && !issue_dp(j + 1)) goto mma_out;
        }
        ptx::mma_commit_elect(bar_addr(c, G::done()));
    mma_out:
        ptx::mma_commit_elect(bar_addr(c, G::drain()));
        wait_drain(bar_addr(c, G::drain()), 0, c.limit);
        __syncwarp();
    } else {
        const int quarter = warp & 3, ch = warp >> 2;
        const int r = quarter * 32 + lane;
        const int row = tile * kT + r;             // query (dQ) or key (dK) of this thread
        const bool live = row < sl.len;
        const uint32_t tl = (uint32_t)(quarter * 32) << 16;
        float* vec = reinterpret_cast<float*>(su.smem + G::kVecOff);
        float lse2 = 0.0f, dlt = 0.0f;
        int limit = sl.len;   // dQ: visible keys are < limit
        if constexpr (kDQ) {
            const size_t vrow = sl.vec0 + (size_t)(live ? row : 0);
            lse2 = live ? p.lse[vrow] * kLog2e : 0.0f;
            if (CAUSAL) limit = min(row + 1, sl.len);
            // delta = sum_d dO * O for this row: this warp's panels 2 ch, 2 ch + 1 (dO from
            // the fixed tile, O from global memory), the two halves added through shared
            // memory after the barrier below
            const size_t erow = sl.row0 + (size_t)(live ? row : 0) * sl.stride;
            const bool okd = wait_warp(c, G::fixed_full(), 0, kRoleSoftmax);
            float acc = 0.0f;
#pragma unroll 1
            for (int pp = 0; pp < 2 && okd && live; ++pp) {
                const int pc = 2 * ch + pp;
                const uint4* orow = reinterpret_cast<const uint4*>(
                    static_cast<const uint16_t*>(p.o) + erow + 64 * pc);
                // the fixed tile's panel pc: rows 0-63 then 64-127, 128 bytes each
                const uint32_t drow = su.sbase + (uint32_t)pc * kFixPanel + (uint32_t)r * 128u;
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const uint4 ov = __ldg(orow + cc);
                    const uint4 dv = ptx::ld_shared_v4(drow + (uint32_t)((cc ^ (r & 7)) * 16));
                    const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        acc = fmaf(unpack_lo<F16>(ow[e]), unpack_lo<F16>(dw[e]), acc);
                        acc = fmaf(unpack_hi<F16>(ow[e]), unpack_hi<F16>(dw[e]), acc);
                    }
                }
            }
            vec[ch * kT + r] = acc;
        }
        if (!row_tile_to_tmem<ROLE>(c, su.sbase, tm, quarter, ch, lane)) goto ew_out;
        if constexpr (kDQ) {
            // both partial sums are published by the barrier inside row_tile_to_tmem
            dlt = vec[r] + vec[kT + r];
            if (live && ch == 0) p.delta[sl.vec0 + (size_t)row] = dlt;   // for the dK kernel
        }
        {
            // dK: LSE (log2 units; +inf past the end, so p = 0 there) and delta of each
            // query column of the next sub-tile, fetched one step ahead by threads 0-127
            const int t = threadIdx.x;
            auto fetch = [&](int s) -> float {
                const int q = (s0 + s) * kSub + (t & (kSub - 1));
                const bool ok = s < n && q < sl.len;
                if (t < kSub) return ok ? p.lse[sl.vec0 + q] * kLog2e : INFINITY;
                return ok ? p.delta[sl.vec0 + q] : 0.0f;
            };
            float next = 0.0f;
            if (!kDQ && t < 2 * kSub) next = fetch(0);
            bool failed = false;
            for (int j = 0; j < n; ++j) {
                const uint32_t par = (uint32_t)j & 1u;
                const int col0 = (s0 + j) * kSub + 32 * ch;   // first key (dQ) / query (dK) of this warp
                const float* vl = vec + par * 128;            // dK: [0, 64) LSE, [64, 128) delta
                float pr[32];
                {   // P (P^T) from S (S^T)
                    bool ok = !failed && wait_warp(c, G::s_ready(0), par, kRoleSoftmax);
                    if constexpr (!kDQ) {
                        if (t < 2 * kSub) vec[par * 128 + t] = next;
                        if (!ew_barrier_and(ok)) goto ew_out;
                        if (t < 2 * kSub) next = fetch(j + 1);
                    } else if (!ok) {
                        failed = true;
                        continue;
                    }
                    ptx::tc_fence_after();
                    uint32_t sv[32];
                    ptx::tmem_ld32_wait(tm + tl + kColS + 32u * (uint32_t)ch, sv);
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(bar_addr(c, G::x_ready(0)));   // S may be overwritten
                    if constexpr (kDQ) {
#pragma unroll
                        for (int cc = 0; cc < 32; cc += 2) {
                            float x0, x1;
                            ptx::fma2(x0, x1, u2f(sv[cc]), u2f(sv[cc + 1]), p.scale_log2, -lse2);
                            pr[cc] = ptx::ex2(x0);
                            pr[cc + 1] = ptx::ex2(x1);
                        }
                        if (__any_sync(0xFFFFFFFFu, col0 + 32 > limit)) {
#pragma unroll
                            for (int cc = 0; cc < 32; ++cc)
                                if (col0 + cc >= limit) pr[cc] = 0.0f;
                        }
                    } else {
                        const float4* l4 = reinterpret_cast<const float4*>(vl + 32 * ch);
#pragma unroll
                        for (int c4 = 0; c4 < 8; ++c4) {
                            const float4 l = l4[c4];
                            const int cc = 4 * c4;
                            float x0, x1, x2, x3;
                            ptx::fma2v(x0, x1, u2f(sv[cc]), u2f(sv[cc + 1]), p.scale_log2, p.scale_log2, -l.x, -l.y);
                            ptx::fma2v(x2, x3, u2f(sv[cc + 2]), u2f(sv[cc + 3]), p.scale_log2, p.scale_log2, -l.z, -l.w);
                            pr[cc] = ptx::ex2(x0);
                            pr[cc + 1] = ptx::ex2(x1);
                            pr[cc + 2] = ptx::ex2(x2);
                            pr[cc + 3] = ptx::ex2(x3);
                        }
                        // queries before this key are masked (only near the diagonal)
                        if (CAUSAL && __any_sync(0xFFFFFFFFu, col0 < row)) {
#pragma unroll
                            for (int cc = 0; cc < 32; ++cc)
                                if (col0 + cc < row) pr[cc] = 0.0f;
                        }
                    }
                }
                {   // dS = P (dP - delta), 16-bit, over the first 16 of this warp's dP columns
                    if (!wait_warp(c, G::dp_ready(), par, kRoleSoftmax)) { failed = true; continue; }
                    ptx::tc_fence_after();
                    const uint32_t tp = tm + tl + kColDP + 32u * (uint32_t)ch;
                    uint32_t dp[32];
                    ptx::tmem_ld32_wait(tp, dp);
                    uint32_t pk[16];
                    if constexpr (kDQ) {
#pragma unroll
                        for (int cc = 0; cc < 32; cc += 2) {
                            float d0 = u2f(dp[cc]), d1 = u2f(dp[cc + 1]);
                            ptx::add2(d0, d1, -dlt, -dlt);
                            ptx::mul2(d0, d1, pr[cc], pr[cc + 1]);
                            pk[cc >> 1] = pack2<F16>(d0, d1);
                        }
                    } else {
                        const float4* d4 = reinterpret_cast<const float4*>(vl + kSub + 32 * ch);
#pragma unroll
                        for (int c4 = 0; c4 < 8; ++c4) {
                            const float4 d = d4[c4];
                            const int cc = 4 * c4;
                            float a0 = u2f(dp[cc]), a1 = u2f(dp[cc + 1]), a2 = u2f(dp[cc + 2]), a3 = u2f(dp[cc + 3]);
                            ptx::add2(a0, a1, -d.x, -d.y);
                            ptx::add2(a2, a3, -d.z, -d.w);
                            ptx::mul2(a0, a1, pr[cc], pr[cc + 1]);
                            ptx::mul2(a2, a3, pr[cc + 2], pr[cc + 3]);
                            pk[cc >> 1] = pack2<F16>(a0, a1);
                            pk[(cc >> 1) + 1] = pack2<F16>(a2, a3);
                        }
                    }
                    ptx::tmem_st16(tp, pk);
                    ptx::tmem_wait_st();
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(bar_addr(c, G::ds_ready()));
                }
            }
            if (failed) goto ew_out;
        }
        if (!wait_warp(c, G::done(), 0, kRoleSoftmax)) goto ew_out;
        ptx::tc_fence_after();
        store_acc<ROLE, F16>(su.sbase, tm, warp, quarter, ch, lane, p.scale, kDQ ? p.dq : p.dk, sl, tile);
    ew_out:;
    }
    teardown_cta(su);
}

// ----------------------------------------------------------------- dV kernel
template <bool CAUSAL, bool F16, int MODE>
__global__ void __launch_bounds__(kThreads, 1) bwd256_dv_kernel(const __grid_constant__ BwdParams p) {
    using G = G256<kRoleDV>;
    int bh, tile;
    cta_tile(p, false, bh, tile);
    const Slice sl = slice_at<MODE, kD>(p, bh);
    if (tile * kT >= sl.len) return;
    const int s0 = CAUSAL ? 2 * tile : 0;
    const int n = (sl.len + kSub - 1) / kSub - s0;
    extern __shared__ uint8_t smem_raw[];
    const Setup su = setup_cta<kRoleDV>(smem_raw, p);
    const Ctl& c = su.c;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const uint32_t tm = su.tmem;

    if (warp == kLoadWarp) {
        if (lane == 0)
            load_role<kRoleDV, MODE>(c, su.sbase, nullptr, &p.tmap_k, tile * kT, &p.tmap_q,
                                     &p.tmap_do, s0, n, bh, sl,
                                     (p.inject_stall == 1 && blockIdx.x == 0) ? 0u : 0xFFFFFFFFu);
        __syncwarp();
    } else if (warp == kMmaWarp) {
        constexpr uint32_t id_s = make_idesc(kT, kSub, false, F16);
        constexpr uint32_t id_acc = make_idesc(kT, kD, true, F16);
        const uint32_t ring = su.sbase + (uint32_t)G::kRingOff;
        uint32_t pos = 2;   // next streamed sub-tile, in the loader's order
        auto issue_s = [&](int s) -> bool {    // S^T(s) = K Q_s^T into buffer s & 1; Q_s is then done
            if (!wait_warp(c, G::ring_full(G::slot(pos)), G::par(pos), kRoleMma)) return false;
            ptx::tc_fence_after();
            mma_rows_x_sub<true>(tm + kColS + 64u * (uint32_t)(s & 1), tm + kColRow,
                                 ring + G::slot(pos) * (uint32_t)kSubBytes, id_s);
            ptx::mma_commit_elect(bar_addr(c, G::s_ready(s & 1)));
            ptx::mma_commit_elect(bar_addr(c, G::ring_empty(G::slot(pos))));
            ++pos;
            return true;
        };
        if (!wait_warp(c, G::row_ready(), 0, kRoleMma)) goto mma_out;
        ptx::tc_fence_after();
        if (!issue_s(0)) goto mma_out;
        if (n > 1 && !issue_s(1)) goto mma_out;
        for (int s = 0; s < n; ++s) {
            const int b = s & 1;
            if (!wait_warp(c, G::x_ready(b), (uint32_t)(s >> 1) & 1u, kRoleMma)) goto mma_out;  // P^T(s) stored
            if (!wait_warp(c, G::ring_full(G::slot(pos)), G::par(pos), kRoleMma)) goto mma_out;  // dO_s
            ptx::tc_fence_after();
            mma_acc(tm + kColAcc, tm + kColS + 64u * (uint32_t)b, ring + G::slot(pos) * (uint32_t)kSubBytes,
                    id_acc, s > 0);   // dV += P^T(s) dO_s
            ptx::mma_commit_elect(bar_addr(c, G::ring_empty(G::slot(pos))));
            ++pos;
            // S^T(s + 2) overwrites P^T(s) in buffer b: products run in issue order
            if (s + 2 < n && !issue_s(s + 2)) goto mma_out;
        }
        ptx::mma_commit_elect(bar_addr(c, G::done()));
    mma_out:
        ptx::mma_commit_elect(bar_addr(c, G::drain()));
        wait_drain(bar_addr(c, G::drain()), 0, c.limit);
        __syncwarp();
    } else {
        const int quarter = warp & 3, ch = warp >> 2;
        const int r = quarter * 32 + lane;
        const int key = tile * kT + r;
        const uint32_t tl = (uint32_t)(quarter * 32) << 16;
        // this warp's staging area: the LSE of its 32 query columns, double-buffered
        float* vw = reinterpret_cast<float*>(su.smem + G::kVecOff) + warp * 64;
        if (!row_tile_to_tmem<kRoleDV>(c, su.sbase, tm, quarter, ch, lane)) goto ew_out;
        {
            // LSE (log2 units; +inf past the end) of this warp's query columns of the next
            // sub-tile, lane l holding column l, fetched one step ahead; staged per warp, so
            // no barrier across warps is needed
            auto fetch = [&](int s) -> float {
                const int q = (s0 + s) * kSub + 32 * ch + lane;
                return (s < n && q < sl.len) ? p.lse[sl.vec0 + q] * kLog2e : INFINITY;
            };
            float next = fetch(0);
            for (int s = 0; s < n; ++s) {
                const int b = s & 1;
                float* vl = vw + b * 32;
                vl[lane] = next;
                __syncwarp();
                if (!wait_warp(c, G::s_ready(b), (uint32_t)(s >> 1) & 1u, kRoleSoftmax)) goto ew_out;
                next = fetch(s + 1);
                ptx::tc_fence_after();
                const int col0 = (s0 + s) * kSub + 32 * ch;   // first query of this warp
                const uint32_t ts = tm + tl + kColS + 64u * (uint32_t)b + 32u * (uint32_t)ch;
                uint32_t sv[32];
                ptx::tmem_ld32_wait(ts, sv);
                const float4* l4 = reinterpret_cast<const float4*>(vl);
                float pr[32];
#pragma unroll
                for (int c4 = 0; c4 < 8; ++c4) {
                    const float4 l = l4[c4];
                    const int cc = 4 * c4;
                    float x0, x1, x2, x3;
                    ptx::fma2v(x0, x1, u2f(sv[cc]), u2f(sv[cc + 1]), p.scale_log2, p.scale_log2, -l.x, -l.y);
                    ptx::fma2v(x2, x3, u2f(sv[cc + 2]), u2f(sv[cc + 3]), p.scale_log2, p.scale_log2, -l.z, -l.w);
                    pr[cc] = ptx::ex2(x0);
                    pr[cc + 1] = ptx::ex2(x1);
                    pr[cc + 2] = ptx::ex2(x2);
                    pr[cc + 3] = ptx::ex2(x3);
                }
                if (CAUSAL && __any_sync(0xFFFFFFFFu, col0 < key)) {
#pragma unroll
                    for (int cc = 0; cc < 32; ++cc)
                        if (col0 + cc < key) pr[cc] = 0.0f;
                }
                uint32_t pk[16];
#pragma unroll
                for (int cc = 0; cc < 32; cc += 2) pk[cc >> 1] = pack2<F16>(pr[cc], pr[cc + 1]);
                ptx::tmem_st16(ts, pk);
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar_addr(c, G::x_ready(b)));
            }
        }
        if (!wait_warp(c, G::done(), 0, kRoleSoftmax)) goto ew_out;
        ptx::tc_fence_after();
        store_acc<kRoleDV, F16>(su.sbase, tm, warp, quarter, ch, lane, 1.0f, p.dv, sl, tile);
    ew_out:;
    }
    teardown_cta(su);
}

// ----------------------------------------------------------------- host side
template <bool CAUSAL, bool F16, int MODE>
cudaError_t prepare_mode() {
    cudaError_t e = cudaFuncSetAttribute(bwd256_kernel<kRoleDQ, CAUSAL, F16, MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, G256<kRoleDQ>::kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bwd256_kernel<kRoleDK, CAUSAL, F16, MODE>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, G256<kRoleDK>::kSmemBytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(bwd256_dv_kernel<CAUSAL, F16, MODE>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, G256<kRoleDV>::kSmemBytes);
    return e;
}

template <bool CAUSAL, bool F16>
cudaError_t prepare2() {
    const cudaError_t e = prepare_mode<CAUSAL, F16, 0>();
    return e != cudaSuccess ? e : prepare_mode<CAUSAL, F16, 1>();
}

// dQ (writes delta), then dV, then dK (reads delta), in stream order.
template <bool CAUSAL, bool F16, int MODE>
cudaError_t launch_mode(const BwdParams& p, unsigned ctas, cudaStream_t stream) {
    bwd256_kernel<kRoleDQ, CAUSAL, F16, MODE><<<ctas, kThreads, G256<kRoleDQ>::kSmemBytes, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd256_dv_kernel<CAUSAL, F16, MODE><<<ctas, kThreads, G256<kRoleDV>::kSmemBytes, stream>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd256_kernel<kRoleDK, CAUSAL, F16, MODE><<<ctas, kThreads, G256<kRoleDK>::kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

template <bool CAUSAL, bool F16>
cudaError_t launch2(const BwdParams& p, int bh, cudaStream_t stream) {
    const long long ctas = (long long)bh * p.ntiles;
    if (ctas > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
    return p.layout == 0 ? launch_mode<CAUSAL, F16, 0>(p, (unsigned)ctas, stream)
                         : launch_mode<CAUSAL, F16, 1>(p, (unsigned)ctas, stream);
}

}  // namespace

cudaError_t bwd256_prepare(bool causal, bool f16) {
    if (causal) return f16 ? prepare2<true, true>() : prepare2<true, false>();
    return f16 ? prepare2<false, true>() : prepare2<false, false>();
}

cudaError_t bwd256_launch(bool causal, bool f16, const BwdParams& p, int bh, cudaStream_t stream) {
    if (causal) return f16 ? launch2<true, true>(p, bh, stream) : launch2<true, false>(p, bh, stream);
    return f16 ? launch2<false, true>(p, bh, stream) : launch2<false, false>(p, bh, stream);
}

cudaError_t bwd256_status_read_reset(uint32_t out[4]) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_status256, sizeof(unsigned int) * 4);
    if (e != cudaSuccess) return e;
    const unsigned int zero[4] = {0, 0, 0, 0};
    return cudaMemcpyToSymbol(g_status256, zero, sizeof(zero));
}

}  // namespace fa
