// fa_bwd.cu -- attention backward on the GB300 tensor cores (tcgen05 + TMEM + TMA).
//
// Gradients of a loss through O = softmax(scale * Q K^T) V, recomputing the probabilities
// from the forward's LSE instead of storing them ("08 · FlashAttention" §三: the backward
// recomputes P from the saved statistics; "第 13 课" §4B):
//     P = exp(scale * Q K^T - LSE),  dP = dO V^T,  delta = rowsum(dO * O),
//     dS = P * (dP - delta),  dV = P^T dO,  dQ = scale * dS K,  dK = scale * dS^T Q.
//
// Two kernels, no atomics (results do not depend on scheduling):
//   * dQ: one CTA per 128-query tile; it also forms delta = rowsum(dO * O) in fp32 for its
//     rows (dO from its shared tile, O from global memory) and writes it for the next kernel.  Q is copied once into TMEM and serves as the A
//     operand of S = Q K_j^T (dO stays in shared memory for dP = dO V_j^T); the
//     elementwise warps (TMEM lane = query row) form P, then dS = P (dP - delta) into a
//     TMEM region of its own (16-bit), so dP of the next key tile can start while dQ +=
//     dS K_j (K_j read as the MN-major operand) waits for dS;
//   * dK, dV: one CTA per 128-key tile with K, V fixed in shared memory; per query tile
//     S^T = K Q_i^T and dP^T = V dO_i^T (TMEM lane = key row), P^T written over S^T feeds
//     dV += P^T dO_i, and dS^T written over dP^T feeds dK += dS^T Q_i.
// All products are M = 128, N = 128 (or N = D), K = 16 steps.  The MMA warp staggers them
// so that each elementwise phase overlaps products of the neighbouring phase: the next S
// is issued as soon as the elementwise warps have read the current one.  Streamed tiles
// pass through a 4-slot ring whose two slots per step swap roles every other step, so the
// tile needed first two steps later lands in the slot that is released first.
// Warps: 0-7 elementwise (warp w: TMEM lanes 32 (w % 4).., columns 64 (w / 4).. of each
// 128-column tile), 8 MMA issuer (converged, one elected lane issues), 9 TMA loader.
// Every wait is bounded as in the forward kernel.
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
__device__ unsigned int g_status[4];

constexpr int kT = 128;          // tile rows (TMEM lanes) and streamed tile rows
constexpr int kThreads = 320;
constexpr int kEwThreads = 256;  // warps 0-7
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

// Rows of a 128 x D tile in shared memory: panels of 128-byte rows (128-byte swizzle), or
// one panel of 64-byte rows (64-byte swizzle) at D = 32, as TMA writes them.
template <int D>
struct Rows {
    static constexpr int kRowBytes = D * 2 < 128 ? D * 2 : 128;
    static constexpr int kCols = kRowBytes / 2;               // 16-bit values per panel row
    static constexpr int kPanelBytes = kT * kRowBytes;        // one 128-row panel
    static constexpr int kPanels = D / kCols;
    static constexpr uint32_t kSBO = 8u * kRowBytes;          // 8-row group stride
    static constexpr uint64_t kLayout = kRowBytes == 128 ? 2ull : 4ull;   // descriptor swizzle
};

// Shared-memory matrix descriptor of a tile with D-dependent rows.
template <int D>
__device__ __forceinline__ uint64_t bdesc(uint32_t saddr, uint32_t lbo) {
    using R = Rows<D>;
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((R::kSBO >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (R::kLayout << 61);
}

// Shared memory: FIXED fixed 128 x D tiles, a ring of SLOTS streamed tiles, the staged
// per-column vectors (dK/dV), then the barriers.
template <int D, int FIXED, int SLOTS>
struct BGeo {
    static constexpr int kPanels = Rows<D>::kPanels;
    static constexpr int kTile = kPanels * Rows<D>::kPanelBytes;   // one 128 x D tile
    static constexpr int kSlots = SLOTS;
    static constexpr int kRingOff = FIXED * kTile;
    // epilogue staging (4 KB per elementwise warp) reuses the ring: it starts only after
    // every product, hence every read of the ring, has completed
    static constexpr int kStageOff = kRingOff;
    // dK/dV: per elementwise warp 2 x 128 floats of staged per-column LSE and delta; dQ:
    // 2 x 128 floats of partial row sums of delta
    static constexpr int kVecOff = kRingOff + kSlots * kTile;
    static constexpr int kBarOff = kVecOff + (FIXED == 2 ? 8 * 2 * 128 * 4 : 2 * 128 * 4);
    // barriers: fixed_full, ring_full[4], ring_empty[4], then the named ones below
    static constexpr int kNumBars = 1 + 2 * kSlots + 9;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;
    static_assert(kSmemBytes <= 232448, "shared memory");
    static_assert(8 * 4096 <= kSlots * kTile, "staging fits the ring");

    static constexpr int fixed_full() { return 0; }
    static constexpr int ring_full(uint32_t slot) { return 1 + (int)slot; }
    static constexpr int ring_empty(uint32_t slot) { return 1 + kSlots + (int)slot; }
    // cyclic use (dQ): streamed tile `pos` in slot pos % SLOTS, its (pos / SLOTS)-th fill
    static __device__ __forceinline__ uint32_t cyc_slot(uint32_t pos) { return pos % SLOTS; }
    static __device__ __forceinline__ uint32_t cyc_par(uint32_t pos) { return (pos / SLOTS) & 1u; }
    static constexpr int s_ready() { return 1 + 2 * kSlots; }    // S (S^T) in TMEM
    static constexpr int dp_ready() { return 2 + 2 * kSlots; }   // dP (dP^T) in TMEM
    static constexpr int x_ready() { return 3 + 2 * kSlots; }    // dQ: S read; dK/dV: P^T stored
    static constexpr int ds_ready() { return 4 + 2 * kSlots; }   // dS (dS^T) stored
    static constexpr int q_ready() { return 5 + 2 * kSlots; }    // dQ: Q copied into TMEM
    static constexpr int dp_free() { return 6 + 2 * kSlots; }    // dQ: dP read
    static constexpr int ds_free() { return 7 + 2 * kSlots; }    // dQ: dQ product read dS
    static constexpr int done() { return 8 + 2 * kSlots; }
    static constexpr int drain() { return 9 + 2 * kSlots; }
};

template <int D> using GeoDq = BGeo<D, 1, 6>;     // dO fixed; Q, then K_j, V_j, streamed
template <int D> using GeoDkdv = BGeo<D, 2, 4>;   // K, V fixed; Q_i, dO_i streamed

// The dK/dV ring: step j streams tile A_j (needed first, released last) and B_j (needed
// second, released first).  A_j takes the slot B_{j-2} used and B_j the slot A_{j-2} used,
// so every slot is filled once per two steps.
__device__ __forceinline__ uint32_t slot_a(int j) { return 2u * (uint32_t)(j & 1) + ((uint32_t)(j >> 1) & 1u); }
__device__ __forceinline__ uint32_t slot_b(int j) { return 2u * (uint32_t)(j & 1) + 1u - ((uint32_t)(j >> 1) & 1u); }
__device__ __forceinline__ uint32_t slot_par(int j) { return (uint32_t)(j >> 1) & 1u; }

// ----------------------------------------------------------------- MMA helpers
// K-major operand: a 16-element K step is 32 bytes of a panel row; panels follow each other.
template <int D>
__device__ __forceinline__ uint64_t kmaj_step(int kk) {
    using R = Rows<D>;
    constexpr int kSteps = R::kRowBytes / 32;   // K steps per panel row
    return ((uint64_t)(kk / kSteps) * R::kPanelBytes + (uint64_t)(kk % kSteps) * 32u) >> 4;
}

// D_tmem = A[128 x D] * B[128 x D]^T, A and B K-major in shared memory.
template <int D>
__device__ __forceinline__ void mma_ss_nt(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc) {
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
        ptx::mma_ss_elect(d_tmem, a_desc + kmaj_step<D>(kk), b_desc + kmaj_step<D>(kk), idesc,
                          kk > 0 ? 1u : 0u);
}

// D_tmem = A_tmem[128 x D] * B[128 x D]^T, A in TMEM (16-bit pairs per column, D/2
// columns), B K-major in shared memory.
template <int D>
__device__ __forceinline__ void mma_ts_nt(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc) {
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
        ptx::mma_ts_elect(d_tmem, a_tmem + (uint32_t)kk * 8u, b_desc + kmaj_step<D>(kk), idesc,
                          kk > 0 ? 1u : 0u);
}

// acc_tmem (+)= A_tmem[128 x 128] * B, B a 128 x D tile read as the MN-major operand (16
// rows per K step).  A holds 16-bit values packed two per TMEM column in two blocks of 32
// columns (64 values each), one per elementwise warp of the lane quarter, at a_tmem and
// a_tmem + BLOCK (BLOCK = 32: contiguous; 64: over the first half of each 64-column fp32
// block the values were computed from).
template <int D, uint32_t BLOCK>
__device__ __forceinline__ void mma_ts_tn(uint32_t acc_tmem, uint32_t a_tmem, uint64_t b_desc,
                                          uint32_t idesc, bool accumulate) {
    constexpr int kStepBytes = 16 * Rows<D>::kRowBytes;
#pragma unroll
    for (int kk = 0; kk < kT / 16; ++kk)
        ptx::mma_ts_elect(acc_tmem, a_tmem + (uint32_t)(kk >> 2) * BLOCK + (uint32_t)(kk & 3) * 8u,
                          b_desc + (uint64_t)((kk * kStepBytes) >> 4), idesc,
                          (accumulate || kk > 0) ? 1u : 0u);
}

// ----------------------------------------------------------------- epilogue
// D = 32: this warp's 32 TMEM lanes x 32 fp32 columns at t_acc, times mul, rounded to 16
// bits, to global rows base + (row0 + r) * stride (64 bytes each; only rows with
// row0 + r < nrows).  Staged with the 16-byte chunks of row r XOR-swizzled by (r >> 1) & 3
// (free of bank conflicts both ways); in [B, H, N, D] the warp's rows are one contiguous
// 2 KB block, so each store instruction then writes 512 contiguous bytes.
template <bool F16>
__device__ __forceinline__ void store_rows32(uint32_t t_acc, float mul, uint32_t stage,
                                             uint16_t* base, size_t stride, int row0, int nrows,
                                             int lane) {
    uint32_t o[32];
    ptx::tmem_ld32_wait(t_acc, o);
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack2<F16>(u2f(o[2 * i]) * mul, u2f(o[2 * i + 1]) * mul);
    const uint32_t sw = (uint32_t)((lane >> 1) & 3);
#pragma unroll
    for (int cc = 0; cc < 4; ++cc)
        ptx::st_shared_v4(stage + (uint32_t)lane * 64u + (((uint32_t)cc ^ sw) * 16u), w[4 * cc],
                          w[4 * cc + 1], w[4 * cc + 2], w[4 * cc + 3]);
    __syncwarp();
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int r = 8 * k + (lane >> 2);
        const int ch = lane & 3;
        const uint4 v = ptx::ld_shared_v4(stage + (uint32_t)r * 64u + (uint32_t)((ch ^ ((r >> 1) & 3)) * 16));
        if (row0 + r < nrows)
            *reinterpret_cast<uint4*>(base + (size_t)(row0 + r) * stride + ch * 8) = v;
    }
    __syncwarp();
}

// ----------------------------------------------------------------- common prologue
struct Setup {
    Ctl c;
    uint32_t sbase, tmem;
};

template <class G>
__device__ __forceinline__ Setup setup_cta(uint8_t* smem_raw, const BwdParams& p) {
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
        ptx::mbar_init(bar_addr(su.c, G::fixed_full()), 1);
        for (int s = 0; s < G::kSlots; ++s) {
            ptx::mbar_init(bar_addr(su.c, G::ring_full(s)), 1);
            ptx::mbar_init(bar_addr(su.c, G::ring_empty(s)), 1);
        }
        ptx::mbar_init(bar_addr(su.c, G::s_ready()), 1);
        ptx::mbar_init(bar_addr(su.c, G::dp_ready()), 1);
        ptx::mbar_init(bar_addr(su.c, G::x_ready()), kEwThreads);
        ptx::mbar_init(bar_addr(su.c, G::ds_ready()), kEwThreads);
        ptx::mbar_init(bar_addr(su.c, G::q_ready()), 1);
        ptx::mbar_init(bar_addr(su.c, G::dp_free()), kEwThreads);
        ptx::mbar_init(bar_addr(su.c, G::ds_free()), 1);
        ptx::mbar_init(bar_addr(su.c, G::done()), 1);
        ptx::mbar_init(bar_addr(su.c, G::drain()), 1);
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

// One 128 x D tile (rows row.. of the slice) into shared memory at dst, completing on
// barrier bar (whose expected bytes the caller has set).  Map dims {D, N, B*H} (MODE 0) or
// {D, H, tokens} (MODE 1).
template <int D, int MODE>
__device__ __forceinline__ void load_tile(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                          int row, int bh, const Slice& sl) {
    using R = Rows<D>;
#pragma unroll
    for (int pc = 0; pc < R::kPanels; ++pc) {
        if (MODE == 0)
            ptx::tma_load_3d(dst + (uint32_t)pc * R::kPanelBytes, map, bar, pc * R::kCols, row, bh);
        else
            ptx::tma_load_3d(dst + (uint32_t)pc * R::kPanelBytes, map, bar, pc * R::kCols, sl.h,
                             sl.tok0 + row);
    }
}

// dK/dV loader: the two fixed tiles (f0, f1 at fixed_row), then for steps j < steps the
// tiles A_j (map ma) and B_j (map mb), rows first_row + 128 j, through the paired ring.
// Waits for its own copies before returning, so no copy is in flight when the CTA leaves.
// withhold (failure-detection test hook): A_0 is never loaded, so the waits for it run out.
template <int D, int MODE>
__device__ void load_pairs(const Ctl& c, uint32_t sbase, const CUtensorMap* f0,
                           const CUtensorMap* f1, int fixed_row, const CUtensorMap* ma,
                           const CUtensorMap* mb, int first_row, int steps, int bh, const Slice& sl,
                           bool withhold) {
    using G = GeoDkdv<D>;
    const uint32_t fb = bar_addr(c, G::fixed_full());
    ptx::mbar_arrive_expect_tx(fb, 2u * G::kTile);
    load_tile<D, MODE>(sbase, f0, fb, fixed_row, bh, sl);
    load_tile<D, MODE>(sbase + (uint32_t)G::kTile, f1, fb, fixed_row, bh, sl);
    int issued = 0;   // tiles issued, A and B alternating
    for (int j = 0; j < steps; ++j) {
        for (int w = 0; w < 2; ++w) {
            const uint32_t slot = w == 0 ? slot_a(j) : slot_b(j);
            if (!wait(c, G::ring_empty(slot), slot_par(j) ^ 1u, kRoleLoad)) goto out;
            if (withhold && issued == 0) {
                ++issued;
                continue;
            }
            const uint32_t bar = bar_addr(c, G::ring_full(slot));
            ptx::mbar_arrive_expect_tx(bar, (uint32_t)G::kTile);
            load_tile<D, MODE>(sbase + (uint32_t)G::kRingOff + slot * (uint32_t)G::kTile, w == 0 ? ma : mb,
                               bar, first_row + j * kT, bh, sl);
            ++issued;
        }
    }
out:
    wait_drain(fb, 0, c.limit);
    // copies of the last two steps may still be in flight
    for (int k = (issued > 4 ? issued - 4 : 0); k < issued; ++k) {
        if (withhold && k == 0) continue;
        const int j = k >> 1;
        wait_drain(bar_addr(c, G::ring_full((k & 1) ? slot_b(j) : slot_a(j))), slot_par(j), c.limit);
    }
}

// dQ loader: the fixed tile dO (rows fixed_row), then streamed tile 0 = Q (rows fixed_row)
// and tiles 1 + 2j = K_j, 2 + 2j = V_j (rows 128 j) through the cyclic ring.  Waits for its
// own copies before returning.  Failure-detection test hook: CTA 0 withholds Q.
template <int D, int MODE>
__device__ void load_dq(const Ctl& c, uint32_t sbase, const BwdParams& p, int fixed_row, int nkv,
                        int bh, const Slice& sl) {
    using G = GeoDq<D>;
    const uint32_t fb = bar_addr(c, G::fixed_full());
    ptx::mbar_arrive_expect_tx(fb, (uint32_t)G::kTile);
    load_tile<D, MODE>(sbase, &p.tmap_do, fb, fixed_row, bh, sl);
    const uint32_t count = 1u + 2u * (uint32_t)nkv;
    const uint32_t skipped = (p.inject_stall == 1 && blockIdx.x == 0) ? 0u : 0xFFFFFFFFu;
    uint32_t pos = 0;
    for (; pos < count; ++pos) {
        const uint32_t slot = G::cyc_slot(pos);
        if (!wait(c, G::ring_empty(slot), G::cyc_par(pos) ^ 1u, kRoleLoad)) break;
        if (pos == skipped) continue;
        const uint32_t bar = bar_addr(c, G::ring_full(slot));
        const CUtensorMap* map = pos == 0 ? &p.tmap_q : ((pos & 1u) ? &p.tmap_k : &p.tmap_v);
        const int row = pos == 0 ? fixed_row : (int)((pos - 1u) >> 1) * kT;
        ptx::mbar_arrive_expect_tx(bar, (uint32_t)G::kTile);
        load_tile<D, MODE>(sbase + (uint32_t)G::kRingOff + slot * (uint32_t)G::kTile, map, bar, row, bh, sl);
    }
    wait_drain(fb, 0, c.limit);
    for (uint32_t i = (pos > (uint32_t)G::kSlots ? pos - G::kSlots : 0u); i < pos; ++i)
        if (i != skipped) wait_drain(bar_addr(c, G::ring_full(G::cyc_slot(i))), G::cyc_par(i), c.limit);
}

// ----------------------------------------------------------------- dQ kernel
// TMEM columns: Q [0, D/2), dS [QC, QC+64), S [QC+64, +128), dP [QC+192, +128), dQ
// accumulator [QC+320, +D) with QC = max(D/2, 32), so every region starts on a multiple of
// 32 columns (512 columns at D = 128).
// Shared memory: dO fixed; ring: Q (copied to TMEM, then released), K_j, V_j.
template <int D, bool CAUSAL, bool F16, int MODE>
__global__ void __launch_bounds__(kThreads, 1) bwd_dq_kernel(const __grid_constant__ BwdParams p) {
    using G = GeoDq<D>;
    // query tiles past a (shorter packed) sequence have nothing to do: the whole CTA leaves.
    // Causal: a slice's last query tile sees the most keys, so it is dispatched first.
    const int bh = blockIdx.x / p.ntiles;
    const int qt = CAUSAL ? p.ntiles - 1 - blockIdx.x % p.ntiles : blockIdx.x % p.ntiles;
    const Slice sl = slice_at<MODE, D>(p, bh);
    if (qt * kT >= sl.len) return;
    constexpr uint32_t kQC = D / 2 < 32 ? 32 : D / 2;
    constexpr uint32_t kColQ = 0, kColDS = kQC, kColS = kQC + 64, kColDP = kColS + 128,
                       kColAcc = kColDP + 128;
    static_assert(kColAcc + D <= kTmemCols, "TMEM columns");
    extern __shared__ uint8_t smem_raw[];
    const Setup su = setup_cta<G>(smem_raw, p);
    const Ctl& c = su.c;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int ntl = (sl.len + kT - 1) / kT;   // key tiles of the slice
    const int nkv = CAUSAL ? min(qt + 1, ntl) : ntl;
    const uint32_t tm = su.tmem;

    if (warp == kLoadWarp) {
        if (lane == 0)
            load_dq<D, MODE>(c, su.sbase, p, qt * kT, nkv, bh, sl);
        __syncwarp();
    } else if (warp == kMmaWarp) {
        constexpr uint32_t id_nt = make_idesc(kT, kT, false, F16);
        constexpr uint32_t id_tn = make_idesc(kT, D, true, F16);
        const uint64_t dDO = bdesc<D>(su.sbase, 16);
        const uint32_t ring = su.sbase + (uint32_t)G::kRingOff;
        auto kdesc = [&](uint32_t pos) {
            return bdesc<D>(ring + G::cyc_slot(pos) * (uint32_t)G::kTile, 16);
        };
        auto mdesc = [&](uint32_t pos) {
            return bdesc<D>(ring + G::cyc_slot(pos) * (uint32_t)G::kTile, (uint32_t)Rows<D>::kPanelBytes);
        };
        auto issue_s = [&](int j) -> bool {    // S = Q K_j^T (Q from TMEM)
            const uint32_t pos = 1u + 2u * (uint32_t)j;
            if (!wait_warp(c, G::ring_full(G::cyc_slot(pos)), G::cyc_par(pos), kRoleMma)) return false;
            ptx::tc_fence_after();
            mma_ts_nt<D>(tm + kColS, tm + kColQ, kdesc(pos), id_nt);
            ptx::mma_commit_elect(bar_addr(c, G::s_ready()));
            return true;
        };
        auto issue_dp = [&](int j) -> bool {   // dP = dO V_j^T; V_j is then done
            const uint32_t pos = 2u + 2u * (uint32_t)j;
            if (!wait_warp(c, G::ring_full(G::cyc_slot(pos)), G::cyc_par(pos), kRoleMma)) return false;
            ptx::tc_fence_after();
            mma_ss_nt<D>(tm + kColDP, dDO, kdesc(pos), id_nt);
            ptx::mma_commit_elect(bar_addr(c, G::dp_ready()));
            ptx::mma_commit_elect(bar_addr(c, G::ring_empty(G::cyc_slot(pos))));
            return true;
        };
        if (!wait_warp(c, G::fixed_full(), 0, kRoleMma)) goto mma_out;
        if (!wait_warp(c, G::q_ready(), 0, kRoleMma)) goto mma_out;
        ptx::tc_fence_after();
        if (!issue_s(0) || !issue_dp(0)) goto mma_out;
        for (int j = 0; j < nkv; ++j) {
            const uint32_t par = (uint32_t)j & 1u;
            if (!wait_warp(c, G::x_ready(), par, kRoleMma)) goto mma_out;    // S(j) read
            if (j + 1 < nkv && !issue_s(j + 1)) goto mma_out;
            if (!wait_warp(c, G::dp_free(), par, kRoleMma)) goto mma_out;    // dP(j) read
            if (j + 1 < nkv && !issue_dp(j + 1)) goto mma_out;
            if (!wait_warp(c, G::ds_ready(), par, kRoleMma)) goto mma_out;
            ptx::tc_fence_after();
            const uint32_t kpos = 1u + 2u * (uint32_t)j;
            mma_ts_tn<D, 32>(tm + kColAcc, tm + kColDS, mdesc(kpos), id_tn, j > 0);   // dQ += dS K_j
            ptx::mma_commit_elect(bar_addr(c, G::ds_free()));
            ptx::mma_commit_elect(bar_addr(c, G::ring_empty(G::cyc_slot(kpos))));
        }
        ptx::mma_commit_elect(bar_addr(c, G::done()));
    mma_out:
        ptx::mma_commit_elect(bar_addr(c, G::drain()));
        wait_drain(bar_addr(c, G::drain()), 0, c.limit);
        __syncwarp();
    } else {
        // elementwise: thread = query row r; this warp's 64 of the 128 keys of each tile
        const int quarter = warp & 3, ch = warp >> 2;
        const int r = quarter * 32 + lane;
        const int i = qt * kT + r;   // row within the slice
        const bool live = i < sl.len;
        const size_t vrow = sl.vec0 + (size_t)(live ? i : 0);                  // lse, delta
        const size_t erow = sl.row0 + (size_t)(live ? i : 0) * sl.stride;      // q, o, dout
        const float lse2 = live ? p.lse[vrow] * kLog2e : 0.0f;
        const int limit = CAUSAL ? min(i + 1, sl.len) : sl.len;    // visible keys: key < limit
        const uint32_t tl = (uint32_t)(quarter * 32) << 16;
        float* part = reinterpret_cast<float*>(smem_raw + (su.sbase - ptx::smem_addr(smem_raw)) + G::kVecOff);
        float dlt = 0.0f;
        if constexpr (D == 32) {
            // delta = sum_d dO * O for this row, both rows (64 bytes each) read from global
            // memory by the first warp of the lane quarter
            const bool mine = live && ch == 0;
            float acc = 0.0f;
            if (mine) {
                const uint4* orow = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.o) + erow);
                const uint4* drow = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.dout) + erow);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    const uint4 ov = __ldg(orow + cc), dv = __ldg(drow + cc);
                    const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        acc = fmaf(unpack_lo<F16>(ow[e]), unpack_lo<F16>(dw[e]), acc);
                        acc = fmaf(unpack_hi<F16>(ow[e]), unpack_hi<F16>(dw[e]), acc);
                    }
                }
            }
            part[ch * kT + r] = acc;
        } else {
            // delta = sum_d dO * O for this row: this warp's 64 columns from dO (the fixed
            // shared tile) and O (global; loaded first so the loads overlap the tile loads),
            // the two halves added through shared memory below
            const bool mine = live && ch < D / 64;
            uint4 ovs[8];
            if (mine) {
                const uint4* orow = reinterpret_cast<const uint4*>(
                    static_cast<const uint16_t*>(p.o) + erow + 64 * ch);
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) ovs[cc] = __ldg(orow + cc);
            }
            const bool okd = wait_warp(c, G::fixed_full(), 0, kRoleSoftmax);
            float acc = 0.0f;
            if (okd && mine) {
                const uint32_t drow = su.sbase + (uint32_t)ch * kPanelBytes + (uint32_t)r * 128u;
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const uint4 ov = ovs[cc];
                    const uint4 dv = ptx::ld_shared_v4(drow + (uint32_t)((cc ^ (r & 7)) * 16));
                    const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, dw[4] = {dv.x, dv.y, dv.z, dv.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        acc = fmaf(unpack_lo<F16>(ow[e]), unpack_lo<F16>(dw[e]), acc);
                        acc = fmaf(unpack_hi<F16>(ow[e]), unpack_hi<F16>(dw[e]), acc);
                    }
                }
            }
            part[ch * kT + r] = acc;
        }
        {
            // Q rows (streamed tile 0) into TMEM as 16-bit pairs (this warp: one 64-column
            // panel; at D = 32 the first warp of the lane quarter copies the 64-byte row
            // from global memory, zeros past N); the ring slot is then released
            const bool ok = wait_warp(c, G::ring_full(0), 0, kRoleSoftmax);
            if constexpr (D == 32) {
                if (ok && ch == 0) {
                    uint32_t w[16];
                    const uint4* qrow = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.q) + erow);
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        const uint4 v = live ? __ldg(qrow + cc) : make_uint4(0u, 0u, 0u, 0u);
                        w[4 * cc] = v.x; w[4 * cc + 1] = v.y; w[4 * cc + 2] = v.z; w[4 * cc + 3] = v.w;
                    }
                    ptx::tmem_st16(tm + tl + kColQ, w);
                    ptx::tmem_wait_st();
                }
            } else if (ok && ch < D / 64) {
                const uint32_t src = su.sbase + (uint32_t)G::kRingOff + (uint32_t)ch * kPanelBytes +
                                     (uint32_t)r * 128u;
                uint32_t w[32];
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const uint4 v = ptx::ld_shared_v4(src + (uint32_t)((cc ^ (r & 7)) * 16));
                    w[4 * cc] = v.x; w[4 * cc + 1] = v.y; w[4 * cc + 2] = v.z; w[4 * cc + 3] = v.w;
                }
                ptx::tmem_st32(tm + tl + kColQ + 32u * (uint32_t)ch, w);
                ptx::tmem_wait_st();
            }
            ptx::tc_fence_before();
            if (!ew_barrier_and(ok)) goto ew_out;
            if (threadIdx.x == 0) {
                ptx::mbar_arrive(bar_addr(c, G::ring_empty(0)));
                ptx::mbar_arrive(bar_addr(c, G::q_ready()));
            }
            // both partial sums are published by the barrier above
            dlt = part[r] + part[kT + r];
            if (live && ch == 0) p.delta[vrow] = dlt;   // for the dK/dV kernel
        }
        for (int j = 0; j < nkv; ++j) {
            const uint32_t par = (uint32_t)j & 1u;
            const int key0 = j * kT + 64 * ch;
            const bool mask = __any_sync(0xFFFFFFFFu, key0 + 64 > limit);
            float pr[64];
            {   // phase a: P from S
                if (!wait_warp(c, G::s_ready(), par, kRoleSoftmax)) goto ew_out;
                ptx::tc_fence_after();
                uint32_t sv[64];
                ptx::tmem_ld64_wait(tm + tl + kColS + 64u * (uint32_t)ch, sv);
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar_addr(c, G::x_ready()));   // S may be overwritten
#pragma unroll
                for (int cc = 0; cc < 64; cc += 2) {
                    float x0, x1;
                    ptx::fma2(x0, x1, u2f(sv[cc]), u2f(sv[cc + 1]), p.scale_log2, -lse2);
                    pr[cc] = ptx::ex2(x0);
                    pr[cc + 1] = ptx::ex2(x1);
                }
                if (mask) {
#pragma unroll
                    for (int cc = 0; cc < 64; ++cc)
                        if (key0 + cc >= limit) pr[cc] = 0.0f;
                }
            }
            {   // phase b: dS = P (dP - delta), 16-bit, into this warp's half of the dS region
                if (!wait_warp(c, G::dp_ready(), par, kRoleSoftmax)) goto ew_out;
                ptx::tc_fence_after();
                uint32_t dp[64];
                ptx::tmem_ld64_wait(tm + tl + kColDP + 64u * (uint32_t)ch, dp);
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar_addr(c, G::dp_free()));   // dP may be overwritten
                uint32_t pk[32];
#pragma unroll
                for (int cc = 0; cc < 64; cc += 2) {
                    float d0 = u2f(dp[cc]), d1 = u2f(dp[cc + 1]);
                    ptx::add2(d0, d1, -dlt, -dlt);
                    ptx::mul2(d0, d1, pr[cc], pr[cc + 1]);
                    pk[cc >> 1] = pack2<F16>(d0, d1);
                }
                // the previous dQ product must have read the dS region
                if (j > 0 && !wait_warp(c, G::ds_free(), par ^ 1u, kRoleSoftmax)) goto ew_out;
                ptx::tc_fence_after();
                ptx::tmem_st32(tm + tl + kColDS + 32u * (uint32_t)ch, pk);
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar_addr(c, G::ds_ready()));
            }
        }
        if (!wait_warp(c, G::done(), 0, kRoleSoftmax)) goto ew_out;
        ptx::tc_fence_after();
        if constexpr (D == 32) {   // the first warp of each lane quarter stores dQ
            if (ch == 0)
                store_rows32<F16>(tm + tl + kColAcc, p.scale,
                                  su.sbase + (uint32_t)G::kStageOff + (uint32_t)warp * 4096u,
                                  reinterpret_cast<uint16_t*>(p.dq) + sl.row0, sl.stride,
                                  qt * kT + quarter * 32, sl.len, lane);
        } else if (ch < D / 64) {   // one 64-column panel of dQ per warp
            store_rows<F16>(tm + tl + kColAcc + 64u * (uint32_t)ch, p.scale,
                            su.sbase + (uint32_t)G::kStageOff + (uint32_t)warp * 4096u,
                            reinterpret_cast<uint16_t*>(p.dq) + sl.row0 + 64 * ch, sl.stride,
                            qt * kT + quarter * 32, sl.len, lane);
        }
    ew_out:;
    }
    teardown_cta(su);
}

// ----------------------------------------------------------------- dK, dV kernel
// TMEM columns: S^T [0, 128), dP^T [128, 256), dV [256, 256+D), dK [256+D, 256+2D)
// (D = 32: dK at 288, a multiple of 32 columns as every other region).
// Shared memory: K, V fixed; ring A_s = Q_i, B_s = dO_i for query tile i = i0 + s.
template <int D, bool CAUSAL, bool F16, int MODE>
__global__ void __launch_bounds__(kThreads, 1) bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
    using G = GeoDkdv<D>;
    // key tiles past a (shorter packed) sequence have nothing to do: the whole CTA leaves
    const int bh = blockIdx.x / p.ntiles, kt = blockIdx.x % p.ntiles;
    const Slice sl = slice_at<MODE, D>(p, bh);
    if (kt * kT >= sl.len) return;
    constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
    extern __shared__ uint8_t smem_raw[];
    const Setup su = setup_cta<G>(smem_raw, p);
    const Ctl& c = su.c;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int ntl = (sl.len + kT - 1) / kT;         // query tiles of the slice
    const int i0 = CAUSAL ? kt : 0;                 // first query tile that sees this key tile
    const int nq = ntl - i0;
    const uint32_t tm = su.tmem;

    if (warp == kLoadWarp) {
        if (lane == 0)
            load_pairs<D, MODE>(c, su.sbase, &p.tmap_k, &p.tmap_v, kt * kT, &p.tmap_q, &p.tmap_do,
                                i0 * kT, nq, bh, sl, p.inject_stall == 1 && blockIdx.x == 0);
        __syncwarp();
    } else if (warp == kMmaWarp) {
        constexpr uint32_t id_nt = make_idesc(kT, kT, false, F16);
        constexpr uint32_t id_tn = make_idesc(kT, D, true, F16);
        const uint64_t dK = bdesc<D>(su.sbase, 16);
        const uint64_t dV = bdesc<D>(su.sbase + (uint32_t)G::kTile, 16);
        const uint32_t ring = su.sbase + (uint32_t)G::kRingOff;
        auto kdesc = [&](uint32_t slot) { return bdesc<D>(ring + slot * (uint32_t)G::kTile, 16); };
        auto mdesc = [&](uint32_t slot) {
            return bdesc<D>(ring + slot * (uint32_t)G::kTile, (uint32_t)Rows<D>::kPanelBytes);
        };
        auto issue_st = [&](int s) -> bool {    // S^T = K Q_i^T
            if (!wait_warp(c, G::ring_full(slot_a(s)), slot_par(s), kRoleMma)) return false;
            ptx::tc_fence_after();
            mma_ss_nt<D>(tm + kColS, dK, kdesc(slot_a(s)), id_nt);
            ptx::mma_commit_elect(bar_addr(c, G::s_ready()));
            return true;
        };
        auto issue_dpt = [&](int s) -> bool {   // dP^T = V dO_i^T
            if (!wait_warp(c, G::ring_full(slot_b(s)), slot_par(s), kRoleMma)) return false;
            ptx::tc_fence_after();
            mma_ss_nt<D>(tm + kColDP, dV, kdesc(slot_b(s)), id_nt);
            ptx::mma_commit_elect(bar_addr(c, G::dp_ready()));
            return true;
        };
        if (!wait_warp(c, G::fixed_full(), 0, kRoleMma)) goto mma_out;
        if (!issue_st(0) || !issue_dpt(0)) goto mma_out;
        for (int s = 0; s < nq; ++s) {
            const uint32_t par = (uint32_t)s & 1u;
            if (!wait_warp(c, G::x_ready(), par, kRoleMma)) goto mma_out;   // P^T stored
            ptx::tc_fence_after();
            mma_ts_tn<D, 64>(tm + kColDV, tm + kColS, mdesc(slot_b(s)), id_tn, s > 0);   // dV += P^T dO_i
            ptx::mma_commit_elect(bar_addr(c, G::ring_empty(slot_b(s))));
            if (s + 1 < nq && !issue_st(s + 1)) goto mma_out;
            if (!wait_warp(c, G::ds_ready(), par, kRoleMma)) goto mma_out;
            ptx::tc_fence_after();
            mma_ts_tn<D, 64>(tm + kColDK, tm + kColDP, mdesc(slot_a(s)), id_tn, s > 0);   // dK += dS^T Q_i
            ptx::mma_commit_elect(bar_addr(c, G::ring_empty(slot_a(s))));
            if (s + 1 < nq && !issue_dpt(s + 1)) goto mma_out;
        }
        ptx::mma_commit_elect(bar_addr(c, G::done()));
    mma_out:
        ptx::mma_commit_elect(bar_addr(c, G::drain()));
        wait_drain(bar_addr(c, G::drain()), 0, c.limit);
        __syncwarp();
    } else {
        // elementwise: thread = key row r; this warp's 64 of the 128 queries of each tile
        const int quarter = warp & 3, ch = warp >> 2;
        const int r = quarter * 32 + lane;
        const int key = kt * kT + r;
        const uint32_t tl = (uint32_t)(quarter * 32) << 16;
        // Per-column LSE (log2 units) and delta of this warp's 64 queries of each query tile,
        // staged in the warp's own area of shared memory, so that no barrier across warps is
        // needed: lane l holds queries l and l + 32 (k = 0, 1: LSE; k = 2, 3: delta), fetched
        // one step ahead into registers.
        float* vw = reinterpret_cast<float*>(smem_raw + (su.sbase - ptx::smem_addr(smem_raw)) + G::kVecOff) +
                    warp * 256;
        auto fetch = [&](int s, int k) -> float {
            const int q = (i0 + s) * kT + 64 * ch + lane + 32 * (k & 1);
            const bool ok = s < nq && q < sl.len;
            if (k < 2) return ok ? p.lse[sl.vec0 + q] * kLog2e : INFINITY;   // p = 0 past the end
            return ok ? p.delta[sl.vec0 + q] : 0.0f;
        };
        float nx[4] = {fetch(0, 0), fetch(0, 1), fetch(0, 2), fetch(0, 3)};
        for (int s = 0; s < nq; ++s) {
            const uint32_t par = (uint32_t)s & 1u;
            float* vl = vw + par * 128;   // [0, 64): LSE * log2 e, [64, 128): delta
            vl[lane] = nx[0];
            vl[lane + 32] = nx[1];
            vl[64 + lane] = nx[2];
            vl[96 + lane] = nx[3];
            __syncwarp();
            if (!wait_warp(c, G::s_ready(), par, kRoleSoftmax)) goto ew_out;
            ptx::tc_fence_after();
#pragma unroll
            for (int k = 0; k < 4; ++k) nx[k] = fetch(s + 1, k);
            const int qbase = (i0 + s) * kT + 64 * ch;
            const bool diag = CAUSAL && (i0 + s == kt);   // queries before this key are masked
            const float4* l4 = reinterpret_cast<const float4*>(vl);
            const float4* d4 = reinterpret_cast<const float4*>(vl + 64);
            float pr[64];
            {   // phase a: P^T from S^T, 16-bit over this warp's S^T columns
                const uint32_t ts = tm + tl + kColS + 64u * (uint32_t)ch;
                uint32_t sv[64];
                ptx::tmem_ld64_wait(ts, sv);
#pragma unroll
                for (int c4 = 0; c4 < 16; ++c4) {
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
                if (diag) {
#pragma unroll
                    for (int cc = 0; cc < 64; ++cc)
                        if (qbase + cc < key) pr[cc] = 0.0f;
                }
                uint32_t pk[32];
#pragma unroll
                for (int cc = 0; cc < 64; cc += 2) pk[cc >> 1] = pack2<F16>(pr[cc], pr[cc + 1]);
                ptx::tmem_st32(ts, pk);
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar_addr(c, G::x_ready()));
            }
            {   // phase b: dS^T = P^T (dP^T - delta), 16-bit over this warp's dP^T columns
                if (!wait_warp(c, G::dp_ready(), par, kRoleSoftmax)) goto ew_out;
                ptx::tc_fence_after();
                const uint32_t tp = tm + tl + kColDP + 64u * (uint32_t)ch;
                uint32_t dp[64];
                ptx::tmem_ld64_wait(tp, dp);
                uint32_t pk[32];
#pragma unroll
                for (int c4 = 0; c4 < 16; ++c4) {
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
                ptx::tmem_st32(tp, pk);
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar_addr(c, G::ds_ready()));
            }
        }
        if (!wait_warp(c, G::done(), 0, kRoleSoftmax)) goto ew_out;
        ptx::tc_fence_after();
        if constexpr (D == 32) {   // dV by the first, dK by the second warp of each quarter
            const uint32_t stage = su.sbase + (uint32_t)G::kStageOff + (uint32_t)warp * 4096u;
            const int row0 = kt * kT + quarter * 32;
            if (ch == 0)
                store_rows32<F16>(tm + tl + kColDV, 1.0f, stage,
                                  reinterpret_cast<uint16_t*>(p.dv) + sl.row0, sl.stride, row0, sl.len, lane);
            else
                store_rows32<F16>(tm + tl + kColDK, p.scale, stage,
                                  reinterpret_cast<uint16_t*>(p.dk) + sl.row0, sl.stride, row0, sl.len, lane);
        } else if (ch < D / 64) {   // one 64-column panel of dV and of dK per warp
            const uint32_t stage = su.sbase + (uint32_t)G::kStageOff + (uint32_t)warp * 4096u;
            const int row0 = kt * kT + quarter * 32;
            const size_t off = sl.row0 + 64 * ch;
            store_rows<F16>(tm + tl + kColDV + 64u * (uint32_t)ch, 1.0f, stage,
                            reinterpret_cast<uint16_t*>(p.dv) + off, sl.stride, row0, sl.len, lane);
            store_rows<F16>(tm + tl + kColDK + 64u * (uint32_t)ch, p.scale, stage,
                            reinterpret_cast<uint16_t*>(p.dk) + off, sl.stride, row0, sl.len, lane);
        }
    ew_out:;
    }
    teardown_cta(su);
}

template <int D, bool CAUSAL, bool F16, int MODE>
cudaError_t prepare_mode() {
    cudaError_t e = cudaFuncSetAttribute(bwd_dq_kernel<D, CAUSAL, F16, MODE>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, GeoDq<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(bwd_dkdv_kernel<D, CAUSAL, F16, MODE>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, GeoDkdv<D>::kSmemBytes);
}

template <int D, bool CAUSAL, bool F16>
cudaError_t prepare3() {
    const cudaError_t e = prepare_mode<D, CAUSAL, F16, 0>();
    return e != cudaSuccess ? e : prepare_mode<D, CAUSAL, F16, 1>();
}

template <int D, bool CAUSAL, bool F16, int MODE>
cudaError_t launch_mode(const BwdParams& p, unsigned ctas, cudaStream_t stream) {
    bwd_dq_kernel<D, CAUSAL, F16, MODE><<<ctas, kThreads, GeoDq<D>::kSmemBytes, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_dkdv_kernel<D, CAUSAL, F16, MODE><<<ctas, kThreads, GeoDkdv<D>::kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

template <int D, bool CAUSAL, bool F16>
cudaError_t launch3(const BwdParams& p, int bh, cudaStream_t stream) {
    const long long ctas = (long long)bh * p.ntiles;
    if (ctas > 0x7FFFFFFFLL) return cudaErrorInvalidConfiguration;
    return p.layout == 0 ? launch_mode<D, CAUSAL, F16, 0>(p, (unsigned)ctas, stream)
                         : launch_mode<D, CAUSAL, F16, 1>(p, (unsigned)ctas, stream);
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

cudaError_t bwd_prepare(int D, bool causal, bool f16) {
    if (D == 32) return dispatch<32>(causal, f16, true, nullptr, 0, nullptr);
    return D == 64 ? dispatch<64>(causal, f16, true, nullptr, 0, nullptr)
                   : dispatch<128>(causal, f16, true, nullptr, 0, nullptr);
}

cudaError_t bwd_launch(int D, bool causal, bool f16, const BwdParams& p, int bh, cudaStream_t stream) {
    if (D == 32) return dispatch<32>(causal, f16, false, &p, bh, stream);
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
