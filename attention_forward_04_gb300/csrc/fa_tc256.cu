// fa_tc256.cu -- attention forward for head dimension D = 256 on the GB300 tensor cores.
//
// Same computation as the D = 64/128 kernel ("08 · FlashAttention" §二: tiles plus the
// online (m, l, O) softmax; "KingOfEgg" §1.1 for the definition), with a layout sized for
// D = 256: the two-query-tile schedule of the smaller head dimensions would need 2 x 256
// TMEM columns of O alone.  Here a persistent CTA (one per SM) takes one 128-row query tile
// at a time and owns all 512 columns:
//     Q [0, 128)       the query tile as 16-bit pairs (A operand of S = Q K^T); e4m3
//                      quadruples fill [0, 64)
//     S/P buffer 0     [128, 192)   64 keys: fp32 scores, then P (16-bit pairs, or e4m3
//                                   quadruples) over them
//     S/P buffer 1     [192, 256)
//     O                [256, 512)   fp32 accumulator
// Element types (ET): 0 bf16, 1 fp16, 2 e4m3 (kind::f8f6f4 products, P rounded to e4m3,
// O in bf16 times V's dequantisation factor, as in the smaller head dimensions).
// Keys advance 64 at a time.  S(j+2) is issued right after O += P(j) V_j, so the softmax
// of step j+1 overlaps both products.  Every product reads only one operand from shared
// memory (K_j or V_j), which keeps shared-memory bandwidth below the tensor rate.
// Warps: 0-3 softmax (thread = query row = TMEM lane), 4 MMA issuer, 5 TMA loader.
// Every wait is bounded; a wait that runs out sets this unit's status word.
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

__device__ unsigned int g_status[4];

constexpr int D = 256;
constexpr int kBM = 128;                       // query rows per CTA
constexpr int kBN = 64;                        // keys per step
constexpr int kThreads = 192;
constexpr int kMmaWarp = 4, kLoadWarp = 5;
constexpr int kSlots = 6;
constexpr int kPanel64 = 64 * 128;             // 64 rows x 128 bytes (64 16-bit or 128 e4m3 columns)
constexpr int kTile = 4 * kPanel64;            // ring slot: a 64 x 256 tile (32 KB at 16 bits)
constexpr int kStageOff = kSlots * kTile;      // 4 warps x 4 KB epilogue staging
constexpr int kBarOff = kStageOff + 4 * 4096;
// barriers: ring_full[6], ring_empty[6], s_full[2], p_full[2], o_done, q_ready, drain
constexpr int kNumBars = 2 * kSlots + 7;
constexpr int kMiscOff = kBarOff + kNumBars * 8;
constexpr int kSmemBytes = kMiscOff + 16 + 1024;
static_assert(kSmemBytes <= 232448, "shared memory");
constexpr uint32_t kColQ = 0, kColS = 128, kColO = 256, kTmemCols = 512;

constexpr int b_ring_full(uint32_t pos) { return (int)(pos % kSlots); }
constexpr int b_ring_empty(uint32_t pos) { return kSlots + (int)(pos % kSlots); }
constexpr int b_s_full(uint32_t b) { return 2 * kSlots + (int)b; }
constexpr int b_p_full(uint32_t b) { return 2 * kSlots + 2 + (int)b; }
constexpr int b_o_done() { return 2 * kSlots + 4; }
constexpr int b_q_ready() { return 2 * kSlots + 5; }
constexpr int b_drain() { return 2 * kSlots + 6; }
__device__ __forceinline__ uint32_t ring_par(uint32_t pos) { return (pos / kSlots) & 1u; }

// Streamed tiles of an item, from its first ring position: 0 and 1 are the two 64-row
// halves of the Q tile, then K_j = 2 + 2j and V_j = 3 + 2j.

// The reference is raised when a step's maximum exceeds it by more than kRescaleLog2 = 8
// log2 units (P stays below 2^8); otherwise the stale reference is kept, which the final
// division cancels.  For bf16 P (8 significant bits) a stale reference alone would leave a
// row's largest P rounded (2^x for fractional x) while the row sum kept the unrounded
// value; so at bf16 O is divided by a second row sum, of the bf16-rounded P that O += P V
// multiplies, and the rounding of P cancels in the quotient (the unrounded sum still gives
// the LSE).  A rescale moves 256 columns of O through TMEM here, four times the work per
// key of the smaller head dimensions, which take the literal reading for bf16 instead.
template <int ET> struct Lazy {
    static constexpr float kRescaleLog2 = 8.0f;
    static constexpr bool kRoundedSum = ET == 0;
};

// Per element type: bytes per value, 128-byte panels per 256-value row, bytes of a tile.
template <int ET> struct Elem {
    static constexpr int kBytes = ET == 2 ? 1 : 2;
    static constexpr int kPanels = D * kBytes / 128;
    static constexpr int kTileBytes = kPanels * kPanel64;
};

// Instruction descriptor: kind::f16 (bf16 or fp16), or kind::f8f6f4 with both operands
// e4m3 (format code 0); fp32 accumulator, A K-major.
template <int ET>
__host__ __device__ constexpr uint32_t idesc_of(int M, int N, bool b_mn_major) {
    return ET == 2 ? ((1u << 4) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
                      ((uint32_t)(M >> 4) << 24))
                   : make_idesc(M, N, b_mn_major, ET == 1);
}

// Named barrier 1 over the 128 softmax threads that also ANDs a predicate, so a stop
// decision is common to the four warps.
__device__ __forceinline__ bool sm_barrier_and(bool ok) {
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

// One 64-key step of one row: running-max update (raised when the step's maximum exceeds
// it by more than kRescaleLog2 log2 units), p = 2^(s * sl2 - m), row sum l_run (of the fp32
// values), and P packed to 16-bit pairs in pk[0, 32), or to e4m3 quadruples in pk[0, 16);
// at bf16 also l_rnd, the row sum of the packed (rounded) values.  Keys at or past `limit`
// count as absent (MASK).  Eight independent max chains and four paired sum chains keep
// the dependent depth short.  Returns the factor the row's O and sums must be scaled by.
template <bool MASK, int ET>
__device__ __forceinline__ float softmax_step(const uint32_t (&s)[64], int key0, int limit,
                                              float sl2, float& m_run, float& l_run, float& l_rnd,
                                              uint32_t (&pk)[32]) {
    float mx[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
#pragma unroll
    for (int cc = 0; cc < 64; cc += 2) {
        float a = u2f(s[cc]), b = u2f(s[cc + 1]);
        if (MASK) {
            if (key0 + cc >= limit) a = -INFINITY;
            if (key0 + cc + 1 >= limit) b = -INFINITY;
        }
        mx[(cc >> 1) & 7] = ptx::max3(mx[(cc >> 1) & 7], a, b);
    }
    const float mt = fmaxf(ptx::max3(mx[0], mx[1], mx[2]),
                           fmaxf(ptx::max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl2;
    float alpha = 1.0f;
    if (mt > m_run + Lazy<ET>::kRescaleLog2) {
        alpha = ptx::ex2(m_run - mt);   // 0 on the first step (m_run = -inf)
        m_run = mt;
    }
    const float neg_m = -m_run;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float accr[4] = {0.f, 0.f, 0.f, 0.f};   // bf16: sums of the rounded values
#pragma unroll
    for (int cc = 0; cc < 64; cc += 4) {
        float x[4], pr[4];
        ptx::fma2(x[0], x[1], u2f(s[cc]), u2f(s[cc + 1]), sl2, neg_m);
        ptx::fma2(x[2], x[3], u2f(s[cc + 2]), u2f(s[cc + 3]), sl2, neg_m);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            pr[e] = ptx::ex2(x[e]);
            if (MASK && key0 + cc + e >= limit) pr[e] = 0.0f;
        }
        const int a = ((cc >> 1) & 3) * 2;   // pairs (cc, cc+1) and (cc+2, cc+3): chains a, a+2
        ptx::add2(acc[a], acc[a + 1], pr[0], pr[1]);
        ptx::add2(acc[a + 2], acc[a + 3], pr[2], pr[3]);
        if constexpr (ET == 2) {
            pk[cc >> 2] = pack4_e4m3(pr[0], pr[1], pr[2], pr[3]);
        } else {
            pk[cc >> 1] = pack2<ET == 1>(pr[0], pr[1]);
            pk[(cc >> 1) + 1] = pack2<ET == 1>(pr[2], pr[3]);
            if constexpr (Lazy<ET>::kRoundedSum) {
                const int ar = ((cc >> 2) & 1) * 2;
                ptx::add2(accr[ar], accr[ar + 1], unpack_lo<false>(pk[cc >> 1]), unpack_hi<false>(pk[cc >> 1]));
                ptx::add2(accr[ar], accr[ar + 1], unpack_lo<false>(pk[(cc >> 1) + 1]),
                          unpack_hi<false>(pk[(cc >> 1) + 1]));
            }
        }
    }
    const float sum = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
    l_run = l_run * alpha + sum;
    if constexpr (Lazy<ET>::kRoundedSum) l_rnd = l_rnd * alpha + ((accr[0] + accr[1]) + (accr[2] + accr[3]));
    return alpha;
}

struct Work {
    int bh, qt, nkv;
    int len;    // sequence length of the slice
    int tok0;   // token-major layouts: token of row 0 of the slice
    int h;      // head
};

// Length and first token of slice bh.  MODE 0, [B, H, N, D]: every slice has N rows.
// MODE 1, token-major [tokens, H, D]: fixed length N (tokens b*N..), or packed sequences
// with offsets cu_seqlens, clamped to [0, total] and lengths to the declared maximum, so
// malformed offsets cannot move an access out of bounds.
template <int MODE>
__device__ __forceinline__ void slice_of(const TcParams& p, int bh, int& len, int& tok0) {
    if (MODE == 0) {
        len = p.n;
        tok0 = 0;
        return;
    }
    const int b = bh / p.heads;
    if (p.cu_seqlens != nullptr) {
        int s0 = __ldg(p.cu_seqlens + b), s1 = __ldg(p.cu_seqlens + b + 1);
        s0 = min(max(s0, 0), p.total);
        s1 = min(max(s1, s0), p.total);
        len = min(s1 - s0, p.n);
        tok0 = s0;
    } else {
        len = p.n;
        tok0 = b * p.n;
    }
}

// Work units of the persistent schedule.  Non-causal: one 128-row query tile per unit,
// slice-major, so the CTAs running together share a few slices' K and V through L2.
// Causal: unit (slice, q) holds tiles ntiles-1-q and q of the slice (one tile when they
// coincide), so units cost about the same; still slice-major.  Units are laid out for
// slices of N (the maximum) rows; a shorter packed sequence leaves some of its units with
// fewer items or none.
__device__ __forceinline__ int ntiles_of(int n) { return (n + kBM - 1) / kBM; }

template <bool CAUSAL, int MODE>
__device__ __forceinline__ int unit_items(const TcParams& p, int u) {
    const int nt = ntiles_of(p.n);
    const int per_slice = CAUSAL ? (nt + 1) / 2 : nt;
    const int q = u % per_slice;
    int len = p.n, tok0 = 0;
    if (MODE == 1) slice_of<MODE>(p, u / per_slice, len, tok0);
    const int ntl = ntiles_of(len);   // tiles of this slice
    if (!CAUSAL) return q < ntl ? 1 : 0;
    if (q >= (ntl + 1) / 2) return 0;
    return (ntl - 1 - q != q) ? 2 : 1;
}

template <bool CAUSAL, int MODE>
__device__ __forceinline__ Work unit_item(const TcParams& p, int u, int sub) {
    const int nt = ntiles_of(p.n);
    const int per_slice = CAUSAL ? (nt + 1) / 2 : nt;
    Work w;
    w.bh = u / per_slice;
    const int q = u % per_slice;
    slice_of<MODE>(p, w.bh, w.len, w.tok0);
    w.h = MODE == 1 ? w.bh % p.heads : 0;
    const int ntl = ntiles_of(w.len);
    w.qt = CAUSAL ? (sub == 0 ? ntl - 1 - q : q) : q;
    const int keys = CAUSAL ? min(w.len, (w.qt + 1) * kBM) : w.len;
    w.nkv = (keys + kBN - 1) / kBN;
    return w;
}

// Every role walks the same items in the same order and keeps running counters: ring
// position (2 Q halves, then K_j, V_j per item), global step index g (S/P buffer g % 2, its
// (g / 2)-th use), products of O done, and items.
template <bool CAUSAL, int ET, int MODE>
__global__ void __launch_bounds__(kThreads, 1) fa_tc256_kernel(const __grid_constant__ TcParams p) {
    constexpr int EB = Elem<ET>::kBytes;
    constexpr int kPanels = Elem<ET>::kPanels;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = ptx::smem_addr(smem);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kMiscOff);
    Ctl c;
    c.bars = sbase + (uint32_t)kBarOff;
    c.abort = reinterpret_cast<volatile int*>(smem + kMiscOff + 4);
    c.limit = p.wait_limit;
    c.status = g_status;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kSlots; ++s) {
            ptx::mbar_init(bar_addr(c, b_ring_full(s)), 1);
            ptx::mbar_init(bar_addr(c, b_ring_empty(s)), 1);
        }
        for (uint32_t b = 0; b < 2; ++b) {
            ptx::mbar_init(bar_addr(c, b_s_full(b)), 1);
            ptx::mbar_init(bar_addr(c, b_p_full(b)), 128);
        }
        ptx::mbar_init(bar_addr(c, b_o_done()), 1);
        ptx::mbar_init(bar_addr(c, b_q_ready()), 1);
        ptx::mbar_init(bar_addr(c, b_drain()), 1);
        *c.abort = 0;
        ptx::fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tm = *tmem_slot;
    const uint32_t ring = sbase;

    if (warp == kLoadWarp) {
        if (lane == 0) {
            uint32_t pos = 0;
            for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
                const int nsub = unit_items<CAUSAL, MODE>(p, u);
                for (int sub = 0; sub < nsub; ++sub) {
                    const Work w = unit_item<CAUSAL, MODE>(p, u, sub);
                    const uint32_t count = 2u + 2u * (uint32_t)w.nkv;
                    for (uint32_t k = 0; k < count; ++k, ++pos) {
                        if (!wait(c, b_ring_empty(pos), ring_par(pos) ^ 1u, kRoleLoad)) goto load_out;
                        const uint32_t bar = bar_addr(c, b_ring_full(pos));
                        const CUtensorMap* map = k < 2 ? &p.tmap_q : ((k & 1u) ? &p.tmap_v : &p.tmap_k);
                        const int row = k < 2 ? w.qt * kBM + (int)k * 64 : (int)((k - 2u) >> 1) * kBN;
                        const uint32_t dst = ring + (pos % kSlots) * (uint32_t)kTile;
                        ptx::mbar_arrive_expect_tx(bar, (uint32_t)Elem<ET>::kTileBytes);
#pragma unroll
                        for (int pc = 0; pc < kPanels; ++pc) {
                            // x = the panel's first column: 64 or 128 values, 128 bytes
                            if (MODE == 0)
                                ptx::tma_load_3d(dst + (uint32_t)pc * kPanel64, map, bar, pc * (128 / EB), row,
                                                 w.bh);
                            else   // token-major: dims {D, H, tokens}
                                ptx::tma_load_3d(dst + (uint32_t)pc * kPanel64, map, bar, pc * (128 / EB), w.h,
                                                 w.tok0 + row);
                        }
                    }
                }
            }
        load_out:
            for (uint32_t i = (pos > (uint32_t)kSlots ? pos - kSlots : 0u); i < pos; ++i)
                wait_drain(bar_addr(c, b_ring_full(i)), ring_par(i), c.limit);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        constexpr uint32_t id_qk = idesc_of<ET>(kBM, kBN, false);
        constexpr uint32_t id_pv = idesc_of<ET>(kBM, D, true);
        constexpr int kKeys = 32 / EB;   // keys per K step of O += P V (32 bytes of P per row)
        auto kdesc = [&](uint32_t pos) {   // K-major 64 x 256 tile (panels of 128 bytes)
            return sw128_desc(ring + (pos % kSlots) * (uint32_t)kTile, 16, 1024);
        };
        auto vdesc = [&](uint32_t pos) {   // the same tile read as the MN-major operand
            return sw128_desc(ring + (pos % kSlots) * (uint32_t)kTile, kPanel64, 1024);
        };
        // S(step g) = Q K^T into buffer g % 2 from the tile at ring position pos; K is then done
        auto issue_s = [&](uint32_t g, uint32_t pos) -> bool {
            const uint32_t b = g & 1u;
            if (!wait_warp(c, b_ring_full(pos), ring_par(pos), kRoleMma)) return false;
            ptx::tc_fence_after();
            const uint64_t kd = kdesc(pos);
            // K steps of 32 bytes: Q's 8 TMEM columns, four steps per 128-byte panel of K
#pragma unroll
            for (int kk = 0; kk < D * EB / 32; ++kk) {
                const uint64_t kb = kd + (((uint64_t)(kk / 4) * kPanel64 + (uint64_t)(kk % 4) * 32u) >> 4);
                if constexpr (ET == 2)
                    ptx::mma_ts_f8_elect(tm + kColS + 64u * b, tm + kColQ + (uint32_t)kk * 8u, kb, id_qk,
                                         kk > 0 ? 1u : 0u);
                else
                    ptx::mma_ts_elect(tm + kColS + 64u * b, tm + kColQ + (uint32_t)kk * 8u, kb, id_qk,
                                      kk > 0 ? 1u : 0u);
            }
            ptx::mma_commit_elect(bar_addr(c, b_s_full(b)));
            ptx::mma_commit_elect(bar_addr(c, b_ring_empty(pos)));
            return true;
        };
        uint32_t g = 0, items = 0, base = 0;
        for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
            const int nsub = unit_items<CAUSAL, MODE>(p, u);
            for (int sub = 0; sub < nsub; ++sub) {
                const Work w = unit_item<CAUSAL, MODE>(p, u, sub);
                if (!wait_warp(c, b_q_ready(), items & 1u, kRoleMma)) goto mma_out;
                ++items;
                ptx::tc_fence_after();
                if (!issue_s(g, base + 2u)) goto mma_out;
                if (w.nkv > 1 && !issue_s(g + 1u, base + 4u)) goto mma_out;
                if (!wait_warp(c, b_ring_full(base + 3u), ring_par(base + 3u), kRoleMma)) goto mma_out;
                for (int j = 0; j < w.nkv; ++j) {
                    const uint32_t gj = g + (uint32_t)j, b = gj & 1u;
                    const uint32_t vpos = base + 3u + 2u * (uint32_t)j;
                    // V_j is resident (waited for before S(j+1) was issued): between the last
                    // product of S(j+1) entering the tensor queue and the first of O += P V,
                    // only the hand-over of P is awaited.
                    if (!wait_warp(c, b_p_full(b), (gj >> 1) & 1u, kRoleMma)) goto mma_out;
                    ptx::tc_fence_after();
                    const uint64_t vd = vdesc(vpos);
                    // K steps of kKeys keys: P's 8 TMEM columns, kKeys rows of 128 bytes of V
#pragma unroll
                    for (int kk = 0; kk < kBN / kKeys; ++kk) {
                        const uint64_t vb = vd + (uint64_t)((kk * kKeys * 128) >> 4);
                        const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
                        if constexpr (ET == 2)
                            ptx::mma_ts_f8_elect(tm + kColO, tm + kColS + 64u * b + (uint32_t)kk * 8u, vb,
                                                 id_pv, acc);
                        else
                            ptx::mma_ts_elect(tm + kColO, tm + kColS + 64u * b + (uint32_t)kk * 8u, vb,
                                              id_pv, acc);
                    }
                    ptx::mma_commit_elect(bar_addr(c, b_o_done()));
                    ptx::mma_commit_elect(bar_addr(c, b_ring_empty(vpos)));
                    if (j + 1 < w.nkv && !wait_warp(c, b_ring_full(vpos + 2u), ring_par(vpos + 2u), kRoleMma))
                        goto mma_out;
                    if (j + 2 < w.nkv && !issue_s(gj + 2u, base + 2u + 2u * (uint32_t)(j + 2))) goto mma_out;
                }
                g += (uint32_t)w.nkv;
                base += 2u + 2u * (uint32_t)w.nkv;
            }
        }
    mma_out:
        ptx::mma_commit_elect(bar_addr(c, b_drain()));
        wait_drain(bar_addr(c, b_drain()), 0, c.limit);
        __syncwarp();
    } else {
        // softmax: thread = query row r (TMEM lane r)
        const int r = warp * 32 + lane;
        const uint32_t tl = (uint32_t)(warp * 32) << 16;
        const float sl2 = p.scale_log2;
        const uint32_t stage = sbase + (uint32_t)kStageOff + (uint32_t)warp * 4096u;
        // Q row r of the query tile at ring positions qpos, qpos + 1 into TMEM as 16-bit pairs
        // (e4m3 quadruples); the two ring slots are then released and the MMA issuer told.
        // No product that reads the previous Q is pending: the caller has seen the last of
        // them complete.
        auto write_q = [&](uint32_t qpos) -> bool {
            const bool ok = wait_warp(c, b_ring_full(qpos), ring_par(qpos), kRoleSoftmax) &&
                            wait_warp(c, b_ring_full(qpos + 1u), ring_par(qpos + 1u), kRoleSoftmax);
            if (ok) {
                const int lr = r & 63;
                const uint32_t src = ring + ((qpos + (uint32_t)(r >> 6)) % kSlots) * kTile + (uint32_t)lr * 128u;
#pragma unroll
                for (int pc = 0; pc < kPanels; ++pc) {
                    uint32_t q[32];
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        const uint4 v = ptx::ld_shared_v4(src + (uint32_t)pc * kPanel64 +
                                                          (uint32_t)((cc ^ (lr & 7)) * 16));
                        q[4 * cc] = v.x; q[4 * cc + 1] = v.y; q[4 * cc + 2] = v.z; q[4 * cc + 3] = v.w;
                    }
                    ptx::tmem_st32(tm + tl + kColQ + 32u * (uint32_t)pc, q);
                }
                ptx::tmem_wait_st();
            }
            ptx::tc_fence_before();
            if (!sm_barrier_and(ok)) return false;
            if (threadIdx.x == 0) {
                ptx::mbar_arrive(bar_addr(c, b_ring_empty(qpos)));
                ptx::mbar_arrive(bar_addr(c, b_ring_empty(qpos + 1u)));
                ptx::mbar_arrive(bar_addr(c, b_q_ready()));
            }
            return true;
        };
        // Whether this CTA has an item after item sub of unit u (units of packed sequences
        // can be empty).
        auto has_next = [&](int u, int sub, int nsub) -> bool {
            if (sub + 1 < nsub) return true;
            for (int u2 = u + (int)gridDim.x; u2 < p.units; u2 += (int)gridDim.x)
                if (unit_items<CAUSAL, MODE>(p, u2) > 0) return true;
            return false;
        };
        uint32_t g = 0, base = 0, pv = 0;   // pv: products of O issued before this item
        bool q_written = false;             // the current item's Q is in TMEM already
        for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
            const int nsub = unit_items<CAUSAL, MODE>(p, u);
            for (int sub = 0; sub < nsub; ++sub) {
                const Work w = unit_item<CAUSAL, MODE>(p, u, sub);
                const int i = w.qt * kBM + r;   // row within the slice
                const int limit = CAUSAL ? min(i + 1, w.len) : w.len;  // visible keys: key < limit
                // A CTA's first item writes its Q here; every later one was written on the
                // previous item's last step.
                if (!q_written && !write_q(base)) goto sm_out;
                q_written = false;
                const bool next = has_next(u, sub, nsub);
                // reference max (log2 units), row sum, and (bf16) row sum of the rounded P
                float m_run = -INFINITY, l_run = 0.0f, l_rnd = 0.0f;
                for (int j = 0; j < w.nkv; ++j) {
                    const uint32_t gj = g + (uint32_t)j, b = gj & 1u;
                    const uint32_t tS = tm + tl + kColS + 64u * b;
                    if (!wait_warp(c, b_s_full(b), (gj >> 1) & 1u, kRoleSoftmax)) goto sm_out;
                    ptx::tc_fence_after();
                    uint32_t s[64];
                    ptx::tmem_ld64_wait(tS, s);
                    const int key0 = j * kBN;
                    const bool mask = __any_sync(0xFFFFFFFFu, key0 + kBN > limit);
                    uint32_t pk[32];
                    const float alpha =
                        mask ? softmax_step<true, ET>(s, key0, limit, sl2, m_run, l_run, l_rnd, pk)
                             : softmax_step<false, ET>(s, key0, limit, sl2, m_run, l_run, l_rnd, pk);
                    // The reference rose for some row: O += P(j-1) V_{j-1} must be complete,
                    // then this row of O is rescaled in TMEM.  The item's last step waits for
                    // that product in any case, so the epilogue's single wait is exact.  (The
                    // product before it is complete: S(j) was issued after it; this step's own
                    // product waits for its hand-over; so the parity wait sees the barrier at
                    // most one phase behind and never ahead.)
                    const bool resc = j > 0 && __any_sync(0xFFFFFFFFu, alpha != 1.0f);
                    if (resc || (j > 0 && j + 1 == w.nkv)) {
                        if (!wait_warp(c, b_o_done(), (pv + (uint32_t)j - 1u) & 1u, kRoleSoftmax)) goto sm_out;
                        ptx::tc_fence_after();
                    }
                    if (resc) {
                        // two 128-column TMEM round trips (this kernel's warps have the
                        // registers), packed multiplies in between
#pragma unroll 1
                        for (int cc = 0; cc < D / 128; ++cc) {
                            uint32_t o[128];
                            ptx::tmem_ld128_wait(tm + tl + kColO + (uint32_t)cc * 128u, o);
#pragma unroll
                            for (int e = 0; e < 128; e += 2) ptx::mul2u(o[e], o[e + 1], alpha);
                            ptx::tmem_st128(tm + tl + kColO + (uint32_t)cc * 128u, o);
                        }
                    }
                    __syncwarp();
                    // P over this buffer's first 32 (e4m3: 16) columns
                    if constexpr (ET == 2) ptx::tmem_st16(tS, pk);
                    else ptx::tmem_st32(tS, pk);
                    ptx::tmem_wait_st();
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(bar_addr(c, b_p_full(b)));
                    // The item's last S product, the last to read this Q, is complete (this
                    // step waited for it): the next item's Q goes into TMEM now, so its first
                    // two S products run during this item's epilogue.
                    if (next && j + 1 == w.nkv) {
                        if (!write_q(base + 2u + 2u * (uint32_t)w.nkv)) goto sm_out;
                        q_written = true;
                    }
                }
                // epilogue: O / l, rounded, staged per warp, whole-line stores; LSE.  The
                // item's second-to-last O product (or the previous item's last one) is known
                // complete and no later O product exists yet (the next item's S products may),
                // so one parity wait for the last O product is exact.  (Two waits in a row, for
                // the last two products, would misread the barrier if both had completed
                // before the first.)
                pv += (uint32_t)w.nkv;
                if (!wait_warp(c, b_o_done(), (pv - 1u) & 1u, kRoleSoftmax)) goto sm_out;
                ptx::tc_fence_after();
                // o_scale: V's dequantisation factor (1 at 16 bits)
                const float inv = p.o_scale / (Lazy<ET>::kRoundedSum ? l_rnd : l_run);
                // row rr of the slice: obase + rr * ostride (elements)
                const size_t ostride = MODE == 0 ? (size_t)D : (size_t)p.heads * D;
                uint16_t* obase = reinterpret_cast<uint16_t*>(p.o) +
                                  (MODE == 0 ? (size_t)w.bh * p.n * D : ((size_t)w.tok0 * p.heads + w.h) * D);
                const int row0 = w.qt * kBM + warp * 32;
#pragma unroll 1
                for (int pc = 0; pc < D / 64; ++pc) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t o[32];
                        ptx::tmem_ld32_wait(tm + tl + kColO + (uint32_t)(pc * 64 + h * 32), o);
                        uint32_t wv[16];
#pragma unroll
                        for (int e = 0; e < 16; ++e)   // fp16 for fp16 storage, else bf16
                            wv[e] = pack2<ET == 1>(u2f(o[2 * e]) * inv, u2f(o[2 * e + 1]) * inv);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const uint32_t chunk = (uint32_t)(h * 4 + e) ^ (uint32_t)(lane & 7);
                            ptx::st_shared_v4(stage + (uint32_t)lane * 128u + chunk * 16u, wv[4 * e],
                                              wv[4 * e + 1], wv[4 * e + 2], wv[4 * e + 3]);
                        }
                    }
                    __syncwarp();
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int rr = 4 * k + (lane >> 3);
                        const int ch = lane & 7;
                        const uint4 v = ptx::ld_shared_v4(stage + (uint32_t)rr * 128u +
                                                          (uint32_t)((ch ^ (rr & 7)) * 16));
                        if (row0 + rr < w.len)
                            *reinterpret_cast<uint4*>(obase + (size_t)(row0 + rr) * ostride + pc * 64 + ch * 8) = v;
                    }
                    __syncwarp();
                }
                if (i < w.len) {
                    // [B, H, N] rows, or [H, total] for packed sequences
                    const size_t lrow = (MODE == 1 && p.cu_seqlens != nullptr)
                                            ? (size_t)w.h * (size_t)p.total + (size_t)w.tok0 + (size_t)i
                                            : (size_t)w.bh * (size_t)p.n + (size_t)i;
                    p.lse[lrow] = (m_run + log2f(l_run)) * kLn2;
                }
                g += (uint32_t)w.nkv;
                base += 2u + 2u * (uint32_t)w.nkv;
            }
        }
    sm_out:;
    }
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tm, kTmemCols);
    }
}

// e4m3 is served for [B, H, N, D] tensors only (MODE 0).
template <bool CAUSAL, int ET>
cudaError_t prepare_modes() {
    auto set = [](const void* fn) {
        return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    };
    const cudaError_t e = set((const void*)fa_tc256_kernel<CAUSAL, ET, 0>);
    if constexpr (ET == 2) return e;
    else return e != cudaSuccess ? e : set((const void*)fa_tc256_kernel<CAUSAL, ET, 1>);
}

template <bool CAUSAL, int ET>
cudaError_t launch_mode(int mode, const TcParams& p, int grid, cudaStream_t stream) {
    if (mode == 0) {
        fa_tc256_kernel<CAUSAL, ET, 0><<<grid, kThreads, kSmemBytes, stream>>>(p);
    } else {
        if constexpr (ET == 2) return cudaErrorInvalidValue;
        else fa_tc256_kernel<CAUSAL, ET, 1><<<grid, kThreads, kSmemBytes, stream>>>(p);
    }
    return cudaGetLastError();
}

template <bool CAUSAL>
cudaError_t prepare_et(int et) {
    return et == 2 ? prepare_modes<CAUSAL, 2>() : et == 1 ? prepare_modes<CAUSAL, 1>() : prepare_modes<CAUSAL, 0>();
}

template <bool CAUSAL>
cudaError_t launch_et(int et, const TcParams& p, int grid, cudaStream_t stream) {
    const int mode = p.layout;   // 0: [B, H, N, D]; 1: token-major
    return et == 2   ? launch_mode<CAUSAL, 2>(mode, p, grid, stream)
           : et == 1 ? launch_mode<CAUSAL, 1>(mode, p, grid, stream)
                     : launch_mode<CAUSAL, 0>(mode, p, grid, stream);
}

}  // namespace

cudaError_t tc256_prepare(bool causal, int et) {
    return causal ? prepare_et<true>(et) : prepare_et<false>(et);
}

int tc256_units(int bh, int n, bool causal) {
    const long long nt = (n + kBM - 1) / kBM;
    const long long u = (long long)bh * (causal ? (nt + 1) / 2 : nt);
    return u > 0x7FFFFFFFLL ? -1 : (int)u;
}

cudaError_t tc256_launch(bool causal, int et, const TcParams& p, int grid, cudaStream_t stream) {
    if (grid < 1 || p.units < 1) return cudaErrorInvalidConfiguration;
    return causal ? launch_et<true>(et, p, grid, stream) : launch_et<false>(et, p, grid, stream);
}

cudaError_t tc256_status_read_reset(uint32_t out[4]) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_status, sizeof(unsigned int) * 4);
    if (e != cudaSuccess) return e;
    const unsigned int zero[4] = {0, 0, 0, 0};
    return cudaMemcpyToSymbol(g_status, zero, sizeof(zero));
}

}  // namespace fa
