// fa_tc.cu -- FlashAttention forward on the GB300 5th-generation tensor cores.
//
// What it computes: O = softmax(scale * Q K^T) V and LSE per row, for every (b, h) slice
// of [B, H, N, D] bf16/fp16 (or e4m3, O in bf16) tensors, D = 32, 64 or 128, or of the
// token-major layouts ("KingOfEgg: Flash Attention v1" §1.1-§1.2), tile
// by tile with the online-softmax (m, l, O) recurrence so that no N x N matrix ever
// reaches HBM ("08 · FlashAttention" §二; "第 13 课：GPU 内核与 FlashAttention"
// Figure 13-2: query blocks outside, key/value blocks inside, O written once).
//
// Design (one persistent CTA per SM, 10 warps, warp-specialised):
//   * warp 9 (loader): TMA loads of two 128-row query tiles (A and B) per work item and
//     a ring of 128-key K and V tiles, each completion counted on an mbarrier
//     (the asynchronous double-buffered copy of "pwwt.cn: FlashAttention 与内存墙" §3.3,
//     here as TMA + mbarrier instead of cp.async groups).
//   * warp 8 (MMA issuer, one thread): tcgen05.mma  S_t = Q_t K_j^T  into TMEM, and
//     O_t += P_t V_j  with P_t read straight from TMEM; completion is signalled with
//     tcgen05.commit onto mbarriers.  Where P is written over S (D = 128), issue order
//     S_A(0) S_B(0) | PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) | ... so the softmax of one tile
//     overlaps the products of the other.  Where TMEM has room for P in columns of its
//     own (D <= 64 at 16 bits, D = 64 at e4m3), S(j+1) is issued as soon as the softmax has
//     loaded S(j), ahead of P(j) V_j.
//   * warps 0-3 / 4-7 (softmax of tile A / tile B): one thread per query row (TMEM lane =
//     row).  Running max m and sum l stay in registers; exp2 with scale*log2(e) folded
//     into one FMA; P is rounded to the input type and stored into TMEM (over S, or into
//     its own columns).
//     bf16: the reference max is raised whenever a tile's max exceeds it, so the largest P
//     of a row is exactly 1 and its bf16 rounding costs nothing; fp16 / e4m3: it is raised
//     only when it grows by more than 2^8 (finer P rounding leaves room), and only then
//     is O rescaled in TMEM ("08 · FlashAttention" §五 and "第 13 课" §4B: old output
//     multiplied by exp(m_old - m_new) when a larger maximum appears; keeping a stale
//     reference is exact after the final division, since O and l share it).  bf16 at
//     D = 128 rescales at most steps, so there the row of O is multiplied inside the
//     softmax step, 32 TMEM columns at a time between quarters of the exponentials.
//   * epilogue: O / l (one division per row at the end, "第 13 课" exercise; "pwwt.cn"
//     §2.2), staged per warp through shared memory in the 128-byte-swizzled layout, then
//     written by one TMA bulk tensor store per 64-column panel ([B, H, N, D], D >= 64) or
//     by row-contiguous stores of whole 128-byte lines (token-major layouts, D = 32);
//     LSE = (m + log2 l) * ln 2.
//   * item prologue: Q_A, then K_0, then Q_B are loaded, so S_A(0) starts as early as
//     possible when a CTA moves to its next work item.
//   * causal: key tiles entirely after a query tile are skipped, only the diagonal tile
//     is masked ("08 · FlashAttention" §四 is_causal).  Work units pair a heavy and a
//     light query-tile pair of the same slice, so every unit costs about the same.
//   * small problems (all B*H*ceil(N/128) query tiles fit on the SMs at once, [B, H, N, D]):
//     a separate instance gives every query tile a CTA of its own (tile B absent).
//
// Every mbarrier wait is bounded: a wait that runs past its limit raises a CTA-wide abort
// flag and a device status word, every role then leaves its loop, in-flight copies and
// products are drained (bounded as well), TMEM is freed, and the kernel returns.
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

constexpr int kBM = 128;            // query rows per tile = TMEM lanes
constexpr int kBN = 128;            // keys per K/V tile
constexpr int kSoftmaxWarps = 8;    // warps 0-3: tile A, warps 4-7: tile B
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr int kThreads = 320;
constexpr uint32_t kTmemCols = 512;
// The running reference is raised when a tile max exceeds it by more than this many log2
// units.  bf16: 0, the literal reading, so the row's largest P is exactly 1: a stale
// reference would leave it at 2^x for fractional x, and its bf16 rounding (2^-9 relative)
// times a large |v|, added to the bf16 rounding of O, can pass 2e-2 on strongly peaked rows.
// fp16 P (11 significant bits, largest value 65504) and e4m3 P (tops out at 448): 8, so
// stored P stays below 2^8.
// Element type of Q, K, V (and P): 0 = bf16, 1 = fp16, 2 = fp8 e4m3 (O is then bf16).
template <int ET> struct Lazy { static constexpr float kRescaleLog2 = ET == 0 ? 0.0f : 8.0f; };
template <int ET> struct Elem {
    static constexpr int kBytes = ET == 2 ? 1 : 2;
};


// Device status word: [0] flags (1 = a wait ran out), [1] role, [2] CTA, [3] wait id.
__device__ unsigned int g_status[4];

template <int D, int EB>
struct Geo {
    // Shared-memory rows of D elements of EB bytes, split into panels of 128-byte rows
    // (128-byte swizzle), or one panel of whole rows when a row is shorter: 64 bytes
    // (64-byte swizzle; D = 32 at 16 bits, D = 64 at 8 bits) or 32 bytes (32-byte swizzle;
    // D = 32 at 8 bits).
    static constexpr int kRowBytesAll = D * EB;
    static constexpr int kRowBytes = kRowBytesAll < 128 ? kRowBytesAll : 128;
    static constexpr int kPanelCols = kRowBytes / EB;          // elements per panel row
    static constexpr int kPanelBytes = 128 * kRowBytes;        // 128 rows of one panel
    static constexpr uint32_t kSBO = 8u * kRowBytes;            // 8-row group stride
    static constexpr int kPanels = kRowBytesAll / kRowBytes;
    static constexpr int kTileBytes = kPanels * kPanelBytes;   // one 128 x D tile
    static constexpr int kSlots = kTileBytes >= 32768 ? 4 : 8; // K/V ring depth
    static constexpr int kKVOff = 2 * kTileBytes;               // after Q_A, Q_B
    // O staging: one 4 KB slot per softmax warp (its 32 rows x one 64-column panel, rows
    // of 128 B with the 16-byte chunks XOR-swizzled by row so both the row-wise writes and
    // the row-contiguous reads are free of bank conflicts)
    static constexpr int kStageOff = kKVOff + kSlots * kTileBytes;
    static constexpr int kStageSlot = 4096;
    static constexpr int kBarOff = kStageOff + kSoftmaxWarps * kStageSlot;
    // barriers: q_full[2] q_empty[2] kv_full[S] kv_empty[S] s_full[2] p_full[2] o_done[2] drain
    // s_read[2]
    static constexpr int kNumBars = 2 + 2 + 2 * kSlots + 2 + 2 + 2 + 1 + 2;
    static constexpr int kMiscOff = kBarOff + kNumBars * 8;     // tmem base, abort flag
    static constexpr int kSmemBytes = kMiscOff + 16 + 1024;     // + alignment slack
    static_assert(kSmemBytes <= 232448, "shared memory per CTA");
    // TMEM columns of one tile's P: 16-bit pairs or e4m3 quadruples of kBN keys
    static constexpr uint32_t kPCols = (uint32_t)(kBN * EB / 4);
    // Where TMEM has room (D <= 64 at 16 bits, D = 64 at 8 bits), P gets columns of its own,
    // so the next S product can be issued as soon as the softmax has read S, without waiting
    // for P V.  Otherwise P overwrites the upper 64 columns of its S region (S columns 0-63
    // stay readable until the next S product).
    static constexpr bool kSepP = 2 * kBN + 2 * kPCols + 2 * D <= 512;
    static constexpr uint32_t col_s(int t) { return (uint32_t)t * kBN; }
    static constexpr uint32_t col_p(int t) {
        return kSepP ? 2u * kBN + (uint32_t)t * kPCols : (uint32_t)t * kBN + 64u;
    }
    static constexpr uint32_t col_o(int t) {
        return (kSepP ? 2u * kBN + 2u * kPCols : 2u * kBN) + (uint32_t)t * D;
    }
};

// Barrier indices.
template <int D, int EB> __device__ __forceinline__ int b_q_full(int t) { return t; }
template <int D, int EB> __device__ __forceinline__ int b_q_empty(int t) { return 2 + t; }
template <int D, int EB> __device__ __forceinline__ int b_kv_full(uint32_t i) { return 4 + (int)(i % Geo<D, EB>::kSlots); }
template <int D, int EB> __device__ __forceinline__ int b_kv_empty(uint32_t i) { return 4 + Geo<D, EB>::kSlots + (int)(i % Geo<D, EB>::kSlots); }
template <int D, int EB> __device__ __forceinline__ int b_s_full(int t) { return 4 + 2 * Geo<D, EB>::kSlots + t; }
template <int D, int EB> __device__ __forceinline__ int b_p_full(int t) { return 6 + 2 * Geo<D, EB>::kSlots + t; }
template <int D, int EB> __device__ __forceinline__ int b_o_done(int t) { return 8 + 2 * Geo<D, EB>::kSlots + t; }
template <int D, int EB> __device__ __forceinline__ int b_drain() { return 10 + 2 * Geo<D, EB>::kSlots; }
template <int D, int EB> __device__ __forceinline__ int b_s_read(int t) { return 11 + 2 * Geo<D, EB>::kSlots + t; }

// Ring position i -> phase parity of its slot.
template <int D, int EB> __device__ __forceinline__ uint32_t ring_parity(uint32_t i) {
    return (i / Geo<D, EB>::kSlots) & 1u;
}

// ----------------------------------------------------------------- work schedule
// Bulk tensor store of one staged 32-row panel of O (shared -> global) with its completion
// tracking, for the [B, H, N, D] epilogue at D >= 64: one lane issues, the copy engine
// reads the staging slot and writes whole lines; rows past N lie outside the map and are
// not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int32_t c0,
                                             int32_t c1, int32_t c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
                 ::"l"(map), "r"(src), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The issuing thread's stores have finished reading shared memory (the slot may be reused).
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// The issuing thread's stores are complete.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// Shared-memory writes of this thread become visible to the copy engine's reads.
__device__ __forceinline__ void fence_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// O leaves through bulk tensor stores where its rows are [B, H, N, D] rows of 64-column
// panels; token-major rows past a sequence belong to the next one, so those layouts (and
// the 64-byte rows of D = 32) keep per-row stores with a length check.
template <int D, int MODE> struct OStore { static constexpr bool kTma = MODE != 1 && D >= 64; };

struct Item {
    int bh;    // slice b*H + h
    int h;     // head
    int pair;  // query rows [256*pair, 256*pair + 256): tile t holds rows 128*(t ^ sw).. of it
    int sw;    // 0: tile A = first 128 rows, tile B = next 128; 1: the other way round
    int nA;    // key/value tiles tile A visits
    int nB;    // key/value tiles tile B visits
    int len;   // sequence length of the slice
    int tok0;  // token-major layout: token index of row 0 of the slice
};

// Length and first token of slice bh.  Packed offsets are clamped to [0, total] and lengths
// to the declared maximum, so malformed offsets cannot move any access out of bounds.
template <int MODE>
__device__ __forceinline__ void slice_geometry(const TcParams& p, int bh, int& len, int& tok0) {
    if (MODE != 1) {   // [B, H, N, D]: every slice has N rows
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

// Work units: non-causal, one unit per (slice, pair), slice-major so concurrently running
// CTAs share the K/V of a few slices in L2.  Causal: unit (slice, q) holds pairs
// npairs-1-q and q of that slice, heavy first, so every unit costs about the same; the
// second pair's rows are swapped between the tiles, so that each tile visits the one
// extra (diagonal) key tile of the upper rows once per unit and neither tile runs a step
// longer than the other over the unit.  Units
// past the end of a (shorter) packed sequence hold nothing.  unit_count gives the number of
// items of unit u, unit_item the s-th one (computed on demand to keep registers free).
//
// MODE 2 is [B, H, N, D] with the single-tile schedule, which the host picks when the
// B*H*ceil(N/128) query tiles fit on the SMs at once: a pair per SM would leave most SMs
// idle and make each SM's two query tiles share its sub-partitions' softmax throughput.
// Unit u is query tile u % nkv of slice u / nkv, placed in tile A; tile B is absent
// (nB = 0), and its buffers, barriers and softmax warps stay unused for the whole launch.
template <bool CAUSAL, int MODE>
__device__ __forceinline__ int unit_count(const TcParams& p, int u) {
    if (MODE == 2) return 1;
    if (MODE == 0) {   // [B, H, N, D]: every unit is full
        if (!CAUSAL) return 1;
        const int q = u % ((p.npairs + 1) / 2);
        return (p.npairs - 1 - q != q) ? 2 : 1;
    }
    const int per_slice = CAUSAL ? (p.npairs + 1) / 2 : p.npairs;
    const int q = u % per_slice;
    int len, tok0;
    slice_geometry<MODE>(p, u / per_slice, len, tok0);
    const int npairs = (len + 2 * kBM - 1) / (2 * kBM);
    if (!CAUSAL) return q < npairs ? 1 : 0;
    if (q >= (npairs + 1) / 2) return 0;
    return (npairs - 1 - q != q) ? 2 : 1;
}

template <bool CAUSAL, int MODE>
__device__ __forceinline__ Item unit_item(const TcParams& p, int u, int s) {
    Item it;
    if constexpr (MODE == 2) {
        const int t = u % p.nkv;   // query tile: rows 128 t ..
        it.bh = u / p.nkv;
        it.h = 0;
        it.len = p.n;
        it.tok0 = 0;
        it.pair = t >> 1;
        it.sw = t & 1;             // tile A holds rows 128 * (t & 1) of the pair
        it.nA = CAUSAL ? min(t + 1, p.nkv) : p.nkv;
        it.nB = 0;
        return it;
    }
    const int per_slice = CAUSAL ? (p.npairs + 1) / 2 : p.npairs;
    if (MODE == 0) {   // [B, H, N, D]: slices of N rows, no head or token bookkeeping
        it.bh = u / per_slice;
        const int q = u % per_slice;
        it.h = 0;
        it.len = p.n;
        it.tok0 = 0;
        it.pair = CAUSAL ? ((s == 0) ? (p.npairs - 1 - q) : q) : q;
        it.sw = (CAUSAL && s == 1) ? 1 : 0;
        const int n_lo = CAUSAL ? min(2 * it.pair + 1, p.nkv) : p.nkv;   // rows 256 pair..
        const int n_hi = CAUSAL ? min(2 * it.pair + 2, p.nkv) : p.nkv;   // rows 256 pair + 128..
        it.nA = it.sw ? n_hi : n_lo;
        it.nB = it.sw ? n_lo : n_hi;
        return it;
    }
    it.bh = u / per_slice;
    it.h = it.bh % p.heads;
    const int q = u % per_slice;
    slice_geometry<MODE>(p, it.bh, it.len, it.tok0);
    const int npairs = (it.len + 2 * kBM - 1) / (2 * kBM);
    const int nkv = (it.len + kBN - 1) / kBN;
    if (!CAUSAL) {
        it.pair = q;
        it.sw = 0;
        it.nA = nkv;
        it.nB = nkv;
    } else {
        it.pair = (s == 0) ? (npairs - 1 - q) : q;
        it.sw = s == 1 ? 1 : 0;
        const int n_lo = min(2 * it.pair + 1, nkv), n_hi = min(2 * it.pair + 2, nkv);
        it.nA = it.sw ? n_hi : n_lo;
        it.nB = it.sw ? n_lo : n_hi;
    }
    return it;
}

// TMA coordinates (dims 1 and 2) of row `row` of the item's slice.
template <int MODE>
__device__ __forceinline__ void tile_coords(const TcParams& p, const Item& it, int row, int& c1,
                                            int& c2) {
    if (MODE != 1) {
        c1 = row;
        c2 = it.bh;
    } else {
        c1 = it.h;
        c2 = it.tok0 + row;
    }
}

// ----------------------------------------------------------------- MMA issue
// Shared-memory descriptor of a tile with D-dependent rows: 128-byte swizzle (layout type
// 2) for 128-byte rows, 64-byte swizzle (type 4) for 64-byte rows (D = 32 at 16 bits, D = 64
// at e4m3), 32-byte swizzle (type 6) for the 32-byte rows of D = 32 at e4m3.
template <int D, int EB>
__device__ __forceinline__ uint64_t tile_desc(uint32_t saddr, uint32_t lbo) {
    using G = Geo<D, EB>;
    static_assert(G::kRowBytes == 128 || G::kRowBytes == 64 || G::kRowBytes == 32, "row width");
    const uint64_t layout = G::kRowBytes == 128 ? 2ull : G::kRowBytes == 64 ? 4ull : 6ull;
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((G::kSBO >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (layout << 61);
}

// Instruction descriptor for the element type: kind::f16 (bf16 or fp16 operands) or
// kind::f8f6f4 with both operands e4m3 (format code 0).
template <int ET>
__host__ __device__ constexpr uint32_t idesc_of(int M, int N, bool b_mn_major) {
    return ET == 2 ? ((1u << 4) | ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) |
                      ((uint32_t)(M >> 4) << 24))
                   : make_idesc(M, N, b_mn_major, ET == 1);
}

// Descriptors are built once per buffer; a K step only adds a constant to the start
// address field (addresses stay below 256 KB, so the 14-bit field never carries).
// All lanes of the MMA warp execute these; one elected lane issues.
template <int D, int ET>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t q_desc, uint64_t k_desc,
                                         uint32_t idesc) {
    using G = Geo<D, Elem<ET>::kBytes>;
    constexpr int kSteps = G::kRowBytesAll / 32;   // 32 bytes (16 or 32 values) per K step
    constexpr int kPerPanel = G::kRowBytes / 32;
#pragma unroll
    for (int kk = 0; kk < kSteps; ++kk) {
        const uint64_t off = ((uint64_t)(kk / kPerPanel) * G::kPanelBytes +
                              (uint64_t)(kk % kPerPanel) * 32u) >> 4;
        if (ET == 2) ptx::mma_ss_f8_elect(d_tmem, q_desc + off, k_desc + off, idesc, kk > 0 ? 1u : 0u);
        else ptx::mma_ss_elect(d_tmem, q_desc + off, k_desc + off, idesc, kk > 0 ? 1u : 0u);
    }
}

template <int D, int ET>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint64_t v_desc,
                                         uint32_t idesc, bool accumulate) {
    using G = Geo<D, Elem<ET>::kBytes>;
    constexpr int kKeys = 32 / Elem<ET>::kBytes;   // keys per K step (32 bytes of P per row)
#pragma unroll
    for (int kk = 0; kk < kBN / kKeys; ++kk) {
        // P: 8 TMEM columns per K step.  V tile: rows = keys (K dimension), one row of
        // head-dim values per key (MN-major); kKeys rows per K step; panels kPanelBytes
        // apart (LBO).
        const uint64_t b = v_desc + (uint64_t)((kk * kKeys * G::kRowBytes) >> 4);
        const uint32_t acc = (accumulate || kk > 0) ? 1u : 0u;
        if (ET == 2) ptx::mma_ts_f8_elect(d_tmem, p_tmem + (uint32_t)kk * 8u, b, idesc, acc);
        else ptx::mma_ts_elect(d_tmem, p_tmem + (uint32_t)kk * 8u, b, idesc, acc);
    }
}

// ----------------------------------------------------------------- roles
// MMA issuer: the whole warp runs this loop (waits are warp-uniform), one lane issues.
template <int D, bool CAUSAL, int ET, int MODE>
__device__ void mma_role(const TcParams& p, const Ctl& c, uint32_t tmem, uint32_t sbase) {
    constexpr int EB = Elem<ET>::kBytes;
    using G = Geo<D, EB>;
    constexpr uint32_t idesc_qk = idesc_of<ET>(kBM, kBN, false);
    constexpr uint32_t idesc_pv = idesc_of<ET>(kBM, D, true);
    const uint64_t dQ[2] = {tile_desc<D, EB>(sbase, 16),
                            tile_desc<D, EB>(sbase + (uint32_t)G::kTileBytes, 16)};
    const uint64_t dK0 = tile_desc<D, EB>(sbase + (uint32_t)G::kKVOff, 16);                  // K-major
    const uint64_t dV0 = tile_desc<D, EB>(sbase + (uint32_t)G::kKVOff, (uint32_t)G::kPanelBytes);  // MN-major
    const uint32_t tS[2] = {tmem + G::col_s(0), tmem + G::col_s(1)};
    const uint32_t tP[2] = {tmem + G::col_p(0), tmem + G::col_p(1)};
    const uint32_t tO[2] = {tmem + G::col_o(0), tmem + G::col_o(1)};
    auto slot_off = [&](uint32_t i) {  // descriptor offset of ring slot i
        return (uint64_t)((i % G::kSlots) * (uint32_t)G::kTileBytes) >> 4;
    };
    uint32_t kv = 0, q_cnt = 0, p_cnt0 = 0, p_cnt1 = 0;

    for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
        const int nsub = unit_count<CAUSAL, MODE>(p, u);
        for (int sub = 0; sub < nsub; ++sub) {
            const Item it = unit_item<CAUSAL, MODE>(p, u, sub);
            if (!wait_warp(c, b_q_full<D, EB>(0), q_cnt & 1u, kRoleMma)) goto out;
            if (!wait_warp(c, b_kv_full<D, EB>(kv), ring_parity<D, EB>(kv), kRoleMma)) goto out;
            ptx::tc_fence_after();
            issue_qk<D, ET>(tS[0], dQ[0], dK0 + slot_off(kv), idesc_qk);
            ptx::mma_commit_elect(bar_addr(c, b_s_full<D, EB>(0)));
            if (it.nA == 1) ptx::mma_commit_elect(bar_addr(c, b_q_empty<D, EB>(0)));
            if constexpr (MODE != 2) {   // tile B (absent in the single-tile schedule)
                if (!wait_warp(c, b_q_full<D, EB>(1), q_cnt & 1u, kRoleMma)) goto out;
                ptx::tc_fence_after();
                issue_qk<D, ET>(tS[1], dQ[1], dK0 + slot_off(kv), idesc_qk);
                ptx::mma_commit_elect(bar_addr(c, b_s_full<D, EB>(1)));
                if (it.nB == 1) ptx::mma_commit_elect(bar_addr(c, b_q_empty<D, EB>(1)));
            }
            ++q_cnt;
            ptx::mma_commit_elect(bar_addr(c, b_kv_empty<D, EB>(kv)));
            ++kv;

            const int nmax = max(it.nA, it.nB);
            for (int j = 0; j < nmax; ++j) {
                const uint32_t vpos = kv;        // V_j
                const uint32_t kpos = kv + 1;    // K_{j+1}
                const bool more = j + 1 < nmax;
                // V_j and K_{j+1} (loaded right after it) are awaited before tile A's P, so
                // that nothing but the hand-over of P stands between O_A += P V_j and S_A(j+1).
                if (!wait_warp(c, b_kv_full<D, EB>(vpos), ring_parity<D, EB>(vpos), kRoleMma)) goto out;
                if (more && !wait_warp(c, b_kv_full<D, EB>(kpos), ring_parity<D, EB>(kpos), kRoleMma)) goto out;
                ptx::tc_fence_after();
                if (j < it.nA) {
                    if (!wait_warp(c, b_p_full<D, EB>(0), p_cnt0 & 1u, kRoleMma)) goto out;
                    ++p_cnt0;
                    ptx::tc_fence_after();
                    issue_pv<D, ET>(tO[0], tP[0], dV0 + slot_off(vpos), idesc_pv, j > 0);
                    ptx::mma_commit_elect(bar_addr(c, b_o_done<D, EB>(0)));
                }
                if (j + 1 < it.nA) {
                    issue_qk<D, ET>(tS[0], dQ[0], dK0 + slot_off(kpos), idesc_qk);
                    ptx::mma_commit_elect(bar_addr(c, b_s_full<D, EB>(0)));
                    if (j + 2 == it.nA) ptx::mma_commit_elect(bar_addr(c, b_q_empty<D, EB>(0)));
                }
                if (j < it.nB) {
                    if (!wait_warp(c, b_p_full<D, EB>(1), p_cnt1 & 1u, kRoleMma)) goto out;
                    ++p_cnt1;
                    ptx::tc_fence_after();
                    issue_pv<D, ET>(tO[1], tP[1], dV0 + slot_off(vpos), idesc_pv, j > 0);
                    ptx::mma_commit_elect(bar_addr(c, b_o_done<D, EB>(1)));
                }
                ptx::mma_commit_elect(bar_addr(c, b_kv_empty<D, EB>(vpos)));
                ++kv;
                if (j + 1 < it.nB) {
                    issue_qk<D, ET>(tS[1], dQ[1], dK0 + slot_off(kpos), idesc_qk);
                    ptx::mma_commit_elect(bar_addr(c, b_s_full<D, EB>(1)));
                    if (j + 2 == it.nB) ptx::mma_commit_elect(bar_addr(c, b_q_empty<D, EB>(1)));
                }
                if (more) {
                    ptx::mma_commit_elect(bar_addr(c, b_kv_empty<D, EB>(kpos)));
                    ++kv;
                }
            }
        }
    }
out:
    // Every product issued so far must finish before TMEM is released.
    ptx::mma_commit_elect(bar_addr(c, b_drain<D, EB>()));
    wait_drain(bar_addr(c, b_drain<D, EB>()), 0, c.limit);
    __syncwarp();
}

// MMA issuer when P has TMEM columns of its own: each tile's next S product is issued as soon
// as the softmax has read the current S (s_read), ahead of O += P V.  Per 128-key step:
// S_A(j+1) S_B(j+1) | PV_A(j) PV_B(j).  The whole warp runs this loop; one lane issues.
template <int D, bool CAUSAL, int ET, int MODE>
__device__ void mma_role_sep(const TcParams& p, const Ctl& c, uint32_t tmem, uint32_t sbase) {
    constexpr int EB = Elem<ET>::kBytes;
    using G = Geo<D, EB>;
    constexpr uint32_t idesc_qk = idesc_of<ET>(kBM, kBN, false);
    constexpr uint32_t idesc_pv = idesc_of<ET>(kBM, D, true);
    const uint64_t dQ[2] = {tile_desc<D, EB>(sbase, 16),
                            tile_desc<D, EB>(sbase + (uint32_t)G::kTileBytes, 16)};
    const uint64_t dK0 = tile_desc<D, EB>(sbase + (uint32_t)G::kKVOff, 16);                       // K-major
    const uint64_t dV0 = tile_desc<D, EB>(sbase + (uint32_t)G::kKVOff, (uint32_t)G::kPanelBytes);  // MN-major
    const uint32_t tS[2] = {tmem + G::col_s(0), tmem + G::col_s(1)};
    const uint32_t tP[2] = {tmem + G::col_p(0), tmem + G::col_p(1)};
    const uint32_t tO[2] = {tmem + G::col_o(0), tmem + G::col_o(1)};
    auto slot_off = [&](uint32_t i) { return (uint64_t)((i % G::kSlots) * (uint32_t)G::kTileBytes) >> 4; };
    uint32_t kv = 0, q_cnt = 0, p_cnt[2] = {0, 0}, sr_cnt[2] = {0, 0}, s_issued[2] = {0, 0};
    // S into tile t's region: the softmax must have read the previous S there
    auto issue_s = [&](int t, uint32_t kpos) -> bool {
        if (s_issued[t] > 0) {
            if (!wait_warp(c, b_s_read<D, EB>(t), sr_cnt[t] & 1u, kRoleMma)) return false;
            ++sr_cnt[t];
        }
        ptx::tc_fence_after();
        issue_qk<D, ET>(tS[t], dQ[t], dK0 + slot_off(kpos), idesc_qk);
        ptx::mma_commit_elect(bar_addr(c, b_s_full<D, EB>(t)));
        ++s_issued[t];
        return true;
    };
    auto issue_o = [&](int t, uint32_t vpos, bool accumulate) -> bool {   // O_t (+)= P_t V_j
        if (!wait_warp(c, b_p_full<D, EB>(t), p_cnt[t] & 1u, kRoleMma)) return false;
        ++p_cnt[t];
        ptx::tc_fence_after();
        issue_pv<D, ET>(tO[t], tP[t], dV0 + slot_off(vpos), idesc_pv, accumulate);
        ptx::mma_commit_elect(bar_addr(c, b_o_done<D, EB>(t)));
        return true;
    };

    for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
        const int nsub = unit_count<CAUSAL, MODE>(p, u);
        for (int sub = 0; sub < nsub; ++sub) {
            const Item it = unit_item<CAUSAL, MODE>(p, u, sub);
            if (!wait_warp(c, b_q_full<D, EB>(0), q_cnt & 1u, kRoleMma)) goto out;
            if (!wait_warp(c, b_kv_full<D, EB>(kv), ring_parity<D, EB>(kv), kRoleMma)) goto out;
            if (!issue_s(0, kv)) goto out;
            if (it.nA == 1) ptx::mma_commit_elect(bar_addr(c, b_q_empty<D, EB>(0)));
            if constexpr (MODE != 2) {   // tile B (absent in the single-tile schedule)
                if (!wait_warp(c, b_q_full<D, EB>(1), q_cnt & 1u, kRoleMma)) goto out;
                if (!issue_s(1, kv)) goto out;
                if (it.nB == 1) ptx::mma_commit_elect(bar_addr(c, b_q_empty<D, EB>(1)));
            }
            ++q_cnt;
            ptx::mma_commit_elect(bar_addr(c, b_kv_empty<D, EB>(kv)));   // K_0
            ++kv;

            const int nmax = max(it.nA, it.nB);
            for (int j = 0; j < nmax; ++j) {
                const uint32_t vpos = kv;        // V_j
                const uint32_t kpos = kv + 1;    // K_{j+1}
                const bool more = j + 1 < nmax;
                if (more) {
                    if (!wait_warp(c, b_kv_full<D, EB>(kpos), ring_parity<D, EB>(kpos), kRoleMma)) goto out;
                    if (j + 1 < it.nA) {
                        if (!issue_s(0, kpos)) goto out;
                        if (j + 2 == it.nA) ptx::mma_commit_elect(bar_addr(c, b_q_empty<D, EB>(0)));
                    }
                    if (j + 1 < it.nB) {
                        if (!issue_s(1, kpos)) goto out;
                        if (j + 2 == it.nB) ptx::mma_commit_elect(bar_addr(c, b_q_empty<D, EB>(1)));
                    }
                    ptx::mma_commit_elect(bar_addr(c, b_kv_empty<D, EB>(kpos)));   // K_{j+1}
                }
                if (!wait_warp(c, b_kv_full<D, EB>(vpos), ring_parity<D, EB>(vpos), kRoleMma)) goto out;
                if (j < it.nA && !issue_o(0, vpos, j > 0)) goto out;
                if (j < it.nB && !issue_o(1, vpos, j > 0)) goto out;
                ptx::mma_commit_elect(bar_addr(c, b_kv_empty<D, EB>(vpos)));      // V_j
                kv += more ? 2u : 1u;
            }
        }
    }
out:
    // Every product issued so far must finish before TMEM is released.
    ptx::mma_commit_elect(bar_addr(c, b_drain<D, EB>()));
    wait_drain(bar_addr(c, b_drain<D, EB>()), 0, c.limit);
    __syncwarp();
}

template <int D, int EB, bool CAUSAL, int MODE>
__device__ void load_role(const TcParams& p, const Ctl& c, uint32_t sbase) {
    using G = Geo<D, EB>;
    const uint32_t sQ[2] = {sbase, sbase + (uint32_t)G::kTileBytes};
    auto slot = [&](uint32_t i) {
        return sbase + (uint32_t)G::kKVOff + (i % G::kSlots) * (uint32_t)G::kTileBytes;
    };
    uint32_t kv = 0, q_cnt = 0;
    uint32_t q_issued[2] = {0, 0};  // Q loads issued per tile buffer
    const uint32_t skipped = (p.inject_stall == 1 && blockIdx.x == 0) ? 0u : 0xFFFFFFFFu;

    for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
        const int nsub = unit_count<CAUSAL, MODE>(p, u);
        for (int sub = 0; sub < nsub; ++sub) {
            const Item it = unit_item<CAUSAL, MODE>(p, u, sub);
            // Q_A first, then K_0 (so S_A(0) can start), then Q_B, then V_0, K_1, V_1, ...
            auto load_q = [&](int t) -> bool {
                if (!wait(c, b_q_empty<D, EB>(t), (q_cnt & 1u) ^ 1u, kRoleLoad)) return false;
                const uint32_t fb = bar_addr(c, b_q_full<D, EB>(t));
                ptx::mbar_arrive_expect_tx(fb, (uint32_t)G::kTileBytes);
                int c1, c2;
                tile_coords<MODE>(p, it, it.pair * 2 * kBM + (t ^ it.sw) * kBM, c1, c2);
#pragma unroll
                for (int pc = 0; pc < G::kPanels; ++pc)
                    ptx::tma_load_3d(sQ[t] + (uint32_t)pc * G::kPanelBytes, &p.tmap_q, fb, pc * G::kPanelCols,
                                     c1, c2);
                ++q_issued[t];
                return true;
            };
            if (!load_q(0)) goto out;
            const int nmax = max(it.nA, it.nB);
            for (int j = 0; j < nmax; ++j) {
                for (int w = 0; w < 2; ++w) {  // K_j then V_j
                    if (!wait(c, b_kv_empty<D, EB>(kv), ring_parity<D, EB>(kv) ^ 1u, kRoleLoad)) goto out;
                    if (kv != skipped) {
                        const uint32_t fb = bar_addr(c, b_kv_full<D, EB>(kv));
                        ptx::mbar_arrive_expect_tx(fb, (uint32_t)G::kTileBytes);
                        const CUtensorMap* map = (w == 0) ? &p.tmap_k : &p.tmap_v;
                        int c1, c2;
                        tile_coords<MODE>(p, it, j * kBN, c1, c2);
#pragma unroll
                        for (int pc = 0; pc < G::kPanels; ++pc)
                            ptx::tma_load_3d(slot(kv) + (uint32_t)pc * G::kPanelBytes, map, fb,
                                             pc * G::kPanelCols, c1, c2);
                    }
                    ++kv;
                    if (MODE != 2 && j == 0 && w == 0 && !load_q(1)) goto out;
                }
            }
            ++q_cnt;
        }
    }
out:
    // No TMA copy may still be writing shared memory when the CTA exits: wait for the
    // last fill of every ring slot and of both query buffers.
    for (uint32_t i = (kv > (uint32_t)G::kSlots ? kv - G::kSlots : 0u); i < kv; ++i)
        if (i != skipped) wait_drain(bar_addr(c, b_kv_full<D, EB>(i)), ring_parity<D, EB>(i), c.limit);
    for (int t = 0; t < 2; ++t)
        if (q_issued[t] > 0) wait_drain(bar_addr(c, b_q_full<D, EB>(t)), (q_issued[t] - 1u) & 1u, c.limit);
}

// Row maximum of the raw scores of NS keys (a 128-key tile, or one 64-key half of it);
// invisible keys (kbase + c >= limit) are left out.
template <bool MASK, int NS>
__device__ __forceinline__ float tile_row_max(const uint32_t (&s)[NS], int kbase, int limit) {
    float mx[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
    if (MASK) {
#pragma unroll
        for (int c = 0; c < NS; ++c) {
            const float x = (kbase + c < limit) ? u2f(s[c]) : -INFINITY;
            mx[c & 7] = fmaxf(mx[c & 7], x);
        }
    } else {
        // eight independent chains keep the dependent depth short
#pragma unroll
        for (int c = 0; c < NS; c += 2)
            mx[(c >> 1) & 7] = ptx::max3(mx[(c >> 1) & 7], u2f(s[c]), u2f(s[c + 1]));
    }
    return fmaxf(ptx::max3(mx[0], mx[1], mx[2]), fmaxf(ptx::max3(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7])));
}

// p = 2^(s * sl2 - m) for columns [C0, C0 + W), partial row sums into acc (four fp32
// pairs), and P packed for TMEM: 16-bit pairs into pk[C0/2 ...], or for e4m3 four values
// per word into pk[C0/4 ...].  Invisible keys give p = 0.
template <int C0, int W, bool MASK, int ET, int NS, int NP>
__device__ __forceinline__ void tile_exp_cols(const uint32_t (&s)[NS], int kbase, int limit,
                                              float sl2, float neg_m, float (&acc)[8],
                                              uint32_t (&pk)[NP]) {
    static_assert(C0 + W <= NS && (ET == 2 ? (C0 + W) / 4 : (C0 + W) / 2) <= NP, "ranges");
#pragma unroll
    for (int c = C0; c < C0 + W; c += 4) {
        float x[4], pr[4];
        ptx::fma2(x[0], x[1], u2f(s[c]), u2f(s[c + 1]), sl2, neg_m);
        ptx::fma2(x[2], x[3], u2f(s[c + 2]), u2f(s[c + 3]), sl2, neg_m);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            pr[e] = ptx::ex2(x[e]);
            if (MASK && kbase + c + e >= limit) pr[e] = 0.f;
        }
        const int a = ((c >> 1) & 3) * 2;
        ptx::add2(acc[a], acc[a + 1], pr[0], pr[1]);
        ptx::add2(acc[a + 2], acc[a + 3], pr[2], pr[3]);
        if constexpr (ET == 2) {
            pk[c >> 2] = pack4_e4m3(pr[0], pr[1], pr[2], pr[3]);
        } else {
            pk[c >> 1] = pack2<ET == 1>(pr[0], pr[1]);
            pk[(c >> 1) + 1] = pack2<ET == 1>(pr[2], pr[3]);
        }
    }
}

// One row of O (NC fp32 columns from TMEM address tO0) times alpha, in place, CH columns
// per TMEM load and store, packed multiplies in between.  Larger chunks mean fewer serial
// TMEM round trips; CH is as large as the instance's registers allow without spills (the
// S and P registers are free once P is stored).
template <int NC, int CH>
__device__ __forceinline__ void rescale_o(uint32_t tO0, float alpha) {
    static_assert(NC % CH == 0, "chunks");
#pragma unroll 1
    for (int cc = 0; cc < NC / CH; ++cc) {
        const uint32_t tO = tO0 + (uint32_t)(cc * CH);
        uint32_t o[CH];
        if constexpr (CH == 128) ptx::tmem_ld128_wait(tO, o);
        else if constexpr (CH == 64) ptx::tmem_ld64_wait(tO, o);
        else if constexpr (CH == 32) ptx::tmem_ld32_wait(tO, o);
        else ptx::tmem_ld16_wait(tO, o);
#pragma unroll
        for (int i = 0; i < CH; i += 2) ptx::mul2u(o[i], o[i + 1], alpha);
        if constexpr (CH == 128) ptx::tmem_st128(tO, o);
        else if constexpr (CH == 64) ptx::tmem_st64(tO, o);
        else if constexpr (CH == 32) ptx::tmem_st32(tO, o);
        else ptx::tmem_st16(tO, o);
    }
}

// 32 lanes x 32 consecutive 32-bit columns, issued without waiting: the registers hold
// the values only after tmem_wait_ld32 on the same array, which the compiler sees as
// rewriting them, so no use can be scheduled between the two.
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld32(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// One 32-column chunk of this row of O, loaded without waiting: the wait, the multiply
// by alpha and the store come later, so the load's latency overlaps the exponentials.
__device__ __forceinline__ void o_chunk_finish(uint32_t tO, uint32_t (&o)[32], float alpha) {
    tmem_wait_ld32(o);
#pragma unroll
    for (int i = 0; i < 32; i += 2) ptx::mul2u(o[i], o[i + 1], alpha);
    ptx::tmem_st32(tO, o);
}

// One 128-key tile of one row: running-max update (raised when the tile max exceeds it by
// more than kRescaleLog2 log2 units), exp2, row sum, and P stored into TMEM at tP in two
// halves (64 columns of 16-bit pairs, or 32 columns of e4m3 quadruples).  before_store()
// runs once, after the first half is computed and before anything is stored; false from
// it abandons the tile (returns false).  alpha receives the O rescale factor.
// RESC (D = 128, P over S: O is final when the step begins): the 128 columns of O at tO
// are multiplied by alpha here, in 32-column chunks woven between quarters of the
// exponentials, every step (alpha = 1 exactly where the reference did not move, and 0 on
// a tile's first step, whose P V then overwrites O; a branch around the chunks costs more
// registers than the multiplies cost time).
template <bool MASK, int ET, bool RESC, class BeforeStore>
__device__ __forceinline__ bool softmax_tile(const uint32_t (&s)[128], int kbase, int limit,
                                             float sl2, float& m_run, float& l_run,
                                             uint32_t tP, uint32_t tO, float& alpha,
                                             BeforeStore&& before_store) {
    const float mt = tile_row_max<MASK, 128>(s, kbase, limit) * sl2;  // log2 units
    alpha = 1.0f;
    if (mt > m_run + Lazy<ET>::kRescaleLog2) {
        alpha = ptx::ex2(m_run - mt);   // m_run = -inf on the first tile: alpha = 0
        m_run = mt;
    }
    const float neg_m = -m_run;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    uint32_t pk[64];
    uint32_t o[32];   // the O chunk in flight (RESC)
    tile_exp_cols<0, 32, MASK, ET>(s, kbase, limit, sl2, neg_m, acc, pk);
    if constexpr (RESC) tmem_ld32_async(tO, o);
    tile_exp_cols<32, 32, MASK, ET>(s, kbase, limit, sl2, neg_m, acc, pk);
    if (!before_store()) return false;
    __syncwarp();
    if constexpr (ET == 2) ptx::tmem_st16(tP, &pk[0]);
    else ptx::tmem_st32p(tP, &pk[0]);
    if constexpr (RESC) {
        o_chunk_finish(tO, o, alpha);
        tmem_ld32_async(tO + 32, o);
    }
    tile_exp_cols<64, 32, MASK, ET>(s, kbase, limit, sl2, neg_m, acc, pk);
    if constexpr (RESC) {
        o_chunk_finish(tO + 32, o, alpha);
        tmem_ld32_async(tO + 64, o);
    }
    tile_exp_cols<96, 32, MASK, ET>(s, kbase, limit, sl2, neg_m, acc, pk);
    __syncwarp();
    if constexpr (ET == 2) ptx::tmem_st16(tP + 16, &pk[16]);
    else ptx::tmem_st32p(tP + 32, &pk[32]);
    if constexpr (RESC) {
        o_chunk_finish(tO + 64, o, alpha);
        tmem_ld32_async(tO + 96, o);
        o_chunk_finish(tO + 96, o, alpha);
    }
    const float sum = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
    l_run = l_run * alpha + sum;
    return true;
}

template <int D, bool CAUSAL, int ET, int MODE>
__device__ void softmax_role(const TcParams& p, const Ctl& c, uint32_t tmem, int warp, int lane,
                             uint32_t stage) {
    constexpr int EB = Elem<ET>::kBytes;
    constexpr bool kOutF16 = ET == 1;   // O storage: fp16, else bf16
    using G = Geo<D, EB>;
    const int t = warp / 4;                       // 0: tile A, 1: tile B
    const int lane_base = (warp % 4) * 32;        // this warp's TMEM lane quarter
    const uint32_t tl = (uint32_t)lane_base << 16;
    const uint32_t tS = tmem + tl + G::col_s(t);
    const uint32_t tP = tmem + tl + G::col_p(t);
    const uint32_t tO = tmem + tl + G::col_o(t);
    // S products read; O products of earlier items (P over S) or O products waited for
    uint32_t s_cnt = 0, o_cnt = 0;

    for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
        const int nsub = unit_count<CAUSAL, MODE>(p, u);
        for (int sub = 0; sub < nsub; ++sub) {
            const Item it = unit_item<CAUSAL, MODE>(p, u, sub);
            const int n = t == 0 ? it.nA : it.nB;
            const int row = it.pair * 2 * kBM + (t ^ it.sw) * kBM + lane_base + lane;
            // sequence length: the kernel parameter for [B, H, N, D] (no register held)
            const int len = MODE != 1 ? p.n : it.len;
            const int limit = CAUSAL ? min(row + 1, len) : len;   // visible keys: j < limit
            float m_run = -INFINITY, l_run = 0.0f;

            for (int j = 0; j < n; ++j) {
                // Where P overwrites S, S(j) was issued after O_t += P(j-1) V(j-1) by the same
                // thread, and the commit behind s_full tracks every product that thread issued
                // before it: O is final once S(j) is complete, and no wait on o_done is needed.
                if (!wait_warp(c, b_s_full<D, EB>(t), s_cnt & 1u, kRoleSoftmax)) return;
                ++s_cnt;
                ptx::tc_fence_after();
                uint32_t s[128];
                ptx::tmem_ld128_wait(tS, s);
                if constexpr (G::kSepP) {   // S may now be overwritten by the next S product
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(bar_addr(c, b_s_read<D, EB>(t)));
                }
                const int kbase = j * kBN;
                const bool mask = __any_sync(0xFFFFFFFFu, kbase + kBN > limit);
                // With separate P columns, O_t += P(j-1) V(j-1) must be complete before P is
                // overwritten (it reads those columns) and before O_t is rescaled below.
                auto before_store = [&]() -> bool {
                    if (!G::kSepP || j == 0) return true;
                    if (!wait_warp(c, b_o_done<D, EB>(t), o_cnt & 1u, kRoleSoftmax)) return false;
                    ++o_cnt;
                    ptx::tc_fence_after();
                    return true;
                };
                // bf16 rows at D = 128 are rescaled at most steps (the reference follows
                // every rise of the maximum): the rescale is woven into the step.  Other
                // cases rescale after the step, when some row's reference rose (rarely
                // for the lazy reference of fp16 and e4m3; at D <= 64 the step waits for
                // the last P V only before its first P store, and the extra registers of
                // a woven O chunk there cost more than they save).
                constexpr bool kWeave = ET == 0 && !G::kSepP;
                float alpha;
                const bool ok =
                    mask ? softmax_tile<true, ET, kWeave>(s, kbase, limit, p.scale_log2, m_run, l_run, tP, tO, alpha, before_store)
                         : softmax_tile<false, ET, kWeave>(s, kbase, limit, p.scale_log2, m_run, l_run, tP, tO, alpha, before_store);
                if (!ok) return;
                if (!kWeave && j > 0 && __any_sync(0xFFFFFFFFu, alpha != 1.0f))
                    rescale_o<D, D == 128 ? 64 : 32>(tO, alpha);   // the running max rose: this row of O times alpha
                ptx::tmem_wait_st();
                ptx::tc_fence_before();
                ptx::mbar_arrive(bar_addr(c, b_p_full<D, EB>(t)));
            }

            // Epilogue: O / l, one 64-column panel at a time through this warp's staging
            // slot, so the global stores are row-contiguous: each store instruction writes
            // four whole 128-byte lines (rows past N are skipped); LSE from registers.
            // Where P overwrites S, only the tile's last O product is awaited: the one before
            // it is complete (S(n-1) was issued after it) and the next item's first one
            // waits for this warp's P, so the parity wait is exact.
            if (!wait_warp(c, b_o_done<D, EB>(t), (G::kSepP ? o_cnt : o_cnt + (uint32_t)n - 1u) & 1u,
                           kRoleSoftmax))
                return;
            o_cnt += G::kSepP ? 1u : (uint32_t)n;
            ptx::tc_fence_after();
            const float inv_l = p.o_scale / l_run;   // o_scale: V's dequantisation factor (1 at 16 bits)
            const int row0 = it.pair * 2 * kBM + (t ^ it.sw) * kBM + lane_base;   // first row of the warp
            // row r of the slice: obase + r * ostride (elements)
            const size_t ostride = MODE != 1 ? (size_t)D : (size_t)p.heads * D;
            uint16_t* obase = reinterpret_cast<uint16_t*>(p.o) +
                              (MODE != 1 ? (size_t)it.bh * (size_t)p.n * D
                                         : ((size_t)it.tok0 * p.heads + it.h) * D);
            if constexpr (D == 32) {
                // one 64-byte row per thread: 4 chunks staged, then 8 rows x 4 chunks per store
                uint32_t o[32];
                ptx::tmem_ld32_wait(tO, o);
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    w[i] = pack2<kOutF16>(u2f(o[2 * i]) * inv_l, u2f(o[2 * i + 1]) * inv_l);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t chunk = (uint32_t)i ^ (uint32_t)(lane & 7);
                    ptx::st_shared_v4(stage + (uint32_t)lane * 128u + chunk * 16u, w[4 * i],
                                      w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                }
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int r = 8 * k + (lane >> 2);   // row within the warp's 32
                    const int ch = lane & 3;             // 16-byte chunk within the 64-byte row
                    const uint4 v = ptx::ld_shared_v4(stage + (uint32_t)r * 128u +
                                                      (uint32_t)((ch ^ (r & 7)) * 16));
                    if (row0 + r < (MODE != 1 ? p.n : it.len))
                        *reinterpret_cast<uint4*>(obase + (size_t)(row0 + r) * ostride + ch * 8) = v;
                }
                __syncwarp();
            }
#pragma unroll 1
            for (int pc = 0; pc < D / 64; ++pc) {
                if constexpr (OStore<D, MODE>::kTma) {   // the slot's last store has read it
                    if (lane == 0) bulk_wait_read_all();
                    __syncwarp();
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t o[32];
                    ptx::tmem_ld32_wait(tO + (uint32_t)(pc * 64 + h * 32), o);
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        w[i] = pack2<kOutF16>(u2f(o[2 * i]) * inv_l, u2f(o[2 * i + 1]) * inv_l);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint32_t chunk = (uint32_t)(h * 4 + i) ^ (uint32_t)(lane & 7);
                        ptx::st_shared_v4(stage + (uint32_t)lane * 128u + chunk * 16u, w[4 * i],
                                          w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                    }
                }
                if constexpr (OStore<D, MODE>::kTma) {
                    // the slot is the store's 128-byte-swizzled 32 x 64 box
                    fence_async_shared();
                    __syncwarp();
                    if (lane == 0 && row0 < p.n) {
                        tma_store_3d(&p.tmap_o, stage, pc * 64, row0, it.bh);
                        bulk_commit();
                    }
                    continue;
                }
                __syncwarp();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int r = 4 * k + (lane >> 3);   // row within the warp's 32
                    const int ch = lane & 7;             // 16-byte chunk within the 128-byte row
                    const uint4 v = ptx::ld_shared_v4(stage + (uint32_t)r * 128u +
                                                      (uint32_t)((ch ^ (r & 7)) * 16));
                    if (row0 + r < (MODE != 1 ? p.n : it.len))
                        *reinterpret_cast<uint4*>(obase + (size_t)(row0 + r) * ostride + pc * 64 + ch * 8) = v;
                }
                __syncwarp();
            }
            if (row < (MODE != 1 ? p.n : it.len)) {
                // [B, H, N] rows, or [H, total] for packed sequences
                const size_t lrow = (MODE == 1 && p.cu_seqlens != nullptr)
                                        ? (size_t)it.h * (size_t)p.total + (size_t)it.tok0 + (size_t)row
                                        : (size_t)it.bh * (size_t)p.n + (size_t)row;
                p.lse[lrow] = (m_run + log2f(l_run)) * kLn2;
            }
            __syncwarp();
        }
    }
}

// ----------------------------------------------------------------- single-tile schedule
// Named barrier 1 + q over the two softmax warps that share TMEM lane quarter q (warps q and
// q + 4), ANDing a predicate.  A warp whose wait gave up still arrives here with false, so
// the pair takes one stop decision and neither warp is left at a barrier the other skips.
__device__ __forceinline__ bool pair_barrier_and(int q, bool ok) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, x;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred x, %2, 64, p;\n\t"
        "selp.u32 %0, 1, 0, x;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)ok), "r"(1 + q)
        : "memory");
    return r != 0;
}
// The same barrier without a predicate, where neither warp can have given up.
__device__ __forceinline__ void pair_barrier(int q) {
    asm volatile("bar.sync %0, 64;" ::"r"(1 + q) : "memory");
}

// Softmax and epilogue of the single-tile schedule (MODE 2), where tile B is absent.  Its
// four warps would idle, so every row of tile A is shared by the two warps of its TMEM lane
// quarter: warp q + 4h (h = 0, 1) takes keys [64h, 64h + 64) of each 128-key tile and O
// columns [h D/2, h D/2 + D/2).  Per tile the two partial row maxima meet in shared memory
// (the unused Q_B buffer) at one barrier, so both warps take the same lazy-rescale decision
// and keep the same running reference; each keeps the row sum of its own keys, and the two
// sums are added once, in the epilogue.  Each warp's serial work per key tile halves.
template <int D, bool CAUSAL, int ET>
__device__ void softmax_role_split(const TcParams& p, const Ctl& c, uint32_t tmem, float* xch,
                                   uint32_t stage_base, int warp, int lane) {
    constexpr int EB = Elem<ET>::kBytes;
    constexpr bool kOutF16 = ET == 1;   // O storage: fp16, else bf16
    constexpr int kHalfO = D / 2;       // O columns of one warp
    using G = Geo<D, EB>;
    const int h = warp / 4;             // key half and O half
    const int q4 = warp % 4;            // TMEM lane quarter, shared by warps q4 and q4 + 4
    const int lane_base = q4 * 32;
    const int r128 = lane_base + lane;  // row within the tile
    const uint32_t tl = (uint32_t)lane_base << 16;
    const uint32_t tS = tmem + tl + G::col_s(0) + (uint32_t)(64 * h);
    const uint32_t tP = tmem + tl + G::col_p(0) + (uint32_t)h * (G::kPCols / 2);
    const uint32_t tO = tmem + tl + G::col_o(0) + (uint32_t)(kHalfO * h);
    // exchange area: partial maxima xm[step parity][half][row], then row sums xl[half][row]
    float* xl = xch + 512;
    uint32_t s_cnt = 0, o_cnt = 0;

    for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
        const Item it = unit_item<CAUSAL, 2>(p, u, 0);
        const int n = it.nA;
        const int row = it.pair * 2 * kBM + it.sw * kBM + r128;
        const int limit = CAUSAL ? min(row + 1, p.n) : p.n;   // visible keys: j < limit
        float m_run = -INFINITY, l_half = 0.0f;
        bool live = true;

        for (int j = 0; j < n; ++j) {
            // Where P overwrites S, S(j) was issued after O += P(j-1) V(j-1) by the same
            // thread, and the commit behind s_full tracks every product issued before it:
            // O is final once S(j) is complete.
            bool ok = live && wait_warp(c, b_s_full<D, EB>(0), s_cnt & 1u, kRoleSoftmax);
            ++s_cnt;
            const int kbase = j * kBN + 64 * h;
            const bool mask = __any_sync(0xFFFFFFFFu, kbase + 64 > limit);
            uint32_t s[64];
            if (ok) {
                ptx::tc_fence_after();
                ptx::tmem_ld64_wait(tS, s);
                if constexpr (G::kSepP) {   // S may now be overwritten by the next S product
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(bar_addr(c, b_s_read<D, EB>(0)));
                }
                xch[((j & 1) * 2 + h) * 128 + r128] =
                    mask ? tile_row_max<true, 64>(s, kbase, limit) : tile_row_max<false, 64>(s, kbase, limit);
            }
            // Both warps' S loads are complete before either stores P (over S at D = 128).
            ptx::tc_fence_before();
            if (!pair_barrier_and(q4, ok)) return;
            ptx::tc_fence_after();
            const float mt = fmaxf(xch[((j & 1) * 2) * 128 + r128],
                                   xch[((j & 1) * 2 + 1) * 128 + r128]) * p.scale_log2;
            float alpha = 1.0f;
            if (mt > m_run + Lazy<ET>::kRescaleLog2) {
                alpha = ptx::ex2(m_run - mt);   // m_run = -inf on the first tile: alpha = 0
                m_run = mt;
            }
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            uint32_t pk[32];
            if (mask) tile_exp_cols<0, 64, true, ET>(s, kbase, limit, p.scale_log2, -m_run, acc, pk);
            else tile_exp_cols<0, 64, false, ET>(s, kbase, limit, p.scale_log2, -m_run, acc, pk);
            // With separate P columns, O += P(j-1) V(j-1) must be complete before P is
            // overwritten and before O is rescaled.
            if (G::kSepP && j > 0) {
                live = wait_warp(c, b_o_done<D, EB>(0), o_cnt & 1u, kRoleSoftmax);
                ++o_cnt;
                if (!live) continue;   // the next barrier ends both warps
                ptx::tc_fence_after();
            }
            __syncwarp();
            if constexpr (ET == 2) ptx::tmem_st16(tP, &pk[0]);
            else ptx::tmem_st32p(tP, &pk[0]);
            const float sum = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
            l_half = l_half * alpha + sum;
            if (j > 0 && __any_sync(0xFFFFFFFFu, alpha != 1.0f))
                rescale_o<kHalfO, kHalfO>(tO, alpha);   // the running max rose: this warp's half of the O row
            ptx::tmem_wait_st();
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar_addr(c, b_p_full<D, EB>(0)));
        }

        // Epilogue: the last O += P V, then the two halves' row sums meet.  Where P overwrites
        // S only that product is awaited (the one before it is complete, S(n-1) having been
        // issued after it), so the parity wait is exact.
        bool ok = live && wait_warp(c, b_o_done<D, EB>(0), (G::kSepP ? o_cnt : o_cnt + (uint32_t)n - 1u) & 1u,
                                    kRoleSoftmax);
        o_cnt += G::kSepP ? 1u : (uint32_t)n;
        xl[h * 128 + r128] = l_half;
        // At D = 64 both warps stage into warp q4's slot: its last bulk store has read it.
        if (OStore<D, 2>::kTma && D == 64 && h == 0 && lane == 0) bulk_wait_read_all();
        if (!pair_barrier_and(q4, ok)) return;
        ptx::tc_fence_after();
        const float l_run = xl[r128] + xl[128 + r128];
        const float inv_l = p.o_scale / l_run;   // o_scale: V's dequantisation factor (1 at 16 bits)
        const int row0 = it.pair * 2 * kBM + it.sw * kBM + lane_base;   // first row of the pair
        if constexpr (D == 128) {
            // one 64-column panel per warp, through the warp's own slot and one bulk store
            const uint32_t stage = stage_base + (uint32_t)(warp * G::kStageSlot);
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t o[32];
                ptx::tmem_ld32_wait(tO + (uint32_t)(hh * 32), o);
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    w[i] = pack2<kOutF16>(u2f(o[2 * i]) * inv_l, u2f(o[2 * i + 1]) * inv_l);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t chunk = (uint32_t)(hh * 4 + i) ^ (uint32_t)(lane & 7);
                    ptx::st_shared_v4(stage + (uint32_t)lane * 128u + chunk * 16u, w[4 * i],
                                      w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                }
            }
            fence_async_shared();
            __syncwarp();
            if (lane == 0 && row0 < p.n) {
                tma_store_3d(&p.tmap_o, stage, h * 64, row0, it.bh);
                bulk_commit();
            }
        } else {
            // D = 64: one panel, each warp stages its 32 columns (16-byte chunks 4h..4h+3);
            // D = 32: one 64-byte row, each warp stages its 16 columns (chunks 2h, 2h+1).
            const uint32_t stage = stage_base + (uint32_t)(q4 * G::kStageSlot);
            constexpr int kChunks = kHalfO / 8;   // 16-byte chunks of this warp's columns
            uint32_t o[kHalfO];
            if constexpr (kHalfO == 32) ptx::tmem_ld32_wait(tO, o);
            else ptx::tmem_ld16_wait(tO, o);
            uint32_t w[kHalfO / 2];
#pragma unroll
            for (int i = 0; i < kHalfO / 2; ++i)
                w[i] = pack2<kOutF16>(u2f(o[2 * i]) * inv_l, u2f(o[2 * i + 1]) * inv_l);
#pragma unroll
            for (int i = 0; i < kChunks; ++i) {
                const uint32_t chunk = (uint32_t)(h * kChunks + i) ^ (uint32_t)(lane & 7);
                ptx::st_shared_v4(stage + (uint32_t)lane * 128u + chunk * 16u, w[4 * i],
                                  w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
            }
            if constexpr (OStore<D, 2>::kTma) fence_async_shared();
            pair_barrier(q4);   // both halves of every row are staged
            if constexpr (OStore<D, 2>::kTma) {
                if (h == 0 && lane == 0 && row0 < p.n) {
                    tma_store_3d(&p.tmap_o, stage, 0, row0, it.bh);
                    bulk_commit();
                }
            } else {
                // 64-byte rows: 8 rows x 4 chunks per store instruction, two of the four
                // row groups per warp
                uint16_t* obase = reinterpret_cast<uint16_t*>(p.o) + (size_t)it.bh * (size_t)p.n * D;
#pragma unroll
                for (int k = 2 * h; k < 2 * h + 2; ++k) {
                    const int r = 8 * k + (lane >> 2);   // row within the warp's 32
                    const int ch = lane & 3;             // 16-byte chunk within the 64-byte row
                    const uint4 v = ptx::ld_shared_v4(stage + (uint32_t)r * 128u +
                                                      (uint32_t)((ch ^ (r & 7)) * 16));
                    if (row0 + r < p.n)
                        *reinterpret_cast<uint4*>(obase + (size_t)(row0 + r) * D + ch * 8) = v;
                }
            }
        }
        if (h == 0 && row < p.n) p.lse[(size_t)it.bh * (size_t)p.n + (size_t)row] = (m_run + log2f(l_run)) * kLn2;
        __syncwarp();
    }
}

template <int D, bool CAUSAL, int ET, int MODE>
__global__ void __launch_bounds__(kThreads, 1) fa_tc_kernel(const __grid_constant__ TcParams p) {
    constexpr int EB = Elem<ET>::kBytes;
    using G = Geo<D, EB>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = ptx::smem_addr(smem);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + G::kMiscOff);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + G::kMiscOff + 4);
    const int warp = threadIdx.x / 32;
    const int lane = threadIdx.x % 32;

    Ctl c;
    c.bars = sbase + (uint32_t)G::kBarOff;
    c.abort = abort_flag;
    c.limit = p.wait_limit;
    c.status = g_status;

    if (threadIdx.x == 0) {
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(bar_addr(c, b_q_full<D, EB>(t)), 1);
            ptx::mbar_init(bar_addr(c, b_q_empty<D, EB>(t)), 1);
            ptx::mbar_init(bar_addr(c, b_s_full<D, EB>(t)), 1);
            // the single-tile schedule's tile A is served by all eight softmax warps
            const uint32_t softmax_threads = (MODE == 2 && t == 0) ? 256u : 128u;
            ptx::mbar_init(bar_addr(c, b_p_full<D, EB>(t)), softmax_threads);
            ptx::mbar_init(bar_addr(c, b_o_done<D, EB>(t)), 1);
            ptx::mbar_init(bar_addr(c, b_s_read<D, EB>(t)), softmax_threads);
        }
        for (int s = 0; s < G::kSlots; ++s) {
            ptx::mbar_init(bar_addr(c, b_kv_full<D, EB>(s)), 1);
            ptx::mbar_init(bar_addr(c, b_kv_empty<D, EB>(s)), 1);
        }
        ptx::mbar_init(bar_addr(c, b_drain<D, EB>()), 1);
        *abort_flag = 0;
        ptx::fence_barrier_init();
    }
    if (warp == kLoadWarp && lane == 0) {
        ptx::prefetch_tensormap(&p.tmap_q);
        ptx::prefetch_tensormap(&p.tmap_k);
        ptx::prefetch_tensormap(&p.tmap_v);
        if constexpr (OStore<D, MODE>::kTma) ptx::prefetch_tensormap(&p.tmap_o);
    }
    if (warp == kMmaWarp) {
        ptx::tmem_alloc(ptx::smem_addr(tmem_slot), kTmemCols);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp < kSoftmaxWarps) {
        if constexpr (MODE == 2)   // the exchange area is the unused Q_B buffer
            softmax_role_split<D, CAUSAL, ET>(p, c, tmem, reinterpret_cast<float*>(smem + G::kTileBytes),
                                              sbase + (uint32_t)G::kStageOff, warp, lane);
        else
            softmax_role<D, CAUSAL, ET, MODE>(p, c, tmem, warp, lane,
                                              sbase + (uint32_t)G::kStageOff + (uint32_t)(warp * G::kStageSlot));
        if constexpr (OStore<D, MODE>::kTma) {   // this warp's O stores complete before exit
            if (lane == 0) bulk_wait_all();
            __syncwarp();
        }
    } else if (warp == kMmaWarp) {
        if constexpr (G::kSepP) mma_role_sep<D, CAUSAL, ET, MODE>(p, c, tmem, sbase);
        else mma_role<D, CAUSAL, ET, MODE>(p, c, tmem, sbase);
    } else {
        if (lane == 0) load_role<D, EB, CAUSAL, MODE>(p, c, sbase);
        __syncwarp();
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

template <int D, bool CAUSAL, int ET, int MODE>
cudaError_t prepare_one() {
    return cudaFuncSetAttribute(fa_tc_kernel<D, CAUSAL, ET, MODE>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Geo<D, Elem<ET>::kBytes>::kSmemBytes);
}

template <int D, bool CAUSAL, int ET, int MODE>
cudaError_t launch_one(const TcParams& p, int grid, cudaStream_t stream) {
    fa_tc_kernel<D, CAUSAL, ET, MODE>
        <<<grid, kThreads, Geo<D, Elem<ET>::kBytes>::kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

// Modes: 0 [B, H, N, D] with query-tile pairs, 2 the same layout with one query tile per
// unit, 1 token-major (16-bit storage only; e4m3 has the [B, H, N, D] modes alone).
template <int D, bool CAUSAL, int ET>
cudaError_t dispatch_mode(int mode, bool prepare, const TcParams* p, int grid, cudaStream_t stream) {
    if (prepare) {
        cudaError_t e = prepare_one<D, CAUSAL, ET, 0>();
        if (e == cudaSuccess) e = prepare_one<D, CAUSAL, ET, 2>();
        if constexpr (ET != 2)
            if (e == cudaSuccess) e = prepare_one<D, CAUSAL, ET, 1>();
        return e;
    }
    if (mode == 0) return launch_one<D, CAUSAL, ET, 0>(*p, grid, stream);
    if (mode == 2) return launch_one<D, CAUSAL, ET, 2>(*p, grid, stream);
    if constexpr (ET != 2) return launch_one<D, CAUSAL, ET, 1>(*p, grid, stream);
    return cudaErrorInvalidValue;
}

template <int D, int ET>
cudaError_t dispatch_et(bool causal, int mode, bool prepare, const TcParams* p, int grid,
                        cudaStream_t stream) {
    return causal ? dispatch_mode<D, true, ET>(mode, prepare, p, grid, stream)
                  : dispatch_mode<D, false, ET>(mode, prepare, p, grid, stream);
}

template <int D>
cudaError_t dispatch(bool causal, int et, int mode, bool prepare, const TcParams* p, int grid,
                     cudaStream_t stream) {
    if (et == 1) return dispatch_et<D, 1>(causal, mode, prepare, p, grid, stream);
    if (et == 2) return dispatch_et<D, 2>(causal, mode, prepare, p, grid, stream);
    return dispatch_et<D, 0>(causal, mode, prepare, p, grid, stream);
}

}  // namespace

int tc_units(int bh, int n, bool causal) {
    const long long npairs = (n + 2 * kBM - 1) / (2 * kBM);
    const long long u = causal ? (long long)bh * ((npairs + 1) / 2) : (long long)bh * npairs;
    return u > 0x7FFFFFFFLL ? -1 : (int)u;
}

int tc_smem_bytes(int D) {
    return D == 32 ? Geo<32, 2>::kSmemBytes : D == 64 ? Geo<64, 2>::kSmemBytes : Geo<128, 2>::kSmemBytes;
}

cudaError_t tc_prepare(int D, bool causal, int et) {
    if (D == 32) return dispatch<32>(causal, et, 0, true, nullptr, 0, nullptr);
    return D == 64 ? dispatch<64>(causal, et, 0, true, nullptr, 0, nullptr)
                   : dispatch<128>(causal, et, 0, true, nullptr, 0, nullptr);
}

cudaError_t tc_launch(int D, bool causal, int et, const TcParams& p, bool single, int grid,
                      cudaStream_t stream) {
    const int mode = p.layout == 0 && single ? 2 : p.layout;
    if (D == 32) return dispatch<32>(causal, et, mode, false, &p, grid, stream);
    return D == 64 ? dispatch<64>(causal, et, mode, false, &p, grid, stream)
                   : dispatch<128>(causal, et, mode, false, &p, grid, stream);
}

cudaError_t tc_status_read_reset(uint32_t out[4]) {
    cudaError_t e = cudaMemcpyFromSymbol(out, g_status, sizeof(unsigned int) * 4);
    if (e != cudaSuccess) return e;
    const unsigned int zero[4] = {0, 0, 0, 0};
    return cudaMemcpyToSymbol(g_status, zero, sizeof(zero));
}

}  // namespace fa
