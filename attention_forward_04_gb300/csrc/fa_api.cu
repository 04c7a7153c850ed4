// fa_api.cu -- the C ABI (include/fa.h): argument checks, TMA descriptor encoding,
// persistent-grid sizing and kernel dispatch.  No call allocates device memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultWaitLimit = 1ull << 32;  // SM cycles (~2 s)

thread_local char g_last_cuda_error[256] = "";

std::atomic<unsigned long long> g_wait_limit{kDefaultWaitLimit};
std::atomic<int> g_inject_stall{0};

struct DeviceInfo {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    int sm_count = 0;
    int major = 0, minor = 0;
    std::once_flag prepared[3][2][3];  // [D = 32, 64, 128][causal][bf16, fp16, fp8]
    cudaError_t prepare_err[3][2][3] = {};
    std::once_flag bwd_prepared[4][2][2];   // [D = 32, 64, 128, 256][causal][f16]
    cudaError_t bwd_prepare_err[4][2][2] = {};
    std::once_flag prepared256[2][3];  // [causal][element type]
    cudaError_t prepare256_err[2][3] = {};
};
DeviceInfo g_dev[kMaxDevices];

int fail_cuda(cudaError_t e, const char* what) {
    std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s (%d)", what,
                  cudaGetErrorString(e), (int)e);
    return FA_ERR_CUDA;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn(cudaError_t* err) {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static cudaError_t e0 = cudaSuccess;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        e0 = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                              &q);
        if (e0 == cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else if (e0 == cudaSuccess)
            e0 = cudaErrorSymbolNotFound;
    });
    *err = e0;
    return fn;
}

// 16-bit tensor viewed as a 3-D TMA map whose box lands in shared memory as 128 rows of
// 64 head-dim values (128 bytes, 128-byte swizzle), which the tensor-core kernel expects.
//   layout 0, [B*H, N, D]: dims {D, N, B*H}, box {64, rows, 1} (rows = 128, 64 for the
//   D = 256 kernel, 32 for the forward's O stores); rows past N read as zero (and are not
//   written by a store).
//   Shorter rows: the box is one whole row wide, 64-byte rows (D = 32 at 16 bits, D = 64
//   at e4m3) with the 64-byte swizzle, 32-byte rows (D = 32 at e4m3) with the 32-byte one.
//   layout 1, token-major [T, H, D]: dims {D, H, T}, box {64, 1, rows}; tokens past T read
//   as zero (tokens of the next packed sequence are masked by the kernel instead).
bool encode_map(CUtensorMap* map, const void* base, int layout, int64_t bh, int64_t n, int64_t h,
                int64_t t, int64_t d, int et, PFN_cuTensorMapEncodeTiled_v12000 fn,
                cuuint32_t rows = 128) {
    // et: 0 bf16, 1 fp16, 2 fp8 e4m3 (raw bytes).  The box spans one panel: 128-byte rows
    // (128-byte swizzle), or whole rows of 64 or 32 bytes (swizzle of the row width).
    const int64_t eb = et == 2 ? 1 : 2;
    const int64_t row_bytes = d * eb < 128 ? d * eb : 128;
    const cuuint32_t box0 = (cuuint32_t)(row_bytes / eb);
    cuuint64_t dims[3], strides[2];
    cuuint32_t box[3];
    if (layout == 0) {
        dims[0] = (cuuint64_t)d; dims[1] = (cuuint64_t)n; dims[2] = (cuuint64_t)bh;
        strides[0] = (cuuint64_t)(d * eb); strides[1] = (cuuint64_t)(n * d * eb);
        box[0] = box0; box[1] = rows; box[2] = 1;
    } else {
        dims[0] = (cuuint64_t)d; dims[1] = (cuuint64_t)h; dims[2] = (cuuint64_t)t;
        strides[0] = (cuuint64_t)(d * eb); strides[1] = (cuuint64_t)(h * d * eb);
        box[0] = box0; box[1] = 1; box[2] = rows;
    }
    cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType type = et == 2   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                     : et == 1 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                               : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUresult r = fn(map, type, 3, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE,
                    row_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                    : row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                      : CU_TENSOR_MAP_SWIZZLE_32B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

}  // namespace

extern "C" {

int fa_version(void) { return 140; }

const char* fa_status_string(int status) {
    switch (status) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
        case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED";
        case FA_ERR_CUDA: return "FA_ERR_CUDA";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
        default: return "FA_ERR_UNKNOWN";
    }
}

const char* fa_last_cuda_error(void) { return g_last_cuda_error; }

int fa_set_watchdog(uint64_t wait_limit_cycles, int inject_stall) {
    if (inject_stall != 0 && inject_stall != 1) return FA_ERR_INVALID_ARG;
    g_wait_limit.store(wait_limit_cycles ? (unsigned long long)wait_limit_cycles : kDefaultWaitLimit);
    g_inject_stall.store(inject_stall);
    return FA_OK;
}

int fa_check_device_status(void* stream, uint32_t* detail) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
    uint32_t w[4] = {0, 0, 0, 0}, wb[4] = {0, 0, 0, 0}, w256[4] = {0, 0, 0, 0},
             wb256[4] = {0, 0, 0, 0};
    e = fa::tc_status_read_reset(w);
    if (e == cudaSuccess) e = fa::bwd_status_read_reset(wb);
    if (e == cudaSuccess) e = fa::tc256_status_read_reset(w256);
    if (e == cudaSuccess) e = fa::bwd256_status_read_reset(wb256);
    if (e != cudaSuccess) return fail_cuda(e, "status word");
    if (!(w[0] & 1u) && (wb[0] & 1u)) std::memcpy(w, wb, sizeof(w));   // report the backward's
    if (!(w[0] & 1u) && (w256[0] & 1u)) std::memcpy(w, w256, sizeof(w));
    if (!(w[0] & 1u) && (wb256[0] & 1u)) std::memcpy(w, wb256, sizeof(w));
    if (detail) std::memcpy(detail, w, sizeof(w));
    return (w[0] & 1u) ? FA_ERR_TIMEOUT : FA_OK;
}

}  // extern "C"

namespace {

// One forward request in any of the three layouts.
struct Request {
    const void *q, *k, *v;
    void* o;
    float* lse;
    int64_t B, H, N, D;    // N: sequence length, or the longest packed sequence
    int64_t T;             // token-major layouts: tokens (B*N, or the packed total)
    int layout;            // 0: [B, H, N, D]; 1: token-major [T, H, D]
    const int* cu;         // packed sequences: [B + 1] token offsets (device), else null
    float scale;
    int causal, dtype;     // dtype: an fa_dtype, or kFp8 (e4m3 in, bf16 out)
    void* stream;
    float descale[3];      // fp8: dequantisation factors of Q, K, V (else 1)
};

constexpr int kFp8 = 3;

int forward(const Request& r) {
    // ---- argument checks: no CUDA call before these pass
    if (!r.q || !r.k || !r.v || !r.o || !r.lse) return FA_ERR_INVALID_ARG;
    if (r.B < 1 || r.H < 1 || r.N < 1 || r.T < 1) return FA_ERR_INVALID_ARG;
    if (r.B > 0x7FFFFFFFLL || r.H > 0x7FFFFFFFLL || r.B * r.H > 0x7FFFFFFFLL ||
        r.N > 0x7FFFFFFFLL || r.T > 0x7FFFFFFFLL)
        return FA_ERR_INVALID_ARG;
    if (r.causal != 0 && r.causal != 1) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(r.scale) || r.scale < 0.0f) return FA_ERR_INVALID_ARG;
    if (r.dtype != FA_FP32 && r.dtype != FA_BF16 && r.dtype != FA_FP16 && r.dtype != kFp8)
        return FA_ERR_INVALID_ARG;
    for (int i = 0; i < 3; ++i)
        if (!std::isfinite(r.descale[i]) || !(r.descale[i] > 0.0f)) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(r.scale * r.descale[0] * r.descale[1])) return FA_ERR_INVALID_ARG;
    if (r.D != 32 && r.D != 64 && r.D != 128 && r.D != 256) return FA_ERR_UNSUPPORTED;
    // fp8: [B, H, N, D] layout only
    if (r.dtype == kFp8 && r.layout != 0) return FA_ERR_UNSUPPORTED;
    const int64_t BH = r.B * r.H;
    const size_t esize = r.dtype == FA_FP32 ? 4 : r.dtype == kFp8 ? 1 : 2;   // Q, K, V
    const size_t osize = r.dtype == FA_FP32 ? 4 : 2;                          // O
    const int64_t rows = r.layout == 0 ? BH * r.N : r.T * r.H;   // rows of D elements
    if (rows / r.H != (r.layout == 0 ? r.B * r.N : r.T)) return FA_ERR_INVALID_ARG;
    const size_t tbytes = (size_t)rows * (size_t)r.D * esize;
    const size_t obytes = (size_t)rows * (size_t)r.D * osize;
    const size_t lbytes = (size_t)(r.cu ? r.T * r.H : BH * r.N) * sizeof(float);
    if (obytes / osize / (size_t)r.D != (size_t)rows) return FA_ERR_INVALID_ARG;
    if (overlaps(r.o, obytes, r.q, tbytes) || overlaps(r.o, obytes, r.k, tbytes) ||
        overlaps(r.o, obytes, r.v, tbytes) || overlaps(r.lse, lbytes, r.q, tbytes) ||
        overlaps(r.lse, lbytes, r.k, tbytes) || overlaps(r.lse, lbytes, r.v, tbytes) ||
        overlaps(r.lse, lbytes, r.o, obytes))
        return FA_ERR_INVALID_ARG;
    for (const void* ptr : {r.q, r.k, r.v, static_cast<const void*>(r.o)})
        if (reinterpret_cast<uintptr_t>(ptr) & 15u) return FA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(r.lse) & 3u) || (reinterpret_cast<uintptr_t>(r.cu) & 3u))
        return FA_ERR_MISALIGNED;
    const bool tc = r.dtype != FA_FP32;
    int units = 0;
    if (tc && r.D != 256) {
        units = fa::tc_units((int)BH, (int)r.N, r.causal != 0);
        if (units < 0) return FA_ERR_UNSUPPORTED;
    }

    // ---- device properties (once per device)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    DeviceInfo& di = g_dev[dev];
    std::call_once(di.once, [&] {
        di.err = cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (di.err == cudaSuccess)
            di.err = cudaDeviceGetAttribute(&di.major, cudaDevAttrComputeCapabilityMajor, dev);
        if (di.err == cudaSuccess)
            di.err = cudaDeviceGetAttribute(&di.minor, cudaDevAttrComputeCapabilityMinor, dev);
    });
    if (di.err != cudaSuccess) return fail_cuda(di.err, "cudaDeviceGetAttribute");
    if (di.major != 10 || di.minor != 3) return FA_ERR_UNSUPPORTED;  // built for sm_103a only
    cudaStream_t st = static_cast<cudaStream_t>(r.stream);

    fa::SliceLayout g;
    g.layout = r.layout;
    g.cu_seqlens = r.cu;
    g.heads = (int)r.H;
    g.total = (int)r.T;
    g.n = (int)r.N;

    if (!tc) {
        e = fa::simt_launch((int)r.D, r.causal != 0, static_cast<const float*>(r.q),
                            static_cast<const float*>(r.k), static_cast<const float*>(r.v),
                            static_cast<float*>(r.o), r.lse, (int)BH, g, r.scale, di.sm_count, st);
        return e == cudaSuccess ? FA_OK : fail_cuda(e, "fp32 kernel launch");
    }

    const bool f16 = r.dtype == FA_FP16;
    const int et = r.dtype == kFp8 ? 2 : f16 ? 1 : 0;   // element type of Q, K, V
    const int dix = r.D == 32 ? 0 : r.D == 64 ? 1 : 2, dic = r.causal != 0, dif = et;
    if (r.D == 256) {
        std::call_once(di.prepared256[dic][dif],
                       [&] { di.prepare256_err[dic][dif] = fa::tc256_prepare(dic, et); });
        if (di.prepare256_err[dic][dif] != cudaSuccess)
            return fail_cuda(di.prepare256_err[dic][dif], "cudaFuncSetAttribute (D = 256)");
        PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn(&e);
        if (!fn) return fail_cuda(e, "cuTensorMapEncodeTiled entry point");
        fa::TcParams p;
        std::memset(&p, 0, sizeof(p));
        if (!encode_map(&p.tmap_q, r.q, r.layout, BH, r.N, r.H, r.T, r.D, et, fn, 64) ||
            !encode_map(&p.tmap_k, r.k, r.layout, BH, r.N, r.H, r.T, r.D, et, fn, 64) ||
            !encode_map(&p.tmap_v, r.v, r.layout, BH, r.N, r.H, r.T, r.D, et, fn, 64))
            return fail_cuda(cudaErrorInvalidValue, "cuTensorMapEncodeTiled");
        p.o = r.o;
        p.lse = r.lse;
        p.layout = r.layout;
        p.cu_seqlens = r.cu;
        p.heads = (int)r.H;
        p.total = (int)r.T;
        p.n = (int)r.N;
        p.bh = (int)BH;
        p.scale_log2 = r.scale * r.descale[0] * r.descale[1] * 1.4426950408889634f;
        p.o_scale = r.descale[2];
        p.wait_limit = g_wait_limit.load();
        p.units = fa::tc256_units((int)BH, (int)r.N, dic != 0);
        if (p.units < 1) return FA_ERR_UNSUPPORTED;
        const int grid = p.units < di.sm_count ? p.units : di.sm_count;
        e = fa::tc256_launch(dic, et, p, grid, st);
        return e == cudaSuccess ? FA_OK : fail_cuda(e, "tensor-core kernel launch (D = 256)");
    }
    std::call_once(di.prepared[dix][dic][dif],
                   [&] { di.prepare_err[dix][dic][dif] = fa::tc_prepare((int)r.D, dic, et); });
    if (di.prepare_err[dix][dic][dif] != cudaSuccess)
        return fail_cuda(di.prepare_err[dix][dic][dif], "cudaFuncSetAttribute");

    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn(&e);
    if (!fn) return fail_cuda(e, "cuTensorMapEncodeTiled entry point");
    fa::TcParams p;
    std::memset(&p, 0, sizeof(p));
    if (!encode_map(&p.tmap_q, r.q, r.layout, BH, r.N, r.H, r.T, r.D, et, fn) ||
        !encode_map(&p.tmap_k, r.k, r.layout, BH, r.N, r.H, r.T, r.D, et, fn) ||
        !encode_map(&p.tmap_v, r.v, r.layout, BH, r.N, r.H, r.T, r.D, et, fn))
        return fail_cuda(cudaErrorInvalidValue, "cuTensorMapEncodeTiled");
    // O of [B, H, N, D] problems at D >= 64 leaves through bulk tensor stores of 32-row
    // panels (O is fp16 for fp16 storage, else bf16)
    if (r.layout == 0 && r.D >= 64 &&
        !encode_map(&p.tmap_o, r.o, 0, BH, r.N, r.H, r.T, r.D, f16 ? 1 : 0, fn, 32))
        return fail_cuda(cudaErrorInvalidValue, "cuTensorMapEncodeTiled (O)");
    p.o = r.o;
    p.lse = r.lse;
    p.layout = r.layout;
    p.cu_seqlens = r.cu;
    p.heads = (int)r.H;
    p.total = (int)r.T;
    p.n = (int)r.N;
    p.bh = (int)BH;
    p.npairs = (int)((r.N + 255) / 256);
    p.nkv = (int)((r.N + 127) / 128);
    // [B, H, N, D] with B*H*ceil(N/128) <= #SM: one query tile per unit, so every tile runs
    // at once on an SM of its own; otherwise pairs of query tiles.
    const long long single_units = BH * (long long)p.nkv;
    const bool single = r.layout == 0 && single_units <= (long long)di.sm_count;
    p.units = single ? (int)single_units : units;
    p.scale_log2 = r.scale * r.descale[0] * r.descale[1] * 1.4426950408889634f;
    p.o_scale = r.descale[2];
    p.wait_limit = g_wait_limit.load();
    p.inject_stall = g_inject_stall.load();
    const int grid = p.units < di.sm_count ? p.units : di.sm_count;
    e = fa::tc_launch((int)r.D, dic, et, p, single, grid, st);
    return e == cudaSuccess ? FA_OK : fail_cuda(e, "tensor-core kernel launch");
}

}  // namespace

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B, int64_t H,
           int64_t N, int64_t D, float scale, int causal, int dtype, void* stream) {
    if (dtype == kFp8) return FA_ERR_INVALID_ARG;   // e4m3 input only through fa_fwd_fp8
    const Request r{q, k, v, o, lse, B, H, N, D, B * N, 0, nullptr, scale, causal, dtype, stream,
                    {1.0f, 1.0f, 1.0f}};
    return forward(r);
}

int fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
               int64_t H, int64_t N, int64_t D, float scale, int causal, float q_descale,
               float k_descale, float v_descale, void* stream) {
    const Request r{q, k, v, o, lse, B, H, N, D, B * N, 0, nullptr, scale, causal, kFp8, stream,
                    {q_descale, k_descale, v_descale}};
    return forward(r);
}

int fa_fwd_bnhd(const void* q, const void* k, const void* v, void* o, float* lse, int64_t B,
                int64_t N, int64_t H, int64_t D, float scale, int causal, int dtype, void* stream) {
    if (dtype == kFp8) return FA_ERR_INVALID_ARG;   // e4m3 input only through fa_fwd_fp8
    const Request r{q, k, v, o, lse, B, H, N, D, B * N, 1, nullptr, scale, causal, dtype, stream,
                    {1.0f, 1.0f, 1.0f}};
    return forward(r);
}

int64_t fa_bwd_workspace_bytes(int64_t B, int64_t H, int64_t N) {
    if (B < 1 || H < 1 || N < 1 || B > 0x7FFFFFFFLL || H > 0x7FFFFFFFLL || N > 0x7FFFFFFFLL ||
        B * H > 0x7FFFFFFFLL)
        return -1;
    const int64_t bytes = B * H * N * (int64_t)sizeof(float);   // delta rows
    return (bytes + 255) / 256 * 256;
}

}  // extern "C"

namespace {

// One backward request: [B, H, N, D] (layout 0), token-major [B, N, H, D] (layout 1, cu
// null, T = B*N) or packed sequences (layout 1, cu set, B = batch, N = max_seqlen, T = total).
struct BwdRequest {
    const void *q, *k, *v, *o, *dout;
    const float* lse;
    void *dq, *dk, *dv, *workspace;
    int64_t workspace_bytes, B, H, N, D, T;
    int layout;
    const int32_t* cu;
    float scale;
    int causal, dtype;
    void* stream;
};

int backward(const BwdRequest& r) {
    // ---- argument checks: no CUDA call before these pass
    if (!r.q || !r.k || !r.v || !r.o || !r.dout || !r.lse || !r.dq || !r.dk || !r.dv || !r.workspace)
        return FA_ERR_INVALID_ARG;
    const bool packed = r.cu != nullptr;
    if (r.layout == 1 && packed && (r.T < 1 || r.T > 0x7FFFFFFFLL)) return FA_ERR_INVALID_ARG;
    // delta is indexed like the LSE: [B*H, N], or [H, total] for packed sequences
    const int64_t need = packed ? fa_bwd_workspace_bytes(1, r.H, r.T) : fa_bwd_workspace_bytes(r.B, r.H, r.N);
    if (need < 0 || fa_bwd_workspace_bytes(r.B, r.H, r.N) < 0) return FA_ERR_INVALID_ARG;
    if (r.workspace_bytes < need) return FA_ERR_INVALID_ARG;
    if (r.causal != 0 && r.causal != 1) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(r.scale) || r.scale < 0.0f) return FA_ERR_INVALID_ARG;
    if (r.dtype != FA_FP32 && r.dtype != FA_BF16 && r.dtype != FA_FP16) return FA_ERR_INVALID_ARG;
    if (r.D != 32 && r.D != 64 && r.D != 128 && r.D != 256) return FA_ERR_UNSUPPORTED;
    const size_t esize = r.dtype == FA_FP32 ? 4 : 2;
    if (r.layout == 1 && !packed && r.B * r.N > 0x7FFFFFFFLL) return FA_ERR_INVALID_ARG;   // tokens
    const int64_t BH = r.B * r.H;
    const int64_t rows = packed ? r.T * r.H : BH * r.N;         // query rows in the tensors
    const size_t tbytes = (size_t)rows * (size_t)r.D * esize;
    const size_t lbytes = (size_t)rows * sizeof(float);
    if (tbytes / esize / (size_t)r.D != (size_t)rows) return FA_ERR_INVALID_ARG;
    const void* ins[7] = {r.q, r.k, r.v, r.o, r.dout, r.lse, r.workspace};
    const size_t in_bytes[7] = {tbytes, tbytes, tbytes, tbytes, tbytes, lbytes, (size_t)need};
    void* outs[3] = {r.dq, r.dk, r.dv};
    for (int a = 0; a < 3; ++a) {
        for (int b = 0; b < 7; ++b)
            if (overlaps(outs[a], tbytes, ins[b], in_bytes[b])) return FA_ERR_INVALID_ARG;
        for (int b = a + 1; b < 3; ++b)
            if (overlaps(outs[a], tbytes, outs[b], tbytes)) return FA_ERR_INVALID_ARG;
    }
    for (const void* t : {r.q, r.k, r.v, r.o, r.dout, static_cast<const void*>(r.lse)})
        if (overlaps(r.workspace, (size_t)need, t, t == static_cast<const void*>(r.lse) ? lbytes : tbytes))
            return FA_ERR_INVALID_ARG;
    for (const void* ptr : {r.q, r.k, r.v, r.o, r.dout, static_cast<const void*>(r.dq),
                            static_cast<const void*>(r.dk), static_cast<const void*>(r.dv)})
        if (reinterpret_cast<uintptr_t>(ptr) & 15u) return FA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(r.lse) & 3u) || (reinterpret_cast<uintptr_t>(r.workspace) & 15u) ||
        (reinterpret_cast<uintptr_t>(r.cu) & 3u))
        return FA_ERR_MISALIGNED;

    // ---- device
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    DeviceInfo& di = g_dev[dev];
    std::call_once(di.once, [&] {
        di.err = cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (di.err == cudaSuccess)
            di.err = cudaDeviceGetAttribute(&di.major, cudaDevAttrComputeCapabilityMajor, dev);
        if (di.err == cudaSuccess)
            di.err = cudaDeviceGetAttribute(&di.minor, cudaDevAttrComputeCapabilityMinor, dev);
    });
    if (di.err != cudaSuccess) return fail_cuda(di.err, "cudaDeviceGetAttribute");
    if (di.major != 10 || di.minor != 3) return FA_ERR_UNSUPPORTED;
    if (r.dtype == FA_FP32) {   // fp32 storage: the CUDA-core kernels
        fa::SliceLayout g;
        g.layout = r.layout;
        g.cu_seqlens = r.cu;
        g.heads = (int)r.H;
        g.total = (int)r.T;
        g.n = (int)r.N;
        e = fa::simt_bwd_launch((int)r.D, r.causal != 0, static_cast<const float*>(r.q),
                                static_cast<const float*>(r.k), static_cast<const float*>(r.v),
                                static_cast<const float*>(r.o), static_cast<const float*>(r.dout),
                                r.lse, static_cast<float*>(r.workspace), static_cast<float*>(r.dq),
                                static_cast<float*>(r.dk), static_cast<float*>(r.dv), (int)BH, g,
                                r.scale, di.sm_count, static_cast<cudaStream_t>(r.stream));
        return e == cudaSuccess ? FA_OK : fail_cuda(e, "CUDA-core backward kernel launch");
    }
    const bool f16 = r.dtype == FA_FP16;
    const bool d256 = r.D == 256;
    const int dix = r.D == 32 ? 0 : r.D == 64 ? 1 : r.D == 128 ? 2 : 3, dic = r.causal != 0, dif = f16;
    std::call_once(di.bwd_prepared[dix][dic][dif], [&] {
        di.bwd_prepare_err[dix][dic][dif] = d256 ? fa::bwd256_prepare(dic, f16)
                                                 : fa::bwd_prepare((int)r.D, dic, f16);
    });
    if (di.bwd_prepare_err[dix][dic][dif] != cudaSuccess)
        return fail_cuda(di.bwd_prepare_err[dix][dic][dif], "cudaFuncSetAttribute (backward)");
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn(&e);
    if (!fn) return fail_cuda(e, "cuTensorMapEncodeTiled entry point");

    fa::BwdParams p;
    std::memset(&p, 0, sizeof(p));
    const int et = f16 ? 1 : 0;
    const cuuint32_t box_rows = d256 ? 64 : 128;   // D = 256 streams 64-row sub-tiles
    if (!encode_map(&p.tmap_q, r.q, r.layout, BH, r.N, r.H, r.T, r.D, et, fn, box_rows) ||
        !encode_map(&p.tmap_k, r.k, r.layout, BH, r.N, r.H, r.T, r.D, et, fn, box_rows) ||
        !encode_map(&p.tmap_v, r.v, r.layout, BH, r.N, r.H, r.T, r.D, et, fn, box_rows) ||
        !encode_map(&p.tmap_do, r.dout, r.layout, BH, r.N, r.H, r.T, r.D, et, fn, box_rows))
        return fail_cuda(cudaErrorInvalidValue, "cuTensorMapEncodeTiled");
    p.lse = r.lse;
    p.o = r.o;
    p.q = r.q;
    p.dout = r.dout;
    p.delta = static_cast<float*>(r.workspace);
    p.dq = r.dq;
    p.dk = r.dk;
    p.dv = r.dv;
    p.n = (int)r.N;
    p.ntiles = (int)((r.N + 127) / 128);
    p.scale = r.scale;
    p.scale_log2 = r.scale * 1.4426950408889634f;
    p.wait_limit = g_wait_limit.load();
    p.layout = r.layout;
    p.heads = (int)r.H;
    p.total = (int)r.T;
    p.cu_seqlens = r.cu;
    p.inject_stall = g_inject_stall.load();
    cudaStream_t st = static_cast<cudaStream_t>(r.stream);
    e = d256 ? fa::bwd256_launch(dic, f16, p, (int)BH, st) : fa::bwd_launch((int)r.D, dic, f16, p, (int)BH, st);
    return e == cudaSuccess ? FA_OK : fail_cuda(e, "backward kernel launch");
}

}  // namespace

extern "C" {

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv, void* workspace, int64_t workspace_bytes,
           int64_t B, int64_t H, int64_t N, int64_t D, float scale, int causal, int dtype,
           void* stream) {
    if (B < 1 || N < 1 || B > 0x7FFFFFFFLL || N > 0x7FFFFFFFLL) return FA_ERR_INVALID_ARG;
    const BwdRequest r{q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes,
                       B, H, N, D, B * N, 0, nullptr, scale, causal, dtype, stream};
    return backward(r);
}

int fa_bwd_bnhd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                const float* lse, void* dq, void* dk, void* dv, void* workspace,
                int64_t workspace_bytes, int64_t B, int64_t N, int64_t H, int64_t D, float scale,
                int causal, int dtype, void* stream) {
    if (B < 1 || N < 1 || B > 0x7FFFFFFFLL || N > 0x7FFFFFFFLL) return FA_ERR_INVALID_ARG;
    const BwdRequest r{q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes,
                       B, H, N, D, B * N, 1, nullptr, scale, causal, dtype, stream};
    return backward(r);
}

int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dout,
                  const float* lse, void* dq, void* dk, void* dv, void* workspace,
                  int64_t workspace_bytes, const int32_t* cu_seqlens, int64_t batch,
                  int64_t max_seqlen, int64_t total, int64_t H, int64_t D, float scale,
                  int causal, int dtype, void* stream) {
    if (!cu_seqlens) return FA_ERR_INVALID_ARG;
    const BwdRequest r{q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes,
                       batch, H, max_seqlen, D, total, 1, cu_seqlens, scale, causal, dtype, stream};
    return backward(r);
}

int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                  const int32_t* cu_seqlens, int64_t batch, int64_t max_seqlen, int64_t total,
                  int64_t H, int64_t D, float scale, int causal, int dtype, void* stream) {
    if (!cu_seqlens) return FA_ERR_INVALID_ARG;
    if (dtype == kFp8) return FA_ERR_INVALID_ARG;   // e4m3 input only through fa_fwd_fp8
    const Request r{q, k, v, o, lse, batch, H, max_seqlen, D, total, 1, cu_seqlens, scale, causal,
                    dtype, stream, {1.0f, 1.0f, 1.0f}};
    return forward(r);
}

}  // extern "C"
