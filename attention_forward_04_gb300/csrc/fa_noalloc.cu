// fa_noalloc.cu -- fa_bwd_noalloc: the backward with its scratch in static device memory.
//
// fa_bwd takes its delta scratch from the caller.  Some callers cannot hand one over:
// code that runs while a memory pool owns every free byte of HBM, code invoked from inside
// an allocator (where allocating again would re-enter it), and code on a latency-critical
// stream that must not pay for cudaMalloc, which can block the host and serialise the
// device.  For them this entry point takes the scratch from one fixed array that the
// library itself defines, so the call allocates nothing.  Its size bounds the problems it
// serves; larger ones are refused before any CUDA call.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "fa.h"

namespace {

constexpr int64_t kScratchBytes = FA_BWD_NOALLOC_MAX_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// One copy per device, created when the library's device code is loaded on that device.
// Nothing in it has to start at zero: the dQ kernel writes every delta row before the dK/dV
// kernel reads it.
static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

// Per device: the array's address once a lookup has succeeded.  A failed lookup (for
// instance an out-of-memory error while the driver loads the library's device code, or a
// call made during stream capture) is not remembered, so a later call retries it.
std::mutex g_scratch_mu;
void* g_scratch[kMaxDevices] = {};

// Checks shared by the three entry points, before any CUDA call: pointers, flags, D, and
// the scratch the call needs (`need`, from fa_bwd_workspace_bytes for its layout).
int check_common(const void* const* ptrs, int64_t need, int64_t D, float scale, int causal,
                 int dtype) {
    for (int a = 0; a < 9; ++a)
        if (!ptrs[a]) return FA_ERR_INVALID_ARG;
    if (need < 0) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (dtype != FA_FP32 && dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_INVALID_ARG;
    if (!std::isfinite(scale) || scale < 0.0f) return FA_ERR_INVALID_ARG;   // as fa_bwd
    if (D != 32 && D != 64 && D != 128 && D != 256) return FA_ERR_UNSUPPORTED;
    if (need > kScratchBytes) return FA_ERR_UNSUPPORTED;
    return FA_OK;
}

// This device's copy of the array (looked up once per device), or null with `status` set.
void* scratch(int* status) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        *status = FA_ERR_CUDA;
        return nullptr;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        *status = FA_ERR_UNSUPPORTED;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch[dev] == nullptr) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_bwd_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();   // leave no sticky error behind for the caller's next call
            *status = FA_ERR_CUDA;
            return nullptr;
        }
        g_scratch[dev] = ptr;
    }
    return g_scratch[dev];
}

}  // namespace

// fa_bwd, fa_bwd_bnhd and fa_bwd_varlen repeat the host checks and add the overlap and
// alignment checks.
extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const void* dout, const float* lse, void* dq, void* dk, void* dv,
                              int64_t B, int64_t H, int64_t N, int64_t D, float scale,
                              int causal, int dtype, void* stream) {
    const void* ptrs[9] = {q, k, v, o, dout, lse, dq, dk, dv};
    const int64_t need = fa_bwd_workspace_bytes(B, H, N);
    int st = check_common(ptrs, need, D, scale, causal, dtype);
    if (st != FA_OK) return st;
    void* ws = scratch(&st);
    if (!ws) return st;
    return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, ws, need, B, H, N, D, scale, causal,
                  dtype, stream);
}

extern "C" int fa_bwd_noalloc_bnhd(const void* q, const void* k, const void* v, const void* o,
                                   const void* dout, const float* lse, void* dq, void* dk,
                                   void* dv, int64_t B, int64_t N, int64_t H, int64_t D,
                                   float scale, int causal, int dtype, void* stream) {
    const void* ptrs[9] = {q, k, v, o, dout, lse, dq, dk, dv};
    const int64_t need = fa_bwd_workspace_bytes(B, H, N);
    int st = check_common(ptrs, need, D, scale, causal, dtype);
    if (st != FA_OK) return st;
    void* ws = scratch(&st);
    if (!ws) return st;
    return fa_bwd_bnhd(q, k, v, o, dout, lse, dq, dk, dv, ws, need, B, N, H, D, scale, causal,
                       dtype, stream);
}

extern "C" int fa_bwd_noalloc_varlen(const void* q, const void* k, const void* v, const void* o,
                                     const void* dout, const float* lse, void* dq, void* dk,
                                     void* dv, const int32_t* cu_seqlens, int64_t batch,
                                     int64_t max_seqlen, int64_t total, int64_t H, int64_t D,
                                     float scale, int causal, int dtype, void* stream) {
    const void* ptrs[9] = {q, k, v, o, dout, lse, dq, dk, dv};
    if (!cu_seqlens) return FA_ERR_INVALID_ARG;
    // delta is indexed like the packed LSE, [H, total]
    const int64_t need = fa_bwd_workspace_bytes(1, H, total);
    if (fa_bwd_workspace_bytes(batch, H, max_seqlen) < 0) return FA_ERR_INVALID_ARG;
    int st = check_common(ptrs, need, D, scale, causal, dtype);
    if (st != FA_OK) return st;
    void* ws = scratch(&st);
    if (!ws) return st;
    return fa_bwd_varlen(q, k, v, o, dout, lse, dq, dk, dv, ws, need, cu_seqlens, batch,
                         max_seqlen, total, H, D, scale, causal, dtype, stream);
}
