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

struct ScratchSlot {
    std::once_flag once;
    cudaError_t err = cudaSuccess;
    void* ptr = nullptr;
};
ScratchSlot g_scratch[kMaxDevices];

}  // namespace

extern "C" int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                              const void* dout, const float* lse, void* dq, void* dk, void* dv,
                              int64_t B, int64_t H, int64_t N, int64_t D, float scale,
                              int causal, int dtype, void* stream) {
    // Host checks before any CUDA call; fa_bwd repeats them and adds the overlap and
    // alignment checks.
    if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
    const int64_t need = fa_bwd_workspace_bytes(B, H, N);
    if (need < 0) return FA_ERR_INVALID_ARG;
    if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
    if (dtype != FA_FP32 && dtype != FA_BF16 && dtype != FA_FP16) return FA_ERR_INVALID_ARG;
    if (!(scale >= 0.0f) || scale > 3.4e38f) return FA_ERR_INVALID_ARG;   // NaN, inf, < 0
    if (D != 32 && D != 64 && D != 128) return FA_ERR_UNSUPPORTED;
    if (need > kScratchBytes) return FA_ERR_UNSUPPORTED;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return FA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
    // Once per device: the address of this device's copy of the array.
    ScratchSlot& s = g_scratch[dev];
    std::call_once(s.once, [&] { s.err = cudaGetSymbolAddress(&s.ptr, g_bwd_scratch); });
    if (s.err != cudaSuccess || !s.ptr) return FA_ERR_CUDA;
    return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, s.ptr, need, B, H, N, D, scale, causal,
                  dtype, stream);
}
