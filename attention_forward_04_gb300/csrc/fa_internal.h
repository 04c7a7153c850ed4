// fa_internal.h -- declarations shared by the C-ABI layer (fa_api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Launch parameters of the tensor-core kernel (bf16/fp16 storage, D = 64 or 128).
struct TcParams {
    CUtensorMap tmap_q;  // 3-D maps over the [B*H, N, D] view, innermost D; box {64, 128, 1},
    CUtensorMap tmap_k;  // 128-byte swizzle, zero fill outside the tensor (ragged N)
    CUtensorMap tmap_v;
    CUtensorMap tmap_o;  // [B*H, N, D] output map, box {64, 32, 1} (D >= 64, [B, H, N, D] only)
    void* o;             // output, same element type and layout as the inputs
    float* lse;          // fp32 LSE: [B, H, N], or [H, total] for packed sequences
    int layout;          // 0: [B, H, N, D] slices; 1: token-major [tokens, H, D]
    const int* cu_seqlens;  // packed sequences: [B + 1] token offsets (device), else null
    int heads;           // H
    int total;           // tokens in the token-major view (B*N, or the packed total)
    int n;               // sequence length N (packed sequences: the longest allowed length)
    int bh;              // B*H
    int npairs;          // ceil(N / 256): query-tile pairs per slice (at most)
    int nkv;             // ceil(N / 128): key/value tiles per slice (at most)
    int units;           // work units of the persistent schedule
    float scale_log2;    // scale * log2(e) (times the Q and K dequantisation factors for fp8)
    float o_scale;       // factor applied to O at the end: V's dequantisation factor (fp8), else 1
    unsigned long long wait_limit;  // cycles a single wait may spin before giving up
    int inject_stall;    // failure-detection test hook (see fa_set_watchdog)
};

// Launch parameters of the backward tensor-core kernels (bf16/fp16, D = 32, 64, 128, 256).
struct BwdParams {
    CUtensorMap tmap_q;   // 3-D maps over [B*H, N, D] exactly as the forward's
    CUtensorMap tmap_k;
    CUtensorMap tmap_v;
    CUtensorMap tmap_do;
    const float* lse;     // [B*H, N] natural-log LSE of the forward
    const void* o;        // [B*H, N, D] the forward's output (16-bit)
    const void* q;        // [B*H, N, D] Q and dO (16-bit), read row by row where D = 32
    const void* dout;
    float* delta;         // [B*H, N] rowsum(dO * O): written by the dQ kernel, read by dK/dV
    void* dq;             // [B*H, N, D] outputs, input element type
    void* dk;
    void* dv;
    int n;                // sequence length N (packed sequences: the maximum length)
    int ntiles;           // ceil(N / 128)
    float scale;          // softmax scale
    float scale_log2;     // scale * log2(e)
    unsigned long long wait_limit;
    int layout;           // 0: [B, H, N, D]; 1: token-major [tokens, H, D] (as the forward's)
    int heads;            // H
    int total;            // tokens (token-major layouts)
    const int* cu_seqlens;   // packed sequences: batch + 1 token offsets; nullptr otherwise
    int inject_stall;     // failure-detection test hook (see fa_set_watchdog)
};

// Raise the dynamic shared-memory limit of the backward tensor-core kernels (once).
cudaError_t bwd_prepare(int D, bool causal, bool f16);
// dQ (one CTA per 128-query tile; also writes delta) and then dK, dV (one CTA per 128-key
// tile), B*H*ntiles CTAs each.
cudaError_t bwd_launch(int D, bool causal, bool f16, const BwdParams& p, int bh,
                       cudaStream_t stream);
// Status word of the backward kernels (same meaning as the forward's).
cudaError_t bwd_status_read_reset(uint32_t out[4]);

// Head dimension 256 (16-bit storage; maps with boxes of 64 rows x 128 bytes): dQ (which
// also writes delta), dV, then dK, B*H*ntiles CTAs each, on `stream`.
cudaError_t bwd256_prepare(bool causal, bool f16);
cudaError_t bwd256_launch(bool causal, bool f16, const BwdParams& p, int bh, cudaStream_t stream);
cudaError_t bwd256_status_read_reset(uint32_t out[4]);

// Work units of the persistent schedule for a given shape.
int tc_units(int bh, int n, bool causal);

// Dynamic shared memory the tensor-core kernel needs for head dimension D.
int tc_smem_bytes(int D);

// One-time per device: raise the dynamic shared-memory limit of the kernel instance.
// et: element type of Q, K, V: 0 bf16, 1 fp16, 2 fp8 e4m3 (layout 0 only).
cudaError_t tc_prepare(int D, bool causal, int et);

// Launch the tensor-core kernel with `grid` persistent CTAs on `stream`.  single: one
// query tile per work unit ([B, H, N, D] only; p.units must then be B*H*nkv) instead of
// pairs of query tiles.
cudaError_t tc_launch(int D, bool causal, int et, const TcParams& p, bool single, int grid,
                      cudaStream_t stream);

// Copy the device status word (4 words) of the tensor-core kernels to `out` and clear it.
cudaError_t tc_status_read_reset(uint32_t out[4]);

// Head dimension 256 (maps with boxes of 64 rows x 128 bytes): persistent CTAs over the
// units tc256_units gives (query tiles; causal: heavy + light tile pairs).  Uses
// tmap_q/k/v, o, lse, n, bh, units, scale_log2, o_scale, wait_limit and the layout fields.
int tc256_units(int bh, int n, bool causal);
cudaError_t tc256_prepare(bool causal, int et);   // et: 0 bf16, 1 fp16, 2 e4m3 ([B, H, N, D] only)
cudaError_t tc256_launch(bool causal, int et, const TcParams& p, int grid, cudaStream_t stream);
cudaError_t tc256_status_read_reset(uint32_t out[4]);

// Geometry shared by both paths: where row r of slice (b, h) lives.
struct SliceLayout {
    int layout;             // 0: [B, H, N, D]; 1: token-major [tokens, H, D]
    const int* cu_seqlens;  // packed sequences (device), else null
    int heads;              // H
    int total;              // tokens in the token-major view
    int n;                  // N, or the longest allowed packed length
};

// fp32 SIMT kernel over the same layouts (fp32 storage); sm_count picks the CTA shape.
cudaError_t simt_launch(int D, bool causal, const float* q, const float* k, const float* v,
                        float* o, float* lse, int bh, const SliceLayout& g, float scale,
                        int sm_count, cudaStream_t stream);

// fp32 SIMT backward over the same layouts: dQ (which also writes delta, indexed like the
// LSE) and then dK, dV, on `stream`; sm_count picks the CTA shape.
cudaError_t simt_bwd_launch(int D, bool causal, const float* q, const float* k, const float* v,
                            const float* o, const float* dout, const float* lse, float* delta,
                            float* dq, float* dk, float* dv, int bh, const SliceLayout& g,
                            float scale, int sm_count, cudaStream_t stream);

}  // namespace fa
