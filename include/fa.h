/*
 * fa.h -- C ABI of the GB300 (sm_103a) FlashAttention forward library (libfa.so).
 *
 * The operation (one call = one whole forward pass over a batch of heads):
 *   For every slice (b, h) of [B, H, N, D] tensors Q, K, V and every query row i,
 *     O[b,h,i,:] = sum_j softmax_j(scale * Q[b,h,i,:] . K[b,h,j,:]) * V[b,h,j,:]
 *     LSE[b,h,i] = ln sum_j exp(scale * Q[b,h,i,:] . K[b,h,j,:])
 *   with j over all N keys, or over j <= i when `causal` is set.
 *   Sources: "KingOfEgg: Flash Attention v1" (dandandamowang.xyz) §1.1 (scaled
 *   dot-product attention) and §1.2 (the [B, H, N, D] layout); "08 · FlashAttention"
 *   §二 (tiles plus online softmax, the N x N matrix never reaches HBM) and §四
 *   (`is_causal`).  LSE is the natural-log row normaliser m + ln l of the scaled
 *   scores; the pages keep m and l separately ("KingOfEgg" §5.2), and one fp32
 *   value per row carries both.
 *
 * All calls are host calls.  No call allocates device memory.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Storage type of Q, K, V and O.  LSE is always fp32. */
typedef enum {
    FA_FP32 = 0, /* fp32 in, fp32 out; SIMT fp32 arithmetic (no TF32)                  */
    FA_BF16 = 1, /* bf16 in, bf16 out; tensor-core products, fp32 accumulation/softmax */
    FA_FP16 = 2  /* fp16 in, fp16 out; same arithmetic as FA_BF16                       */
} fa_dtype;

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1, /* null pointer, size out of range, bad flag, output overlaps an input */
    FA_ERR_UNSUPPORTED = 2, /* valid request the library does not serve (D, dtype, GPU model)      */
    FA_ERR_MISALIGNED = 3,  /* a tensor pointer is not 16-byte aligned (TMA needs 16 B)             */
    FA_ERR_CUDA = 4,        /* a CUDA runtime call or the kernel launch failed                      */
    FA_ERR_TIMEOUT = 5      /* a kernel wait ran past its limit (reported by fa_check_device_status) */
} fa_status;

/*
 * fa_fwd -- attention forward pass, asynchronous on `stream`.
 *
 *   q, k, v : device pointers, [B, H, N, D] contiguous (row-major), element type `dtype`.
 *   o       : device pointer, [B, H, N, D] contiguous, element type `dtype`; written fully.
 *   lse     : device pointer, [B, H, N] contiguous fp32; written fully.
 *   B, H, N : >= 1.  B*H < 2^31 and N < 2^31.  Any N is accepted (a ragged last tile is
 *             masked; keys >= N never contribute).
 *   D       : head dimension: 32, 64, 128 or 256.
 *   scale   : finite, >= 0 (normally 1/sqrt(D)).
 *   causal  : 0 = all keys; 1 = key j <= query i (square N x N).
 *   dtype   : an fa_dtype value.
 *   stream  : a cudaStream_t (CUstream) cast to void*, or NULL for the legacy default stream.
 *
 * Ownership: the caller owns every buffer and keeps it alive until the stream has
 * finished the call.  o and lse need no initialisation.  o and lse must not overlap
 * q, k, v or each other.  The call allocates nothing and does not synchronise.
 *
 * Errors: arguments are checked before any CUDA call; on a bad argument nothing is
 * launched and FA_ERR_INVALID_ARG / FA_ERR_UNSUPPORTED / FA_ERR_MISALIGNED is returned.
 * A failed launch returns FA_ERR_CUDA (see fa_last_cuda_error).  Faults inside the
 * kernel never trap: every wait in the kernel is bounded, and a wait that runs out sets
 * a device status word that fa_check_device_status reports as FA_ERR_TIMEOUT.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int64_t B, int64_t H, int64_t N, int64_t D,
           float scale, int causal, int dtype, void* stream);

/*
 * fa_fwd_bnhd -- the same forward pass over token-major tensors.
 *
 *   q, k, v, o : device pointers, [B, N, H, D] contiguous ("batch, sequence, head, dim"):
 *                row i of head h of batch b starts at element ((b*N + i)*H + h)*D.  Reading
 *                and writing this layout directly saves the [B,N,H,D] <-> [B,H,N,D] copies
 *                around the attention ("pwwt.cn: FlashAttention 与内存墙" §5.2).
 *   lse        : device pointer, [B, H, N] contiguous fp32.
 *   Everything else as fa_fwd (same limits, ownership, errors, asynchrony).
 */
int fa_fwd_bnhd(const void* q, const void* k, const void* v, void* o, float* lse,
                int64_t B, int64_t N, int64_t H, int64_t D,
                float scale, int causal, int dtype, void* stream);

/*
 * fa_fwd_varlen -- the forward pass over packed sequences of different lengths, without
 * padding ("08 · FlashAttention" §四: packing with cu_seqlens instead of a padding mask).
 *
 *   q, k, v, o : device pointers, [total, H, D] contiguous: the tokens of all sequences one
 *                after another; sequence b owns tokens cu_seqlens[b] .. cu_seqlens[b+1]-1.
 *   lse        : device pointer, [H, total] contiguous fp32 (entry h*total + token).
 *   cu_seqlens : device pointer, batch + 1 int32 values: 0 = cu[0] <= cu[1] <= ... <=
 *                cu[batch] = total, and cu[b+1] - cu[b] <= max_seqlen.  Each sequence
 *                attends only to its own tokens (causal: token j <= token i within it).
 *                Empty sequences are allowed.  The kernel clamps offsets to [0, total] and
 *                lengths to max_seqlen, so malformed offsets give wrong results but never an
 *                access outside the tensors; they are not otherwise checked (checking would
 *                need a device-to-host copy).
 *   batch, max_seqlen, total, H : >= 1; batch*H < 2^31; total < 2^31.
 *   Everything else as fa_fwd.
 */
int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                  const int32_t* cu_seqlens, int64_t batch, int64_t max_seqlen, int64_t total,
                  int64_t H, int64_t D, float scale, int causal, int dtype, void* stream);

/*
 * fa_fwd_fp8 -- the forward pass on fp8 inputs (the FP8 tensor-core direction that
 * "第 13 课：GPU 内核与 FlashAttention", answer to question 3, names for FlashAttention-3),
 * asynchronous on `stream`.
 *
 *   q, k, v : device pointers, [B, H, N, D] contiguous fp8 e4m3 (1 byte per element); the
 *             values are q_descale * Q, k_descale * K, v_descale * V (per-tensor factors).
 *   o       : device pointer, [B, H, N, D] contiguous bf16; written fully.
 *   lse     : device pointer, [B, H, N] fp32; written fully.
 *   B, H, N, scale, causal, stream : as for fa_fwd.
 *   D       : 32, 64, 128 or 256.
 *   q_descale, k_descale, v_descale : finite, > 0.
 *
 * Computes O = softmax(scale * (q_descale Q)(k_descale K)^T) (v_descale V) and its LSE:
 * Q K^T and P V on the tensor cores from e4m3 operands (kind::f8f6f4) with fp32
 * accumulation; P is rounded to e4m3 before P V (l is summed from the fp32 values);
 * O is rounded to bf16.  Errors as fa_fwd.
 */
int fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse,
               int64_t B, int64_t H, int64_t N, int64_t D, float scale, int causal,
               float q_descale, float k_descale, float v_descale, void* stream);

/*
 * fa_bwd_workspace_bytes -- bytes of device workspace fa_bwd needs for a [B, H, N, D]
 * problem (one fp32 value per query row, rounded up to 256 bytes); -1 if B, H or N is out
 * of range.  Pure host arithmetic.
 */
int64_t fa_bwd_workspace_bytes(int64_t B, int64_t H, int64_t N);

/*
 * fa_bwd -- attention backward pass, asynchronous on `stream`.
 *
 * Given dO = dL/dO for the forward above, writes the gradients of L:
 *     P = exp(scale * Q K^T - LSE) (causal: P_ij = 0 for j > i),
 *     delta_i = sum_d dO_id O_id,  dS = P * (dO V^T - delta),
 *     dV = P^T dO,  dQ = scale * dS K,  dK = scale * dS^T Q.
 * P is rebuilt from the forward's LSE instead of being stored ("08 · FlashAttention" §三
 * 反向传播; "第 13 课：GPU 内核与 FlashAttention" §4B); the formulas are the chain rule through the
 * softmax of "KingOfEgg: Flash Attention v1" §1.1.
 *
 *   q, k, v, o, dout : device pointers, [B, H, N, D] contiguous, element type `dtype`;
 *                      o and lse are the outputs of fa_fwd on the same q, k, v, scale, causal.
 *   lse              : device pointer, [B, H, N] fp32 (fa_fwd's lse).
 *   dq, dk, dv       : device pointers, [B, H, N, D] contiguous, element type `dtype`;
 *                      written fully (no accumulation into existing contents).
 *   workspace        : device pointer of at least fa_bwd_workspace_bytes(B, H, N) bytes,
 *                      16-byte aligned; scratch for delta, needs no initialisation, and
 *                      must not be shared by two calls in flight at once.
 *   B, H, N, scale, causal, stream : as for fa_fwd.
 *   D                : 32, 64, 128 or 256.
 *   dtype            : FA_BF16 or FA_FP16 (tensor cores), or FA_FP32 (CUDA cores, fp32
 *                      arithmetic throughout).
 *
 * Arithmetic: 16-bit storage: products on the tensor cores from 16-bit operands (P and dS
 * are rounded to `dtype` before their products, like P in the forward), fp32 accumulation,
 * results rounded to `dtype` (D <= 128: a dQ and a dK/dV kernel; D = 256: a dQ, a dV and a
 * dK kernel); fp32 storage: fp32 throughout.  No atomics: results do not depend on
 * scheduling.
 * Errors: as fa_fwd; additionally FA_ERR_INVALID_ARG when the workspace is too small or any
 * output overlaps an input, the workspace or another output.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv, void* workspace,
           int64_t workspace_bytes, int64_t B, int64_t H, int64_t N, int64_t D, float scale,
           int causal, int dtype, void* stream);

/*
 * fa_bwd_bnhd -- the backward pass over token-major tensors: q, k, v, o, dout, dq, dk, dv
 * are [B, N, H, D] contiguous as for fa_fwd_bnhd, lse is [B, H, N] fp32 (fa_fwd_bnhd's
 * lse).  Everything else as fa_bwd (workspace of fa_bwd_workspace_bytes(B, H, N) bytes).
 */
int fa_bwd_bnhd(const void* q, const void* k, const void* v, const void* o, const void* dout,
                const float* lse, void* dq, void* dk, void* dv, void* workspace,
                int64_t workspace_bytes, int64_t B, int64_t N, int64_t H, int64_t D, float scale,
                int causal, int dtype, void* stream);

/*
 * fa_bwd_varlen -- the backward pass over packed sequences: q, k, v, o, dout, dq, dk, dv
 * are [total, H, D] and lse [H, total] fp32 as for fa_fwd_varlen (same cu_seqlens,
 * batch, max_seqlen, total, with the same clamping of malformed offsets).  The workspace
 * holds delta indexed like lse: at least fa_bwd_workspace_bytes(1, H, total) bytes.
 * Gradient rows of tokens that belong to no sequence (past cu_seqlens[batch]) are not
 * written.  Everything else as fa_bwd.
 */
int fa_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dout,
                  const float* lse, void* dq, void* dk, void* dv, void* workspace,
                  int64_t workspace_bytes, const int32_t* cu_seqlens, int64_t batch,
                  int64_t max_seqlen, int64_t total, int64_t H, int64_t D, float scale,
                  int causal, int dtype, void* stream);

/*
 * fa_bwd_noalloc -- fa_bwd with its scratch taken from a fixed array inside the library
 * instead of from the caller.  The pages have no counterpart: it serves callers that
 * cannot provide or allocate device memory at the call site (a pool holding all free HBM,
 * code running inside an allocator, a stream that must not wait on cudaMalloc).
 *
 *   Arguments, results, arithmetic and errors: as fa_bwd, without workspace arguments.
 *   Limit: fa_bwd_workspace_bytes(B, H, N) <= FA_BWD_NOALLOC_MAX_SCRATCH_BYTES (4 MiB, i.e.
 *          B*H*N <= 1,048,576 query rows); larger problems return FA_ERR_UNSUPPORTED before
 *          any CUDA call.
 *   Allocation: none, by this call or anything it calls.
 *   Set-up: the first call on each device looks up that device's copy of the array
 *          (cudaGetSymbolAddress) and keeps the address.  That first call may make the
 *          driver load the library's device code on the device, which itself needs device
 *          memory (the 4 MiB array among it), so make it early: before a memory pool takes
 *          all free HBM, and before any stream capture begins on the device.  A lookup that
 *          fails returns FA_ERR_CUDA and is retried by the next call.
 *   Scale:  any finite scale >= 0, as fa_bwd.
 *   Concurrency: every call on one device uses the same array.  Two calls whose work can
 *          overlap on the device (different streams not ordered by events, or two host
 *          threads' streams) race on it and give wrong results; order them on one stream.
 */
#define FA_BWD_NOALLOC_MAX_SCRATCH_BYTES (4 * 1024 * 1024)
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                   const void* dout, const float* lse, void* dq, void* dk, void* dv,
                   int64_t B, int64_t H, int64_t N, int64_t D, float scale, int causal,
                   int dtype, void* stream);

/*
 * fa_bwd_noalloc_bnhd -- fa_bwd_bnhd with the scratch of fa_bwd_noalloc: token-major
 * [B, N, H, D] tensors, lse [B, H, N].  Limit: fa_bwd_workspace_bytes(B, H, N) <=
 * FA_BWD_NOALLOC_MAX_SCRATCH_BYTES.  Set-up and concurrency as fa_bwd_noalloc (the three
 * no-alloc entry points share one array per device).
 */
int fa_bwd_noalloc_bnhd(const void* q, const void* k, const void* v, const void* o,
                        const void* dout, const float* lse, void* dq, void* dk, void* dv,
                        int64_t B, int64_t N, int64_t H, int64_t D, float scale, int causal,
                        int dtype, void* stream);

/*
 * fa_bwd_noalloc_varlen -- fa_bwd_varlen with the scratch of fa_bwd_noalloc: packed
 * [total, H, D] tensors, lse [H, total], the same cu_seqlens.  Limit:
 * fa_bwd_workspace_bytes(1, H, total) <= FA_BWD_NOALLOC_MAX_SCRATCH_BYTES (H*total <=
 * 1,048,576).  cu_seqlens == NULL is FA_ERR_INVALID_ARG.  Set-up and concurrency as
 * fa_bwd_noalloc.
 */
int fa_bwd_noalloc_varlen(const void* q, const void* k, const void* v, const void* o,
                          const void* dout, const float* lse, void* dq, void* dk, void* dv,
                          const int32_t* cu_seqlens, int64_t batch, int64_t max_seqlen,
                          int64_t total, int64_t H, int64_t D, float scale, int causal,
                          int dtype, void* stream);

/* Human-readable name of a status code (static string; never NULL). */
const char* fa_status_string(int status);

/* Text of the last CUDA error seen by this library in the calling thread, or "". */
const char* fa_last_cuda_error(void);

/*
 * fa_check_device_status -- synchronises `stream`, then reads and clears the device
 * status word the tensor-core kernels set when a bounded wait runs out.
 * Returns FA_OK, FA_ERR_TIMEOUT, or FA_ERR_CUDA if the synchronisation itself failed.
 * If `detail` is not NULL it receives 4 words: flags, role that gave up, CTA index, wait id.
 */
int fa_check_device_status(void* stream, uint32_t* detail);

/*
 * fa_set_watchdog -- failure-detection control for the tensor-core kernels (affects
 * launches made after the call, in this process).
 *   wait_limit_cycles : SM clock cycles any single wait may spin before the kernel gives
 *                       up; 0 restores the default (2^32 cycles, about two seconds).
 *   inject_stall      : 0 = normal.  1 = in CTA 0 of each tensor-core kernel the loader
 *                       withholds one tile (the forward: the first K/V tile of its first
 *                       work item; the backward kernels: the first tile they stream), so
 *                       the waits for it run out.  This exists so tests can check that a
 *                       stuck pipeline ends with FA_ERR_TIMEOUT instead of a hang; the
 *                       outputs of that call are then undefined.
 * Returns FA_OK, or FA_ERR_INVALID_ARG for an unknown inject_stall value.
 */
int fa_set_watchdog(uint64_t wait_limit_cycles, int inject_stall);

/* Library ABI version (major * 100 + minor). */
int fa_version(void);   /* 140: adds fa_bwd_bnhd, fa_bwd_varlen */

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
