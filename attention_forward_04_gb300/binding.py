"""ctypes binding of libfa.so (include/fa.h): argument marshalling only.

Every step of the attention forward runs in the library's CUDA kernels; this module
turns torch tensors into pointers, sizes and a stream handle.  torch provides device
memory and streams, nothing else.  If the library is missing the import fails loudly:
there is no fallback path.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfa.so")

FA_FP32, FA_BF16, FA_FP16 = 0, 1, 2
STATUS = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_MISALIGNED",
          4: "FA_ERR_CUDA", 5: "FA_ERR_TIMEOUT"}

# Every symbol include/fa.h declares, with its ctypes signature.
_c = ctypes
SIGNATURES = {
    "fa_fwd": (_c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                          _c.c_int64, _c.c_int64, _c.c_int64, _c.c_int64, _c.c_float, _c.c_int,
                          _c.c_int, _c.c_void_p]),
    "fa_fwd_bnhd": (_c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                               _c.c_int64, _c.c_int64, _c.c_int64, _c.c_int64, _c.c_float,
                               _c.c_int, _c.c_int, _c.c_void_p]),
    "fa_fwd_varlen": (_c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                                 _c.c_void_p, _c.c_int64, _c.c_int64, _c.c_int64, _c.c_int64,
                                 _c.c_int64, _c.c_float, _c.c_int, _c.c_int, _c.c_void_p]),
    "fa_fwd_fp8": (_c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                              _c.c_int64, _c.c_int64, _c.c_int64, _c.c_int64, _c.c_float,
                              _c.c_int, _c.c_float, _c.c_float, _c.c_float, _c.c_void_p]),
    "fa_bwd_workspace_bytes": (_c.c_int64, [_c.c_int64, _c.c_int64, _c.c_int64]),
    "fa_bwd": (_c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                          _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                          _c.c_int64, _c.c_int64, _c.c_int64, _c.c_int64, _c.c_int64,
                          _c.c_float, _c.c_int, _c.c_int, _c.c_void_p]),
    "fa_bwd_bnhd": (_c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                               _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                               _c.c_int64, _c.c_int64, _c.c_int64, _c.c_int64, _c.c_int64,
                               _c.c_float, _c.c_int, _c.c_int, _c.c_void_p]),
    "fa_bwd_varlen": (_c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                                 _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                                 _c.c_int64, _c.c_void_p, _c.c_int64, _c.c_int64, _c.c_int64,
                                 _c.c_int64, _c.c_int64, _c.c_float, _c.c_int, _c.c_int,
                                 _c.c_void_p]),
    "fa_bwd_noalloc": (_c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                                  _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                                  _c.c_void_p, _c.c_int64, _c.c_int64, _c.c_int64, _c.c_int64,
                                  _c.c_float, _c.c_int, _c.c_int, _c.c_void_p]),
    "fa_bwd_noalloc_bnhd": (_c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                                       _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                                       _c.c_void_p, _c.c_int64, _c.c_int64, _c.c_int64,
                                       _c.c_int64, _c.c_float, _c.c_int, _c.c_int,
                                       _c.c_void_p]),
    "fa_bwd_noalloc_varlen": (_c.c_int, [_c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                                         _c.c_void_p, _c.c_void_p, _c.c_void_p, _c.c_void_p,
                                         _c.c_void_p, _c.c_void_p, _c.c_int64, _c.c_int64,
                                         _c.c_int64, _c.c_int64, _c.c_int64, _c.c_float,
                                         _c.c_int, _c.c_int, _c.c_void_p]),
    "fa_status_string": (_c.c_char_p, [_c.c_int]),
    "fa_last_cuda_error": (_c.c_char_p, []),
    "fa_check_device_status": (_c.c_int, [_c.c_void_p, _c.POINTER(_c.c_uint32)]),
    "fa_set_watchdog": (_c.c_int, [_c.c_uint64, _c.c_int]),
    "fa_version": (_c.c_int, []),
}


class FaError(RuntimeError):
    def __init__(self, status: int, detail: str = ""):
        self.status = status
        msg = STATUS.get(status, "FA_ERR_UNKNOWN(%d)" % status)
        super().__init__(msg + (": " + detail if detail else ""))


_lib = None
_lock = threading.Lock()


def load_library(path: str = LIB_PATH):
    """Load libfa.so and declare every exported signature. Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None and path == LIB_PATH:
            return _lib
        if not os.path.exists(path):
            raise FileNotFoundError(
                "libfa.so not found at %s: build it first (attention_forward_04_gb300.build)" % path)
        lib = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        if path == LIB_PATH:
            _lib = lib
        return lib


def _dtype_code(t):
    import torch
    codes = {torch.float32: FA_FP32, torch.bfloat16: FA_BF16, torch.float16: FA_FP16}
    if t.dtype not in codes:
        raise TypeError("unsupported dtype %s (fp32, bf16 or fp16)" % t.dtype)
    return codes[t.dtype]


def _check(status: int):
    if status != 0:
        lib = load_library()
        detail = lib.fa_last_cuda_error().decode() if status == 4 else ""
        raise FaError(status, detail)


def fwd_ptr(q, k, v, o, lse, B, H, N, D, scale, causal, dtype, stream=0) -> int:
    """Raw pointer form of fa_fwd; returns the status code."""
    return int(load_library().fa_fwd(q, k, v, o, lse, B, H, N, D, float(scale), int(causal),
                                      int(dtype), stream))


def fwd(q, k, v, scale=None, causal=False, out=None, lse=None, stream=None):
    """Attention forward through the C ABI.

    q, k, v: CUDA tensors [B, H, N, D], contiguous, one dtype (fp32, bf16 or fp16).
    Returns (o [B,H,N,D] in the input dtype, lse [B,H,N] fp32).  The call is
    asynchronous on ``stream`` (default: torch's current stream).
    """
    import torch
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one [B, H, N, D] shape")
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous [B, H, N, D]")
    _same_device(q, k, v)
    B, H, N, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    _check_buffer(out, "out", q.shape, q.dtype, q.device)
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check_buffer(lse, "lse", (B, H, N), torch.float32, q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    with torch.cuda.device(q.device):
        _check(fwd_ptr(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                       B, H, N, D, scale, causal, _dtype_code(q), handle))
    return out, lse


def fwd_fp8(q, k, v, q_descale, k_descale, v_descale, scale=None, causal=False, out=None,
            lse=None, stream=None):
    """Forward pass on fp8 e4m3 inputs (fa_fwd_fp8).

    q, k, v: contiguous CUDA tensors [B, H, N, D] of torch.float8_e4m3fn; the descale factors
    are the per-tensor dequantisation multipliers.  Returns (o [B, H, N, D] bf16, lse fp32)."""
    import torch
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if q.dim() != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one [B, H, N, D] shape")
    for t in (q, k, v):
        if t.dtype != torch.float8_e4m3fn or not t.is_contiguous():
            raise TypeError("q, k, v must be contiguous torch.float8_e4m3fn tensors")
    _same_device(q, k, v)
    B, H, N, D = q.shape
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    out = torch.empty((B, H, N, D), dtype=torch.bfloat16, device=q.device) if out is None else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_buffer(out, "out", (B, H, N, D), torch.bfloat16, q.device)
    _check_buffer(lse, "lse", (B, H, N), torch.float32, q.device)
    with torch.cuda.device(q.device):
        _check(int(load_library().fa_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                             out.data_ptr(), lse.data_ptr(), B, H, N, D,
                                             float(scale), int(causal), float(q_descale),
                                             float(k_descale), float(v_descale),
                                             _stream_handle(q, stream))))
    return out, lse


def _common(q, k, v, ndim):
    if not (q.is_cuda and k.is_cuda and v.is_cuda):
        raise ValueError("q, k, v must be CUDA tensors")
    if q.dim() != ndim or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one %d-D shape" % ndim)
    if k.dtype != q.dtype or v.dtype != q.dtype:
        raise TypeError("q, k, v must share one dtype")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    _same_device(q, k, v)


def _check_buffer(t, name, shape, dtype, device):
    """A caller-supplied tensor the library writes or reads by pointer: it must have exactly
    the shape and dtype the call implies, be contiguous, and live on the inputs' device
    (the library cannot see buffer sizes, so a mismatch is refused here)."""
    if not t.is_cuda or t.device != device:
        raise ValueError("%s must be a CUDA tensor on %s" % (name, device))
    if tuple(t.shape) != tuple(shape) or t.dtype != dtype or not t.is_contiguous():
        raise ValueError("%s must be a contiguous %s tensor of shape %s" % (name, dtype, tuple(shape)))


def _same_device(q, *others):
    for t in others:
        if t.device != q.device:
            raise ValueError("all tensors must be on %s" % q.device)


def _stream_handle(q, stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def fwd_bnhd(q, k, v, scale=None, causal=False, out=None, lse=None, stream=None):
    """Forward pass over token-major tensors q, k, v [B, N, H, D] (fa_fwd_bnhd).

    Returns (o [B, N, H, D], lse [B, H, N] fp32)."""
    import torch
    _common(q, k, v, 4)
    B, N, H, D = q.shape
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_buffer(out, "out", q.shape, q.dtype, q.device)
    _check_buffer(lse, "lse", (B, H, N), torch.float32, q.device)
    with torch.cuda.device(q.device):
        _check(int(load_library().fa_fwd_bnhd(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                              out.data_ptr(), lse.data_ptr(), B, N, H, D,
                                              float(scale), int(causal), _dtype_code(q),
                                              _stream_handle(q, stream))))
    return out, lse


def fwd_varlen(q, k, v, cu_seqlens, max_seqlen, scale=None, causal=False, out=None, lse=None,
               stream=None):
    """Forward pass over packed sequences (fa_fwd_varlen).

    q, k, v: [total, H, D]; cu_seqlens: int32 CUDA tensor [batch + 1] of token offsets.
    Returns (o [total, H, D], lse [H, total] fp32)."""
    import torch
    _common(q, k, v, 3)
    if not (cu_seqlens.is_cuda and cu_seqlens.dtype == torch.int32 and cu_seqlens.dim() == 1
            and cu_seqlens.is_contiguous() and cu_seqlens.device == q.device):
        raise ValueError("cu_seqlens must be a contiguous 1-D int32 tensor on %s" % q.device)
    T, H, D = q.shape
    batch = cu_seqlens.numel() - 1
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((H, T), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_buffer(out, "out", q.shape, q.dtype, q.device)
    _check_buffer(lse, "lse", (H, T), torch.float32, q.device)
    with torch.cuda.device(q.device):
        _check(int(load_library().fa_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                                out.data_ptr(), lse.data_ptr(),
                                                cu_seqlens.data_ptr(), batch, int(max_seqlen), T,
                                                H, D, float(scale), int(causal), _dtype_code(q),
                                                _stream_handle(q, stream))))
    return out, lse


def bwd_workspace_bytes(B, H, N) -> int:
    return int(load_library().fa_bwd_workspace_bytes(int(B), int(H), int(N)))


def bwd(q, k, v, o, lse, dout, scale=None, causal=False, dq=None, dk=None, dv=None,
        workspace=None, stream=None):
    """Attention backward through the C ABI (fa_bwd).

    q, k, v, o, dout: CUDA tensors [B, H, N, D], contiguous, bf16 or fp16; o and lse are the
    forward's outputs.  Returns (dq, dk, dv) in the input dtype.  ``workspace`` (a uint8
    CUDA tensor of at least bwd_workspace_bytes(B, H, N) bytes) is allocated when omitted.
    """
    import torch
    _common(q, k, v, 4)
    B, H, N, D = q.shape
    _check_buffer(o, "o", q.shape, q.dtype, q.device)
    _check_buffer(dout, "dout", q.shape, q.dtype, q.device)
    _check_buffer(lse, "lse", (B, H, N), torch.float32, q.device)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check_buffer(t, name, q.shape, q.dtype, q.device)
    need = bwd_workspace_bytes(B, H, N)
    if need < 0:
        raise FaError(1, "B, H or N out of range")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if not (workspace.is_cuda and workspace.device == q.device and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor on %s" % q.device)
    with torch.cuda.device(q.device):
        _check(int(load_library().fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         dout.data_ptr(), lse.data_ptr(), dq.data_ptr(),
                                         dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
                                         workspace.numel() * workspace.element_size(), B, H, N,
                                         D, float(scale), int(causal), _dtype_code(q),
                                         _stream_handle(q, stream))))
    return dq, dk, dv


def _bwd_buffers(q, o, dout, lse, lse_shape, dq, dk, dv, workspace, need):
    """Check and allocate the backward's buffers (shared by the layout variants)."""
    import torch
    _check_buffer(o, "o", q.shape, q.dtype, q.device)
    _check_buffer(dout, "dout", q.shape, q.dtype, q.device)
    _check_buffer(lse, "lse", lse_shape, torch.float32, q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check_buffer(t, name, q.shape, q.dtype, q.device)
    if need < 0:
        raise FaError(1, "sizes out of range")
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    if not (workspace.is_cuda and workspace.device == q.device and workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor on %s" % q.device)
    return dq, dk, dv, workspace


def bwd_bnhd(q, k, v, o, lse, dout, scale=None, causal=False, dq=None, dk=None, dv=None,
             workspace=None, stream=None):
    """Backward over token-major tensors [B, N, H, D] (fa_bwd_bnhd); lse [B, H, N] as
    fwd_bnhd returns it.  Returns (dq, dk, dv) in [B, N, H, D]."""
    import torch
    _common(q, k, v, 4)
    B, N, H, D = q.shape
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    dq, dk, dv, workspace = _bwd_buffers(q, o, dout, lse, (B, H, N), dq, dk, dv, workspace,
                                         bwd_workspace_bytes(B, H, N))
    with torch.cuda.device(q.device):
        _check(int(load_library().fa_bwd_bnhd(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
            lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), B, N, H, D, float(scale), int(causal),
            _dtype_code(q), _stream_handle(q, stream))))
    return dq, dk, dv


def bwd_varlen(q, k, v, o, lse, dout, cu_seqlens, max_seqlen, scale=None, causal=False,
               dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Backward over packed sequences (fa_bwd_varlen): q, k, v, o, dout [total, H, D],
    lse [H, total] as fwd_varlen returns it, the same cu_seqlens.  Returns (dq, dk, dv)."""
    import torch
    _common(q, k, v, 3)
    if not (cu_seqlens.is_cuda and cu_seqlens.dtype == torch.int32 and cu_seqlens.dim() == 1
            and cu_seqlens.is_contiguous() and cu_seqlens.device == q.device):
        raise ValueError("cu_seqlens must be a contiguous 1-D int32 tensor on %s" % q.device)
    T, H, D = q.shape
    batch = cu_seqlens.numel() - 1
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    dq, dk, dv, workspace = _bwd_buffers(q, o, dout, lse, (H, T), dq, dk, dv, workspace,
                                         bwd_workspace_bytes(1, H, T))
    with torch.cuda.device(q.device):
        _check(int(load_library().fa_bwd_varlen(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
            lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), cu_seqlens.data_ptr(), batch,
            int(max_seqlen), T, H, D, float(scale), int(causal), _dtype_code(q),
            _stream_handle(q, stream))))
    return dq, dk, dv


def bwd_noalloc(q, k, v, o, lse, dout, dq, dk, dv, scale=None, causal=False, stream=None):
    """fa_bwd_noalloc: the backward with library-owned scratch.  The caller provides the
    gradient buffers dq, dk, dv (same shape and dtype as q); nothing is allocated."""
    import torch
    _common(q, k, v, 4)
    B, H, N, D = q.shape
    for name, t in (("o", o), ("dout", dout), ("dq", dq), ("dk", dk), ("dv", dv)):
        _check_buffer(t, name, q.shape, q.dtype, q.device)
    _check_buffer(lse, "lse", (B, H, N), torch.float32, q.device)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    with torch.cuda.device(q.device):
        _check(int(load_library().fa_bwd_noalloc(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
            lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, N, D,
            float(scale), int(causal), _dtype_code(q), _stream_handle(q, stream))))
    return dq, dk, dv


def bwd_noalloc_bnhd(q, k, v, o, lse, dout, dq, dk, dv, scale=None, causal=False, stream=None):
    """fa_bwd_noalloc_bnhd: bwd_bnhd with library-owned scratch; the caller provides dq,
    dk, dv ([B, N, H, D], the dtype of q)."""
    import torch
    _common(q, k, v, 4)
    B, N, H, D = q.shape
    for name, t in (("o", o), ("dout", dout), ("dq", dq), ("dk", dk), ("dv", dv)):
        _check_buffer(t, name, q.shape, q.dtype, q.device)
    _check_buffer(lse, "lse", (B, H, N), torch.float32, q.device)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    with torch.cuda.device(q.device):
        _check(int(load_library().fa_bwd_noalloc_bnhd(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
            lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, N, H, D,
            float(scale), int(causal), _dtype_code(q), _stream_handle(q, stream))))
    return dq, dk, dv


def bwd_noalloc_varlen(q, k, v, o, lse, dout, dq, dk, dv, cu_seqlens, max_seqlen, scale=None,
                       causal=False, stream=None):
    """fa_bwd_noalloc_varlen: bwd_varlen with library-owned scratch; the caller provides
    dq, dk, dv ([total, H, D], the dtype of q)."""
    import torch
    _common(q, k, v, 3)
    if not (cu_seqlens.is_cuda and cu_seqlens.dtype == torch.int32 and cu_seqlens.dim() == 1
            and cu_seqlens.is_contiguous() and cu_seqlens.device == q.device):
        raise ValueError("cu_seqlens must be a contiguous 1-D int32 tensor on %s" % q.device)
    T, H, D = q.shape
    for name, t in (("o", o), ("dout", dout), ("dq", dq), ("dk", dk), ("dv", dv)):
        _check_buffer(t, name, q.shape, q.dtype, q.device)
    _check_buffer(lse, "lse", (H, T), torch.float32, q.device)
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    with torch.cuda.device(q.device):
        _check(int(load_library().fa_bwd_noalloc_varlen(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
            lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), cu_seqlens.data_ptr(),
            cu_seqlens.numel() - 1, int(max_seqlen), T, H, D, float(scale), int(causal),
            _dtype_code(q), _stream_handle(q, stream))))
    return dq, dk, dv


def check_device_status(stream=None):
    """Synchronise the stream and return (status, detail words) of the kernel watchdog."""
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    detail = (ctypes.c_uint32 * 4)()
    st = int(load_library().fa_check_device_status(handle, detail))
    return st, list(detail)


def set_watchdog(wait_limit_cycles: int = 0, inject_stall: int = 0):
    _check(int(load_library().fa_set_watchdog(int(wait_limit_cycles), int(inject_stall))))
