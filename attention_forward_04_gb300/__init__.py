"""GB300 (sm_103a) FlashAttention: forward O = softmax(scale * Q K^T) V with the row LSE,
and the backward that rebuilds P from the LSE.

The compute lives in ``libfa.so`` (C ABI declared in ``include/fa.h``); this package
holds the ctypes binding, the in-tree build, and the seeded synthetic inputs.
"""
from .binding import (FA_BF16, FA_FP16, FA_FP32, FaError, bwd, bwd_bnhd, bwd_noalloc,
                      bwd_noalloc_bnhd, bwd_noalloc_varlen, bwd_varlen, bwd_workspace_bytes, check_device_status, fwd, fwd_bnhd,
                      fwd_fp8, fwd_ptr, fwd_varlen, load_library, set_watchdog)

__all__ = ["fwd", "fwd_bnhd", "fwd_varlen", "fwd_fp8", "fwd_ptr", "bwd", "bwd_bnhd",
           "bwd_varlen", "bwd_noalloc", "bwd_noalloc_bnhd", "bwd_noalloc_varlen", "bwd_workspace_bytes",
           "load_library", "check_device_status", "set_watchdog", "FaError", "FA_FP32",
           "FA_BF16", "FA_FP16"]
