"""Attention oracle: a plain fp64 CPU statement of what the attention forward computes.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The GPU library in
``attention_forward_04_gb300`` never imports it, and the two share no code.

Two independent statements of the method live here:

* ``attention_fwd`` / ``attention_rows`` -- the definition itself, three passes
  per block of rows (materialise S, stable row softmax, multiply by V), in C,
  fp64 (``attention_oracle.c``).  Sources: "KingOfEgg: Flash Attention v1"
  (dandandamowang.xyz) §1.1-§1.2; "08 · FlashAttention" §一 and §四
  (``is_causal``); "第 13 课：GPU 内核与 FlashAttention", exercise
  ``standard_attention``.
* ``tiled.attention_tiled`` -- the tiled online-softmax algorithm (query blocks
  outside, key/value blocks inside, running max m, running sum l, rescaled
  accumulator, one division at the end), in numpy.  It exists to pin the
  three-pass definition: the pages state that the two are exactly equal.

Inputs are numpy float64 arrays of shape [B, H, N, D]; callers convert stored
bf16/fp32 tensors to float64, which is exact.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``attention_oracle.c`` with gcc (OpenMP if available). Returns the .so path."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    base = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        # No OpenMP runtime: the pragmas are ignored and the oracle runs on one thread.
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            i64p = ctypes.POINTER(ctypes.c_int64)
            i64 = ctypes.c_int64
            lib.oracle_attention_fwd.argtypes = [dp, dp, dp, dp, dp, i64, i64, i64,
                                                 ctypes.c_double, ctypes.c_int, ctypes.c_int, dp]
            lib.oracle_attention_fwd.restype = ctypes.c_int
            lib.oracle_attention_rows.argtypes = [dp, dp, dp, i64, i64, i64, ctypes.c_double,
                                                  ctypes.c_int, i64p, i64p, i64, dp, dp,
                                                  ctypes.c_int]
            lib.oracle_attention_rows.restype = ctypes.c_int
            lib.oracle_default_threads.argtypes = []
            lib.oracle_default_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f64(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray, ty=ctypes.c_double):
    return a.ctypes.data_as(ctypes.POINTER(ty))


def default_threads() -> int:
    return int(_load().oracle_default_threads())


def attention_fwd(q, k, v, scale: float, causal: bool = False, threads: int = 0,
                  return_rowsum_err: bool = False):
    """O = softmax(scale * Q K^T) V and LSE over [B, H, N, D] fp64 arrays.

    Returns (o [B,H,N,D] float64, lse [B,H,N] float64) and, if asked, the largest
    |sum_j P_ij - 1| over all rows.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim != 4 or k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must share one [B, H, N, D] shape")
    B, H, N, D = q.shape
    o = np.empty_like(q)
    lse = np.empty((B, H, N), dtype=np.float64)
    err = ctypes.c_double(0.0)
    rc = _load().oracle_attention_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                      B * H, N, D, float(scale), int(bool(causal)),
                                      int(threads), ctypes.byref(err))
    if rc != 0:
        raise RuntimeError("oracle_attention_fwd failed with code %d" % rc)
    if return_rowsum_err:
        return o, lse, float(err.value)
    return o, lse


def attention_rows(q, k, v, scale: float, causal: bool, bh_idx, row_idx, threads: int = 0):
    """The same definition for sampled rows.

    Row r of the result is query row ``row_idx[r]`` of slice ``bh_idx[r]`` (slice =
    b*H + h).  Returns (o_rows [n, D], lse_rows [n]) as float64.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, D = q.shape
    bh = np.ascontiguousarray(bh_idx, dtype=np.int64)
    rows = np.ascontiguousarray(row_idx, dtype=np.int64)
    if bh.shape != rows.shape or bh.ndim != 1:
        raise ValueError("bh_idx and row_idx must be 1-D and of equal length")
    n = bh.shape[0]
    o = np.empty((n, D), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    rc = _load().oracle_attention_rows(_ptr(q), _ptr(k), _ptr(v), B * H, N, D, float(scale),
                                       int(bool(causal)), _ptr(bh, ctypes.c_int64),
                                       _ptr(rows, ctypes.c_int64), n, _ptr(o), _ptr(lse),
                                       int(threads))
    if rc != 0:
        raise RuntimeError("oracle_attention_rows failed with code %d" % rc)
    return o, lse
