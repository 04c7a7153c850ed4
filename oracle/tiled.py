"""Tiled online-softmax attention in numpy (fp64) -- TEST INFRASTRUCTURE ONLY.

This is the algorithm the pages teach, written out from its description, and
used only to pin the three-pass oracle (the pages state the two are exactly
equal, "第 13 课：GPU 内核与 FlashAttention" exercise result and
"pwwt.cn: FlashAttention 与内存墙" §4.2):

* "08 · FlashAttention" §二 and "第 13 课" Figure 13-2: queries in blocks on the
  outside; for each query block, key/value blocks on the inside;
* running maximum m and running sum l per query row; when a larger maximum
  appears, the old sum and the old accumulator are multiplied by
  exp(m_old - m_new) before the new block is added
  ("KingOfEgg: Flash Attention v1" §2; "08 · FlashAttention" §二);
* one division by l at the very end ("第 13 课" exercise; "pwwt.cn" §2.2).

The causal mask (key j <= query i, "08 · FlashAttention" §四) is applied inside
each block before the block maximum is taken.
"""
from __future__ import annotations

import numpy as np


def attention_tiled_slice(q, k, v, scale: float, causal: bool = False,
                          block_q: int = 64, block_kv: int = 64):
    """One [N, D] slice. Returns (O [N, D], m [N], l [N]) with O already divided by l."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, d = q.shape
    O = np.zeros((n, d))
    l = np.zeros(n)
    m = np.full(n, -np.inf)
    for i0 in range(0, n, block_q):
        i1 = min(n, i0 + block_q)
        Oi = O[i0:i1].copy()
        li = l[i0:i1].copy()
        mi = m[i0:i1].copy()
        rows = np.arange(i0, i1)
        for j0 in range(0, n, block_kv):
            j1 = min(n, j0 + block_kv)
            if causal and j0 > i1 - 1:
                break  # every key of this block lies after every query of the block
            S = scale * (q[i0:i1] @ k[j0:j1].T)
            if causal:
                cols = np.arange(j0, j1)
                S = np.where(cols[None, :] <= rows[:, None], S, -np.inf)
            m_new = np.maximum(mi, S.max(axis=1))
            shrink = np.exp(mi - m_new)                 # rescales what was summed so far
            p = np.exp(S - m_new[:, None])
            li = li * shrink + p.sum(axis=1)
            Oi = Oi * shrink[:, None] + p @ v[j0:j1]
            mi = m_new
        O[i0:i1] = Oi
        l[i0:i1] = li
        m[i0:i1] = mi
    return O / l[:, None], m, l


def attention_tiled(q, k, v, scale: float, causal: bool = False,
                    block_q: int = 64, block_kv: int = 64):
    """[B, H, N, D] fp64 inputs. Returns (O [B,H,N,D], LSE [B,H,N]) with LSE = m + ln l."""
    q = np.asarray(q, dtype=np.float64)
    B, H, N, D = q.shape
    O = np.empty((B, H, N, D))
    LSE = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            o, m, l = attention_tiled_slice(q[b, h], k[b, h], v[b, h], scale, causal,
                                            block_q, block_kv)
            O[b, h] = o
            LSE[b, h] = m + np.log(l)
    return O, LSE
