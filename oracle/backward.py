"""Attention backward oracle (fp64, numpy) -- TEST INFRASTRUCTURE ONLY.

Gradients of a scalar loss L with dL/dO = dO through the forward definition
O = softmax(scale * Q K^T) V ("KingOfEgg: Flash Attention v1" §1.1), written out as the
plain chain rule on materialised matrices, one (b, h) slice at a time:

    S  = scale * Q K^T        (causal: S_ij = -inf for j > i, "08 · FlashAttention" §四)
    P  = softmax_row(S)
    dV = P^T dO
    dP = dO V^T
    delta_i = sum_j P_ij dP_ij            (= sum_d dO_id O_id)
    dS = P * (dP - delta)                 (derivative of the row softmax)
    dQ = scale * dS K
    dK = scale * dS^T Q

The pages state only that the backward recomputes P from the saved O, l, m instead of
storing it ("08 · FlashAttention" §三 反向传播; "第 13 课" §4B); the formulas above are
calculus, pinned in the tests against finite differences of the forward oracle.
Inputs are [B, H, N, D] float64 arrays.
"""
from __future__ import annotations

import numpy as np


def _slice_bwd(q, k, v, do, scale, causal):
    N = q.shape[0]
    S = scale * (q @ k.T)
    if causal:
        S = np.where(np.tril(np.ones((N, N), dtype=bool)), S, -np.inf)
    m = S.max(axis=1, keepdims=True)
    P = np.exp(S - m)
    l = P.sum(axis=1, keepdims=True)
    P = P / l
    o = P @ v
    dv = P.T @ do
    dP = do @ v.T
    delta = (P * dP).sum(axis=1)
    dS = P * (dP - delta[:, None])
    dq = scale * (dS @ k)
    dk = scale * (dS.T @ q)
    lse = (m + np.log(l))[:, 0]
    return dq, dk, dv, o, lse, delta


def attention_bwd(q, k, v, do, scale: float, causal: bool = False):
    """Returns (dq, dk, dv, o, lse, delta); gradients have the inputs' shape, lse and delta
    are [B, H, N]."""
    q, k, v, do = (np.asarray(t, dtype=np.float64) for t in (q, k, v, do))
    B, H, N, D = q.shape
    dq, dk, dv, o = (np.empty_like(q) for _ in range(4))
    lse = np.empty((B, H, N))
    delta = np.empty((B, H, N))
    for b in range(B):
        for h in range(H):
            r = _slice_bwd(q[b, h], k[b, h], v[b, h], do[b, h], scale, causal)
            dq[b, h], dk[b, h], dv[b, h], o[b, h], lse[b, h], delta[b, h] = r
    return dq, dk, dv, o, lse, delta
