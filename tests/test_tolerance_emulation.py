"""The derived GPU tolerances, checked on the CPU against a numpy emulation of the kernels'
rounding points.

A tolerance is only useful if it holds for what the kernel does and fails for a plausible
mistake.  These tests restate, in numpy, where the tensor-core kernels round (P to e4m3
or bf16 before its product, O, dS and the gradients to bf16, a lazy softmax reference up
to 2^8 below the row maximum) and check that

  * the element-wise bounds of ``test_fp8_gpu.py`` and ``test_backward_gpu.py`` cover the
    emulated results with room to spare, and
  * the same bounds reject results with one planted mistake (a dropped dequantisation
    factor, a dropped delta, a missing scale, a transposed operand).

No GPU is needed; the oracle is the fp64 reference the GPU tests use.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_forward_04_gb300.inputs import Workload, make_qkv_fp8, make_shape, make_shape_dout
from oracle.backward import attention_bwd


def e4m3(x):
    return torch.from_numpy(np.ascontiguousarray(x)).float().to(torch.float8_e4m3fn).double().numpy()


def bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x)).float().to(torch.bfloat16).double().numpy()


def causal_mask(n):
    return np.tril(np.ones((n, n), dtype=bool))


# ------------------------------------------------------------------ fp8 forward
def fp8_emulated_output(q, k, v8, vd, scale, causal, mistake=None):
    """O as the e4m3 kernel forms it: scores in full precision, p = exp(s - m_ref) with a
    reference up to 2^8 below the row maximum (the lazy rescale), P rounded to e4m3 before
    P V, l summed from the unrounded p, O rounded to bf16."""
    n = q.shape[0]
    s = scale * (q @ k.T)
    if causal:
        s = np.where(causal_mask(n), s, -np.inf)
    m_ref = s.max(1, keepdims=True) - 8 * math.log(2)
    p = np.exp(s - m_ref)
    l = p.sum(1, keepdims=True)
    factor = 1.0 if mistake == "no_v_descale" else vd
    return bf16((e4m3(p) @ v8) * factor / l)


@pytest.mark.parametrize("n,d,causal,mult", [(300, 128, False, 1.0), (700, 64, True, 1.0),
                                             (500, 128, True, 4.0), (200, 256, False, 1.0),
                                             (129, 32, True, 1.0)])
def test_fp8_bound_covers_emulated_rounding(n, d, causal, mult):
    from test_fp8_gpu import bound, deq
    w = Workload("emulated", 1, 1, n, d, "fp8", causal, 5 + n, qk_mult=mult)
    (q8, k8, v8), (qd, kd, vd) = make_qkv_fp8(w)
    q, k, v = (deq(a, s)[0, 0] for a, s in ((q8, qd), (k8, kd), (v8, vd)))
    v8n = v8.double().numpy()[0, 0]
    o_ref, lse_ref = oracle.attention_fwd(q[None, None], k[None, None], v[None, None], w.scale,
                                          causal)
    o_ref, lse_ref = o_ref[0, 0], lse_ref[0, 0]
    tol = bound(q, k, v8n, vd, w.scale, causal, o_ref, lse_ref)
    good = np.max(np.abs(fp8_emulated_output(q, k, v8n, vd, w.scale, causal) - o_ref) / tol)
    bad = np.max(np.abs(fp8_emulated_output(q, k, v8n, vd, w.scale, causal, "no_v_descale")
                        - o_ref) / tol)
    assert good <= 0.5, good          # the bound has room for what the kernel does
    assert bad > 1.0, bad             # and rejects a dropped V factor


# ------------------------------------------------------------------ backward
def bwd_emulated(q, k, v, do, scale, causal, mistake=None):
    """Forward and backward as the bf16 tensor-core kernels round them: S in fp32, P rounded
    to bf16 before P V, O rounded to bf16; the backward rebuilds P from the LSE, forms delta
    from the stored O, rounds dS and P to bf16 before their products and the gradients to
    bf16 at the end."""
    n = q.shape[0]
    s = scale * (q.astype(np.float32) @ k.T.astype(np.float32)).astype(np.float64)
    if causal:
        s = np.where(causal_mask(n), s, -np.inf)
    m = s.max(1, keepdims=True)
    p = np.exp(s - m)
    l = p.sum(1, keepdims=True)
    lse = (m + np.log(l))[:, 0]
    o = bf16((bf16(p) @ v) / l)
    p2 = np.exp(s - lse[:, None])
    delta = (do * o).sum(1)
    if mistake == "no_delta":
        delta = 0.0 * delta
    ds = bf16(p2 * (do @ v.T - delta[:, None]))
    dv = bf16(bf16(p2).T @ do)
    dq = bf16((1.0 if mistake == "dq_no_scale" else scale) * ds @ k)
    dk = bf16(scale * (ds if mistake == "dk_untransposed" else ds.T) @ q)
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("n,d,causal", [(1, 128, False), (300, 128, True), (640, 64, False),
                                        (513, 32, True)])
def test_backward_bound_covers_emulated_rounding(n, d, causal):
    from test_backward_gpu import U, bounds
    q, k, v = make_shape(1, 1, n, d, "bf16", seed=n + d)
    do = make_shape_dout(1, 1, n, d, "bf16", seed=n + d)
    args = [t[0, 0].double().numpy() for t in (q, k, v, do)]
    scale = 1.0 / math.sqrt(d)
    ref = [r[0, 0] for r in attention_bwd(*[a[None, None] for a in args], scale, causal)]
    o, lse, dq, dk, dv = bwd_emulated(*args, scale, causal)
    tol = bounds(*args, scale, causal, o, lse, ref, U["bf16"])
    for name, g, r, t in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref[:3], tol):
        ratio = float(np.max(np.abs(g - r) / t))
        assert ratio <= 0.8, (name, ratio)


@pytest.mark.parametrize("mistake", ["no_delta", "dq_no_scale", "dk_untransposed"])
def test_backward_bound_rejects_planted_mistakes(mistake):
    from test_backward_gpu import U, bounds
    n, d = 300, 64
    q, k, v = make_shape(1, 1, n, d, "bf16", seed=77)
    do = make_shape_dout(1, 1, n, d, "bf16", seed=77)
    args = [t[0, 0].double().numpy() for t in (q, k, v, do)]
    scale = 1.0 / math.sqrt(d)
    ref = [r[0, 0] for r in attention_bwd(*[a[None, None] for a in args], scale, False)]
    o, lse, dq, dk, dv = bwd_emulated(*args, scale, False, mistake)
    tol = bounds(*args, scale, False, o, lse, ref, U["bf16"])
    worst = max(float(np.max(np.abs(g - r) / t)) for g, r, t in zip((dq, dk, dv), ref[:3], tol))
    assert worst > 1.0, (mistake, worst)
