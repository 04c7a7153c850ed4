"""GPU parity of the fp8 forward (fa_fwd_fp8) against the fp64 oracle.

The oracle reads the dequantised inputs descale * x8 exactly (fp8 values times fp32
factors, in fp64).  Tolerance, element-wise on O, derived from the kernel's rounding
points: P is rounded to e4m3 before P V (unit roundoff u8 = 2^-4 for normal values, and at
most 2^-10 absolute below the smallest normal 2^-6; P never exceeds 2^8 < 448, so nothing
saturates), then O is rounded to bf16 (u = 2^-8: 8 significant bits).  With P the oracle's probabilities and
l >= 1 the oracle's row sum relative to the row maximum (the kernel's own sum relative to
its reference maximum is never smaller):
    |O - O_oracle| <= v_descale * (u8 * sum_j P_ij |v8_j| + 2^-10 * sum_j |v8_j| / l_i)
                      + 2^-8 |O_oracle| + 1e-4 * sum_j P_ij |v_j|
(the last term covers fp32 score accumulation and ex2).  The test allows twice the bound
plus 1e-5.  LSE is formed from fp32 sums and keeps the bf16 path's 1e-3.
"""

import numpy as np
import pytest
import torch

import oracle
from attention_forward_04_gb300 import binding, build
from attention_forward_04_gb300.inputs import WORKLOADS, make_qkv_fp8, Workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    binding.load_library()


def deq(x8, ds):
    return x8.to(torch.float64).numpy() * float(ds)


def bound(q, k, v8, vd, scale, causal, o_ref, lse_ref, rows=None):
    """Element-wise error bound (module docstring) for the rows `rows` (default: all) of one
    [N, D] slice; o_ref and lse_ref hold the oracle's values of those rows."""
    N = q.shape[0]
    rows = np.arange(N) if rows is None else np.asarray(rows)
    S = scale * (q[rows] @ k.T)
    vis = (np.arange(N)[None, :] <= rows[:, None]) if causal else np.ones((rows.size, N), dtype=bool)
    P = np.where(vis, np.exp(S - lse_ref[:, None]), 0.0)
    m = np.where(vis, S, -np.inf).max(1)
    l = np.exp(lse_ref - m)              # row sum relative to the row maximum (>= 1)
    av = np.abs(v8)
    t = vd * (2.0 ** -4 * (P @ av) + 2.0 ** -10 * (vis.astype(np.float64) @ av) / l[:, None])
    t += 2.0 ** -8 * np.abs(o_ref) + 1e-4 * (P @ (vd * av))
    return 2.0 * t + 1e-5


def compare(w, slices=None, what=""):
    (q8, k8, v8), (qd, kd, vd) = make_qkv_fp8(w)
    o, lse = binding.fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), qd, kd, vd, scale=w.scale,
                             causal=w.causal)
    torch.cuda.synchronize()
    st, detail = binding.check_device_status()
    assert st == 0, (st, detail)
    o = o.double().cpu().numpy()
    lse = lse.double().cpu().numpy()
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), what
    q, k, v = deq(q8, qd), deq(k8, kd), deq(v8, vd)
    v8n = v8.to(torch.float64).numpy()
    BH = w.B * w.H
    if slices is None:
        slices = range(BH)
    for s in slices:
        b, h = divmod(s, w.H)
        o_ref, lse_ref = oracle.attention_fwd(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1],
                                              v[b:b + 1, h:h + 1], w.scale, w.causal)
        o_ref, lse_ref = o_ref[0, 0], lse_ref[0, 0]
        tol = bound(q[b, h], k[b, h], v8n[b, h], vd, w.scale, w.causal, o_ref, lse_ref)
        err = np.abs(o[b, h] - o_ref)
        worst = np.unravel_index(np.argmax(err / tol), err.shape)
        assert np.all(err <= tol), "%s slice %d: O err %.3e > tol %.3e at %s (max err %.3e)" % (
            what, s, err[worst], tol[worst], worst, err.max())
        el = np.max(np.abs(lse[b, h] - lse_ref))
        assert el <= 1e-3, "%s slice %d: LSE err %.3e" % (what, s, el)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [32, 64, 128, 256])
@pytest.mark.parametrize("N", [1, 17, 128, 129, 300, 1000])
def test_fp8_edge_shapes(N, D, causal):
    w = Workload("adhoc", 1, 2, N, D, "fp8", causal, N * 3 + D)
    compare(w, what="fp8 N=%d D=%d causal=%d" % (N, D, causal))


@pytest.mark.parametrize("D", [128, 256])
def test_fp8_large_scores_force_rescales(D):
    for causal in (False, True):
        w = Workload("adhoc", 1, 2, 700, D, "fp8", causal, 91, qk_mult=4.0)
        compare(w, what="fp8 x4 D=%d causal=%d" % (D, causal))


def test_fp8_rejects_bad_arguments():
    (q8, k8, v8), (qd, kd, vd) = make_qkv_fp8(Workload("adhoc", 1, 1, 64, 64, "fp8", False, 5))
    q8, k8, v8 = q8.cuda(), k8.cuda(), v8.cuda()
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        with pytest.raises(binding.FaError):
            binding.fwd_fp8(q8, k8, v8, bad, kd, vd)
    with pytest.raises(TypeError):
        binding.fwd_fp8(q8.float(), k8, v8, qd, kd, vd)
