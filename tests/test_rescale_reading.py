"""The rescale condition: a stale running reference is exact after the final division.

"08 · FlashAttention" §五 and "第 13 课：GPU 内核与 FlashAttention" §4B rescale the old
output by exp(m_old - m_new) whenever a larger maximum appears (the literal reading,
tau = 0).  The head-dimension 32-128 kernels take the literal reading for bf16 P, and for
fp16 and e4m3 P raise the reference only when a key tile's maximum exceeds it by more than
tau = 8 log2 units; below that, the exponentials are taken against the stale reference.  O
and l share the reference, so the final division cancels it.  Why bf16 needs more than a
stale reference: a row's largest P is then 2^x for fractional x, and its bf16 rounding
times a large |v|, added to the bf16 rounding of O, can pass the 2e-2 tolerance (the
constructed rows of test_literal_reading_on_a_dominant_key).  Two cures: the literal
reading (the largest P is exactly 1), or dividing O by the row sum of the rounded P that
P V multiplies, so that the rounding of P cancels in the quotient (the LSE keeps the
unrounded sum); the head-dimension-256 kernel takes the second with tau = 8 for bf16.

These CPU tests state that recurrence in fp64 (the order of the kernels' steps, not their
code) and check it against the three-pass fp64 oracle for tau in {0, 8, 16}: exact (to
fp64 rounding) with P kept in fp64, and within the bf16 / fp16 output tolerances and the
derived rounding bound with P rounded to the storage type before the P V product, as the
kernels do.  A planted mistake (the reference raised without rescaling O and l) must fail.
"""
import math

import numpy as np
import pytest
import torch

import oracle

LOG2E = 1.0 / math.log(2.0)


def lazy_attention(q, k, v, scale, causal, tau, p_dtype=None, plant=None, block=128,
                   rounded_sum=False):
    """One [N, D] slice by the lazy-reference online softmax.  The reference m (log2 units)
    is raised to the tile maximum only when that maximum exceeds it by more than tau; O and
    l are then multiplied by 2^(m_old - m_new).  P is optionally rounded to p_dtype before
    P V (l keeps the unrounded values).  With rounded_sum, O is divided by a second row sum
    l_o of the rounded P (rescaled with O), while the LSE keeps l.  Returns (O, LSE)."""
    n, d = q.shape
    O = np.zeros((n, d))
    l = np.zeros(n)
    l_o = np.zeros(n)
    m = np.full(n, -np.inf)
    rows = np.arange(n)
    for j0 in range(0, n, block):
        j1 = min(n, j0 + block)
        x = scale * LOG2E * (q @ k[j0:j1].T)            # scores in log2 units
        if causal:
            x = np.where(np.arange(j0, j1)[None, :] <= rows[:, None], x, -np.inf)
        live = np.isfinite(x).any(axis=1)
        tmax = np.where(live, x.max(axis=1, initial=-np.inf), -np.inf)
        raise_ = live & (tmax > m + tau)
        alpha = np.where(raise_, np.exp2(np.where(raise_, m - tmax, 0.0)), 1.0)
        m = np.where(raise_, tmax, m)
        if plant != "no_rescale":
            O = O * alpha[:, None]
            l = l * alpha
            l_o = l_o * alpha
        p = np.where(live[:, None], np.exp2(x - np.where(live, m, 0.0)[:, None]), 0.0)
        l = l + p.sum(axis=1)
        if p_dtype is not None:
            p = torch.from_numpy(p).to(p_dtype).double().numpy()
        l_o = l_o + p.sum(axis=1)
        O = O + p @ v[j0:j1]
    return O / (l_o if rounded_sum else l)[:, None], (m + np.log2(l)) * math.log(2.0)


def rnd(shape, seed, mult=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * mult


def compare(n, d, causal, mult, seed, tau, p_dtype=None, plant=None, rounded_sum=False):
    q, k, v = rnd((n, d), seed, mult), rnd((n, d), seed + 1, mult), rnd((n, d), seed + 2)
    scale = 1.0 / math.sqrt(d)
    o_ref, l_ref = oracle.attention_fwd(q[None, None], k[None, None], v[None, None], scale, causal)
    o, lse = lazy_attention(q, k, v, scale, causal, tau, p_dtype, plant, rounded_sum=rounded_sum)
    return float(np.max(np.abs(o - o_ref[0, 0]))), float(np.max(np.abs(lse - l_ref[0, 0])))


@pytest.mark.parametrize("tau", [0.0, 8.0, 16.0])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("mult", [1.0, 4.0])
def test_stale_reference_is_exact_in_fp64(tau, causal, mult):
    # mult = 4 spreads the scores over tens of log2 units, so the reference is raised
    # several times along each row for every tau
    eo, el = compare(700, 64, causal, mult, 31, tau)
    assert eo < 1e-12 and el < 1e-12, (eo, el)


@pytest.mark.parametrize("rounded_sum", [False, True])
@pytest.mark.parametrize("tau", [0.0, 8.0, 16.0])
@pytest.mark.parametrize("p_dtype,tol_o", [(torch.bfloat16, 2e-2), (torch.float16, 2e-3)])
def test_rounded_p_within_tolerance_for_every_tau(tau, p_dtype, tol_o, rounded_sum):
    for causal in (False, True):
        for mult in (1.0, 4.0):
            eo, el = compare(600, 128, causal, mult, 57, tau, p_dtype, rounded_sum=rounded_sum)
            assert eo < tol_o and el < 1e-6, (causal, mult, eo, el)


@pytest.mark.parametrize("tau", [0.0, 8.0, 16.0])
def test_rounded_sum_error_bound(tau):
    # With O divided by the sum of the rounded weights p~_j = p_j (1 + delta_j), O is a
    # convex combination of the v_j whose weights moved by w_j (delta_j - dbar) / (1 + dbar),
    # dbar = sum_j w_j delta_j; those shifts sum to zero, so
    # |O_err| <= 2u / (1 - u) * max_j |v_j - O| per column, whatever the reference: the row's
    # dominant key (v_j close to O) contributes little, which is the point of the sum.
    for p_dtype, u in ((torch.bfloat16, 2.0 ** -8), (torch.float16, 2.0 ** -11)):
        for causal in (False, True):
            n, d, seed = 900, 64, 77
            q, k, v = rnd((n, d), seed, 4.0), rnd((n, d), seed + 1, 4.0), rnd((n, d), seed + 2)
            scale = 1.0 / math.sqrt(d)
            o_ref, _ = oracle.attention_fwd(q[None, None], k[None, None], v[None, None], scale, causal)
            o, _ = lazy_attention(q, k, v, scale, causal, tau, p_dtype, rounded_sum=True)
            o_ref = o_ref[0, 0]
            err = np.abs(o - o_ref)
            for i in range(0, n, 7):
                keys = v[: i + 1] if causal else v
                bound = 2 * u / (1 - u) * np.abs(keys - o_ref[i]).max(axis=0)
                assert np.all(err[i] <= bound * (1 + 1e-9) + 1e-12), (p_dtype, causal, i)


@pytest.mark.parametrize("tau", [0.0, 8.0, 16.0])
def test_rounded_p_error_bound(tau):
    # P rounded to nearest (unit roundoff u) with l summed from the unrounded values and
    # O accumulated exactly: O_err = sum_j delta_j p_j v_j / l with |delta_j| <= u, so
    # |O_err| <= u * max_j |v_j| per column, whatever the reference.  A fresh reference
    # makes the row maximum's p exactly 1 (no rounding), so on peaked rows (scores x4) the
    # literal reading's error sits well below the bound and the stale reference's nearer
    # to it; both stay inside it.
    for p_dtype, u in ((torch.bfloat16, 2.0 ** -8), (torch.float16, 2.0 ** -11)):
        for causal in (False, True):
            n, d, seed = 900, 64, 77
            q, k, v = rnd((n, d), seed, 4.0), rnd((n, d), seed + 1, 4.0), rnd((n, d), seed + 2)
            scale = 1.0 / math.sqrt(d)
            o_ref, _ = oracle.attention_fwd(q[None, None], k[None, None], v[None, None], scale, causal)
            o, _ = lazy_attention(q, k, v, scale, causal, tau, p_dtype)
            err = np.abs(o - o_ref[0, 0])
            if causal:   # row i sees keys 0..i only
                vmax = np.maximum.accumulate(np.abs(v), axis=0)
            else:
                vmax = np.broadcast_to(np.abs(v).max(axis=0), v.shape)
            assert np.all(err <= u * vmax * (1 + 1e-9) + 1e-12), (p_dtype, causal, float(err.max()))


@pytest.mark.parametrize("tau", [0.0, 16.0])
def test_planted_missing_rescale_fails(tau):
    # raising the reference without rescaling O and l must be caught (scores spread wide
    # enough that the reference moves after the first tile even with tau = 16)
    eo, el = compare(700, 64, False, 6.0, 91, tau, plant="no_rescale")
    assert eo > 1e-3 or el > 1e-3, (eo, el)


def dominant_key_slice(d=64, score=6.25):
    """Q = e_0, K = s_j e_0, V = 0.5 except one row: row 0 of K scores 0, row 200 scores
    `score` with V = 7.96875, every other key scores -100.  Every row then has one dominant
    key with a large value, stored exactly in bf16.  6.25 is 9.02 log2 units above key 0
    (below a 16-unit lazy threshold, above an 8-unit one); 3.5 is 5.05 units above it
    (below both), and its p = 2^5.05 = 33.115 rounds to 33.0 in bf16, a relative error of
    0.35 %, near the unit roundoff 2^-8."""
    n = 256
    q = np.zeros((n, d)); q[:, 0] = 1.0
    k = np.zeros((n, d)); k[:, 0] = -100.0; k[0, 0] = 0.0; k[200, 0] = score
    v = np.full((n, d), 0.5); v[200, :] = 7.96875
    return q, k, v


def test_literal_reading_on_a_dominant_key():
    # The kernels' rounding points for bf16 storage: P to bf16 before P V, O to bf16 at the
    # end.  With a stale reference (tau = 16) the dominant p is 2^9.02 and its rounding
    # (unit roundoff 2^-8) moves O by up to 2^-8 * 7.97; with the literal reading (tau = 0)
    # it is exactly 1 and only the rounding of O itself (half an ulp, 2^-6 near 8) remains.
    q, k, v = dominant_key_slice()
    o_ref, _ = oracle.attention_fwd(q[None, None], k[None, None], v[None, None], 1.0, False)
    err = {}
    for tau in (0.0, 16.0):
        o, _ = lazy_attention(q, k, v, 1.0, False, tau, torch.bfloat16)
        o_bf16 = torch.from_numpy(o).to(torch.bfloat16).double().numpy()
        err[tau] = float(np.abs(o_bf16 - o_ref[0, 0]).max())
    assert err[0.0] <= 2.0 ** -6 + 1e-9 < 2e-2 < err[16.0], err


def test_rounded_sum_on_a_dominant_key():
    # The head-dimension-256 kernel's bf16 reading: tau = 8 with O divided by the row sum of
    # the rounded P.  On the row whose dominant key sits 5.05 log2 units above the first
    # (inside tau = 8, so the reference stays stale), the unrounded sum leaves the dominant
    # p's rounding in O and passes the bound; the rounded sum cancels it, leaving about the
    # literal reading's error (the rounding of O).
    q, k, v = dominant_key_slice(score=3.5)
    o_ref, l_ref = oracle.attention_fwd(q[None, None], k[None, None], v[None, None], 1.0, False)
    err, lse_err = {}, {}
    for name, tau, rs in (("literal", 0.0, False), ("stale", 8.0, False), ("stale+sum", 8.0, True)):
        o, lse = lazy_attention(q, k, v, 1.0, False, tau, torch.bfloat16, rounded_sum=rs)
        o_bf16 = torch.from_numpy(o).to(torch.bfloat16).double().numpy()
        err[name] = float(np.abs(o_bf16 - o_ref[0, 0]).max())
        lse_err[name] = float(np.abs(lse - l_ref[0, 0]).max())
    assert err["stale"] > 2e-2, err
    assert err["stale+sum"] <= 2.0 ** -6 + 1e-9 and err["literal"] <= 2.0 ** -6 + 1e-9, err
    # the LSE comes from the unrounded sum in every reading
    assert max(lse_err.values()) < 1e-12, lse_err


def test_planted_rounded_sum_for_the_lse_fails():
    # taking the LSE from the rounded sum as well moves it by about the dominant p's relative
    # rounding (0.35 %), past the 1e-3 tolerance: the kernel keeps both sums
    q, k, v = dominant_key_slice(score=3.5)
    _, l_ref = oracle.attention_fwd(q[None, None], k[None, None], v[None, None], 1.0, False)
    x = (q @ k.T) / math.log(2.0)
    m = x[:, 0]   # the stale reference: key 0's score, the maximum of the first key tile
    p = torch.from_numpy(np.exp2(x - m[:, None])).to(torch.bfloat16).double().numpy()
    lse_rounded = (m + np.log2(p.sum(axis=1))) * math.log(2.0)
    assert np.abs(lse_rounded - l_ref[0, 0]).max() > 1e-3
