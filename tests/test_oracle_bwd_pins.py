"""Pins for the backward oracle.

The decisive pin is numerical differentiation of the (separately pinned) forward oracle:
for L = sum(O * G), central differences of L in every input entry must equal the
backward oracle's gradient.  The others are closed forms and sum rules of the softmax
derivative.  A mutation test plants plausible mistakes in numpy copies of the backward and
checks each fails at least one pin.
"""
import numpy as np
import pytest

import oracle
from oracle.backward import attention_bwd


def rnd(shape, seed, mult=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * mult


def c_bwd(q, k, v, do, scale, causal):
    dq, dk, dv, *_ = attention_bwd(q, k, v, do, scale, causal)
    return dq, dk, dv


def pin_finite_differences(impl):
    """dL/dx for L = sum(O * G) by central differences of the C forward oracle."""
    for causal in (False, True):
        B, H, N, D, scale = 1, 2, 6, 4, 0.7
        q, k, v, g = (rnd((B, H, N, D), s) for s in (1, 2, 3, 4))
        dq, dk, dv = impl(q, k, v, g, scale, causal)
        h = 1e-5

        def loss(qq, kk, vv):
            o, _ = oracle.attention_fwd(qq, kk, vv, scale, causal)
            return float(np.sum(o * g))
        for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
                args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
                num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * h)
            assert np.max(np.abs(num - grad)) < 1e-7, (name, causal, np.max(np.abs(num - grad)))


def pin_single_key(impl):
    """N = 1: the softmax weight is the constant 1, so dQ = dK = 0 and dV = dO."""
    q, k, v, g = (rnd((2, 1, 1, 8), s) for s in (5, 6, 7, 8))
    dq, dk, dv = impl(q, k, v, g, 0.9, False)
    assert np.max(np.abs(dq)) < 1e-14 and np.max(np.abs(dk)) < 1e-14
    assert np.max(np.abs(dv - g)) < 1e-14


def pin_sum_rules(impl):
    """Rows of P sum to one: sum_j dV_j = sum_i dO_i, and rows of dS sum to zero, so
    sum_j dK_j = 0 (per slice)."""
    for causal in (False, True):
        q, k, v, g = (rnd((1, 2, 23, 8), s) for s in (9, 10, 11, 12))
        dq, dk, dv = impl(q, k, v, g, 0.4, causal)
        assert np.max(np.abs(dv.sum(axis=2) - g.sum(axis=2))) < 1e-12
        assert np.max(np.abs(dk.sum(axis=2))) < 1e-12


def pin_constant_values(impl):
    """All value rows equal: O does not depend on Q or K, so dQ = dK = 0."""
    q, k, g = (rnd((1, 1, 17, 8), s) for s in (13, 14, 15))
    v = np.broadcast_to(rnd((8,), 16), (1, 1, 17, 8)).copy()
    for causal in (False, True):
        dq, dk, _ = impl(q, k, v, g, 0.6, causal)
        assert np.max(np.abs(dq)) < 1e-12 and np.max(np.abs(dk)) < 1e-12


def pin_causal_last_key(impl):
    """Causal: only the last query sees the last key, so dV_{N-1} = P_{N-1,N-1} dO_{N-1}
    and dK, dV of key j do not depend on queries before j."""
    q, k, v, g = (rnd((1, 1, 9, 4), s) for s in (17, 18, 19, 20))
    _, dk, dv = impl(q, k, v, g, 0.8, True)
    s = 0.8 * q[0, 0, 8] @ k[0, 0].T
    p_last = np.exp(s[8] - s.max()) / np.exp(s - s.max()).sum()
    assert np.max(np.abs(dv[0, 0, 8] - p_last * g[0, 0, 8])) < 1e-13
    g2 = g.copy()
    g2[0, 0, :4] = rnd((4, 4), 21)   # change dO for queries 0..3 only
    _, dk2, dv2 = impl(q, k, v, g2, 0.8, True)
    assert np.max(np.abs(dk2[0, 0, 4:] - dk[0, 0, 4:])) < 1e-13
    assert np.max(np.abs(dv2[0, 0, 4:] - dv[0, 0, 4:])) < 1e-13


PINS = [pin_finite_differences, pin_single_key, pin_sum_rules, pin_constant_values,
        pin_causal_last_key]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_backward_oracle_meets_pin(pin):
    pin(c_bwd)


def test_delta_is_row_dot_of_dout_and_out():
    q, k, v, g = (rnd((1, 2, 31, 16), s) for s in (22, 23, 24, 25))
    for causal in (False, True):
        _, _, _, o, lse, delta = attention_bwd(q, k, v, g, 0.3, causal)
        o_f, lse_f = oracle.attention_fwd(q, k, v, 0.3, causal)
        assert np.max(np.abs(o - o_f)) < 1e-13 and np.max(np.abs(lse - lse_f)) < 1e-13
        assert np.max(np.abs(delta - (g * o).sum(axis=-1))) < 1e-13


def _mutant(q, k, v, do, scale, causal, mutate):
    dq, dk, dv = [], [], []
    B, H, N, D = q.shape
    out = [np.empty_like(q) for _ in range(3)]
    for b in range(B):
        for h in range(H):
            S = scale * q[b, h] @ k[b, h].T
            if causal:
                S = np.where(np.tril(np.ones((N, N), dtype=bool)), S, -np.inf)
            P = np.exp(S - S.max(1, keepdims=True))
            P /= P.sum(1, keepdims=True)
            dP = do[b, h] @ v[b, h].T
            delta = (P * dP).sum(1)
            if mutate == "no_delta":
                delta = 0 * delta
            dS = P * (dP - delta[:, None])
            sq = 1.0 if mutate == "dq_no_scale" else scale
            out[0][b, h] = sq * dS @ k[b, h]
            out[1][b, h] = scale * (dS @ q[b, h] if mutate == "dk_untransposed" else dS.T @ q[b, h])
            out[2][b, h] = (P @ do[b, h]) if mutate == "dv_untransposed" else (P.T @ do[b, h])
    return tuple(out)


@pytest.mark.parametrize("mutant", ["no_delta", "dq_no_scale", "dk_untransposed",
                                    "dv_untransposed"])
def test_each_planted_backward_mistake_fails_a_pin(mutant):
    impl = lambda q, k, v, do, s, c: _mutant(q, k, v, do, s, c, mutant)  # noqa: E731
    caught = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(impl)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, mutant


def test_unmutated_copy_meets_pins():
    for pin in PINS:
        pin(lambda q, k, v, do, s, c: _mutant(q, k, v, do, s, c, None))
