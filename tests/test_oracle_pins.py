"""Pins for the attention oracle: checks against what the pages and the mathematics fix.

None of these re-derives the oracle's formula.  Each pin is a fact that holds for
the true result whatever the implementation: closed forms, invariants, the tiled
online algorithm of the pages, brute force in plain Python, and the worked
exercise of "第 13 课：GPU 内核与 FlashAttention".  The mutation test at the end
plants plausible mistakes in numpy copies of the definition (on the CPU) and
checks that every one of them fails at least one pin.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle.tiled import attention_tiled

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed, mult=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * mult


def c_oracle(q, k, v, scale, causal):
    return oracle.attention_fwd(q, k, v, scale, causal)


# --------------------------------------------------------------------------- pins
# Each pin takes an implementation impl(q, k, v, scale, causal) -> (o, lse) over
# [B, H, N, D] float64 arrays and raises AssertionError if the fact fails.

def pin_constant_value_column(impl):
    """Rows of P sum to one ("KingOfEgg" §1.1), so a constant column of V passes through."""
    for causal in (False, True):
        q, k, v = rnd((1, 2, 37, 16), 1), rnd((1, 2, 37, 16), 2), rnd((1, 2, 37, 16), 3)
        v[..., 5] = 0.7
        v[..., 9] = -3.25
        o, _ = impl(q, k, v, 0.3, causal)
        assert np.max(np.abs(o[..., 5] - 0.7)) < 1e-13
        assert np.max(np.abs(o[..., 9] + 3.25)) < 1e-13


def pin_identical_keys(impl):
    """All keys equal: weights are uniform over A(i), O_i = mean of those V rows,
    LSE_i = scale*q_i.u + ln|A(i)|."""
    N, D, scale = 29, 8, 0.4
    u = rnd((D,), 11)
    q = rnd((1, 1, N, D), 12)
    k = np.broadcast_to(u, (1, 1, N, D)).copy()
    v = rnd((1, 1, N, D), 13)
    for causal in (False, True):
        o, lse = impl(q, k, v, scale, causal)
        for i in range(N):
            na = i + 1 if causal else N
            assert np.max(np.abs(o[0, 0, i] - v[0, 0, :na].mean(axis=0))) < 1e-12
            assert abs(lse[0, 0, i] - (scale * q[0, 0, i] @ u + math.log(na))) < 1e-12


def pin_tiled_online_equals(impl):
    """The pages' tiled online-softmax algorithm equals the definition
    ("第 13 课" exercise; "pwwt.cn" §4.2 "严格等价"), including ragged blocks."""
    for (N, D, bq, bk) in ((100, 16, 32, 32), (130, 32, 64, 48), (64, 8, 17, 23)):
        q, k, v = rnd((2, 1, N, D), N), rnd((2, 1, N, D), N + 1), rnd((2, 1, N, D), N + 2)
        for causal in (False, True):
            o, lse = impl(q, k, v, 0.25, causal)
            ot, lset = attention_tiled(q, k, v, 0.25, causal, bq, bk)
            assert np.max(np.abs(o - ot)) < 1e-12
            assert np.max(np.abs(lse - lset)) < 1e-12


def _brute_force_slice(q, k, v, scale, causal):
    """Plain-Python loops with math.exp and math.fsum; no numpy arithmetic."""
    N, D = len(q), len(q[0])
    O, L = [], []
    for i in range(N):
        keys = range(i + 1) if causal else range(N)
        s = [scale * math.fsum(q[i][d] * k[j][d] for d in range(D)) for j in keys]
        w = [math.exp(x) for x in s]           # inputs are small: no overflow
        tot = math.fsum(w)
        O.append([math.fsum(w[t] * v[j][d] for t, j in enumerate(keys)) / tot for d in range(D)])
        L.append(math.log(tot))
    return O, L


def pin_brute_force_tiny(impl):
    """Brute force on tiny inputs (N <= 7)."""
    for N in (1, 2, 3, 7):
        D = 4
        q, k, v = rnd((1, 1, N, D), 40 + N), rnd((1, 1, N, D), 50 + N), rnd((1, 1, N, D), 60 + N)
        for causal in (False, True):
            o, lse = impl(q, k, v, 0.6, causal)
            ob, lb = _brute_force_slice(q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist(),
                                        0.6, causal)
            assert np.max(np.abs(o[0, 0] - np.array(ob))) < 1e-12
            assert np.max(np.abs(lse[0, 0] - np.array(lb))) < 1e-12


def pin_two_keys_closed_form(impl):
    """N=2 non-causal: O_0 = sigmoid(s00-s01) v0 + sigmoid(s01-s00) v1, LSE = logaddexp."""
    q, k, v = rnd((1, 1, 2, 3), 71), rnd((1, 1, 2, 3), 72), rnd((1, 1, 2, 3), 73)
    o, lse = impl(q, k, v, 0.9, False)
    for i in range(2):
        s0 = 0.9 * float(q[0, 0, i] @ k[0, 0, 0])
        s1 = 0.9 * float(q[0, 0, i] @ k[0, 0, 1])
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        expect = w0 * v[0, 0, 0] + (1.0 - w0) * v[0, 0, 1]
        assert np.max(np.abs(o[0, 0, i] - expect)) < 1e-13
        assert abs(lse[0, 0, i] - np.logaddexp(s0, s1)) < 1e-13


def pin_zero_scale(impl):
    """scale = 0: uniform weights, O_i = mean of V over A(i), LSE_i = ln|A(i)|;
    causal row 0 returns V_0."""
    N = 21
    q, k, v = rnd((1, 1, N, 8), 81), rnd((1, 1, N, 8), 82), rnd((1, 1, N, 8), 83)
    for causal in (False, True):
        o, lse = impl(q, k, v, 0.0, causal)
        for i in range(N):
            na = i + 1 if causal else N
            assert np.max(np.abs(o[0, 0, i] - v[0, 0, :na].mean(axis=0))) < 1e-13
            assert abs(lse[0, 0, i] - math.log(na)) < 1e-13
    o, _ = impl(q, k, v, 1.3, True)
    assert np.max(np.abs(o[0, 0, 0] - v[0, 0, 0])) < 1e-14


def pin_key_shift(impl):
    """Adding a vector u to every key leaves O unchanged and adds scale*q_i.u to LSE_i."""
    N, D, scale = 40, 16, 0.35
    q, k, v = rnd((1, 2, N, D), 91), rnd((1, 2, N, D), 92), rnd((1, 2, N, D), 93)
    u = rnd((D,), 94)
    for causal in (False, True):
        o1, l1 = impl(q, k, v, scale, causal)
        o2, l2 = impl(q, k + u, v, scale, causal)
        assert np.max(np.abs(o1 - o2)) < 1e-12
        assert np.max(np.abs(l2 - l1 - scale * (q @ u))) < 1e-12


def pin_permutations(impl):
    """Permuting K and V rows together leaves non-causal O unchanged; permuting Q rows
    permutes O and LSE the same way."""
    N, D = 33, 8
    q, k, v = rnd((1, 1, N, D), 101), rnd((1, 1, N, D), 102), rnd((1, 1, N, D), 103)
    o, lse = impl(q, k, v, 0.5, False)
    perm = np.random.default_rng(104).permutation(N)
    o2, lse2 = impl(q, k[:, :, perm], v[:, :, perm], 0.5, False)
    assert np.max(np.abs(o - o2)) < 1e-12 and np.max(np.abs(lse - lse2)) < 1e-12
    o3, lse3 = impl(q[:, :, perm], k, v, 0.5, False)
    assert np.max(np.abs(o[:, :, perm] - o3)) < 1e-12
    assert np.max(np.abs(lse[:, :, perm] - lse3)) < 1e-12


def pin_golden_closed_forms(impl):
    """Hand-derived closed-form cases stored in tests/golden/closed_forms.json."""
    with open(os.path.join(GOLDEN, "closed_forms.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        q = np.array(c["q"])[None, None]
        k = np.array(c["k"])[None, None]
        v = np.array(c["v"])[None, None]
        o, lse = impl(q, k, v, c["scale"], c["causal"])
        assert np.max(np.abs(o[0, 0] - np.array(c["o"]))) < 1e-13, c["name"]
        assert np.max(np.abs(lse[0, 0] - np.array(c["lse"]))) < 1e-13, c["name"]


def pin_head_independence(impl):
    """Each (b, h) slice is its own attention problem ("KingOfEgg" §1.2, §3)."""
    q, k, v = rnd((2, 3, 19, 8), 111), rnd((2, 3, 19, 8), 112), rnd((2, 3, 19, 8), 113)
    o, lse = impl(q, k, v, 0.7, True)
    for b in range(2):
        for h in range(3):
            os_, ls_ = impl(q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1], 0.7, True)
            assert np.max(np.abs(o[b, h] - os_[0, 0])) < 1e-14
            assert np.max(np.abs(lse[b, h] - ls_[0, 0])) < 1e-14


PINS = [pin_constant_value_column, pin_identical_keys, pin_tiled_online_equals,
        pin_brute_force_tiny, pin_two_keys_closed_form, pin_zero_scale, pin_key_shift,
        pin_permutations, pin_golden_closed_forms, pin_head_independence]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_meets_pin(pin):
    pin(c_oracle)


def test_rows_of_p_sum_to_one():
    """The oracle's own normalised P rows sum to one ("KingOfEgg" §1.1)."""
    for causal in (False, True):
        q, k, v = rnd((2, 2, 150, 32), 5, 2.0), rnd((2, 2, 150, 32), 6, 2.0), rnd((2, 2, 150, 32), 7)
        _, _, err = oracle.attention_fwd(q, k, v, 0.2, causal, return_rowsum_err=True)
        assert err < 1e-12


def test_lesson13_exercise():
    """The worked exercise of "第 13 课": rng(0), n=256, d=32, Q,K x0.5, scale 1, block 32.
    The page prints a max abs error ~1e-15 between the tiled and materialising
    versions, an S of 65536 elements, and asserts allclose(atol=1e-6)."""
    with open(os.path.join(GOLDEN, "lesson13_exercise.json")) as f:
        g = json.load(f)
    rng = np.random.default_rng(g["seed"])
    n, d = g["n"], g["d"]
    Q = rng.standard_normal((n, d)) * g["q_mult"]
    K = rng.standard_normal((n, d)) * g["k_mult"]
    V = rng.standard_normal((n, d)) * g["v_mult"]
    o_ref, _ = oracle.attention_fwd(Q[None, None], K[None, None], V[None, None], g["scale"])
    o_flash, _ = attention_tiled(Q[None, None], K[None, None], V[None, None], g["scale"],
                                 False, g["block_size"], g["block_size"])
    err = np.max(np.abs(o_ref - o_flash))
    assert err < 100 * g["printed_max_abs_error"]
    assert np.allclose(o_ref, o_flash, atol=g["page_atol"])
    assert n * n == g["printed_S_size"]


def test_rows_api_matches_full():
    q, k, v = rnd((2, 3, 77, 16), 21), rnd((2, 3, 77, 16), 22), rnd((2, 3, 77, 16), 23)
    for causal in (False, True):
        o, lse = oracle.attention_fwd(q, k, v, 0.3, causal)
        bh = np.array([0, 5, 3, 3, 1])
        rows = np.array([0, 76, 40, 1, 63])
        orow, lrow = oracle.attention_rows(q, k, v, 0.3, causal, bh, rows)
        of = o.reshape(6, 77, 16)
        lf = lse.reshape(6, 77)
        assert np.array_equal(orow, of[bh, rows])
        assert np.array_equal(lrow, lf[bh, rows])


def test_thread_count_does_not_change_result():
    q, k, v = rnd((1, 4, 200, 32), 31), rnd((1, 4, 200, 32), 32), rnd((1, 4, 200, 32), 33)
    o1, l1 = oracle.attention_fwd(q, k, v, 0.2, True, threads=1)
    o4, l4 = oracle.attention_fwd(q, k, v, 0.2, True, threads=4)
    assert np.array_equal(o1, o4) and np.array_equal(l1, l4)


# ------------------------------------------------------------------ mutation test
def _definition(q, k, v, scale, causal, mutate=None):
    """numpy copy of the definition with one planted mistake (CPU only)."""
    S = scale * np.einsum("bhid,bhjd->bhij", q, k)
    if mutate == "no_scale":
        S = np.einsum("bhid,bhjd->bhij", q, k)
    N = q.shape[2]
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    if causal:
        keep = {"causal_upper": j >= i, "causal_off_by_one": j <= i + 1}.get(mutate, j <= i)
        S = np.where(keep, S, -np.inf)
    m = S.max(axis=-1, keepdims=True)
    if mutate == "column_softmax":
        m = S.max(axis=-2, keepdims=True)
        p = np.exp(S - m)
        l = p.sum(axis=-2, keepdims=True)
        return (p / l) @ v, (m + np.log(l))[..., 0, :]
    p = np.exp(m - S) if mutate == "exp_sign" else np.exp(S - m)
    p = np.where(np.isfinite(p), p, 0.0)
    l = p.sum(axis=-1, keepdims=True)
    P = p if mutate == "no_normalise" else p / l
    if mutate == "transposed_p":
        P = np.swapaxes(P, -1, -2)
    o = P @ v
    lse = np.log(l)[..., 0] if mutate == "lse_no_max" else (m + np.log(l))[..., 0]
    if mutate == "lse_log2":
        lse = (m + np.log2(l))[..., 0]
    if mutate == "dropped_first_key":
        o = P[..., 1:] @ v[..., 1:, :]
    return o, lse


MUTANTS = ["no_scale", "causal_upper", "causal_off_by_one", "column_softmax", "exp_sign",
           "no_normalise", "transposed_p", "lse_no_max", "lse_log2", "dropped_first_key"]


def test_unmutated_definition_meets_pins():
    for pin in PINS:
        pin(lambda q, k, v, s, c: _definition(q, k, v, s, c))


@pytest.mark.parametrize("mutant", MUTANTS)
def test_each_planted_mistake_fails_a_pin(mutant):
    impl = lambda q, k, v, s, c: _definition(q, k, v, s, c, mutate=mutant)  # noqa: E731
    caught = []
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin(impl)
        except AssertionError:
            caught.append(pin.__name__)
    assert caught, "planted mistake %r passed every pin" % mutant
