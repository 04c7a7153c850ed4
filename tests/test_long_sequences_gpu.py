"""Long sequences: the largest single-slice shapes the tests run, checked on sampled rows.

Rows are independent, so the oracle's per-row routine (no N x N matrix) gives exactly the
full oracle's values for the sampled rows.  Tolerances as in test_parity_gpu.py (bf16:
2e-2 on O, 1e-3 on LSE).  N = 131072 is the 128K context the pages cite for O(N) memory
("08 · FlashAttention" §五): here 100 MB of inputs, never an N x N buffer.
"""

import numpy as np
import pytest
import torch

import oracle
from attention_forward_04_gb300 import binding, build
from attention_forward_04_gb300.inputs import Workload, make_qkv, make_qkv_fp8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    binding.load_library()


def sample_rows(N, seed):
    rng = np.random.default_rng(seed)
    rows = {0, 1, 127, 128, N // 2, N - 129, N - 128, N - 2, N - 1}
    rows.update(rng.integers(0, N, size=12).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < N), dtype=np.int64)


def check_rows(q64, k64, v64, o, lse, scale, causal, rows, tol_o, tol_l, what):
    o_ref, l_ref = oracle.attention_rows(q64, k64, v64, scale, causal, np.zeros_like(rows), rows)
    og = o[0, 0, rows].float().cpu().numpy().astype(np.float64)
    lg = lse[0, 0, rows].cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(og)) and np.all(np.isfinite(lg)), what
    eo, el = np.max(np.abs(og - o_ref)), np.max(np.abs(lg - l_ref))
    assert eo <= tol_o and el <= tol_l, "%s: O err %.3e, LSE err %.3e" % (what, eo, el)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_131072_tokens_one_slice(dtype, causal):
    w = Workload("long", 1, 1, 131072, 128, dtype, causal, 9100)
    q, k, v = make_qkv(w)
    o, lse = binding.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    assert binding.check_device_status()[0] == 0
    check_rows(*(t.double().numpy() for t in (q, k, v)), o, lse, w.scale, causal,
               sample_rows(w.N, 1), 2e-2, 1e-3, "%s N=131072 causal=%d" % (dtype, causal))


@pytest.mark.parametrize("causal", [False, True])
def test_65536_tokens_head_dim_256(causal):
    w = Workload("long256", 1, 1, 65536, 256, "bf16", causal, 9200)
    q, k, v = make_qkv(w)
    o, lse = binding.fwd(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    assert binding.check_device_status()[0] == 0
    check_rows(*(t.double().numpy() for t in (q, k, v)), o, lse, w.scale, causal,
               sample_rows(w.N, 2), 2e-2, 1e-3, "D=256 N=65536 causal=%d" % causal)


def test_131072_tokens_fp8():
    # fp8: the element-wise bound of test_fp8_gpu.py, evaluated for each sampled row from that
    # row's probabilities (an N-vector per row)
    w = Workload("long8", 1, 1, 131072, 128, "fp8", True, 9300)
    (q8, k8, v8), (qd, kd, vd) = make_qkv_fp8(w)
    o, lse = binding.fwd_fp8(q8.cuda(), k8.cuda(), v8.cuda(), qd, kd, vd, causal=True)
    torch.cuda.synchronize()
    assert binding.check_device_status()[0] == 0
    q, k, v = (t.double().numpy()[0, 0] * d for t, d in zip((q8, k8, v8), (qd, kd, vd)))
    av = np.abs(v8.double().numpy()[0, 0])
    rows = sample_rows(w.N, 3)
    o_ref, l_ref = oracle.attention_rows(q[None, None], k[None, None], v[None, None], w.scale,
                                         True, np.zeros_like(rows), rows)
    og = o[0, 0, rows].float().cpu().numpy().astype(np.float64)
    lg = lse[0, 0, rows].cpu().numpy().astype(np.float64)
    for n_, r in enumerate(rows):
        s = w.scale * (k[: r + 1] @ q[r])                  # visible keys 0..r
        P = np.exp(s - l_ref[n_])
        l = np.exp(l_ref[n_] - s.max())                    # row sum relative to the maximum
        t = vd * (2.0 ** -4 * (P @ av[: r + 1]) + 2.0 ** -10 * av[: r + 1].sum(0) / l)
        t += 2.0 ** -8 * np.abs(o_ref[n_]) + 1e-4 * vd * (P @ av[: r + 1])
        err = np.abs(og[n_] - o_ref[n_])
        assert np.all(err <= 2.0 * t + 1e-5), "fp8 N=131072 row %d: err %.3e" % (r, err.max())
        assert abs(lg[n_] - l_ref[n_]) <= 1e-3, "fp8 N=131072 row %d LSE" % r
