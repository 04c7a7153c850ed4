"""GPU parity of the backward over token-major [B, N, H, D] tensors (fa_bwd_bnhd) and over
packed sequences (fa_bwd_varlen) against the fp64 backward oracle, per (b, h) slice or per
(sequence, head), with the element-wise bound derived for the [B, H, N, D] backward (the
arithmetic is the same; only the addressing differs).  O and LSE come from the GPU forward
in the same layout, as in training."""
import math

import numpy as np
import pytest
import torch

from attention_forward_04_gb300 import binding, build
from attention_forward_04_gb300.inputs import make_shape, make_shape_dout
from oracle.backward import attention_bwd

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    binding.load_library()


def f64(t):
    return t.detach().cpu().to(torch.float64).numpy()


def check_slice(q, k, v, do, o, lse, grads, scale, causal, dtype, what):
    """q, k, v, do, o: [N, D] fp64 of one slice; lse [N]; grads: (dq, dk, dv) [N, D]."""
    from test_backward_gpu import P_FLOOR, U, bounds
    ref = [r[0, 0] for r in attention_bwd(q[None, None], k[None, None], v[None, None],
                                           do[None, None], scale, causal)]
    tol = bounds(q, k, v, do, scale, causal, o, lse, ref, U[dtype], P_FLOOR[dtype])
    for name, g, r, t in zip(("dQ", "dK", "dV"), grads, ref[:3], tol):
        assert np.all(np.isfinite(g)), (what, name)
        err = np.abs(g - r)
        assert np.all(err <= t), "%s %s: max err %.3e (max err/tol %.2f)" % (
            what, name, err.max(), (err / t).max())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [32, 64, 128])
def test_bnhd_backward(D, causal):
    B, N, H = 2, 333, 3
    to_bnhd = lambda t: t.permute(0, 2, 1, 3).contiguous().cuda()  # noqa: E731
    q, k, v = (to_bnhd(t) for t in make_shape(B, H, N, D, "bf16", seed=D + 40))
    do = to_bnhd(make_shape_dout(B, H, N, D, "bf16", seed=D + 40))
    scale = 1.0 / math.sqrt(D)
    o, lse = binding.fwd_bnhd(q, k, v, scale=scale, causal=causal)
    grads = binding.bwd_bnhd(q, k, v, o, lse, do, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert binding.check_device_status()[0] == 0
    for b in range(B):
        for h in range(H):
            sl = lambda t: f64(t[b, :, h])  # noqa: E731
            check_slice(sl(q), sl(k), sl(v), sl(do), sl(o), f64(lse[b, h]),
                        [sl(g) for g in grads], scale, causal, "bf16",
                        "bnhd D=%d causal=%d (b=%d, h=%d)" % (D, causal, b, h))


@pytest.mark.parametrize("dtype,D", [("fp16", 64), ("fp32", 64), ("fp32", 256), ("bf16", 256),
                                     ("fp16", 256)])
def test_bnhd_backward_other_dtypes(dtype, D):
    B, N, H = 1, 200, 2
    to_bnhd = lambda t: t.permute(0, 2, 1, 3).contiguous().cuda()  # noqa: E731
    q, k, v = (to_bnhd(t) for t in make_shape(B, H, N, D, dtype, seed=9))
    do = to_bnhd(make_shape_dout(B, H, N, D, dtype, seed=9))
    o, lse = binding.fwd_bnhd(q, k, v, causal=True)
    grads = binding.bwd_bnhd(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    assert binding.check_device_status()[0] == 0
    for h in range(H):
        sl = lambda t: f64(t[0, :, h])  # noqa: E731
        check_slice(sl(q), sl(k), sl(v), sl(do), sl(o), f64(lse[0, h]), [sl(g) for g in grads],
                    1.0 / math.sqrt(D), True, dtype, "bnhd %s D=%d h=%d" % (dtype, D, h))


LENGTHS = [[1, 17, 300, 129, 0, 256], [640], [257, 3, 500]]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [32, 128])
@pytest.mark.parametrize("mix", range(len(LENGTHS)))
def test_varlen_backward(mix, D, causal):
    run_varlen_backward(LENGTHS[mix], D, causal, "bf16", 100 + mix * 7 + D)


@pytest.mark.parametrize("D", [64, 256])
def test_varlen_backward_fp32(D):
    run_varlen_backward([0, 40, 129, 7], D, True, "fp32", 5)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_backward_bf16_head_dim_256(causal):
    run_varlen_backward([0, 40, 129, 7, 300], 256, causal, "bf16", 6)


def run_varlen_backward(lengths, D, causal, dtype, seed):
    H = 2
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    g = torch.Generator().manual_seed(seed)
    tdt = {"bf16": torch.bfloat16, "fp32": torch.float32}[dtype]
    q, k, v, do = (torch.randn((T, H, D), generator=g).to(tdt).cuda() for _ in range(4))
    cu_t = torch.from_numpy(cu).cuda()
    scale = 1.0 / math.sqrt(D)
    o, lse = binding.fwd_varlen(q, k, v, cu_t, max(lengths), scale=scale, causal=causal)
    grads = binding.bwd_varlen(q, k, v, o, lse, do, cu_t, max(lengths), scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert binding.check_device_status()[0] == 0
    for b, L in enumerate(lengths):
        if L == 0:
            continue
        s0, s1 = int(cu[b]), int(cu[b + 1])
        for h in range(H):
            sl = lambda t: f64(t[s0:s1, h])  # noqa: E731
            check_slice(sl(q), sl(k), sl(v), sl(do), sl(o), f64(lse[h, s0:s1]),
                        [sl(x) for x in grads], scale, causal, dtype,
                        "varlen seq %d (len %d) h=%d D=%d causal=%d" % (b, L, h, D, causal))
