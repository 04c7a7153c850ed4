"""Tensors of more than 2^31 elements (2.18 G per tensor, 4.4 GB at 16 bits): every
element offset past 2^31 must be formed in 64 bits.  Whole (b, h) slices at the start, the
middle and the end of each tensor (the last slice lies entirely past element 2^31) are
compared with the fp64 oracle; bf16 and fp16 forward, e4m3 forward, the head-dimension-256
forward, and the backward.

The inputs are drawn on the device from a seeded torch generator (drawing 2.18 G values on
the host would take minutes); the compared slices are copied to the host and handed to the
oracle as they are.  Peak device memory is about 45 GB (the backward)."""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_forward_04_gb300 import binding, build
from attention_forward_04_gb300.inputs import quantize_e4m3
from oracle.backward import attention_bwd

pytestmark = pytest.mark.gpu

H, N, D = 16640, 1024, 128             # 16640 * 1024 * 128 = 2,181,038,080 > 2^31
SLICES = (0, H // 2, H - 1)


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    binding.load_library()


def draw(shape, seed, dtype):
    """Seeded N(0, 1) values drawn on the device, cast to dtype one tensor at a time."""
    g = torch.Generator(device="cuda").manual_seed(seed)
    x = torch.randn(shape, generator=g, device="cuda", dtype=torch.float32)
    out = x.to(dtype)
    del x
    return out


def f64(t):
    """A (small) slice, copied to the host first, as fp64."""
    return t.detach().cpu().to(torch.float64).numpy()


def free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_forward_past_2_31_elements(dtype):
    td = torch.bfloat16 if dtype == "bf16" else torch.float16
    shape = (1, H, N, D)
    assert math.prod(shape) > 2 ** 31
    q, k, v = (draw(shape, 900 + i, td) for i in range(3))
    scale = 1.0 / math.sqrt(D)
    o, lse = binding.fwd(q, k, v, scale=scale, causal=True)
    torch.cuda.synchronize()
    assert binding.check_device_status()[0] == 0
    for h in SLICES:
        o_ref, l_ref = oracle.attention_fwd(f64(q[:, h:h + 1]), f64(k[:, h:h + 1]),
                                            f64(v[:, h:h + 1]), scale, True)
        eo = float(np.max(np.abs(f64(o[:, h:h + 1]) - o_ref)))
        el = float(np.max(np.abs(f64(lse[:, h:h + 1]) - l_ref)))
        assert eo <= 2e-2 and el <= 1e-3, (dtype, h, eo, el)
    del q, k, v, o, lse
    free()


def test_fp8_forward_past_2_31_elements():
    shape = (1, H, N, D)
    x8, ds = [], []
    for i in range(3):
        x = draw(shape, 950 + i, torch.float32)
        a, d = quantize_e4m3(x)
        del x
        x8.append(a)
        ds.append(d)
    scale = 1.0 / math.sqrt(D)
    o, lse = binding.fwd_fp8(*x8, *ds, scale=scale, causal=False)
    torch.cuda.synchronize()
    assert binding.check_device_status()[0] == 0
    from test_fp8_gpu import bound
    for h in SLICES:
        q, k, v = (f64(t[0, h]) * d for t, d in zip(x8, ds))
        o_ref, l_ref = oracle.attention_fwd(q[None, None], k[None, None], v[None, None], scale, False)
        o_ref, l_ref = o_ref[0, 0], l_ref[0, 0]
        tol = bound(q, k, f64(x8[2][0, h]), ds[2], scale, False, o_ref, l_ref)
        err = np.abs(f64(o[0, h]) - o_ref)
        el = float(np.max(np.abs(f64(lse[0, h]) - l_ref)))
        assert np.all(err <= tol) and el <= 1e-3, (h, float(err.max()), el)
    del x8, o, lse
    free()


def test_head_dim_256_forward_past_2_31_elements():
    h256 = 8320                          # 8320 * 1024 * 256 = 2,181,038,080
    shape = (1, h256, N, 256)
    q, k, v = (draw(shape, 970 + i, torch.bfloat16) for i in range(3))
    scale = 1.0 / 16.0
    o, lse = binding.fwd(q, k, v, scale=scale, causal=False)
    torch.cuda.synchronize()
    assert binding.check_device_status()[0] == 0
    for h in (0, h256 // 2, h256 - 1):
        o_ref, l_ref = oracle.attention_fwd(f64(q[:, h:h + 1]), f64(k[:, h:h + 1]),
                                            f64(v[:, h:h + 1]), scale, False)
        eo = float(np.max(np.abs(f64(o[:, h:h + 1]) - o_ref)))
        el = float(np.max(np.abs(f64(lse[:, h:h + 1]) - l_ref)))
        assert eo <= 2e-2 and el <= 1e-3, (h, eo, el)
    del q, k, v, o, lse
    free()


def test_backward_past_2_31_elements():
    from test_backward_gpu import U, bounds
    shape = (1, H, N, D)
    q, k, v, do = (draw(shape, 990 + i, torch.bfloat16) for i in range(4))
    scale = 1.0 / math.sqrt(D)
    o, lse = binding.fwd(q, k, v, scale=scale, causal=False)
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, scale=scale, causal=False)
    torch.cuda.synchronize()
    assert binding.check_device_status()[0] == 0
    for h in (0, H - 1):
        args = [f64(t[:, h:h + 1]) for t in (q, k, v, do)]
        ref = [r[0, 0] for r in attention_bwd(*args, scale, False)]
        tol = bounds(*(a[0, 0] for a in args), scale, False, f64(o[0, h]), f64(lse[0, h]), ref,
                     U["bf16"])
        for name, g, r, t in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref[:3], tol):
            err = np.abs(f64(g[0, h]) - r)
            assert np.all(err <= t), (name, h, float(err.max()))
    del q, k, v, do, o, lse, dq, dk, dv
    free()
