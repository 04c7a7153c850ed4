"""The seeded input recipe, pinned on the CPU: every test and benchmark input comes from
``inputs.py``, so its draws must be exactly the stated recipe (seeds s, s+1, s+2 for Q, K,
V and s+3 for dO; float32 torch.randn on the CPU; the Q/K multiplier before the cast; the
cast to the storage type; per-tensor e4m3 scaling by max|x| / 448)."""
import math

import torch

from attention_forward_04_gb300.inputs import (WORKLOADS, Workload, make_dout, make_qkv,
                                               make_qkv_fp8, quantize_e4m3)


def draw(seed, shape):
    return torch.randn(shape, generator=torch.Generator().manual_seed(seed), dtype=torch.float32)


def test_qkv_and_dout_follow_the_seeds():
    w = Workload("recipe", 2, 3, 40, 64, "bf16", False, 123)
    shape = (2, 3, 40, 64)
    q, k, v = make_qkv(w)
    for t, x in enumerate((q, k, v)):
        assert x.dtype == torch.bfloat16 and tuple(x.shape) == shape
        assert torch.equal(x, draw(123 + t, shape).to(torch.bfloat16))
    assert torch.equal(make_dout(w), draw(126, shape).to(torch.bfloat16))


def test_multiplier_applies_to_q_and_k_only():
    w = Workload("recipe", 1, 2, 33, 32, "fp16", True, 7, qk_mult=2.0)
    shape = (1, 2, 33, 32)
    q, k, v = make_qkv(w)
    assert torch.equal(q, (2.0 * draw(7, shape)).to(torch.float16))
    assert torch.equal(k, (2.0 * draw(8, shape)).to(torch.float16))
    assert torch.equal(v, draw(9, shape).to(torch.float16))


def test_fp8_is_a_per_tensor_scaling_of_the_same_draws():
    w = Workload("recipe", 1, 2, 50, 64, "fp8", False, 31)
    shape = (1, 2, 50, 64)
    (q8, k8, v8), scales = make_qkv_fp8(w)
    for t, (x8, s) in enumerate(zip((q8, k8, v8), scales)):
        x = draw(31 + t, shape)
        assert s == float(x.abs().max()) / 448.0
        assert x8.dtype == torch.float8_e4m3fn
        assert torch.equal(x8, (x / s).to(torch.float8_e4m3fn))
        # the stored values times the factor are within e4m3's relative rounding of x
        err = (x8.double() * s - x.double()).abs()
        assert bool((err <= 2.0 ** -4 * x.double().abs() + 2.0 ** -9 * s).all())


def test_quantize_keeps_zero_tensors_finite():
    x8, s = quantize_e4m3(torch.zeros(4, 4))
    assert s == 1.0 and bool((x8.float() == 0).all())


def test_workload_table():
    head = WORKLOADS["bf16_b4h16n4096d128"]
    assert (head.B, head.H, head.N, head.D, head.dtype, head.causal) == (4, 16, 4096, 128, "bf16", False)
    assert head.scale == 1.0 / math.sqrt(128)
    assert head.flops == 4.0 * 4 * 16 * 4096 ** 2 * 128
    causal = WORKLOADS["bf16_b8h32n4096d128_causal"]
    assert causal.causal and causal.flops == 4.0 * 8 * 32 * 4096 ** 2 * 128 / 2
    long = WORKLOADS["bf16_b1h32n16384d128_x2"]
    assert (long.N, long.qk_mult) == (16384, 2.0)
    small = WORKLOADS["fp32_b1h1n256d64"]
    assert (small.B, small.H, small.N, small.D, small.dtype) == (1, 1, 256, 64, "fp32")
    for name, w in WORKLOADS.items():
        assert w.name == name
