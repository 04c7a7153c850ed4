"""Seeded synthetic inputs for the attention forward.

This module only draws numbers: it holds none of the attention arithmetic, and it
is the one module that both the GPU tests/benchmark and the oracle side use.

Recipe (the same for every caller): for a workload with seed base ``s`` the
three tensors are drawn with ``torch.Generator().manual_seed(s + t)`` for
t = 0 (Q), 1 (K), 2 (V) as ``torch.randn(..., dtype=float32)`` on the CPU,
multiplied by the workload's Q/K multiplier (1, or 2 for the long-sequence
workload; multiplying by 2 is exact in binary floating point), then cast to the
workload's storage dtype.  The backward's upstream gradient dO is drawn the same way
with t = 3 (no multiplier).  Shapes follow the pages' workloads: [B, H, N, D]
with N = 4096 and d = 128 (the shape the pages analyse), d = 64, and N up to
16k.  There is no dataset on the pages; everything here is synthetic.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    D: int
    dtype: str          # "fp32", "bf16", "fp16" or "fp8" (e4m3 Q, K, V; bf16 O)
    causal: bool
    seed: int           # seed base: Q uses seed, K seed+1, V seed+2
    qk_mult: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def flops(self) -> float:
        """Attention FLOPs counted as 4*B*H*N^2*D, halved for the causal mask."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.D
        return f / 2 if self.causal else f

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


TORCH_DTYPES = {"fp32": torch.float32, "bf16": torch.bfloat16, "fp16": torch.float16,
                "fp8": torch.float8_e4m3fn}

# The workloads; seeds are 1000*c + {0,1,2} for workload number c.
WORKLOADS = {
    "fp32_b1h1n256d64": Workload("fp32_b1h1n256d64", 1, 1, 256, 64, "fp32", False, 1000),
    "bf16_b2h8n1024d64": Workload("bf16_b2h8n1024d64", 2, 8, 1024, 64, "bf16", False, 2000),
    "bf16_b4h16n4096d128": Workload("bf16_b4h16n4096d128", 4, 16, 4096, 128, "bf16", False, 3000),
    "bf16_b8h32n4096d128_causal": Workload("bf16_b8h32n4096d128_causal", 8, 32, 4096, 128,
                                           "bf16", True, 4000),
    "bf16_b1h32n16384d128_x2": Workload("bf16_b1h32n16384d128_x2", 1, 32, 16384, 128, "bf16",
                                        False, 5000, 2.0),
    "bf16_b1h32n16384d128_x2_causal": Workload("bf16_b1h32n16384d128_x2_causal", 1, 32, 16384,
                                               128, "bf16", True, 5000, 2.0),
    # head dimension 256 (the largest head dimension the pages name), same FLOPs as the
    # headline workload
    "bf16_b4h8n4096d256": Workload("bf16_b4h8n4096d256", 4, 8, 4096, 256, "bf16", False, 6000),
    "bf16_b4h8n4096d256_causal": Workload("bf16_b4h8n4096d256_causal", 4, 8, 4096, 256, "bf16",
                                          True, 6000),
    # fp8 e4m3 inputs (per-tensor scales), the headline shape
    "fp8_b4h16n4096d128": Workload("fp8_b4h16n4096d128", 4, 16, 4096, 128, "fp8", False, 8000),
    "fp8_b8h32n4096d128_causal": Workload("fp8_b8h32n4096d128_causal", 8, 32, 4096, 128, "fp8",
                                          True, 8100),
    # head dimension 32 (the "第 13 课" exercise's d), same FLOPs as the headline workload
    "bf16_b8h32n4096d32": Workload("bf16_b8h32n4096d32", 8, 32, 4096, 32, "bf16", False, 7000),
    # head dimension 64 (the small shape's d) at full size, 16-bit and e4m3 inputs
    "bf16_b8h16n4096d64": Workload("bf16_b8h16n4096d64", 8, 16, 4096, 64, "bf16", False, 7100),
    "fp8_b8h16n4096d64": Workload("fp8_b8h16n4096d64", 8, 16, 4096, 64, "fp8", False, 8200),
    # head dimension 256 with e4m3 inputs
    "fp8_b4h8n4096d256": Workload("fp8_b4h8n4096d256", 4, 8, 4096, 256, "fp8", False, 8300),
    "fp8_b4h8n4096d256_causal": Workload("fp8_b4h8n4096d256_causal", 4, 8, 4096, 256, "fp8",
                                         True, 8300),
}

# The workload the throughput metric is quoted on.
HEADLINE = "bf16_b4h16n4096d128"


def make_qkv(w: Workload, seed_offset: int = 0):
    """Q, K, V as CPU tensors of shape [B, H, N, D] in the workload's dtype."""
    shape = (w.B, w.H, w.N, w.D)
    out = []
    for t in range(3):
        g = torch.Generator().manual_seed(w.seed + seed_offset + t)
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if t < 2 and w.qk_mult != 1.0:
            x = x * w.qk_mult
        out.append(x.to(TORCH_DTYPES[w.dtype]).contiguous())
    return tuple(out)


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor fp8 e4m3 quantisation of an fp32 tensor: returns (x8, descale) with
    x8 = round(x / descale) in torch.float8_e4m3fn and descale = max|x| / 448, so that
    descale * x8 is the value the fp8 path computes on."""
    amax = float(x.abs().max())
    descale = amax / 448.0 if amax > 0 else 1.0
    return (x / descale).to(torch.float8_e4m3fn).contiguous(), descale


def make_qkv_fp8(w: Workload, seed_offset: int = 0):
    """Q, K, V drawn as make_qkv draws them (fp32, before the cast), then quantised per
    tensor to e4m3: returns ((q8, k8, v8), (q_descale, k_descale, v_descale))."""
    shape = (w.B, w.H, w.N, w.D)
    out, scales = [], []
    for t in range(3):
        g = torch.Generator().manual_seed(w.seed + seed_offset + t)
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if t < 2 and w.qk_mult != 1.0:
            x = x * w.qk_mult
        x8, ds = quantize_e4m3(x)
        out.append(x8)
        scales.append(ds)
    return tuple(out), tuple(scales)


def make_shape(B, H, N, D, dtype="bf16", seed=7, qk_mult=1.0):
    """Seeded Q, K, V for an arbitrary shape (edge cases in the tests)."""
    w = Workload("adhoc", B, H, N, D, dtype, False, seed, qk_mult)
    return make_qkv(w)


def make_dout(w: Workload, seed_offset: int = 0):
    """dO = dL/dO for the backward: CPU tensor [B, H, N, D] in the workload's dtype."""
    g = torch.Generator().manual_seed(w.seed + seed_offset + 3)
    x = torch.randn((w.B, w.H, w.N, w.D), generator=g, dtype=torch.float32)
    return x.to(TORCH_DTYPES[w.dtype]).contiguous()


def make_shape_dout(B, H, N, D, dtype="bf16", seed=7):
    """Seeded dO for an arbitrary shape (same recipe as make_dout)."""
    return make_dout(Workload("adhoc", B, H, N, D, dtype, False, seed))
