"""GPU parity of the backward (fa_bwd through the C ABI) against the fp64 backward oracle.

Tolerance, derived from the kernel's arithmetic and applied element by element.  With u the
unit roundoff of the storage type (2^-8 bf16, 2^-11 fp16, 2^-24 fp32: 8, 11 and 24
significant bits), P and dS the oracle's probabilities and softmax derivative, and
e_p = |LSE_gpu - LSE_oracle| + f the relative error of the kernel's rebuilt P (its forward
LSE error, plus f = 1e-4 for fp32 accumulation of S and ex2 on the tensor cores, or
f = 2e-5 for the fp32 kernels' S over D terms and expf):
  * dV = P^T dO with P rounded to 16 bits before the product:
        |err| <= (P (u + e_p))^T |dO| + u |dV|                  (the last term: output rounding)
  * delta is formed from the forward's stored O, so it is off by
        e_delta_i = sum_d |dO_id| |O_gpu - O_oracle|_id + D 2^-24 sum_d |dO_id| |O_id|,
    dP = dO V^T carries fp32 accumulation error e_dP = D 2^-24 |dO| |V|^T, and dS is rounded
    to 16 bits:
        |dS_gpu - dS| <= P (e_delta + e_dP) + (u + e_p) |dS|
  * dQ = scale dS K, dK = scale dS^T Q:
        |err_dQ| <= scale (|dS_gpu - dS| bound) |K| + u |dQ|,
        |err_dK| <= scale (|dS_gpu - dS| bound)^T |Q| + u |dK|.
For fp32 storage nothing is rounded to 16 bits and the same bound holds with u = 2^-24.
The test allows twice each bound plus 1e-5 absolute.  The oracle reads the same stored
Q, K, V, dO, converted exactly to fp64; O and LSE come from the GPU forward, as in
training.
"""
import math

import numpy as np
import pytest
import torch

from attention_forward_04_gb300 import binding, build
from attention_forward_04_gb300.inputs import (WORKLOADS, make_dout, make_qkv, make_shape,
                                               make_shape_dout)
from oracle.backward import attention_bwd

pytestmark = pytest.mark.gpu

U = {"bf16": 2.0 ** -8, "fp16": 2.0 ** -11, "fp32": 2.0 ** -24}
# floor on the relative error of the rebuilt P beyond the LSE difference: fp32 accumulation of
# S and exp2 on the tensor cores (16-bit storage); fp32 S over D terms and expf (fp32 storage)
P_FLOOR = {"bf16": 1e-4, "fp16": 1e-4, "fp32": 2e-5}


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    binding.load_library()


def f64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def gpu_fwd_bwd(q, k, v, do, scale, causal):
    q, k, v, do = (t.cuda() for t in (q, k, v, do))
    o, lse = binding.fwd(q, k, v, scale=scale, causal=causal)
    dq, dk, dv = binding.bwd(q, k, v, o, lse, do, scale=scale, causal=causal)
    torch.cuda.synchronize()
    st, detail = binding.check_device_status()
    assert st == 0, (st, detail)
    return o, lse, dq, dk, dv


def bounds(q, k, v, do, scale, causal, o_gpu, lse_gpu, ref, u, p_floor=1e-4):
    """Element-wise error bounds (see the module docstring) for one [N, D] slice."""
    dq_r, dk_r, dv_r, o_r, lse_r, delta_r = ref
    N, D = q.shape
    S = scale * (q @ k.T)
    P = np.exp(S - lse_r[:, None])
    if causal:
        P = np.where(np.tril(np.ones((N, N), dtype=bool)), P, 0.0)
    dS = P * (do @ v.T - delta_r[:, None])
    gam = D * 2.0 ** -24
    e_p = np.abs(lse_gpu - lse_r) + p_floor
    e_delta = (np.abs(do) * np.abs(o_gpu - o_r)).sum(1) + gam * (np.abs(do) * np.abs(o_r)).sum(1)
    e_dp = gam * (np.abs(do) @ np.abs(v).T)
    e_ds = P * (e_delta[:, None] + e_dp) + (u + e_p[:, None]) * np.abs(dS)
    t_dv = (P * (u + e_p[:, None])).T @ np.abs(do) + u * np.abs(dv_r)
    t_dq = scale * (e_ds @ np.abs(k)) + u * np.abs(dq_r)
    t_dk = scale * (e_ds.T @ np.abs(q)) + u * np.abs(dk_r)
    return [2.0 * t + 1e-5 for t in (t_dq, t_dk, t_dv)]


def compare_slices(q, k, v, do, scale, causal, dtype, slices, what=""):
    o, lse, dq, dk, dv = gpu_fwd_bwd(q, k, v, do, scale, causal)
    got = [f64(t) for t in (dq, dk, dv)]
    o_g, lse_g = f64(o), f64(lse)
    for (b, h) in slices:
        args = [f64(t[b:b + 1, h:h + 1]) for t in (q, k, v, do)]
        ref = attention_bwd(*args, scale, causal)
        ref = [r[0, 0] for r in ref]
        tol = bounds(*(a[0, 0] for a in args), scale, causal, o_g[b, h], lse_g[b, h], ref,
                     U[dtype], P_FLOOR[dtype])
        for name, g, r, t in zip(("dQ", "dK", "dV"), got, ref[:3], tol):
            x = g[b, h]
            assert np.all(np.isfinite(x)), (what, name)
            err = np.abs(x - r)
            worst = np.unravel_index(np.argmax(err / t), err.shape)
            assert np.all(err <= t), "%s %s slice (%d,%d): err %.3e > tol %.3e at %s (max err %.3e)" % (
                what, name, b, h, err[worst], t[worst], worst, err.max())


# ------------------------------------------------------------ small and edge shapes
EDGE_N = [1, 17, 127, 128, 129, 256, 300, 640, 1000]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("N", EDGE_N)
def test_bf16_backward_edge_shapes(N, D, causal):
    q, k, v = make_shape(1, 2, N, D, "bf16", seed=N * 13 + D)
    do = make_shape_dout(1, 2, N, D, "bf16", seed=N * 13 + D)
    compare_slices(q, k, v, do, 1.0 / math.sqrt(D), causal, "bf16", [(0, 0), (0, 1)],
                   "N=%d D=%d causal=%d" % (N, D, causal))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [32, 64, 128, 256])
@pytest.mark.parametrize("N", [1, 17, 129, 300])
def test_fp32_backward(N, D, causal):
    q, k, v = make_shape(2, 1, N, D, "fp32", seed=N * 19 + D)
    do = make_shape_dout(2, 1, N, D, "fp32", seed=N * 19 + D)
    compare_slices(q, k, v, do, 1.0 / math.sqrt(D), causal, "fp32", [(0, 0), (1, 0)],
                   "fp32 N=%d D=%d causal=%d" % (N, D, causal))


# The fp32 backward runs 32-row CTAs (16 at D = 256) of 4 (8) threads per row, or 8-row
# CTAs of 16 threads per row when those would not give every SM (152 on GB300) one; the
# small shapes above take the second form, these (32 slices) the first.
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 256])
def test_fp32_backward_narrow_cta_shape(D, causal):
    q, k, v = make_shape(4, 8, 200, D, "fp32", seed=200 + D)
    do = make_shape_dout(4, 8, 200, D, "fp32", seed=200 + D)
    assert 4 * 8 * ((200 + 31) // 32) >= 152
    compare_slices(q, k, v, do, 1.0 / math.sqrt(D), causal, "fp32", [(0, 0), (1, 3), (3, 7)],
                   "fp32 narrow CTAs D=%d causal=%d" % (D, causal))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("N", [1, 200, 384])
def test_fp16_backward(N, D, causal):
    q, k, v = make_shape(2, 1, N, D, "fp16", seed=N * 17 + D)
    do = make_shape_dout(2, 1, N, D, "fp16", seed=N * 17 + D)
    compare_slices(q, k, v, do, 1.0 / math.sqrt(D), causal, "fp16", [(0, 0), (1, 0)],
                   "fp16 N=%d D=%d causal=%d" % (N, D, causal))


# Head dimension 256 with 16-bit storage: three tensor-core kernels (dQ, dV, dK), each CTA
# on one 128-row tile and the other side streamed in 64-row sub-tiles.  The lengths put the
# sequence end inside and on the edges of both (63/64/65: one sub-tile; 127/128/129 and
# 191/192/193: the tile edge and the second sub-tile of a tile).
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("N", [1, 17, 63, 64, 65, 127, 128, 129, 191, 193, 300, 640])
def test_16bit_backward_head_dim_256(N, dtype, causal):
    q, k, v = make_shape(2, 1, N, 256, dtype, seed=N * 23 + 256)
    do = make_shape_dout(2, 1, N, 256, dtype, seed=N * 23 + 256)
    compare_slices(q, k, v, do, 1.0 / 16.0, causal, dtype, [(0, 0), (1, 0)],
                   "%s D=256 N=%d causal=%d" % (dtype, N, causal))


# 32 slices of 2 tiles: more CTAs than SMs in each of the three kernels.
@pytest.mark.parametrize("causal", [False, True])
def test_16bit_backward_head_dim_256_many_slices(causal):
    q, k, v = make_shape(4, 8, 200, 256, "bf16", seed=456)
    do = make_shape_dout(4, 8, 200, 256, "bf16", seed=456)
    compare_slices(q, k, v, do, 1.0 / 16.0, causal, "bf16", [(0, 0), (1, 3), (3, 7)],
                   "bf16 D=256 32 slices causal=%d" % causal)


@pytest.mark.parametrize("D", [32, 128, 256])
def test_backward_scale_zero_and_large_scores(D):
    # scale 0: P is uniform over the visible keys; scores x4: a peaked softmax
    q, k, v = make_shape(1, 2, 300, D, "bf16", seed=91, qk_mult=4.0)
    do = make_shape_dout(1, 2, 300, D, "bf16", seed=91)
    for scale in (0.0, 1.0 / math.sqrt(D)):
        for causal in (False, True):
            compare_slices(q, k, v, do, scale, causal, "bf16", [(0, 0), (0, 1)],
                           "scale=%g causal=%d" % (scale, causal))


# ------------------------------------------------------------ full-size workloads, sampled
@pytest.mark.parametrize("name", ["bf16_b2h8n1024d64", "bf16_b4h16n4096d128",
                                  "bf16_b8h32n4096d128_causal", "bf16_b8h32n4096d32",
                                  "bf16_b4h8n4096d256", "bf16_b4h8n4096d256_causal"])
def test_backward_full_size_sampled_slices(name):
    w = WORKLOADS[name]
    q, k, v = make_qkv(w)
    do = make_dout(w)
    slices = [(0, 0), (w.B - 1, w.H - 1), (w.B // 2, w.H // 3)]
    compare_slices(q, k, v, do, w.scale, w.causal, "bf16", slices, name)


# ------------------------------------------------------------ contract
@pytest.mark.parametrize("D", [128, 256])
def test_backward_overwrites_outputs_and_is_deterministic(D):
    q, k, v = (t.cuda() for t in make_shape(2, 3, 700, D, "bf16", seed=5))
    do = make_shape_dout(2, 3, 700, D, "bf16", seed=5).cuda()
    o, lse = binding.fwd(q, k, v, causal=True)
    first = binding.bwd(q, k, v, o, lse, do, causal=True)
    outs = [torch.full_like(q, float("nan")) for _ in range(3)]
    ws = torch.full((binding.bwd_workspace_bytes(2, 3, 700),), 0xFF, dtype=torch.uint8,
                    device="cuda")   # workspace needs no initialisation
    second = binding.bwd(q, k, v, o, lse, do, causal=True, dq=outs[0], dk=outs[1], dv=outs[2],
                         workspace=ws)
    torch.cuda.synchronize()
    assert binding.check_device_status()[0] == 0
    for a, b in zip(first, second):
        assert torch.equal(a, b)


def test_backward_rejects_small_workspace():
    q, k, v = (t.cuda() for t in make_shape(1, 1, 128, 64, "bf16", seed=3))
    o, lse = binding.fwd(q, k, v)
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.FaError):
        binding.bwd(q, k, v, o, lse, o.clone(), workspace=ws)
