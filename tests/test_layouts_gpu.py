"""GPU parity of the token-major [B, N, H, D] entry point and of packed variable-length
sequences (cu_seqlens) against the fp64 oracle.  The oracle is applied per sequence to the
same stored inputs, moved into its [B, H, N, D] layout (a transpose, no arithmetic)."""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_forward_04_gb300 import binding, build
from attention_forward_04_gb300.inputs import make_shape

pytestmark = pytest.mark.gpu

TOL = {"fp32": (1e-5, 1e-5), "bf16": (2e-2, 1e-3), "fp16": (2e-2, 1e-3)}


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    binding.load_library()


def check(o, lse, o_ref, lse_ref, dtype, what):
    tol_o, tol_l = TOL[dtype]
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), what
    eo, el = np.max(np.abs(o - o_ref)), np.max(np.abs(lse - lse_ref))
    assert eo <= tol_o and el <= tol_l, "%s: O err %.3e, LSE err %.3e" % (what, eo, el)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [32, 64, 128])
def test_bnhd_matches_oracle(D, causal, dtype):
    B, N, H = 2, 333, 3
    q, k, v = (t.permute(0, 2, 1, 3).contiguous() for t in make_shape(B, H, N, D, dtype, seed=D + 5))
    o, lse = binding.fwd_bnhd(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    assert binding.check_device_status()[0] == 0
    to_bhnd = lambda t: t.permute(0, 2, 1, 3).double().numpy()  # noqa: E731
    o_ref, lse_ref = oracle.attention_fwd(to_bhnd(q), to_bhnd(k), to_bhnd(v), 1 / math.sqrt(D), causal)
    check(o.permute(0, 2, 1, 3).double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, lse_ref,
          dtype, "bnhd D=%d causal=%d" % (D, causal))


LENGTH_MIXES = [[1, 17, 300, 1000, 129, 0, 256], [4096], [257, 3, 640]]


def run_varlen(lengths, H, D, dtype, causal, seed):
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    T = int(cu[-1])
    g = torch.Generator().manual_seed(seed)
    dt = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[dtype]
    q, k, v = (torch.randn((T, H, D), generator=g).to(dt) for _ in range(3))
    o, lse = binding.fwd_varlen(q.cuda(), k.cuda(), v.cuda(), torch.from_numpy(cu).cuda(),
                                max(lengths), causal=causal)
    torch.cuda.synchronize()
    assert binding.check_device_status()[0] == 0
    o = o.double().cpu().numpy()
    lse = lse.double().cpu().numpy()
    for b, L in enumerate(lengths):
        if L == 0:
            continue
        s0, s1 = cu[b], cu[b + 1]
        seq = lambda t: t[s0:s1].permute(1, 0, 2).unsqueeze(0).double().numpy()  # noqa: E731
        o_ref, lse_ref = oracle.attention_fwd(seq(q), seq(k), seq(v), 1 / math.sqrt(D), causal)
        check(o[s0:s1].transpose(1, 0, 2), lse[:, s0:s1], o_ref[0], lse_ref[0], dtype,
              "varlen seq %d (len %d) D=%d causal=%d" % (b, L, D, causal))


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_pair_schedule(causal):
    # 40 heads x 6 sequences x ceil(300 / 128) = 720 single-tile units > 152 SMs: the
    # paired schedule, with empty, single-token and ragged sequences
    run_varlen([1, 17, 300, 0, 129, 256], 40, 64, "bf16", causal, seed=41)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [32, 64, 128])
@pytest.mark.parametrize("mix", range(len(LENGTH_MIXES)))
def test_varlen_bf16(mix, D, causal):
    run_varlen(LENGTH_MIXES[mix], 2, D, "bf16", causal, seed=mix * 10 + D)


@pytest.mark.parametrize("dtype", ["fp16", "fp32"])
def test_varlen_other_dtypes(dtype):
    run_varlen([5, 200, 129], 2, 64, dtype, True, seed=77)


def test_varlen_all_empty_but_one():
    run_varlen([0, 0, 77, 0], 1, 128, "bf16", False, seed=3)


def test_varlen_malformed_offsets_stay_in_bounds():
    """Offsets that decrease or run past `total` are clamped in the kernel: the call must
    return, the device must report no error and every output must be finite (values for the
    malformed sequences are unspecified)."""
    T, H, D = 200, 2, 64
    q, k, v = (torch.randn((T, H, D)).to(torch.bfloat16).cuda() for _ in range(3))
    cu = torch.tensor([0, 100, 50, 300], dtype=torch.int32).cuda()
    o = torch.zeros_like(q)
    lse = torch.zeros((H, T), dtype=torch.float32, device="cuda")
    binding.fwd_varlen(q, k, v, cu, 400, out=o, lse=lse)
    torch.cuda.synchronize()
    assert binding.check_device_status()[0] == 0
    assert bool(torch.isfinite(o).all()) and bool(torch.isfinite(lse).all())


# ------------------------------------------------------------ head dimension 256
@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("causal", [False, True])
def test_bnhd_head_dim_256(causal, dtype):
    B, N, H, D = 2, 333, 3, 256
    q, k, v = (t.permute(0, 2, 1, 3).contiguous() for t in make_shape(B, H, N, D, dtype, seed=261))
    o, lse = binding.fwd_bnhd(q.cuda(), k.cuda(), v.cuda(), causal=causal)
    torch.cuda.synchronize()
    assert binding.check_device_status()[0] == 0
    to_bhnd = lambda t: t.permute(0, 2, 1, 3).double().numpy()  # noqa: E731
    o_ref, lse_ref = oracle.attention_fwd(to_bhnd(q), to_bhnd(k), to_bhnd(v), 1 / math.sqrt(D), causal)
    check(o.permute(0, 2, 1, 3).double().cpu().numpy(), lse.double().cpu().numpy(), o_ref, lse_ref,
          dtype, "bnhd D=256 causal=%d" % causal)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("mix", range(len(LENGTH_MIXES)))
def test_varlen_head_dim_256(mix, causal):
    run_varlen(LENGTH_MIXES[mix], 2, 256, "bf16", causal, seed=mix * 10 + 256)


def test_varlen_head_dim_256_fp16_and_empty():
    run_varlen([0, 65, 0, 190], 2, 256, "fp16", True, seed=257)


@pytest.mark.parametrize("causal", [False, True])
def test_varlen_head_dim_256_fp32(causal):
    run_varlen([1, 17, 300, 0, 129], 2, 256, "fp32", causal, seed=258)
