"""fa_bwd_noalloc: the backward with library-owned scratch, against fa_bwd.

Both run the same kernels; only where the delta scratch lives differs, so results must be
bit-identical.  Two calls in a row check that the second call's reuse of the fixed scratch
does not disturb the first call's results and that nothing depends on the scratch's prior
contents.  This file sorts last so that it also runs after every other test has used the
library on the same device.
"""
import pytest
import torch

from attention_forward_04_gb300 import binding, build
from attention_forward_04_gb300.inputs import make_shape, make_shape_dout

MAX_ROWS = 4 * 1024 * 1024 // 4   # FA_BWD_NOALLOC_MAX_SCRATCH_BYTES / sizeof(float)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load_library()


def test_noalloc_refuses_before_cuda(lib):
    base, sz = 1 << 40, 1 << 36
    ptrs = [base + i * sz for i in range(9)]
    # one row beyond the fixed scratch: refused (FA_ERR_UNSUPPORTED) with fake pointers,
    # so no CUDA call can have been made
    assert lib.fa_bwd_noalloc(*ptrs, 1, 1, MAX_ROWS + 1, 128, 0.1, 0, 1, None) == 2
    assert lib.fa_bwd_noalloc(*ptrs, 2, 4, MAX_ROWS // 8 + 1, 64, 0.1, 1, 1, None) == 2
    assert lib.fa_bwd_noalloc(0, *ptrs[1:], 1, 1, 128, 128, 0.1, 0, 1, None) == 1
    assert lib.fa_bwd_noalloc(*ptrs, 1, 1, 0, 128, 0.1, 0, 1, None) == 1
    assert lib.fa_bwd_noalloc(*ptrs, 1, 1, 128, 128, 0.1, 2, 1, None) == 1
    assert lib.fa_bwd_noalloc(*ptrs, 1, 1, 128, 128, float("nan"), 0, 1, None) == 1
    assert lib.fa_bwd_noalloc(*ptrs, 1, 1, 128, 96, 0.1, 0, 1, None) == 2
    assert lib.fa_bwd_noalloc(*ptrs, 1, 1, 128, 128, 0.1, 0, 7, None) == 1   # unknown dtype
    # token-major: the same limit on B*H*N rows
    assert lib.fa_bwd_noalloc_bnhd(*ptrs, 1, MAX_ROWS + 1, 1, 128, 0.1, 0, 1, None) == 2
    assert lib.fa_bwd_noalloc_bnhd(*ptrs, 1, 128, 1, 96, 0.1, 0, 1, None) == 2
    assert lib.fa_bwd_noalloc_bnhd(*ptrs, 0, 128, 1, 128, 0.1, 0, 1, None) == 1
    # packed: the limit is on H*total (delta indexed like the [H, total] LSE)
    cu = base + 9 * sz
    assert lib.fa_bwd_noalloc_varlen(*ptrs, cu, 2, 512, MAX_ROWS // 4 + 1, 4, 128, 0.1, 0, 1,
                                     None) == 2
    assert lib.fa_bwd_noalloc_varlen(*ptrs, None, 2, 512, 1000, 4, 128, 0.1, 0, 1, None) == 1
    assert lib.fa_bwd_noalloc_varlen(*ptrs, cu, 0, 512, 1000, 4, 128, 0.1, 0, 1, None) == 1
    assert lib.fa_bwd_noalloc_varlen(*ptrs, cu, 2, 512, 1000, 4, 128, 0.1, 3, 1, None) == 1


def _problem(B, H, N, D, dtype, seed, causal):
    q, k, v = (t.cuda() for t in make_shape(B, H, N, D, dtype, seed=seed))
    do = make_shape_dout(B, H, N, D, dtype, seed=seed).cuda()
    o, lse = binding.fwd(q, k, v, causal=causal)
    return q, k, v, o, lse, do


@pytest.mark.gpu
@pytest.mark.parametrize("shape,dtype,causal", [
    ((2, 3, 700, 128), "bf16", False),
    ((1, 4, 1000, 64), "fp16", True),
    ((1, 4, 500, 256), "bf16", True),          # head dimension 256: dQ, dV and dK kernels
    ((1, 256, 4096, 64), "bf16", True),        # B*H*N = 1,048,576 rows: exactly the limit
])
def test_noalloc_matches_fa_bwd_on_two_calls_in_a_row(lib, shape, dtype, causal):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    B, H, N, D = shape
    pa = _problem(B, H, N, D, dtype, 11, causal)
    pb = _problem(B, H, N, D, dtype, 12, causal)
    ga = [torch.full_like(pa[0], float("nan")) for _ in range(3)]
    gb = [torch.full_like(pa[0], float("nan")) for _ in range(3)]
    torch.cuda.synchronize()
    # two calls back to back on one stream, sharing the fixed scratch
    binding.bwd_noalloc(pa[0], pa[1], pa[2], pa[3], pa[4], pa[5], *ga, causal=causal)
    binding.bwd_noalloc(pb[0], pb[1], pb[2], pb[3], pb[4], pb[5], *gb, causal=causal)
    torch.cuda.synchronize()
    assert binding.check_device_status()[0] == 0
    ra = binding.bwd(pa[0], pa[1], pa[2], pa[3], pa[4], pa[5], causal=causal)
    rb = binding.bwd(pb[0], pb[1], pb[2], pb[3], pb[4], pb[5], causal=causal)
    torch.cuda.synchronize()
    for got, ref in zip(ga + gb, list(ra) + list(rb)):
        assert torch.equal(got, ref)
    assert not torch.equal(ga[0], gb[0])


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,causal", [("bf16", True), ("fp16", False), ("fp32", True)])
def test_noalloc_token_major_and_packed_match(lib, dtype, causal):
    """The token-major and packed no-alloc entry points give the bits of fa_bwd_bnhd and
    fa_bwd_varlen on the same inputs."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    B, N, H, D = 2, 333, 3, 64
    q, k, v = (t.permute(0, 2, 1, 3).contiguous().cuda()
               for t in make_shape(B, H, N, D, dtype, seed=41))
    do = make_shape_dout(B, H, N, D, dtype, seed=41).permute(0, 2, 1, 3).contiguous().cuda()
    o, lse = binding.fwd_bnhd(q, k, v, causal=causal)
    got = [torch.full_like(q, float("nan")) for _ in range(3)]
    binding.bwd_noalloc_bnhd(q, k, v, o, lse, do, *got, causal=causal)
    ref = binding.bwd_bnhd(q, k, v, o, lse, do, causal=causal)
    torch.cuda.synchronize()
    assert binding.check_device_status()[0] == 0
    for a, b in zip(got, ref):
        assert torch.equal(a, b)

    lengths = [1, 300, 0, 129]
    cu = torch.tensor([0, 1, 301, 301, 430], dtype=torch.int32).cuda()
    T = sum(lengths)
    g = torch.Generator().manual_seed(43)
    dt = {"bf16": torch.bfloat16, "fp16": torch.float16, "fp32": torch.float32}[dtype]
    qv, kv, vv, dov = (torch.randn((T, H, D), generator=g).to(dt).cuda() for _ in range(4))
    ov, lv = binding.fwd_varlen(qv, kv, vv, cu, max(lengths), causal=causal)
    got = [torch.full_like(qv, float("nan")) for _ in range(3)]
    binding.bwd_noalloc_varlen(qv, kv, vv, ov, lv, dov, *got, cu, max(lengths), causal=causal)
    ref = binding.bwd_varlen(qv, kv, vv, ov, lv, dov, cu, max(lengths), causal=causal)
    torch.cuda.synchronize()
    assert binding.check_device_status()[0] == 0
    for a, b in zip(got, ref):
        assert torch.equal(a, b)
