"""The Python binding refuses caller-supplied buffers whose shape, dtype, layout or device
does not match the call (the C ABI cannot see buffer sizes), before anything is launched."""
import pytest
import torch

from attention_forward_04_gb300 import binding, build
from attention_forward_04_gb300.inputs import make_shape, make_shape_dout

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    binding.load_library()


def qkv(B=1, H=2, N=200, D=64):
    return [t.cuda() for t in make_shape(B, H, N, D, "bf16", seed=3)]


def test_forward_refuses_mismatched_out_and_lse():
    q, k, v = qkv()
    bad_outs = [torch.empty(1, 2, 199, 64, dtype=torch.bfloat16, device="cuda"),   # shape
                torch.empty(1, 2, 200, 64, dtype=torch.float16, device="cuda"),    # dtype
                torch.empty(1, 2, 64, 200, dtype=torch.bfloat16, device="cuda").transpose(2, 3),
                torch.empty(1, 2, 200, 64, dtype=torch.bfloat16)]                  # host
    for out in bad_outs:
        with pytest.raises(ValueError):
            binding.fwd(q, k, v, out=out)
    for lse in (torch.empty(1, 2, 100, device="cuda"), torch.empty(1, 2, 200, device="cuda",
                dtype=torch.float64), torch.empty(1, 2, 200)):
        with pytest.raises(ValueError):
            binding.fwd(q, k, v, lse=lse)
    # well-formed buffers are used as given
    out = torch.empty_like(q)
    lse = torch.empty(1, 2, 200, device="cuda")
    o2, l2 = binding.fwd(q, k, v, out=out, lse=lse)
    torch.cuda.synchronize()
    assert o2.data_ptr() == out.data_ptr() and l2.data_ptr() == lse.data_ptr()
    assert bool(torch.isfinite(out.float()).all())


def test_layout_variants_refuse_mismatched_buffers():
    q, k, v = (t.transpose(1, 2).contiguous() for t in qkv())          # [B, N, H, D]
    with pytest.raises(ValueError):
        binding.fwd_bnhd(q, k, v, out=torch.empty(1, 2, 200, 64, dtype=torch.bfloat16, device="cuda"))
    qp, kp, vp = (t.reshape(200, 2, 64) for t in (q, k, v))              # [total, H, D]
    cu = torch.tensor([0, 120, 200], dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError):
        binding.fwd_varlen(qp, kp, vp, cu, 120, lse=torch.empty(200, 2, device="cuda"))
    with pytest.raises(ValueError):
        binding.fwd_varlen(qp, kp, vp, cu.cpu(), 120)


def test_backward_refuses_mismatched_buffers():
    q, k, v = qkv()
    do = make_shape_dout(1, 2, 200, 64, "bf16", seed=3).cuda()
    o, lse = binding.fwd(q, k, v)
    with pytest.raises(ValueError):
        binding.bwd(q, k, v, o, lse.cpu(), do)
    with pytest.raises(ValueError):
        binding.bwd(q, k, v, o, lse, do, dq=torch.empty(1, 2, 200, 32, dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):
        binding.bwd(q, k, v, o, lse, do, workspace=torch.empty(4096, dtype=torch.uint8))
    with pytest.raises(ValueError):
        binding.bwd_noalloc(q, k, v, o, lse, do, torch.empty_like(q), torch.empty_like(q),
                            torch.empty(1, 2, 200, 64, dtype=torch.float16, device="cuda"))
    torch.cuda.synchronize()
    assert binding.check_device_status()[0] == 0
