"""The entry points inside CUDA graphs: a forward or backward captured into a
torch.cuda.CUDAGraph and replayed on new inputs (written in place into the captured
buffers) gives the same bits as an eager call on those inputs.  The calls allocate nothing
and never synchronise, so they capture as plain kernel launches."""
import pytest
import torch

from attention_forward_04_gb300 import binding, build
from attention_forward_04_gb300.inputs import make_qkv_fp8, make_shape, make_shape_dout, Workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    binding.load_library()


def inputs(seed, B=2, H=3, N=700, D=128, dtype="bf16"):
    return [t.cuda() for t in make_shape(B, H, N, D, dtype, seed=seed)]


@pytest.mark.parametrize("D,causal", [(128, False), (64, True), (256, True)])
def test_forward_graph_replay_matches_eager(D, causal):
    q, k, v = inputs(1, D=D)
    binding.fwd(q, k, v, causal=causal)              # first call: one-time set-up, outside
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        o_g, lse_g = binding.fwd(q, k, v, causal=causal)
    for seed in (2, 3):
        for dst, src in zip((q, k, v), inputs(seed, D=D)):
            dst.copy_(src)
        g.replay()
        o_e, lse_e = binding.fwd(q, k, v, causal=causal)
        torch.cuda.synchronize()
        assert binding.check_device_status()[0] == 0
        assert torch.equal(o_g, o_e) and torch.equal(lse_g, lse_e)


def test_fp8_forward_graph_replay_matches_eager():
    w = Workload("graph", 1, 2, 600, 128, "fp8", True, 7)
    (q8, k8, v8), ds = make_qkv_fp8(w)
    q8, k8, v8 = q8.cuda(), k8.cuda(), v8.cuda()
    binding.fwd_fp8(q8, k8, v8, *ds, causal=True)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        o_g, lse_g = binding.fwd_fp8(q8, k8, v8, *ds, causal=True)
    (q2, k2, v2), _ = make_qkv_fp8(w.with_(seed=17))
    for dst, src in zip((q8, k8, v8), (q2, k2, v2)):
        dst.copy_(src.cuda())
    g.replay()
    o_e, lse_e = binding.fwd_fp8(q8, k8, v8, *ds, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o_g, o_e) and torch.equal(lse_g, lse_e)


@pytest.mark.parametrize("D", [128, 256])
def test_backward_graph_replay_matches_eager(D):
    q, k, v = inputs(4, D=D)
    do = make_shape_dout(2, 3, 700, D, "bf16", seed=4).cuda()
    o, lse = binding.fwd(q, k, v, causal=True)
    binding.bwd(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        o_g, lse_g = binding.fwd(q, k, v, causal=True)
        grads_g = binding.bwd(q, k, v, o_g, lse_g, do, causal=True)
    for dst, src in zip((q, k, v), inputs(5, D=D)):
        dst.copy_(src)
    do.copy_(make_shape_dout(2, 3, 700, D, "bf16", seed=5).cuda())
    g.replay()
    o_e, lse_e = binding.fwd(q, k, v, causal=True)
    grads_e = binding.bwd(q, k, v, o_e, lse_e, do, causal=True)
    torch.cuda.synchronize()
    assert binding.check_device_status()[0] == 0
    assert torch.equal(o_g, o_e)
    for a, b in zip(grads_g, grads_e):
        assert torch.equal(a, b)
