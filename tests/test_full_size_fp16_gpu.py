"""Full-size backward parity for fp16 storage, on whole slices, with the derived
element-wise bound of test_backward_gpu.py.  The inputs are the seeded headline workload
of ``inputs.py`` stored as fp16.  (The full-size fp16 forward is compared on every row by
test_workloads_full_gpu.py.)"""
import pytest
import torch

from attention_forward_04_gb300 import binding, build
from attention_forward_04_gb300.inputs import WORKLOADS, make_dout, make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    binding.load_library()


@pytest.mark.parametrize("causal", [False, True])
def test_fp16_backward_full_size_slices(causal):
    from test_backward_gpu import compare_slices
    w = WORKLOADS["bf16_b4h16n4096d128"].with_(dtype="fp16", causal=causal)
    q, k, v = make_qkv(w)
    do = make_dout(w)
    compare_slices(q, k, v, do, w.scale, causal, "fp16", [(0, 0), (w.B - 1, w.H - 1)],
                   "fp16 backward causal=%d" % causal)
