"""Failure detection without a GPU fault.

The tensor-core kernel bounds every mbarrier wait.  With a short wait limit and the
loader of CTA 0 told to withhold its first K tile, the waits for that tile run out: the
kernel must raise its status word, leave cleanly (drain copies and products, free TMEM),
and the host must read FA_ERR_TIMEOUT.  The context must stay usable: the next normal
call on the same stream returns correct results.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attention_forward_04_gb300 import binding, build
from attention_forward_04_gb300.inputs import make_shape

pytestmark = pytest.mark.gpu

FA_OK, FA_ERR_TIMEOUT = 0, 5


@pytest.fixture(scope="module", autouse=True)
def gpu_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build.build()
    binding.load_library()


def test_stalled_pipeline_reports_timeout_and_context_survives():
    q, k, v = make_shape(1, 4, 1024, 128, "bf16", seed=41)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    assert binding.check_device_status()[0] == FA_OK   # clears anything left before
    try:
        binding.set_watchdog(1 << 22, 1)   # ~2 ms per wait; CTA 0 withholds its first K tile
        binding.fwd(qc, kc, vc)
        st, detail = binding.check_device_status()
    finally:
        binding.set_watchdog(0, 0)
    assert st == FA_ERR_TIMEOUT, (st, detail)
    assert detail[0] == 1 and detail[2] == 0, detail   # a wait in CTA 0 gave up
    assert detail[1] in (1, 2, 3), detail             # softmax, MMA or loader role

    # the status word is cleared by the read, and a normal call still works
    assert binding.check_device_status()[0] == FA_OK
    o, lse = binding.fwd(qc, kc, vc)
    st, _ = binding.check_device_status()
    assert st == FA_OK
    o_ref, l_ref = oracle.attention_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                        1.0 / math.sqrt(128), False)
    assert np.max(np.abs(o.double().cpu().numpy() - o_ref)) <= 2e-2
    assert np.max(np.abs(lse.double().cpu().numpy() - l_ref)) <= 1e-3


def test_short_limit_alone_does_not_fire():
    """A short but sane wait limit must not fire on a healthy pipeline."""
    q, k, v = make_shape(2, 8, 2048, 128, "bf16", seed=43)
    try:
        binding.set_watchdog(1 << 24, 0)
        o, lse = binding.fwd(q.cuda(), k.cuda(), v.cuda(), causal=True)
        st, detail = binding.check_device_status()
    finally:
        binding.set_watchdog(0, 0)
    assert st == FA_OK, detail
    assert bool(torch.isfinite(o).all())


# The backward kernels bound their waits the same way: dQ (and, at D = 256, dV and dK) and
# the dK/dV kernel each withhold one streamed tile in CTA 0.  Every kernel of the call must
# give up and leave; the next call on the same context must give exactly the results of a
# call made before the stall (the backward is deterministic).
@pytest.mark.parametrize("D", [128, 256])
def test_stalled_backward_reports_timeout_and_context_survives(D):
    from attention_forward_04_gb300.inputs import make_shape_dout
    q, k, v = (t.cuda() for t in make_shape(1, 4, 640, D, "bf16", seed=47))
    do = make_shape_dout(1, 4, 640, D, "bf16", seed=47).cuda()
    assert binding.check_device_status()[0] == FA_OK
    o, lse = binding.fwd(q, k, v, causal=True)
    before = binding.bwd(q, k, v, o, lse, do, causal=True)
    assert binding.check_device_status()[0] == FA_OK
    try:
        binding.set_watchdog(1 << 22, 1)   # ~2 ms per wait; CTA 0 of each kernel withholds a tile
        binding.bwd(q, k, v, o, lse, do, causal=True)
        st, detail = binding.check_device_status()
    finally:
        binding.set_watchdog(0, 0)
    assert st == FA_ERR_TIMEOUT, (st, detail)
    assert detail[0] == 1 and detail[2] == 0, detail   # a wait in CTA 0 gave up
    assert detail[1] in (1, 2, 3), detail             # elementwise, MMA or loader role

    assert binding.check_device_status()[0] == FA_OK
    after = binding.bwd(q, k, v, o, lse, do, causal=True)
    assert binding.check_device_status()[0] == FA_OK
    for a, b in zip(before, after):
        assert torch.equal(a, b)
