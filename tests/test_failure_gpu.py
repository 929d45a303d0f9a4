"""Failure detection on the GPU without a fault: a bounded wait that runs out
reports SWIGLU_ERR_TIMEOUT to the host and leaves the context usable."""
import time

import pytest
import torch

import oracle
import swiglu_mlp_projection_gb300 as swg
from swiglu_mlp_projection_gb300 import _lib, inputs
from tests.parity import compare

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(cuda_lib):
    swg.check_device_status()                      # starts clean
    t0 = time.time()
    st = cuda_lib.swiglu_selftest_wait_timeout(50, None)
    assert st == 0
    with pytest.raises(swg.SwiGLUError) as e:
        swg.check_device_status()
    assert e.value.status == 6
    assert time.time() - t0 < 30
    swg.check_device_status()                      # the word was cleared
    # the context still runs the real kernels correctly
    dev = torch.device("cuda", 0)
    for M, path in [(4, "skinny"), (40, "tc")]:
        x, wg, wu = inputs.make_inputs(M, 256, 520, "bf16", seed=3)
        h = swg.swiglu_up(x.to(dev), wg.to(dev), wu.to(dev), path=path)
        torch.cuda.synchronize()
        raw = inputs.raw_bits
        h64, _, s = oracle.swiglu_up(raw(x), raw(wg), raw(wu), oracle.BF16)
        assert compare(h.cpu().double().numpy(), h64, s, "bf16", 256)["ok"]
    swg.check_device_status()


def test_selftest_rejects_bad_limits(cuda_lib):
    assert cuda_lib.swiglu_selftest_wait_timeout(0, None) == 1
    assert cuda_lib.swiglu_selftest_wait_timeout(20000, None) == 1
