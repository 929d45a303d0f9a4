"""swiglu_up_noalloc: the entry point for callers that cannot allocate device
memory (an operator enqueued from a framework callback that forbids
allocation, a process whose device memory another allocator has reserved, a
latency-critical loop that must not block on cudaMalloc/cudaFree).  It uses
a fixed scratch array held by the library instead of a workspace.

The test calls it through the C ABI and checks every output against the CPU
oracle's fp64 result, within the tolerance the parity tests use, and also
against the regular swiglu_up entry point, on two calls in a row with
different shapes and inputs (the scratch keeps the first call's contents when
the second one runs).  This file sorts last so that a
run stopping at the first failure has run every other test before it.
"""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_projection_gb300 as swg
from swiglu_mlp_projection_gb300 import _lib, inputs
from tests.parity import compare

pytestmark = pytest.mark.gpu

CASES = {
    "bf16": [(16, 4096, 14336, 1), (3, 1000, 1032, 2)],
    "f32": [(1, 512, 2048, 1), (5, 520, 264, 2)],
}


def _to64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def _noalloc(lib, x, wg, wu, h, code):
    M, d = x.shape
    d_ff = wg.shape[1]
    stream = torch.cuda.current_stream()
    return lib.swiglu_up_noalloc(x.data_ptr(), wg.data_ptr(), wu.data_ptr(), h.data_ptr(),
                                 M, d, d_ff, code, stream.cuda_stream)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_noalloc_matches_swiglu_up_on_two_calls(cuda_lib, dtype):
    dev = torch.device("cuda", 0)
    code = _lib.BF16 if dtype == "bf16" else _lib.F32
    od = oracle.BF16 if dtype == "bf16" else oracle.F32
    for (M, d, d_ff, seed) in CASES[dtype]:
        x, wg, wu = inputs.make_inputs(M, d, d_ff, dtype, seed=seed)
        xd, wgd, wud = x.to(dev), wg.to(dev), wu.to(dev)
        ref = swg.swiglu_up(xd, wgd, wud)
        out = torch.full((M, d_ff), float("nan"), dtype=xd.dtype, device=dev)
        st = _noalloc(cuda_lib, xd, wgd, wud, out, code)
        assert st == 0, cuda_lib.swiglu_last_error_string()
        torch.cuda.synchronize()
        raw = inputs.raw_bits
        h64, _, sens = oracle.swiglu_up(raw(x), raw(wg), raw(wu), od)
        res = compare(_to64(out), h64, sens, dtype, d)
        assert res["ok"], (M, d, d_ff, dtype, res)
        # and within the same tolerance of the regular entry point
        res = compare(_to64(out), _to64(ref), sens, dtype, d)
        assert res["ok"], (M, d, d_ff, dtype, "vs swiglu_up", res)
    swg.check_device_status()


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_lib):
    dev = torch.device("cuda", 0)
    M, d, d_ff = 256, 4096, 14336          # needs far more than the fixed scratch
    x = torch.zeros(M, d, dtype=torch.bfloat16, device=dev)
    w = torch.zeros(d, d_ff, dtype=torch.bfloat16, device=dev)
    h = torch.full((M, d_ff), 3.0, dtype=torch.bfloat16, device=dev)
    st = _noalloc(cuda_lib, x, w, w, h, _lib.BF16)
    assert st == 8
    assert b"scratch" in cuda_lib.swiglu_last_error_string()
    # a rejected call enqueues nothing: h keeps its contents
    torch.cuda.synchronize()
    assert bool((h == 3.0).all())
