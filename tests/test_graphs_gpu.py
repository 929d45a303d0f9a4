"""Calls captured into a CUDA graph and replayed (the launch-overhead remedy
that "Ou part le temps d'un token" discusses in "Ce qui reste : les
lancements"): every path records into a graph, and replays with new inputs
in the captured buffers match the oracle."""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_projection_gb300 as swg
from swiglu_mlp_projection_gb300 import inputs
from tests.parity import compare

pytestmark = pytest.mark.gpu

CASES = [("bf16", "skinny", 4, 512, 1032), ("bf16", "tc", 40, 256, 520),
         ("f32", "simt", 3, 256, 264), ("bf16", "auto", 16, 1024, 2048)]


def _check(h, x, wg, wu, dtype, d):
    od = oracle.BF16 if dtype == "bf16" else oracle.F32
    raw = inputs.raw_bits
    h64, _, s = oracle.swiglu_up(raw(x), raw(wg), raw(wu), od)
    return compare(h.detach().to("cpu", torch.float64).numpy(), h64, s, dtype, d)


@pytest.mark.parametrize("case", CASES)
def test_capture_and_replay(case):
    dtype, path, M, d, d_ff = case
    dev = torch.device("cuda", 0)
    x0, wg, wu = inputs.make_inputs(M, d, d_ff, dtype, seed=50)
    xs, wgs, wus = x0.to(dev), wg.to(dev), wu.to(dev)
    hs = torch.empty(M, d_ff, dtype=xs.dtype, device=dev)
    swg.swiglu_up(xs, wgs, wus, out=hs, path=path)          # warm-up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(3):                                   # several calls per graph
            swg.swiglu_up(xs, wgs, wus, out=hs, path=path)
    for seed in (51, 52):
        xn = inputs.make_inputs(M, d, d_ff, dtype, seed=seed, x_only=True)[0]
        xs.copy_(xn.to(dev))
        g.replay()
        torch.cuda.synchronize()
        res = _check(hs, xn, wg, wu, dtype, d)
        assert res["ok"], (case, seed, res)
    # calls outside the graph still work on the same stream afterwards
    h2 = swg.swiglu_up(xs, wgs, wus, path=path)
    torch.cuda.synchronize()
    assert torch.equal(h2.view(torch.int16 if dtype == "bf16" else torch.int32),
                       hs.view(torch.int16 if dtype == "bf16" else torch.int32))
    swg.check_device_status()
