"""Weights in the [N, K] layout (torch.nn.Linear.weight, shared dimension
contiguous), read without a copy: parity with the oracle on the same values
in the [K, N] layout, for the up and down projections on both tensor-core
paths."""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_projection_gb300 as swg
from swiglu_mlp_projection_gb300 import inputs
from tests.parity import compare

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def to64(t):
    return t.detach().to("cpu", torch.float64).numpy()


SHAPES = [(1, 64, 64), (3, 520, 264), (16, 1032, 520), (17, 96, 1032), (40, 264, 136),
          (200, 520, 264)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("path", ["skinny", "tc", "auto"])
def test_up_nk(shape, path):
    M, d, d_ff = shape
    x, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=M + d_ff)
    h = swg.swiglu_up(x.to(DEV), wg.t().contiguous().to(DEV), wu.t().contiguous().to(DEV),
                      path=path, layout="nk")
    torch.cuda.synchronize()
    raw = inputs.raw_bits
    h64, _, s = oracle.swiglu_up(raw(x), raw(wg), raw(wu), oracle.BF16)
    res = compare(to64(h), h64, s, "bf16", d)
    assert res["ok"], (shape, path, res)


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("path", ["skinny", "tc"])
def test_down_nk(shape, path):
    M, d_ff, d = shape
    h = inputs.make_inputs(M, d_ff, 8, "bf16", seed=M, x_only=True)[0]
    _, wd, _ = inputs.make_inputs(1, d_ff, d, "bf16", seed=M + 1)
    r = inputs.make_inputs(M, d, 8, "bf16", seed=M + 2, x_only=True)[0]
    y = swg.swiglu_down(h.to(DEV), wd.t().contiguous().to(DEV), r.to(DEV), path=path,
                        layout="nk")
    torch.cuda.synchronize()
    raw = inputs.raw_bits
    y64, _, s = oracle.down_proj(raw(h), raw(wd), oracle.BF16, raw(r))
    res = compare(to64(y), y64, s, "bf16", d_ff)
    assert res["ok"], (shape, path, res)


def test_decode_shape_nk_full():
    M, d, d_ff = 16, 4096, 14336
    x, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=3)
    h = swg.swiglu_up(x.to(DEV), wg.t().contiguous().to(DEV), wu.t().contiguous().to(DEV),
                      layout="nk")
    torch.cuda.synchronize()
    raw = inputs.raw_bits
    h64, _, s = oracle.swiglu_up(raw(x), raw(wg), raw(wu), oracle.BF16)
    assert compare(to64(h), h64, s, "bf16", d)["ok"]


def test_nk_unsupported_paths():
    x, wg, wu = inputs.make_inputs(2, 64, 64, "f32", seed=5)
    with pytest.raises(swg.SwiGLUError) as e:
        swg.swiglu_up(x.to(DEV), wg.t().contiguous().to(DEV), wu.t().contiguous().to(DEV),
                      layout="nk")
    assert e.value.status == 2
    xb, wgb, wub = (t.to(torch.bfloat16).to(DEV) for t in (x, wg, wu))
    with pytest.raises(swg.SwiGLUError) as e:
        swg.swiglu_up(xb, wgb.t().contiguous(), wub.t().contiguous(), layout="nk", path="simt")
    assert e.value.status == 2
