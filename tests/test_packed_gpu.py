"""Weight packing (step a0, the SwiGLU paper's Kernel-2 interleave in
64-column blocks) on the GPU: the packing kernel against the oracle's packing
bit for bit, and the up projection from packed weights against the oracle on
the unpacked weights, on every path; the same path with packed and unpacked
weights must agree bit for bit (same products, same order)."""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_projection_gb300 as swg
from swiglu_mlp_projection_gb300 import _lib, inputs
from tests.parity import compare

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
RAW = inputs.raw_bits


def to64(t):
    return t.detach().to("cpu", torch.float64).numpy()


@pytest.mark.parametrize("dtype,shape", [("bf16", (64, 520)), ("bf16", (8, 200)),
                                         ("f32", (4, 1032)), ("bf16", (4096, 14336))])
def test_pack_matches_oracle_bitwise(dtype, shape):
    d, d_ff = shape
    _, wg, wu = inputs.make_inputs(1, d, d_ff, dtype, seed=d + d_ff)
    od = oracle.BF16 if dtype == "bf16" else oracle.F32
    want = oracle.pack(RAW(wg), RAW(wu), od)
    out = torch.full(want.shape, 7.0, dtype=wg.dtype, device=DEV)   # no stale zeros
    got = swg.pack_weights(wg.to(DEV), wu.to(DEV), out=out)
    torch.cuda.synchronize()
    assert got.data_ptr() == out.data_ptr()
    assert swg.packed_weight_bytes(d, d_ff, dtype) == want.nbytes
    assert np.array_equal(RAW(got.cpu()).view(np.uint8), want.view(np.uint8))


PATHS = {"f32": ["simt"], "bf16": ["simt", "skinny", "tc"]}
SHAPES = [(1, 64, 136), (3, 520, 264), (16, 1032, 520), (17, 264, 1032), (200, 520, 392),
          (300, 1032, 200)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES)
def test_up_packed_matches_oracle_and_unpacked(dtype, shape):
    M, d, d_ff = shape
    x, wg, wu = inputs.make_inputs(M, d, d_ff, dtype, seed=M + d_ff)
    od = oracle.BF16 if dtype == "bf16" else oracle.F32
    h64, _, s = oracle.swiglu_up(RAW(x), RAW(wg), RAW(wu), od)
    xd, wgd, wud = x.to(DEV), wg.to(DEV), wu.to(DEV)
    wp = swg.pack_weights(wgd, wud)
    view = torch.int16 if dtype == "bf16" else torch.int32
    for path in PATHS[dtype] + ["auto"]:
        if path == "skinny" and M > 256:
            continue
        hp = swg.swiglu_up_packed(xd, wp, d_ff, path=path)
        hu = swg.swiglu_up(xd, wgd, wud, path=path)
        torch.cuda.synchronize()
        res = compare(to64(hp), h64, s, dtype, d)
        assert res["ok"], (shape, dtype, path, res)
        assert torch.equal(hp.view(view), hu.view(view)), (shape, dtype, path)


@pytest.mark.parametrize("env", [("SWIGLU_TILE_PAIR", "0"), ("SWIGLU_TILE_PAIR", "1"),
                                 ("SWIGLU_TILE_SK", "1"), ("SWIGLU_SK_CLUSTER", "4")])
def test_up_packed_kernel_modes(env, monkeypatch):
    monkeypatch.setenv(*env)
    M, d, d_ff = (300, 520, 392) if env[0] != "SWIGLU_SK_CLUSTER" else (7, 1032, 1032)
    path = "skinny" if env[0] == "SWIGLU_SK_CLUSTER" else "tc"
    x, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=5)
    h64, _, s = oracle.swiglu_up(RAW(x), RAW(wg), RAW(wu), oracle.BF16)
    wp = swg.pack_weights(wg.to(DEV), wu.to(DEV))
    hp = swg.swiglu_up_packed(x.to(DEV), wp, d_ff, path=path)
    torch.cuda.synchronize()
    res = compare(to64(hp), h64, s, "bf16", d)
    assert res["ok"], (env, res)


def test_decode_and_prefill_shapes():
    d, d_ff = 4096, 14336
    _, wg, wu = inputs.make_inputs(1, d, d_ff, "bf16", seed=0)
    wgd, wud = wg.to(DEV), wu.to(DEV)
    wp = swg.pack_weights(wgd, wud)
    for M in (1, 16, 4096):
        x = inputs.make_inputs(M, d, d_ff, "bf16", seed=M, x_only=True)[0]
        xd = x.to(DEV)
        hp = swg.swiglu_up_packed(xd, wp, d_ff)
        hu = swg.swiglu_up(xd, wgd, wud)
        torch.cuda.synchronize()
        assert torch.equal(hp.view(torch.int16), hu.view(torch.int16)), M
        rows = [0, M - 1] if M > 1 else [0]
        cols = np.arange(0, d_ff, 97)
        rr = np.repeat(rows, cols.size)
        cc = np.tile(cols, len(rows))
        h64, s = oracle.swiglu_up_at(RAW(x), RAW(wg), RAW(wu), oracle.BF16, rr, cc)
        got = to64(hp)[rr, cc]
        res = compare(got, h64, s, "bf16", d)
        assert res["ok"], (M, res)
    swg.check_device_status()


def test_packed_errors():
    lib = _lib.load()
    x = torch.zeros(2, 64, dtype=torch.bfloat16, device=DEV)
    wp = torch.zeros(64, 128, dtype=torch.bfloat16, device=DEV)
    h = torch.zeros(2 * 64 + 8, dtype=torch.bfloat16, device=DEV)
    st = lib.swiglu_up_packed(x.data_ptr(), wp.data_ptr(), h.data_ptr() + 2, 2, 64, 64,
                              _lib.BF16, 0, None, 0, None)
    assert st == 3                                       # h not 16-byte aligned
    st = lib.swiglu_up_packed(x.data_ptr(), None, h.data_ptr(), 2, 64, 64, _lib.BF16, 0,
                              None, 0, None)
    assert st == 1                                       # null weights
    st = lib.swiglu_up_packed(x.data_ptr(), wp.data_ptr(), wp.data_ptr(), 2, 64, 64,
                              _lib.BF16, 0, None, 0, None)
    assert st == 1                                       # h overlaps the weights
    w = torch.zeros(64, 64, dtype=torch.bfloat16, device=DEV)
    st = lib.swiglu_pack_weights(w.data_ptr(), w.data_ptr(), w.data_ptr(), 64, 64, _lib.BF16,
                                 None)
    assert st == 1                                       # output overlaps an input
    with pytest.raises(ValueError):
        swg.swiglu_up_packed(x, wp[:, :64].contiguous(), 64)
