"""The tensor-core tile path in its two forms: one CTA per 128-row tile, and
a 2-CTA cluster per 256-row tile whose MMAs run on the CTA pair
(tcgen05 cta_group::2).  Both are compared with the oracle on every output,
for the SwiGLU up projection and the plain down projection, in both weight
layouts, at row counts around the 128- and 256-row tile edges (a pair whose
second CTA has no rows inside M included)."""
import pytest
import torch

import oracle
import swiglu_mlp_projection_gb300 as swg
from swiglu_mlp_projection_gb300 import inputs
from tests.parity import compare

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
RAW = inputs.raw_bits


def to64(t):
    return t.detach().to("cpu", torch.float64).numpy()


UP_SHAPES = [(1, 64, 136), (17, 264, 520), (128, 520, 264), (129, 136, 1032),
             (256, 1032, 264), (300, 520, 392), (513, 264, 136)]
DOWN_SHAPES = [(3, 264, 520), (129, 520, 264), (256, 136, 1032), (300, 1032, 392),
               (513, 264, 136)]


@pytest.mark.parametrize("pair", ["0", "1"])
@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("shape", UP_SHAPES)
def test_up_tiles(shape, layout, pair, monkeypatch):
    monkeypatch.setenv("SWIGLU_TILE_PAIR", pair)
    M, d, d_ff = shape
    assert swg.plan(M, d, d_ff, "bf16", "tc")["cluster"] == (2 if pair == "1" else 1)
    x, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=M + d)
    if layout == "nk":
        wgd, wud = wg.t().contiguous().to(DEV), wu.t().contiguous().to(DEV)
    else:
        wgd, wud = wg.to(DEV), wu.to(DEV)
    h = swg.swiglu_up(x.to(DEV), wgd, wud, path="tc", layout=layout)
    torch.cuda.synchronize()
    h64, _, s = oracle.swiglu_up(RAW(x), RAW(wg), RAW(wu), oracle.BF16)
    res = compare(to64(h), h64, s, "bf16", d)
    assert res["ok"], (shape, layout, pair, res)


@pytest.mark.parametrize("pair", ["0", "1"])
@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("shape", DOWN_SHAPES)
def test_down_tiles(shape, layout, pair, monkeypatch):
    monkeypatch.setenv("SWIGLU_TILE_PAIR", pair)
    M, d_ff, d = shape
    h = inputs.make_inputs(M, d_ff, 8, "bf16", seed=M, x_only=True)[0]
    _, wd, _ = inputs.make_inputs(1, d_ff, d, "bf16", seed=M + 1)
    r = inputs.make_inputs(M, d, 8, "bf16", seed=M + 2, x_only=True)[0]
    wdd = wd.t().contiguous().to(DEV) if layout == "nk" else wd.to(DEV)
    y = swg.swiglu_down(h.to(DEV), wdd, r.to(DEV), path="tc", layout=layout)
    torch.cuda.synchronize()
    y64, _, s = oracle.down_proj(RAW(h), RAW(wd), oracle.BF16, RAW(r))
    res = compare(to64(y), y64, s, "bf16", d_ff)
    assert res["ok"], (shape, layout, pair, res)


def test_guard_rows_and_columns_untouched(monkeypatch):
    # A pair tile reaching past M must not write past the output's last row.
    monkeypatch.setenv("SWIGLU_TILE_PAIR", "1")
    M, d, d_ff = 140, 264, 392
    x, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=5)
    buf = torch.full(((M + 300) * d_ff,), 7.0, dtype=torch.bfloat16, device=DEV)
    h = buf[: M * d_ff].view(M, d_ff)
    swg.swiglu_up(x.to(DEV), wg.to(DEV), wu.to(DEV), out=h, path="tc")
    torch.cuda.synchronize()
    assert bool((buf[M * d_ff:] == 7.0).all())
    h64, _, s = oracle.swiglu_up(RAW(x), RAW(wg), RAW(wu), oracle.BF16)
    assert compare(to64(h), h64, s, "bf16", d)["ok"]


def test_pair_tiles_at_prefill_size_sampled_rows():
    # d = 4096, d_ff = 14336, M = 4096 (the prefill call) in pair mode, checked
    # on rows from both CTAs of several pairs and from the last tile.
    M, d, d_ff = 4096, 4096, 14336
    assert swg.plan(M, d, d_ff, "bf16", "auto")["cluster"] == 2
    x, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=0)
    h = swg.swiglu_up(x.to(DEV), wg.to(DEV), wu.to(DEV))
    torch.cuda.synchronize()
    rows = [0, 127, 128, 255, 1000, 2175, 4095]
    h64, _, s = oracle.swiglu_up(RAW(x[rows].contiguous()), RAW(wg), RAW(wu), oracle.BF16)
    res = compare(to64(h)[rows], h64, s, "bf16", d)
    assert res["ok"], res
    swg.check_device_status()


@pytest.mark.parametrize("layout", ["kn", "nk", "packed"])
@pytest.mark.parametrize("shape", [(17, 264, 520), (300, 520, 392), (513, 1032, 136)])
def test_sequential_gate_then_up_order(shape, layout, monkeypatch):
    # The SwiGLU paper's Kernel-1 order: per tile, a k loop over W_gate, then
    # one over W_up (each N = 128), instead of one interleaved N = 256 loop.
    monkeypatch.setenv("SWIGLU_TILE_SEQ", "1")
    M, d, d_ff = shape
    assert swg.plan(M, d, d_ff, "bf16", "tc")["cluster"] == 1     # single-CTA tiles
    x, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=M + 3)
    xd = x.to(DEV)
    if layout == "nk":
        h = swg.swiglu_up(xd, wg.t().contiguous().to(DEV), wu.t().contiguous().to(DEV),
                          path="tc", layout="nk")
    elif layout == "packed":
        h = swg.swiglu_up_packed(xd, swg.pack_weights(wg.to(DEV), wu.to(DEV)), d_ff, path="tc")
    else:
        h = swg.swiglu_up(xd, wg.to(DEV), wu.to(DEV), path="tc")
    torch.cuda.synchronize()
    h64, _, s = oracle.swiglu_up(RAW(x), RAW(wg), RAW(wu), oracle.BF16)
    res = compare(to64(h), h64, s, "bf16", d)
    assert res["ok"], (shape, layout, res)


@pytest.mark.parametrize("band", ["1", "2", "3"])
@pytest.mark.parametrize("pair", ["0", "1"])
def test_banded_tile_order(band, pair, monkeypatch):
    # tiles run in bands of row blocks (the last band shorter when the band
    # does not divide the row blocks); every tile is computed exactly once
    monkeypatch.setenv("SWIGLU_TILE_BAND", band)
    monkeypatch.setenv("SWIGLU_TILE_PAIR", pair)
    monkeypatch.setenv("SWIGLU_TILE_SK", "0")
    M, d, d_ff = 1100, 264, 904          # 9 / 5 row blocks, 8 column blocks
    x, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=int(band) + 10 * int(pair))
    buf = torch.full(((M + 40) * d_ff,), 7.0, dtype=torch.bfloat16, device=DEV)
    h = buf[: M * d_ff].view(M, d_ff)
    swg.swiglu_up(x.to(DEV), wg.to(DEV), wu.to(DEV), out=h, path="tc")
    torch.cuda.synchronize()
    assert bool((buf[M * d_ff:] == 7.0).all())
    h64, _, s = oracle.swiglu_up(RAW(x), RAW(wg), RAW(wu), oracle.BF16)
    res = compare(to64(h), h64, s, "bf16", d)
    assert res["ok"], (band, pair, res)
    # the down projection's plain tiles too
    _, wd, _ = inputs.make_inputs(1, d_ff, d, "bf16", seed=3)
    hb = h[:, :].contiguous()
    y = swg.swiglu_down(hb, wd.to(DEV), path="tc")
    torch.cuda.synchronize()
    y64, _, ys = oracle.down_proj(RAW(hb.cpu()), RAW(wd), oracle.BF16)
    assert compare(to64(y), y64, ys, "bf16", d_ff)["ok"]
