"""Stream-K tail of the tensor-core tile path.  When the tiles leave the last
wave of the GPU partly idle, the (tile, k-block) iterations of the last waves
are shared out evenly over all CTAs (or CTA pairs); a tile whose k range is
split writes f32 partial tiles, and the last of its CTAs to finish adds them
in k order and runs the epilogue.  These tests force the tail on and off for
shapes that split tiles in every way (two to many segments per tile, whole
tiles inside a share, tiles done whole before the tail) and compare both with
the oracle on every output."""
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


def up_check(M, d, d_ff, layout="kn", seed=0, rows=None):
    x, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=seed)
    if layout == "nk":
        wgd, wud = wg.t().contiguous().to(DEV), wu.t().contiguous().to(DEV)
    else:
        wgd, wud = wg.to(DEV), wu.to(DEV)
    h = swg.swiglu_up(x.to(DEV), wgd, wud, path="tc", layout=layout)
    torch.cuda.synchronize()
    xs = x if rows is None else x[rows].contiguous()
    h64, _, s = oracle.swiglu_up(RAW(xs), RAW(wg), RAW(wu), oracle.BF16)
    got = to64(h) if rows is None else to64(h)[rows]
    res = compare(got, h64, s, "bf16", d)
    assert res["ok"], (M, d, d_ff, layout, res)
    return h


def down_check(M, d_ff, d, layout="kn", seed=0, rows=None):
    h = inputs.make_inputs(M, d_ff, 8, "bf16", seed=seed, x_only=True)[0]
    _, wd, _ = inputs.make_inputs(1, d_ff, d, "bf16", seed=seed + 1)
    r = inputs.make_inputs(M, d, 8, "bf16", seed=seed + 2, x_only=True)[0]
    wdd = wd.t().contiguous().to(DEV) if layout == "nk" else wd.to(DEV)
    y = swg.swiglu_down(h.to(DEV), wdd, r.to(DEV), path="tc", layout=layout)
    torch.cuda.synchronize()
    sel = slice(None) if rows is None else rows
    y64, _, s = oracle.down_proj(RAW(h[sel].contiguous()), RAW(wd), oracle.BF16,
                                 RAW(r[sel].contiguous()))
    res = compare(to64(y)[sel], y64, s, "bf16", d_ff)
    assert res["ok"], (M, d_ff, d, layout, res)
    return y


# (M, d, d_ff): one 128- or 256-row block with few tiles (every tile split),
# and shapes with whole-tile waves before the tail (1-CTA: 310 tiles on 152
# CTAs; pairs: 160 tiles on 76 pairs)
UP = [(17, 264, 520), (128, 520, 1032), (300, 520, 392), (100, 136, 39680),
      (300, 200, 10240)]
DOWN = [(40, 1032, 520), (300, 1032, 392), (513, 520, 264)]


@pytest.mark.parametrize("sk", ["0", "1"])
@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("shape", UP)
def test_up_stream_k(shape, layout, sk, monkeypatch):
    monkeypatch.setenv("SWIGLU_TILE_SK", sk)
    M, d, d_ff = shape
    ws = swg.workspace_bytes(M, d, d_ff, "bf16", "tc")
    assert (ws > 0) == (sk == "1")
    up_check(M, d, d_ff, layout, seed=M + d_ff)


@pytest.mark.parametrize("sk", ["0", "1"])
@pytest.mark.parametrize("layout", ["kn", "nk"])
@pytest.mark.parametrize("shape", DOWN)
def test_down_stream_k(shape, layout, sk, monkeypatch):
    monkeypatch.setenv("SWIGLU_TILE_SK", sk)
    down_check(*shape, layout, seed=shape[0])


@pytest.mark.parametrize("split", ["2", "8", "64"])
def test_split_caps(split, monkeypatch):
    # at most `split` CTAs (pairs) per tile when all tiles fit in one wave
    monkeypatch.setenv("SWIGLU_TILE_SK", "1")
    monkeypatch.setenv("SWIGLU_TILE_SK_SPLIT", split)
    up_check(17, 1032, 264, seed=int(split))
    down_check(300, 2056, 264, seed=int(split))


@pytest.mark.parametrize("pair", ["0", "1"])
def test_stream_k_is_deterministic(pair, monkeypatch):
    monkeypatch.setenv("SWIGLU_TILE_SK", "1")
    monkeypatch.setenv("SWIGLU_TILE_PAIR", pair)
    x, wg, wu = (t.to(DEV) for t in inputs.make_inputs(200, 1032, 392, "bf16", seed=3))
    a = swg.swiglu_up(x, wg, wu, path="tc")
    b = swg.swiglu_up(x, wg, wu, path="tc")
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    swg.check_device_status()


def test_caller_workspace_for_the_tail(monkeypatch):
    monkeypatch.setenv("SWIGLU_TILE_SK", "1")
    M, d, d_ff = 300, 520, 392
    x, wg, wu = (t.to(DEV) for t in inputs.make_inputs(M, d, d_ff, "bf16", seed=9))
    need = swg.workspace_bytes(M, d, d_ff, "bf16", "tc")
    assert need > 0
    ws = torch.full((need,), 0xAB, dtype=torch.uint8, device=DEV)   # stale contents
    a = swg.swiglu_up(x, wg, wu, path="tc", workspace=ws)
    b = swg.swiglu_up(x, wg, wu, path="tc")
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_default_plans_at_full_size():
    # The down projection at d = 4096 with M = 64 (16 single-CTA tiles) and
    # M = 256 (16 pair tiles) takes the stream-K tail by default; checked on
    # rows of both CTAs of a pair.
    for M, rows in ((64, [0, 31, 63]), (256, [0, 127, 128, 255])):
        assert swg.down_workspace_bytes(M, 14336, 4096, "bf16", "tc") > 0
        down_check(M, 14336, 4096, seed=11 + M, rows=rows)
    # whole waves, or most of one, keep whole tiles
    assert swg.down_workspace_bytes(4096, 14336, 4096, "bf16", "tc") == 0
    assert swg.workspace_bytes(256, 4096, 14336, "bf16", "tc") == 0
    swg.check_device_status()
