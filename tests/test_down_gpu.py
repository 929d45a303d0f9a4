"""Parity of the down projection y = h.W_down (+ residual) and of the
two-kernel MLP with the oracle (anatomy chapter, section 1.6, kernels #10
and #11)."""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_projection_gb300 as swg
from swiglu_mlp_projection_gb300 import inputs
from tests.parity import compare, tile_rows

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


def to64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def make(M, d_ff, d, seed, with_resid=True):
    h = inputs.make_inputs(M, d_ff, 8, "bf16", seed=seed, x_only=True)[0]
    _, wd, _ = inputs.make_inputs(1, d_ff, d, "bf16", seed=seed + 1)
    r = inputs.make_inputs(M, d, 8, "bf16", seed=seed + 2, x_only=True)[0] if with_resid else None
    return h, wd, r


def check(M, d_ff, d, path, seed=0, with_resid=True, rows=None):
    h, wd, r = make(M, d_ff, d, seed, with_resid)
    y = swg.swiglu_down(h.to(DEV), wd.to(DEV), r.to(DEV) if r is not None else None, path=path)
    torch.cuda.synchronize()
    raw = inputs.raw_bits
    sel = slice(None) if rows is None else rows
    hs = h[sel].contiguous()
    rs = r[sel].contiguous() if r is not None else None
    y64, _, s = oracle.down_proj(raw(hs), raw(wd), oracle.BF16, raw(rs) if rs is not None else None)
    res = compare(to64(y)[sel], y64, s, "bf16", d_ff)
    assert res["ok"], (M, d_ff, d, path, with_resid, res)
    return y


RAGGED = [(1, 64, 64), (3, 200, 136), (16, 1032, 520), (17, 96, 264), (40, 520, 1032),
          (5, 4104, 264), (130, 264, 520)]


@pytest.mark.parametrize("shape", RAGGED)
@pytest.mark.parametrize("path", ["skinny", "tc", "auto"])
def test_ragged(shape, path):
    M, d_ff, d = shape
    if path == "skinny" and M > 256:
        pytest.skip("skinny path serves M <= 256")
    check(M, d_ff, d, path, seed=M + d, with_resid=True)
    check(M, d_ff, d, path, seed=M + d + 7, with_resid=False)


@pytest.mark.parametrize("cluster", ["0", "4", "8"])
def test_skinny_plain_cluster_modes(cluster, monkeypatch):
    monkeypatch.setenv("SWIGLU_SK_CLUSTER", cluster)
    for shape in [(1, 4864, 896), (16, 1032, 520), (7, 520, 1032)]:
        check(*shape, "skinny", seed=int(cluster) + shape[0])


@pytest.mark.parametrize("M", [1, 4, 16, 48])
def test_decode_shape_full(M):
    # d_ff=14336 -> d=4096; M = 48 takes 4-CTA clusters of 128-column groups
    check(M, 14336, 4096, "auto", seed=M)


@pytest.mark.parametrize("M", [1, 96, 256])
def test_small_model_full(M):
    # d_ff = 4864 -> d = 896 (8.7 MB of weights): AUTO serves every M up to
    # 256 on the skinny kernel's cluster mode
    assert swg.down_plan(M, 4864, 896)["path"] == "skinny"
    check(M, 4864, 896, "auto", seed=M + 5)


@pytest.mark.parametrize("M", [33, 48, 64, 256])
def test_skinny_cluster4_rows(M, monkeypatch):
    # the skinny kernel in 4-CTA clusters of 128-column groups (the K quarters
    # meet on chip; AUTO takes it for FP8 at 16-64 rows), forced for bf16
    monkeypatch.setenv("SWIGLU_SK_CLUSTER", "4")
    monkeypatch.setenv("SWIGLU_SK_NB", "1")
    p = swg.down_plan(M, 14336, 4096)
    assert p["path"] == "skinny" and p["cluster"] == 4 and p["workspace"] == 0
    check(M, 14336, 4096, "auto", seed=M, rows=tile_rows(M, seed=M))


@pytest.mark.parametrize("M", [1, 16, 32, 48, 65, 128, 256])
def test_skinny_two_kernel_rows(M):
    # AUTO runs the bf16 down projection on the skinny kernel's stream-K
    # form on every SM and adds the partial sums in a second kernel; every
    # column of rows of every 128-row block against the oracle
    p = swg.down_plan(M, 14336, 4096, "bf16", "auto", 0)
    assert p["path"] == "skinny" and p["cluster"] == 1 and p["launches"] == 2
    rows = np.arange(M) if M <= 32 else tile_rows(M, seed=M)
    check(M, 14336, 4096, "auto", seed=M + 3, rows=rows)
    swg.check_device_status()


@pytest.mark.parametrize("shape", [(1, 14336, 4096), (16, 14336, 4096), (200, 14336, 4096),
                                   (40, 4104, 1032), (7, 29568, 8192)])
def test_two_kernel_sums_equal_one_kernel_sums(shape, monkeypatch):
    # Stream-K mode: the second kernel (SWIGLU_SK_SPLIT=1) adds each column
    # group's partial sums in the order the group's last CTA does in the
    # one-kernel form (SWIGLU_SK_SPLIT=0, sums staged by bulk copies or read
    # from L2): the bits must agree, and match the oracle
    M, d_ff, d = shape
    h, wd, r = make(M, d_ff, d, seed=M + 11)
    monkeypatch.setenv("SWIGLU_SK_CLUSTER", "0")
    outs = []
    for split, bulk in (("1", "1"), ("0", "1"), ("0", "0")):
        monkeypatch.setenv("SWIGLU_SK_SPLIT", split)
        monkeypatch.setenv("SWIGLU_SK_BULK", bulk)
        p = swg.down_plan(M, d_ff, d, "bf16", "skinny", 0)
        assert p["cluster"] == 1 and p["launches"] == (2 if split == "1" else 1)
        y = swg.swiglu_down(h.to(DEV), wd.to(DEV), r.to(DEV), path="skinny")
        torch.cuda.synchronize()
        outs.append(y)
    for y in outs[1:]:
        assert torch.equal(outs[0].view(torch.int16), y.view(torch.int16))
    raw = inputs.raw_bits
    rows = np.unique(np.linspace(0, M - 1, min(M, 6)).astype(int))
    y64, _, s = oracle.down_proj(raw(h[rows].contiguous()), raw(wd), oracle.BF16,
                                 raw(r[rows].contiguous()))
    assert compare(to64(outs[0])[rows], y64, s, "bf16", d_ff)["ok"]
    swg.check_device_status()


def test_cluster4_and_stream_k_agree(monkeypatch):
    # both modes of the skinny kernel serve the same call
    M, d_ff, d = 40, 14336, 4096
    h, wd, r = make(M, d_ff, d, seed=77)
    outs = {}
    for mode in ("0", "4"):
        monkeypatch.setenv("SWIGLU_SK_CLUSTER", mode)
        monkeypatch.setenv("SWIGLU_SK_NB", "1")
        assert swg.down_plan(M, d_ff, d, "bf16", "skinny")["cluster"] == (4 if mode == "4" else 1)
        y = swg.swiglu_down(h.to(DEV), wd.to(DEV), r.to(DEV), path="skinny")
        torch.cuda.synchronize()
        outs[mode] = to64(y)
    raw = inputs.raw_bits
    y64, _, s = oracle.down_proj(raw(h), raw(wd), oracle.BF16, raw(r))
    for mode, y in outs.items():
        assert compare(y, y64, s, "bf16", d_ff)["ok"], mode


def test_prefill_shape_tile_rows():
    # M = 4096 (16 row blocks of CTA-pair tiles): every column of 2 rows of
    # every 128-row block, so every 256-column output tile is reached
    check(4096, 14336, 4096, "auto", seed=9, rows=tile_rows(4096, seed=9))


def test_in_place_residual_and_paths_agree():
    M, d_ff, d = 24, 640, 520
    h, wd, r = make(M, d_ff, d, seed=31)
    raw = inputs.raw_bits
    y64, _, s = oracle.down_proj(raw(h), raw(wd), oracle.BF16, raw(r))
    outs = {}
    for path in ("skinny", "tc"):
        y = r.to(DEV).clone()
        swg.swiglu_down(h.to(DEV), wd.to(DEV), residual=y, out=y, path=path)   # y += h.W
        torch.cuda.synchronize()
        outs[path] = to64(y)
        assert compare(outs[path], y64, s, "bf16", d_ff)["ok"], path
    assert compare(outs["skinny"], outs["tc"], s, "bf16", d_ff)["ok"]


def test_deterministic_and_errors():
    h, wd, r = make(7, 1024, 512, seed=41)
    a = swg.swiglu_down(h.to(DEV), wd.to(DEV), r.to(DEV), path="skinny")
    b = swg.swiglu_down(h.to(DEV), wd.to(DEV), r.to(DEV), path="skinny")
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    with pytest.raises(swg.SwiGLUError) as e:
        swg.swiglu_down(h.float().to(DEV), wd.float().to(DEV))
    assert e.value.status == 2
    with pytest.raises(swg.SwiGLUError) as e:
        swg.swiglu_down(h.to(DEV), wd.to(DEV), path="simt")
    assert e.value.status == 2
    # d_ff = 0: y = residual
    y = swg.swiglu_down(torch.empty(3, 0, dtype=torch.bfloat16, device=DEV),
                        torch.empty(0, 16, dtype=torch.bfloat16, device=DEV),
                        torch.ones(3, 16, dtype=torch.bfloat16, device=DEV))
    torch.cuda.synchronize()
    assert torch.all(y == 1)


@pytest.mark.parametrize("M", [1, 16, 200])
def test_mlp_matches_oracle(M):
    d, d_ff = 512, 1536
    x, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=60 + M)
    _, wd, _ = inputs.make_inputs(1, d_ff, d, "bf16", seed=70 + M)
    y, h = swg.swiglu_mlp(x.to(DEV), wg.to(DEV), wu.to(DEV), wd.to(DEV), residual=x.to(DEV))
    torch.cuda.synchronize()
    raw = inputs.raw_bits
    # the intermediate is the up projection's output: check it on its own ...
    h64, _, hs = oracle.swiglu_up(raw(x), raw(wg), raw(wu), oracle.BF16)
    assert compare(to64(h), h64, hs, "bf16", d)["ok"]
    # ... and the second step from the GPU's own bf16 intermediate
    y64, _, ys = oracle.down_proj(inputs.raw_bits(h.cpu()), raw(wd), oracle.BF16, raw(x))
    assert compare(to64(y), y64, ys, "bf16", d_ff)["ok"]
    swg.check_device_status()


@pytest.mark.parametrize("shape", [(16, 14336, 4096), (64, 14336, 4096), (128, 14336, 4096),
                                   (40, 4104, 1032), (200, 2056, 520)])
def test_bulk_staged_final_sums_equal_l2_sums(shape, monkeypatch):
    # The skinny kernel's final sums, staged in shared memory by bulk copies
    # (SWIGLU_SK_BULK=1, the default) or read from L2 (0), add the same
    # partials in the same order: the bits must agree, and match the oracle.
    M, d_ff, d = shape
    h, wd, r = make(M, d_ff, d, seed=M + 1)
    outs = []
    monkeypatch.setenv("SWIGLU_SK_SPLIT", "0")     # the one-kernel form's final sums
    for bulk in ("1", "0"):
        monkeypatch.setenv("SWIGLU_SK_BULK", bulk)
        monkeypatch.setenv("SWIGLU_SK_CLUSTER", "0")
        y = swg.swiglu_down(h.to(DEV), wd.to(DEV), r.to(DEV), path="skinny")
        torch.cuda.synchronize()
        outs.append(y)
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    raw = inputs.raw_bits
    rows = np.unique(np.linspace(0, M - 1, min(M, 8)).astype(int))
    y64, _, s = oracle.down_proj(raw(h[rows].contiguous()), raw(wd), oracle.BF16,
                                 raw(r[rows].contiguous()))
    assert compare(to64(outs[0])[rows], y64, s, "bf16", d_ff)["ok"]
    swg.check_device_status()


def test_large_model_stream_k_with_bulk_final_sums():
    # d_ff = 29568 -> d = 8192 at M = 64: stream-K mode (its 64 groups do not
    # fit as 4-CTA clusters), 128-column groups, the sums added by the second
    # kernel; every column of rows from both halves of the call
    M, d_ff, d = 64, 29568, 8192
    p = swg.down_plan(M, d_ff, d)
    assert p["path"] == "skinny" and p["cluster"] == 1 and p["workspace"] > 0
    assert p["launches"] == 2
    check(M, d_ff, d, "auto", seed=91, rows=np.array([0, 17, 40, 63]))


@pytest.mark.parametrize("M", [1, 16, 48])
def test_back_to_back_calls_on_two_weight_sets(M):
    # d_ff = 14336 -> d = 4096, two kernels per call, whose sum kernel lets
    # the next call's GEMM start (and prefetch its weights) before the sums
    # are done: six calls back to back, alternating two weight matrices and
    # each with its own h and output, equal the same calls made one at a
    # time bit for bit, and match the oracle
    d_ff, d = 14336, 4096
    ws = [inputs.make_inputs(1, d_ff, d, "bf16", seed=300 + j)[1] for j in range(2)]
    wds = [w.to(DEV) for w in ws]
    hs = [inputs.make_inputs(M, d_ff, 8, "bf16", seed=310 + i, x_only=True)[0] for i in range(6)]
    r = inputs.make_inputs(M, d, 8, "bf16", seed=320, x_only=True)[0]
    hd, rd = [h.to(DEV) for h in hs], r.to(DEV)
    assert swg.down_plan(M, d_ff, d)["launches"] == 2
    alone = []
    for i in range(6):
        alone.append(swg.swiglu_down(hd[i], wds[i % 2], residual=rd))
        torch.cuda.synchronize()
    ys = [torch.full((M, d), float("nan"), dtype=torch.bfloat16, device=DEV) for _ in range(6)]
    for i in range(6):
        swg.swiglu_down(hd[i], wds[i % 2], residual=rd, out=ys[i])
    torch.cuda.synchronize()
    for i in range(6):
        assert torch.equal(alone[i].view(torch.int16), ys[i].view(torch.int16)), (M, i)
    raw = inputs.raw_bits
    rows = np.unique(np.linspace(0, M - 1, 3).astype(int))
    for i in (0, 5):
        y64, _, s = oracle.down_proj(raw(hs[i][rows].contiguous()), raw(ws[i % 2]), oracle.BF16,
                                     raw(r[rows].contiguous()))
        res = compare(to64(ys[i])[rows], y64, s, "bf16", d_ff)
        assert res["ok"], (M, i, res)
    swg.check_device_status()
