"""The FP8 up projection (e4m3 weights per output column, e4m3 activations
per row, tcgen05 kind::f8f6f4, scaled f32 sums, SwiGLU epilogue): the
quantizers against the oracle bit for bit, and h against the oracle's FP8
definition (the fused definition on the dequantized operands) on every
tensor-core path and mode."""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_projection_gb300 as swg
from swiglu_mlp_projection_gb300 import _lib, inputs
from tests.parity import compare, tile_rows

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
RAW = inputs.raw_bits


def to64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def make(M, d, d_ff, seed):
    x, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=seed)
    return x, wg, wu


@pytest.mark.parametrize("shape", [(64, 136), (1040, 264), (16, 8)])
def test_weight_quantizer_bitwise(shape):
    d, d_ff = shape
    _, wg, wu = make(1, d, d_ff, seed=d)
    w = swg.quantize_weights_fp8(wg.to(DEV), wu.to(DEV))
    torch.cuda.synchronize()
    for got8, gots, ref in ((w.w8_gate, w.s_gate, wg), (w.w8_up, w.s_up, wu)):
        c, s = oracle.quantize_cols_e4m3(RAW(ref))
        assert np.array_equal(got8.cpu().numpy(), c)
        assert np.array_equal(gots.cpu().numpy().view(np.uint32), s.view(np.uint32))


def test_activation_quantizer_bitwise_through_the_workspace():
    # a caller workspace holds x's codes [M, d] at offset 0 and the row scales
    # from byte M d rounded up to 256
    M, d, d_ff = 5, 1040, 264
    x, wg, wu = make(M, d, d_ff, seed=3)
    xb = RAW(x)
    xb[4] = 0                                    # an all-zero row: scale 0
    xd = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(DEV)
    w = swg.quantize_weights_fp8(wg.to(DEV), wu.to(DEV))
    for path in ("skinny", "tc"):
        need = swg.fp8_workspace_bytes(M, d, d_ff, path)
        ws = torch.full((need,), 0xCD, dtype=torch.uint8, device=DEV)
        swg.swiglu_up_fp8(xd, w, path=path, workspace=ws)
        torch.cuda.synchronize()
        c, s = oracle.quantize_rows_e4m3(xb)
        off = -(-M * d // 256) * 256
        wsn = ws.cpu().numpy()
        assert np.array_equal(wsn[:M * d].reshape(M, d), c), path
        assert np.array_equal(wsn[off:off + 4 * M].view(np.float32), s), path


def check(M, d, d_ff, path, seed=0, **env):
    x, wg, wu = make(M, d, d_ff, seed)
    h64, sens, _ = oracle.swiglu_up_fp8(RAW(x), RAW(wg), RAW(wu))
    w = swg.quantize_weights_fp8(wg.to(DEV), wu.to(DEV))
    h = swg.swiglu_up_fp8(x.to(DEV), w, path=path)
    torch.cuda.synchronize()
    res = compare(to64(h), h64, sens, "bf16", d)
    assert res["ok"], (M, d, d_ff, path, res)
    return h


SHAPES = [(1, 64, 136), (3, 528, 264), (16, 1040, 520), (17, 256, 1032), (200, 528, 392),
          (300, 1040, 200)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("path", ["skinny", "tc", "auto"])
def test_fp8_matches_oracle(shape, path):
    if path == "skinny" and shape[0] > 256:
        pytest.skip("skinny path serves M <= 256")
    check(*shape, path, seed=sum(shape))


@pytest.mark.parametrize("env,path,shape", [
    (("SWIGLU_TILE_PAIR", "0"), "tc", (300, 528, 392)),
    (("SWIGLU_TILE_PAIR", "1"), "tc", (300, 528, 392)),
    (("SWIGLU_TILE_SK", "1"), "tc", (40, 1040, 520)),
    (("SWIGLU_SK_CLUSTER", "4"), "skinny", (7, 1040, 1032)),
    (("SWIGLU_SK_CLUSTER", "0"), "skinny", (7, 1040, 1032))])
def test_fp8_kernel_modes(env, path, shape, monkeypatch):
    monkeypatch.setenv(*env)
    check(*shape, path, seed=7)


def test_fp8_deterministic_and_errors():
    M, d, d_ff = 9, 1040, 520
    x, wg, wu = make(M, d, d_ff, seed=1)
    w = swg.quantize_weights_fp8(wg.to(DEV), wu.to(DEV))
    xd = x.to(DEV)
    a = swg.swiglu_up_fp8(xd, w)
    b = swg.swiglu_up_fp8(xd, w)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    with pytest.raises(swg.SwiGLUError) as e:
        swg.swiglu_up_fp8(xd, w, path="simt")
    assert e.value.status == 2
    lib = _lib.load()
    h = torch.empty(M, d_ff, dtype=torch.bfloat16, device=DEV)
    st = lib.swiglu_up_fp8(xd.data_ptr(), w.w8_gate.data_ptr(), w.w8_up.data_ptr(),
                           w.s_gate.data_ptr(), w.s_up.data_ptr(), h.data_ptr(), M, 1032,
                           d_ff, 0, None, 0, None)
    assert st == 3                                   # d not a multiple of 16
    st = lib.swiglu_up_fp8(xd.data_ptr(), w.w8_gate.data_ptr(), w.w8_up.data_ptr(),
                           w.s_gate.data_ptr() + 4, w.s_up.data_ptr(), h.data_ptr(), M, d,
                           d_ff, 0, None, 0, None)
    assert st == 3                                   # scales not 16-byte aligned
    swg.check_device_status()


@pytest.mark.parametrize("M,d,d_ff", [(1, 4096, 14336), (16, 4096, 14336), (4096, 4096, 14336),
                                       (16, 8192, 29568), (2048, 8192, 29568)])
def test_fp8_full_size_sampled(M, d, d_ff):
    # the decode, prefill and large-model shapes: the weight codes are checked
    # against the oracle on sampled columns, and h on those columns for
    # sampled rows
    x, wg, wu = make(M, d, d_ff, seed=M)
    w = swg.quantize_weights_fp8(wg.to(DEV), wu.to(DEV))
    h = swg.swiglu_up_fp8(x.to(DEV), w)
    torch.cuda.synchronize()
    cols = np.arange(3, d_ff, 211 if d_ff < 20000 else 421)
    rows = np.unique(np.linspace(0, M - 1, min(M, 6)).astype(int))
    gsub, usub = RAW(wg)[:, cols].copy(), RAW(wu)[:, cols].copy()
    cg, sg = oracle.quantize_cols_e4m3(gsub)
    cu, su = oracle.quantize_cols_e4m3(usub)
    assert np.array_equal(w.w8_gate[cols].cpu().numpy(), cg)
    assert np.array_equal(w.w8_up[cols].cpu().numpy(), cu)
    x8, sx = oracle.quantize_rows_e4m3(RAW(x)[rows].copy())
    xdq = oracle.dequant_rows_e4m3(x8, sx)
    gdq = np.ascontiguousarray(oracle.dequant_rows_e4m3(cg, sg).T)
    udq = np.ascontiguousarray(oracle.dequant_rows_e4m3(cu, su).T)
    h64, _, sens = oracle.swiglu_up(xdq, gdq, udq, oracle.F64, want_rounded=False)
    res = compare(to64(h)[np.ix_(rows, cols)], h64, sens, "bf16", d)
    assert res["ok"], (M, res)
    swg.check_device_status()


def test_fp8_prefill_tile_rows():
    # M = 4096, d = 4096, d_ff = 14336 on the FP8 tile kernel (CTA pairs):
    # every column of 2 rows of every 128-row block, against the oracle's
    # quantization and fp64 definition on the dequantized operands
    M, d, d_ff = 4096, 4096, 14336
    x, wg, wu = make(M, d, d_ff, seed=11)
    w = swg.quantize_weights_fp8(wg.to(DEV), wu.to(DEV))
    h = swg.swiglu_up_fp8(x.to(DEV), w)
    torch.cuda.synchronize()
    rows = tile_rows(M, seed=11)
    cg, sg = oracle.quantize_cols_e4m3(RAW(wg))
    cu, su = oracle.quantize_cols_e4m3(RAW(wu))
    assert np.array_equal(w.w8_gate.cpu().numpy(), cg)
    assert np.array_equal(w.w8_up.cpu().numpy(), cu)
    x8, sx = oracle.quantize_rows_e4m3(RAW(x)[rows].copy())
    xdq = oracle.dequant_rows_e4m3(x8, sx)
    gdq = np.ascontiguousarray(oracle.dequant_rows_e4m3(cg, sg).T)
    udq = np.ascontiguousarray(oracle.dequant_rows_e4m3(cu, su).T)
    h64, _, sens = oracle.swiglu_up(xdq, gdq, udq, oracle.F64, want_rounded=False)
    res = compare(to64(h)[rows], h64, sens, "bf16", d)
    assert res["ok"], res
    swg.check_device_status()


# ---------------------------------------------------------------------------
# The FP8 down projection
# ---------------------------------------------------------------------------

def down_check(M, d_ff, d, path, seed=0, rows=None):
    h = inputs.make_inputs(M, d_ff, 8, "bf16", seed=seed, x_only=True)[0]
    _, wd, _ = inputs.make_inputs(1, d_ff, d, "bf16", seed=seed + 1)
    r = inputs.make_inputs(M, d, 8, "bf16", seed=seed + 2, x_only=True)[0]
    w8 = swg.quantize_weight_fp8(wd.to(DEV))
    y = swg.swiglu_down_fp8(h.to(DEV), w8, residual=r.to(DEV), path=path)
    torch.cuda.synchronize()
    sel = slice(None) if rows is None else rows
    y64, sens = oracle.down_proj_fp8(RAW(h[sel].contiguous()), RAW(wd), RAW(r[sel].contiguous()))
    res = compare(to64(y)[sel], y64, sens, "bf16", d_ff)
    assert res["ok"], (M, d_ff, d, path, res)
    return w8, wd


@pytest.mark.parametrize("shape", [(1, 528, 136), (16, 1040, 264), (65, 528, 520),
                                   (300, 1040, 392)])
@pytest.mark.parametrize("path", ["skinny", "tc", "auto"])
def test_fp8_down_matches_oracle(shape, path):
    if path == "skinny" and shape[0] > 256:
        pytest.skip("skinny path serves M <= 256")
    w8, wd = down_check(*shape, path, seed=sum(shape))
    c, s = oracle.quantize_cols_e4m3(RAW(wd))
    assert np.array_equal(w8.w8.cpu().numpy(), c)
    assert np.array_equal(w8.s.cpu().numpy().view(np.uint32), s.view(np.uint32))


@pytest.mark.parametrize("env,path,shape", [
    (("SWIGLU_TILE_PAIR", "0"), "tc", (300, 528, 392)),
    (("SWIGLU_TILE_SK", "1"), "tc", (40, 1040, 520)),
    (("SWIGLU_SK_CLUSTER", "8"), "skinny", (3, 4864, 896)),
    (("SWIGLU_SK_CLUSTER", "0"), "skinny", (3, 4864, 896))])
def test_fp8_down_kernel_modes(env, path, shape, monkeypatch):
    monkeypatch.setenv(*env)
    down_check(*shape, path, seed=9)


def test_fp8_down_full_size_rows():
    # d = 4096, d_ff = 14336 at decode and prefill sizes: every column of the
    # chosen rows (at M = 4096, 2 rows of every 128-row block)
    for M, rows in ((16, np.arange(16)), (128, [0, 63, 127]), (4096, tile_rows(4096, seed=4))):
        down_check(M, 14336, 4096, "auto", seed=M, rows=rows)
    swg.check_device_status()


@pytest.mark.parametrize("M", [1, 16, 64, 256])
def test_fp8_down_final_sum_routes(M, monkeypatch):
    # FP8 down projection in stream-K mode at d = 4096: the second kernel's
    # sums and the one-kernel form's (bulk-staged or read from L2) agree bit
    # for bit and match the oracle
    h = inputs.make_inputs(M, 14336, 8, "bf16", seed=M, x_only=True)[0]
    _, wd, _ = inputs.make_inputs(1, 14336, 4096, "bf16", seed=M + 1)
    r = inputs.make_inputs(M, 4096, 8, "bf16", seed=M + 2, x_only=True)[0]
    w8 = swg.quantize_weight_fp8(wd.to(DEV))
    monkeypatch.setenv("SWIGLU_SK_CLUSTER", "0")
    outs = []
    for split, bulk in (("1", "1"), ("0", "1"), ("0", "0")):
        monkeypatch.setenv("SWIGLU_SK_SPLIT", split)
        monkeypatch.setenv("SWIGLU_SK_BULK", bulk)
        outs.append(swg.swiglu_down_fp8(h.to(DEV), w8, residual=r.to(DEV), path="skinny"))
        torch.cuda.synchronize()
    for y in outs[1:]:
        assert torch.equal(outs[0].view(torch.int16), y.view(torch.int16))
    rows = [0, M - 1]
    y64, sens = oracle.down_proj_fp8(RAW(h[rows].contiguous()), RAW(wd), RAW(r[rows].contiguous()))
    assert compare(to64(outs[0])[rows], y64, sens, "bf16", 14336)["ok"]


@pytest.mark.parametrize("M", [16, 64, 128, 256])
def test_fp8_down_cluster4(M):
    # FP8 down projection at d = 4096: 4-CTA clusters of 128-column groups
    # for M = 16 .. 64, stream-K with the second kernel's sums above; every
    # column of rows of every 128-row block
    down_check(M, 14336, 4096, "auto", seed=M + 9, rows=tile_rows(M, seed=M))


@pytest.mark.parametrize("op,mode,shape", [
    ("up", "0", (5, 1040, 1032)), ("up", "0", (16, 4096, 1040)), ("up", "2", (3, 1040, 264)),
    ("down", "0", (7, 1040, 520)), ("down", "4", (33, 14336, 4096)), ("down", "4", (16, 1040, 264))])
def test_fp8_two_k_blocks_per_unit(op, mode, shape, monkeypatch):
    # Units of two 64-deep k blocks (256 code bytes of every weight row), the
    # 4-CTA cluster form's default and SWIGLU_SK_KB=2 elsewhere, in stream-K
    # (mode 0) and cluster modes.  K = 1040 codes (520 pairs, 9 blocks) leaves
    # the last unit's second block past K, which the kernel skips.
    monkeypatch.setenv("SWIGLU_SK_KB", "2")
    monkeypatch.setenv("SWIGLU_SK_CLUSTER", mode)
    if op == "up":
        check(*shape, "skinny", seed=sum(shape))
    else:
        down_check(*shape, "skinny", seed=sum(shape))
    swg.check_device_status()


@pytest.mark.parametrize("shape", [(7, 1040, 520), (12, 14336, 4096)])
def test_fp8_down_one_k_block_per_unit(shape, monkeypatch):
    # The FP8 down projection's stream-K units default to two k blocks above
    # 32 MB of weights; one block per unit (SWIGLU_SK_KB=1) stays a valid
    # form, and is the default for small weights and above 64 rows
    monkeypatch.setenv("SWIGLU_SK_KB", "1")
    monkeypatch.setenv("SWIGLU_SK_CLUSTER", "0")
    down_check(*shape, "skinny", seed=sum(shape), rows=[0, shape[0] - 1])
    swg.check_device_status()
