"""Parity of the CUDA path with the CPU oracle, element by element.

Small and ragged shapes are compared on every output; the full-size
workloads on every output where the oracle finishes in seconds, otherwise on
every column of rows chosen so that each 128-row block (each CTA of each
row block of tiles) contributes rows from different epilogue warps.  Every row
of h is independent of the others, so a row is checked exactly as a full
comparison would check it, and every output tile of the call is reached.
"""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_projection_gb300 as swg
from swiglu_mlp_projection_gb300 import _lib, inputs, workload
from tests.parity import TOL, compare, tile_rows

pytestmark = pytest.mark.gpu

PATHS_BY_DTYPE = {"f32": ["simt"], "bf16": ["simt", "skinny", "tc"]}


def odt(dtype):
    return oracle.BF16 if dtype == "bf16" else oracle.F32


def to64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def gpu_run(x, wg, wu, path="auto", **kw):
    dev = torch.device("cuda", 0)
    h = swg.swiglu_up(x.to(dev), wg.to(dev), wu.to(dev), path=path, **kw)
    torch.cuda.synchronize()
    return h


def full_check(M, d, d_ff, dtype, path, seed=0):
    x, wg, wu = inputs.make_inputs(M, d, d_ff, dtype, seed=seed)
    raw = inputs.raw_bits
    h64, _, sens = oracle.swiglu_up(raw(x), raw(wg), raw(wu), odt(dtype))
    h = gpu_run(x, wg, wu, path)
    res = compare(to64(h), h64, sens, dtype, d)
    assert res["ok"], (M, d, d_ff, dtype, path, res)
    return res


RAGGED = [
    (1, 8, 8), (1, 24, 40), (2, 520, 264), (3, 1000, 1000), (5, 64, 2056),
    (16, 136, 520), (17, 256, 264), (33, 96, 1032), (4, 2048, 4104),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", RAGGED)
def test_ragged_shapes_all_paths(dtype, shape):
    for path in PATHS_BY_DTYPE[dtype] + ["auto"]:
        full_check(*shape, dtype, path, seed=sum(shape))


def test_f32_decode_step_full():
    # d=512, d_ff=2048, M=1, f32: every output
    cfg = workload.CONFIG_BY_NAME["f32_decode_d512"]
    for (M, d, d_ff) in cfg.shapes():
        full_check(M, d, d_ff, "f32", "auto")


@pytest.mark.parametrize("M", [1, 2, 4, 8, 16])
def test_bf16_decode_sweep_full(M):
    full_check(M, 4096, 14336, "bf16", "auto", seed=M)


@pytest.mark.parametrize("M", [1, 64, 512])
def test_bf16_small_model_full(M):
    full_check(M, 896, 4864, "bf16", "auto", seed=M)


def rows_check(M, d, d_ff, dtype, path, seed=0, rows=None):
    """Every column of the rows ``tile_rows`` picks (all rows if ``rows`` is
    "all"), against the oracle evaluated on exactly those rows of x."""
    x, wg, wu = inputs.make_inputs(M, d, d_ff, dtype, seed=seed)
    h = gpu_run(x, wg, wu, path)
    if rows is None:
        rows = tile_rows(M, seed=seed)
    elif isinstance(rows, str):
        rows = np.arange(M)
    raw = inputs.raw_bits
    h64, _, sens = oracle.swiglu_up(raw(x[rows].contiguous()), raw(wg), raw(wu), odt(dtype))
    hr = to64(h)[rows]
    res = compare(hr, h64, sens, dtype, d)
    assert res["ok"], (M, d, d_ff, dtype, path, res)
    assert bool(torch.isfinite(h).all())
    return res


def test_bf16_prefill_tile_rows():
    # M = 4096: 16 row blocks of CTA pairs; 2 rows of every 128-row half
    rows_check(4096, 4096, 14336, "bf16", "auto")


@pytest.mark.parametrize("M", [16, 2048, 8192])
def test_bf16_large_model_tile_rows(M):
    # d = 8192, d_ff = 29568: M = 16 on every output, M = 2048 and 8192 on
    # 2 rows of every 128-row block (32 / 128 blocks of 231 column tiles)
    rows_check(M, 8192, 29568, "bf16", "auto", seed=M, rows="all" if M <= 16 else None)


@pytest.mark.parametrize("M", [17, 64, 256])
def test_forced_paths_agree(M):
    # the three kernels serve the same call; each must match the oracle
    d, d_ff = 640, 1160
    x, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=40 + M)
    raw = inputs.raw_bits
    h64, _, sens = oracle.swiglu_up(raw(x), raw(wg), raw(wu), oracle.BF16)
    outs = {}
    for path in PATHS_BY_DTYPE["bf16"]:
        outs[path] = to64(gpu_run(x, wg, wu, path))
        assert compare(outs[path], h64, sens, "bf16", d)["ok"], path
    for a in outs:
        for b in outs:
            assert compare(outs[a], outs[b], sens, "bf16", d)["ok"], (a, b)


@pytest.mark.parametrize("cluster", ["0", "2", "4", "8"])
def test_skinny_cluster_and_stream_k_modes(cluster, monkeypatch):
    # the skinny kernel's two reductions: stream-K (global partials, last
    # arriver) and cluster mode (on-chip, through distributed shared memory)
    monkeypatch.setenv("SWIGLU_SK_CLUSTER", cluster)
    for (M, d, d_ff) in [(1, 896, 4864), (16, 896, 4864), (3, 520, 264), (40, 1024, 1032),
                         (130, 640, 520)]:
        full_check(M, d, d_ff, "bf16", "skinny", seed=M + int(cluster))


def test_cluster_mode_selection():
    # Small weights (<= 32 MB) run the skinny kernel in the largest clusters
    # that all fit at once, with no workspace: the small model's down
    # projection in 8-CTA clusters (7 groups of 128 columns), its up projection in 2-CTA
    # clusters (38 or 76 groups: too many for one wave of 4-CTA clusters).
    # The d = 4096 decode stays on stream-K.
    for M in (1, 16):
        p = swg.down_plan(M, 4864, 896, "bf16", "auto", 152)
        assert p["path"] == "skinny" and p["workspace"] == 0 and p["grid"] == 7 * 8
        assert p["cluster"] == 8
        assert swg.down_workspace_bytes(M, 4864, 896, "bf16", "auto") == 0
        # (from 16 rows in 64-column groups: 76 clusters of 2)
        p = swg.plan(M, 896, 4864, "bf16", "skinny", 152)
        assert p["cluster"] == 2 and p["grid"] == (76 if M >= 16 else 38) * 2
        assert p["workspace"] == 0
        assert swg.workspace_bytes(M, 896, 4864, "bf16", "skinny") == 0
    # AUTO: one row takes the SIMT path's cluster form (8 K slices, no workspace)
    p = swg.plan(1, 896, 4864, "bf16", "auto", 152)
    assert p["path"] == "simt" and p["cluster"] == 8 and p["workspace"] == 0
    assert swg.plan(16, 4096, 14336, "bf16", "auto", 152)["workspace"] > 0
    assert swg.workspace_bytes(16, 4096, 14336, "bf16", "auto") > 0


# --------------------------------------------------------------------------
# Invariants and edge cases
# --------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_deterministic_bits(dtype):
    x, wg, wu = inputs.make_inputs(7, 1024, 3072, dtype, seed=31)
    for path in PATHS_BY_DTYPE[dtype]:
        a = gpu_run(x, wg, wu, path)
        b = gpu_run(x, wg, wu, path)
        assert torch.equal(a.view(torch.int16 if dtype == "bf16" else torch.int32),
                           b.view(torch.int16 if dtype == "bf16" else torch.int32))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_one_hot_rows_and_zero_columns(dtype):
    d, d_ff = 256, 520
    _, wg, wu = inputs.make_inputs(1, d, d_ff, dtype, seed=32)
    wg, wu = wg.clone(), wu.clone()
    wu[:, 3] = 0
    wg[:, 7] = 0
    ks = [0, 5, 130, d - 1]
    x = torch.zeros(len(ks), d, dtype=wg.dtype)
    for r, k in enumerate(ks):
        x[r, k] = 1.0
    raw = inputs.raw_bits
    h64, _, sens = oracle.swiglu_up(raw(x), raw(wg), raw(wu), odt(dtype))
    for path in PATHS_BY_DTYPE[dtype]:
        h = to64(gpu_run(x, wg, wu, path))
        assert np.all(h[:, 3] == 0) and np.all(h[:, 7] == 0)
        res = compare(h, h64, sens, dtype, d)
        assert res["ok"], res
        # g and u are single weights here: only silu and the final rounding differ
        tight = 2.0 ** -7 if dtype == "bf16" else 4e-7
        nz = np.abs(h64) > 0
        assert np.all(np.abs(h[nz] - h64[nz]) <= tight * np.abs(h64[nz]))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_rows_independent(dtype):
    x, wg, wu = inputs.make_inputs(6, 512, 1024, dtype, seed=33)
    full = to64(gpu_run(x, wg, wu))
    raw = inputs.raw_bits
    h64, _, sens = oracle.swiglu_up(raw(x), raw(wg), raw(wu), odt(dtype))
    for i in range(6):
        hi = to64(gpu_run(x[i:i + 1].contiguous(), wg, wu))
        assert compare(hi, full[i:i + 1], sens[i:i + 1], dtype, 512)["ok"]


def test_empty_and_degenerate_sizes():
    dev = torch.device("cuda", 0)
    for dtype in ("f32", "bf16"):
        td = inputs.TORCH_DTYPE[dtype]
        # M = 0: no-op
        h = swg.swiglu_up(torch.empty(0, 64, dtype=td, device=dev),
                          torch.zeros(64, 32, dtype=td, device=dev),
                          torch.zeros(64, 32, dtype=td, device=dev))
        assert h.shape == (0, 32)
        # d = 0: empty sums, h = silu(0) * 0 = 0
        out = torch.full((3, 16), 7.0, dtype=td, device=dev)
        swg.swiglu_up(torch.empty(3, 0, dtype=td, device=dev),
                      torch.empty(0, 16, dtype=td, device=dev),
                      torch.empty(0, 16, dtype=td, device=dev), out=out)
        torch.cuda.synchronize()
        assert torch.all(out == 0)
        # d_ff = 0
        h = swg.swiglu_up(torch.ones(2, 8, dtype=td, device=dev),
                          torch.empty(8, 0, dtype=td, device=dev),
                          torch.empty(8, 0, dtype=td, device=dev))
        assert h.shape == (2, 0)


def test_large_magnitude_gate_is_finite():
    # g far below -88 makes e^-g overflow: silu must give -0, not NaN
    d, d_ff = 64, 64
    x = torch.full((2, d), 8.0, dtype=torch.bfloat16)
    wg = torch.full((d, d_ff), -1.0, dtype=torch.bfloat16)
    wg[:, 1::2] = 1.0
    wu = torch.ones(d, d_ff, dtype=torch.bfloat16)
    for path in PATHS_BY_DTYPE["bf16"]:
        h = to64(gpu_run(x, wg, wu, path))
        assert np.all(np.isfinite(h))
        assert np.all(h[:, 0::2] == 0)                 # silu(-512) * 512 -> 0
        assert np.all(h[:, 1::2] == 512.0 * 512.0)     # silu(512) * 512


def test_output_guard_band_untouched():
    dev = torch.device("cuda", 0)
    M, d, d_ff = 5, 256, 1032
    for dtype in ("f32", "bf16"):
        x, wg, wu = inputs.make_inputs(M, d, d_ff, dtype, seed=34)
        td = inputs.TORCH_DTYPE[dtype]
        pad = 4096
        buf = torch.full((M * d_ff + 2 * pad,), -3.0, dtype=td, device=dev)
        out = buf[pad:pad + M * d_ff].view(M, d_ff)
        for path in PATHS_BY_DTYPE[dtype]:
            swg.swiglu_up(x.to(dev), wg.to(dev), wu.to(dev), out=out, path=path)
            torch.cuda.synchronize()
            assert torch.all(buf[:pad] == -3.0) and torch.all(buf[-pad:] == -3.0)


@pytest.mark.parametrize("path", ["simt", "skinny"])
def test_caller_workspace_and_errors(path, monkeypatch):
    monkeypatch.setenv("SWIGLU_SK_CLUSTER", "0")     # the split-K workspace of stream-K mode
    monkeypatch.setenv("SWIGLU_SIMT_CLUSTER", "0")   # (the SIMT path's cluster form has none)
    dev = torch.device("cuda", 0)
    M, d, d_ff = 3, 1024, 2048
    x, wg, wu = (t.to(dev) for t in inputs.make_inputs(M, d, d_ff, "bf16", seed=35))
    need = swg.workspace_bytes(M, d, d_ff, "bf16", path)
    assert need > 0
    ws = torch.full((need + 256,), 0xAB, dtype=torch.uint8, device=dev)   # stale contents
    a = swg.swiglu_up(x, wg, wu, path=path, workspace=ws[:need])
    b = swg.swiglu_up(x, wg, wu, path=path)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    with pytest.raises(swg.SwiGLUError) as e:
        swg.swiglu_up(x, wg, wu, path=path, workspace=ws[:need - 256])
    assert e.value.status == 8
    with pytest.raises(swg.SwiGLUError) as e:
        swg.swiglu_up(x, wg, wu, path=path, workspace=ws[16:16 + need])
    assert e.value.status == 8
    # tc: M = 3 is one 128-row tile per 128 columns, 16 tiles < SMs: stream-K
    assert swg.workspace_bytes(M, d, d_ff, "bf16", "tc") > 0
    # whole waves (prefill shape, 1792 pair tiles) need none
    assert swg.workspace_bytes(4096, 4096, 14336, "bf16", "tc") == 0


def test_misaligned_pointer_rejected():
    dev = torch.device("cuda", 0)
    x, wg, wu = (t.to(dev) for t in inputs.make_inputs(2, 64, 64, "bf16", seed=36))
    big = torch.zeros(2 * 64 + 8, dtype=torch.bfloat16, device=dev)
    lib = _lib.load()
    st = lib.swiglu_up(x.data_ptr(), wg.data_ptr(), wu.data_ptr(), big.data_ptr() + 2,
                       2, 64, 64, _lib.BF16, None)
    assert st == 3


def test_non_default_stream_and_raw_abi():
    dev = torch.device("cuda", 0)
    M, d, d_ff = 4, 512, 1024
    x, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=37)
    xd, wgd, wud = x.to(dev), wg.to(dev), wu.to(dev)
    h = torch.empty(M, d_ff, dtype=torch.bfloat16, device=dev)
    s = torch.cuda.Stream()
    lib = _lib.load()
    with torch.cuda.stream(s):
        st = lib.swiglu_up(xd.data_ptr(), wgd.data_ptr(), wud.data_ptr(), h.data_ptr(),
                           M, d, d_ff, _lib.BF16, s.cuda_stream)
    assert st == 0
    s.synchronize()
    raw = inputs.raw_bits
    h64, _, sens = oracle.swiglu_up(raw(x), raw(wg), raw(wu), oracle.BF16)
    assert compare(to64(h), h64, sens, "bf16", d)["ok"]
    swg.check_device_status()


@pytest.mark.parametrize("dtype,shape", [("f32", (1, 512, 2048)), ("f32", (5, 1000, 1032)),
                                         ("bf16", (3, 520, 264)), ("f32", (17, 64, 2056))])
def test_simt_single_launch_matches_two_launches(dtype, shape, monkeypatch):
    # The SIMT path reduces its K slices either in a second kernel or, in one
    # launch, in the last CTA of each column block; both add the slices in
    # the same order, so the results are bit-identical.
    M, d, d_ff = shape
    monkeypatch.setenv("SWIGLU_SIMT_CLUSTER", "0")   # the split-K form's two reductions
    dev = torch.device("cuda", 0)
    x, wg, wu = (t.to(dev) for t in inputs.make_inputs(M, d, d_ff, dtype, seed=M + d))
    out = {}
    for fused in ("0", "1"):
        monkeypatch.setenv("SWIGLU_SIMT_FUSED", fused)
        assert swg.plan(M, d, d_ff, dtype, "simt", 152)["launches"] == (1 if fused == "1" else 2)
        out[fused] = swg.swiglu_up(x, wg, wu, path="simt")
        swg.swiglu_up(x, wg, wu, path="simt", out=out[fused])   # counters left at zero
    torch.cuda.synchronize()
    view = torch.int32 if dtype == "f32" else torch.int16
    assert torch.equal(out["0"].view(view), out["1"].view(view))
    full_check(M, d, d_ff, dtype, "simt", seed=M + d)


@pytest.mark.parametrize("M,d,d_ff", [(16, 4096, 14336), (32, 4096, 14336), (130, 640, 1032),
                                      (7, 1024, 4104)])
def test_skinny_bulk_staged_final_sums_equal_l2_sums(M, d, d_ff, monkeypatch):
    # the up projection's final sums by every route (the group's last CTA
    # with bulk-staged or L2 loads, or the second kernel that
    # SWIGLU_SK_SPLIT=1 adds): identical bits
    x, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=M + 2)
    outs = []
    monkeypatch.setenv("SWIGLU_SK_CLUSTER", "0")
    for split, bulk in (("0", "1"), ("0", "0"), ("1", "0")):
        monkeypatch.setenv("SWIGLU_SK_SPLIT", split)
        monkeypatch.setenv("SWIGLU_SK_BULK", bulk)
        assert swg.plan(M, d, d_ff, "bf16", "skinny", 0)["launches"] == (2 if split == "1" else 1)
        outs.append(gpu_run(x, wg, wu, "skinny"))
    for h in outs[1:]:
        assert torch.equal(outs[0].view(torch.int16), h.view(torch.int16))
    raw = inputs.raw_bits
    h64, _, sens = oracle.swiglu_up(raw(x), raw(wg), raw(wu), oracle.BF16)
    assert compare(to64(outs[0]), h64, sens, "bf16", d)["ok"]
