"""The cluster form of the SIMT path (one row, weights <= 32 MB, d <= 2048):
the K slices of a column block meet in distributed shared memory instead of
a workspace.  Parity with the oracle on every output, for f32 and bf16, ragged
shapes, packed weights, graph capture and run-to-run determinism."""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_projection_gb300 as swg
from swiglu_mlp_projection_gb300 import inputs
from tests.parity import compare

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
RAW = inputs.raw_bits

SHAPES = [(8, 8), (24, 40), (64, 264), (512, 2048), (520, 264), (896, 4864), (1000, 1032),
          (2048, 1032), (1024, 4104)]


def oracle_h(x, wg, wu, dtype):
    return oracle.swiglu_up(RAW(x), RAW(wg), RAW(wu), oracle.BF16 if dtype == "bf16" else oracle.F32)


def run(x, wg, wu, path="simt"):
    h = swg.swiglu_up(x.to(DEV), wg.to(DEV), wu.to(DEV), path=path)
    torch.cuda.synchronize()
    return h


CASES = [("bf16", s) for s in SHAPES] + \
    [("f32", s) for s in SHAPES if 2 * s[0] * s[1] * 4 <= 32 << 20]   # f32: <= 32 MB of weights


@pytest.mark.parametrize("seed", [0, 1])
@pytest.mark.parametrize("dtype,shape", CASES)
def test_cluster_form_matches_oracle(dtype, seed, shape):
    M = 1
    d, d_ff = shape
    assert swg.plan(M, d, d_ff, dtype, "simt")["cluster"] == 8
    # on the device: 8 slices, or fewer where 8-CTA clusters would not all fit
    assert swg.plan(M, d, d_ff, dtype, "simt", 0)["cluster"] in (4, 5, 6, 7, 8)
    x, wg, wu = inputs.make_inputs(M, d, d_ff, dtype, seed=seed * 7 + d)
    h = run(x, wg, wu)
    h64, _, s = oracle_h(x, wg, wu, dtype)
    res = compare(h.cpu().double().numpy(), h64, s, dtype, d)
    assert res["ok"], (dtype, M, shape, res)


@pytest.mark.parametrize("ks", [4, 5, 6, 7, 8])
@pytest.mark.parametrize("dtype,shape", [("f32", (512, 2048)), ("bf16", (512, 2048)),
                                         ("bf16", (520, 264)), ("bf16", (896, 4864)),
                                         ("f32", (24, 40))])
def test_every_cluster_size_matches_oracle(dtype, shape, ks, monkeypatch):
    # SWIGLU_SIMT_CLUSTER=S forces S K slices per cluster where a slice holds
    # at most 4 rows of W per thread (8 slices: 8 rows)
    d, d_ff = shape
    monkeypatch.setenv("SWIGLU_SIMT_CLUSTER", str(ks))
    kn = -(-d // ks)
    if not (kn <= 256 if ks == 8 else kn <= 128):
        assert swg.plan(1, d, d_ff, dtype, "simt", 0)["cluster"] == 1
        return
    p = swg.plan(1, d, d_ff, dtype, "simt", 0)
    assert p["cluster"] == p["slices"] == ks and p["workspace"] == 0
    x, wg, wu = inputs.make_inputs(1, d, d_ff, dtype, seed=ks + d)
    h = run(x, wg, wu)
    h64, _, s = oracle_h(x, wg, wu, dtype)
    res = compare(h.cpu().double().numpy(), h64, s, dtype, d)
    assert res["ok"], (dtype, shape, ks, res)
    h2 = run(x, wg, wu)
    view = torch.int16 if dtype == "bf16" else torch.int32
    assert torch.equal(h.view(view), h2.view(view))      # same bits every run


def test_small_model_clusters_fit_at_once():
    # the d = 896 model's 76 column blocks: the device plan takes the largest
    # cluster whose 76 clusters all run at once (on GB300, 4 CTAs per SM hold
    # 74 clusters of 8 but 81 of 7)
    p = swg.plan(1, 896, 4864, "bf16", "auto", 0)
    assert p["path"] == "simt" and p["cluster"] in (7, 8)
    assert p["grid"] == 76 * p["cluster"] and p["workspace"] == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_cluster_form_equals_split_k_kernel_within_tolerance(dtype, monkeypatch):
    # both forms of the SIMT path serve the same call; each matches the oracle
    M, d, d_ff = 1, 896, 2048
    x, wg, wu = inputs.make_inputs(M, d, d_ff, dtype, seed=5)
    h64, _, s = oracle_h(x, wg, wu, dtype)
    a = run(x, wg, wu)
    monkeypatch.setenv("SWIGLU_SIMT_CLUSTER", "0")
    assert swg.plan(M, d, d_ff, dtype, "simt")["cluster"] == 1
    b = run(x, wg, wu)
    for h in (a, b):
        assert compare(h.cpu().double().numpy(), h64, s, dtype, d)["ok"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_cluster_form_packed_weights_and_determinism(dtype):
    M, d, d_ff = 1, 520, 1000
    x, wg, wu = inputs.make_inputs(M, d, d_ff, dtype, seed=11)
    xd = x.to(DEV)
    wp = swg.pack_weights(wg.to(DEV), wu.to(DEV))
    hp = swg.swiglu_up_packed(xd, wp, d_ff, path="simt")
    h1 = swg.swiglu_up(xd, wg.to(DEV), wu.to(DEV), path="simt")
    h2 = swg.swiglu_up(xd, wg.to(DEV), wu.to(DEV), path="simt")
    torch.cuda.synchronize()
    view = torch.int16 if dtype == "bf16" else torch.int32
    assert torch.equal(h1.view(view), h2.view(view))      # same bits every run
    assert torch.equal(hp.view(view), h1.view(view))      # packed: same arithmetic
    h64, _, s = oracle_h(x, wg, wu, dtype)
    assert compare(h1.cpu().double().numpy(), h64, s, dtype, d)["ok"]


def test_cluster_form_in_a_cuda_graph():
    # no workspace: the captured call is one kernel node; replays match the oracle
    M, d, d_ff = 1, 512, 2048
    x, wg, wu = inputs.make_inputs(M, d, d_ff, "f32", seed=3)
    xd, wgd, wud = x.to(DEV), wg.to(DEV), wu.to(DEV)
    h = torch.empty(M, d_ff, device=DEV)
    s = torch.cuda.Stream(DEV)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        swg.swiglu_up(xd, wgd, wud, out=h)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        swg.swiglu_up(xd, wgd, wud, out=h)
    h.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    h64, _, sens = oracle_h(x, wg, wu, "f32")
    assert compare(h.cpu().double().numpy(), h64, sens, "f32", d)["ok"]
    swg.check_device_status()


def test_guard_band_around_h():
    # outputs past the last column or row are never written
    M, d, d_ff = 1, 896, 520
    x, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=8)
    buf = torch.full(((M + 2) * d_ff,), 7.0, dtype=torch.bfloat16, device=DEV)
    assert swg.plan(M, d, d_ff, "bf16", "simt")["cluster"] == 8
    h = buf[: M * d_ff].view(M, d_ff)
    swg.swiglu_up(x.to(DEV), wg.to(DEV), wu.to(DEV), out=h, path="simt")
    torch.cuda.synchronize()
    assert bool((buf[M * d_ff:] == 7.0).all())
    h64, _, s = oracle_h(x, wg, wu, "bf16")
    assert compare(h.cpu().double().numpy(), h64, s, "bf16", d)["ok"]


def test_more_rows_take_the_split_k_kernel():
    # M > 1 is served by the split-K kernel of the SIMT path
    assert swg.plan(2, 512, 2048, "f32", "simt")["cluster"] == 1
    x, wg, wu = inputs.make_inputs(3, 512, 2048, "f32", seed=4)
    h = run(x, wg, wu)
    h64, _, s = oracle_h(x, wg, wu, "f32")
    assert compare(h.cpu().double().numpy(), h64, s, "f32", 512)["ok"]
