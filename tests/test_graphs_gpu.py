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


@pytest.mark.parametrize("env,path,shape", [
    (("SWIGLU_SK_CLUSTER", "0"), "skinny", (4, 512, 1032)),    # stream-K: arrival counters
    (("SWIGLU_TILE_SK", "1"), "tc", (40, 1040, 520)),           # tile stream-K tail
    (None, "auto", (16, 4096, 14336))])                         # the decode shape
def test_graphs_with_arrival_counters(env, path, shape, monkeypatch):
    # Captured calls whose kernels count arrivals take their counters from a
    # region that stays zero between replays; two graphs of the same call,
    # replayed alternately, each keep their own.
    if env:
        monkeypatch.setenv(*env)
    M, d, d_ff = shape
    dev = torch.device("cuda", 0)
    x0, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=60)
    xs, wgs, wus = x0.to(dev), wg.to(dev), wu.to(dev)
    ha = torch.empty(M, d_ff, dtype=xs.dtype, device=dev)
    hb = torch.empty(M, d_ff, dtype=xs.dtype, device=dev)
    swg.swiglu_up(xs, wgs, wus, out=ha, path=path)          # outside capture first
    torch.cuda.synchronize()
    graphs = []
    for h in (ha, hb):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(2):
                swg.swiglu_up(xs, wgs, wus, out=h, path=path)
        graphs.append(g)
    for rep, seed in enumerate((61, 62, 63)):
        xn = inputs.make_inputs(M, d, d_ff, "bf16", seed=seed, x_only=True)[0]
        xs.copy_(xn.to(dev))
        for g in graphs:
            g.replay()
        torch.cuda.synchronize()
        for h in (ha, hb):
            if M * d_ff <= 2 ** 16:
                res = _check(h, xn, wg, wu, "bf16", d)
                assert res["ok"], (shape, rep, res)
        assert torch.equal(ha.view(torch.int16), hb.view(torch.int16))
    ref = swg.swiglu_up(xs, wgs, wus, path=path)
    torch.cuda.synchronize()
    assert torch.equal(ref.view(torch.int16), ha.view(torch.int16))
    swg.check_device_status()


def test_fp8_call_in_a_graph():
    M, d, d_ff = 8, 1040, 1032
    dev = torch.device("cuda", 0)
    x0, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=70)
    w8 = swg.quantize_weights_fp8(wg.to(dev), wu.to(dev))
    xs = x0.to(dev)
    h = torch.empty(M, d_ff, dtype=xs.dtype, device=dev)
    swg.swiglu_up_fp8(xs, w8, out=h)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        swg.swiglu_up_fp8(xs, w8, out=h)
    xn = inputs.make_inputs(M, d, d_ff, "bf16", seed=71, x_only=True)[0]
    xs.copy_(xn.to(dev))
    g.replay()
    torch.cuda.synchronize()
    raw = inputs.raw_bits
    h64, sens, _ = oracle.swiglu_up_fp8(raw(xn), raw(wg), raw(wu))
    res = compare(h.to("cpu", torch.float64).numpy(), h64, sens, "bf16", d)
    assert res["ok"], res


@pytest.mark.parametrize("M", [16, 64])
def test_down_projection_in_a_graph(M):
    # d_ff = 14336 -> d = 4096: stream-K, two kernel nodes (the partial sums
    # and their sum); replays with a new h match the oracle and the direct
    # call bit for bit
    d_ff, d = 14336, 4096
    dev = torch.device("cuda", 0)
    h0 = inputs.make_inputs(M, d_ff, 8, "bf16", seed=80, x_only=True)[0]
    _, wd, _ = inputs.make_inputs(1, d_ff, d, "bf16", seed=81)
    r = inputs.make_inputs(M, d, 8, "bf16", seed=82, x_only=True)[0]
    hs, wds, rs = h0.to(dev), wd.to(dev), r.to(dev)
    y = torch.empty(M, d, dtype=torch.bfloat16, device=dev)
    assert swg.down_plan(M, d_ff, d)["launches"] == 2
    swg.swiglu_down(hs, wds, residual=rs, out=y)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        swg.swiglu_down(hs, wds, residual=rs, out=y)
    hn = inputs.make_inputs(M, d_ff, 8, "bf16", seed=83, x_only=True)[0]
    hs.copy_(hn.to(dev))
    g.replay()
    torch.cuda.synchronize()
    raw = inputs.raw_bits
    rows = np.unique(np.linspace(0, M - 1, 4).astype(int))
    y64, _, s = oracle.down_proj(raw(hn[rows].contiguous()), raw(wd), oracle.BF16,
                                 raw(r[rows].contiguous()))
    res = compare(y.to("cpu", torch.float64).numpy()[rows], y64, s, "bf16", d_ff)
    assert res["ok"], (M, res)
    ref = swg.swiglu_down(hs, wds, residual=rs)
    torch.cuda.synchronize()
    assert torch.equal(ref.view(torch.int16), y.view(torch.int16))
    swg.check_device_status()


@pytest.mark.parametrize("M", [1, 16])
def test_down_chain_in_a_graph(M):
    # Three bf16 down projections (d_ff = 14336 -> d = 4096) captured back to
    # back, each on its own h and output: every call's sum kernel releases
    # the next call's GEMM early.  Replays equal the direct calls bit for bit
    # and match the oracle.
    d_ff, d = 14336, 4096
    dev = torch.device("cuda", 0)
    _, wd, _ = inputs.make_inputs(1, d_ff, d, "bf16", seed=191)
    wds = wd.to(dev)
    hs = [inputs.make_inputs(M, d_ff, 8, "bf16", seed=192 + i, x_only=True)[0].to(dev)
          for i in range(3)]
    r = inputs.make_inputs(M, d, 8, "bf16", seed=195, x_only=True)[0]
    rs = r.to(dev)
    ys = [torch.empty(M, d, dtype=torch.bfloat16, device=dev) for _ in range(3)]
    for i in range(3):
        swg.swiglu_down(hs[i], wds, residual=rs, out=ys[i])
        torch.cuda.synchronize()
    direct = [y.clone() for y in ys]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(3):
            swg.swiglu_down(hs[i], wds, residual=rs, out=ys[i])
    for y in ys:
        y.fill_(float("nan"))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for i in range(3):
        assert torch.equal(direct[i].view(torch.int16), ys[i].view(torch.int16)), i
    raw = inputs.raw_bits
    h_host = hs[1].cpu()
    rows = np.unique(np.linspace(0, M - 1, 4).astype(int))
    y64, _, s = oracle.down_proj(raw(h_host[rows].contiguous()), raw(wd), oracle.BF16,
                                 raw(r[rows].contiguous()))
    res = compare(ys[1].to("cpu", torch.float64).numpy()[rows], y64, s, "bf16", d_ff)
    assert res["ok"], (M, res)
    swg.check_device_status()


@pytest.mark.parametrize("M", [1, 16])
def test_fp8_down_chain_in_a_graph(M):
    # The FP8 down projection, d_ff = 14336 -> d = 4096: M = 1 runs three
    # kernels (quantize h, partial sums, their sum, which releases the next
    # kernel early), M = 16 two (quantize, 4-CTA clusters).  Three calls
    # captured back to back, each on its own h and output: replays match the
    # oracle and the direct calls bit for bit.
    d_ff, d = 14336, 4096
    dev = torch.device("cuda", 0)
    _, wd, _ = inputs.make_inputs(1, d_ff, d, "bf16", seed=91)
    w8 = swg.quantize_weight_fp8(wd.to(dev))
    hs = [inputs.make_inputs(M, d_ff, 8, "bf16", seed=92 + i, x_only=True)[0].to(dev)
          for i in range(3)]
    r = inputs.make_inputs(M, d, 8, "bf16", seed=95, x_only=True)[0]
    rs = r.to(dev)
    ys = [torch.empty(M, d, dtype=torch.bfloat16, device=dev) for _ in range(3)]
    for i in range(3):
        swg.swiglu_down_fp8(hs[i], w8, residual=rs, out=ys[i])
    torch.cuda.synchronize()
    direct = [y.clone() for y in ys]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(3):
            swg.swiglu_down_fp8(hs[i], w8, residual=rs, out=ys[i])
    for y in ys:
        y.fill_(float("nan"))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    raw = inputs.raw_bits
    for i in range(3):
        assert torch.equal(direct[i].view(torch.int16), ys[i].view(torch.int16)), i
    h_host = hs[2].cpu()
    rows = np.unique(np.linspace(0, M - 1, 4).astype(int))
    y64, sens = oracle.down_proj_fp8(raw(h_host[rows].contiguous()), raw(wd), raw(r[rows].contiguous()))
    res = compare(ys[2].to("cpu", torch.float64).numpy()[rows], y64, sens, "bf16", d_ff)
    assert res["ok"], (M, res)
    swg.check_device_status()


def _graph_node_types(graph):
    # node types of a captured CUDA graph, through the driver API
    import ctypes
    cu = ctypes.CDLL("libcuda.so.1")
    raw = graph.raw_cuda_graph()
    count = ctypes.c_size_t(0)
    assert cu.cuGraphGetNodes(ctypes.c_void_p(raw), None, ctypes.byref(count)) == 0
    nodes = (ctypes.c_void_p * count.value)()
    assert cu.cuGraphGetNodes(ctypes.c_void_p(raw), nodes, ctypes.byref(count)) == 0
    types = []
    for i in range(count.value):
        t = ctypes.c_int(-1)
        assert cu.cuGraphNodeGetType(ctypes.c_void_p(nodes[i]), ctypes.byref(t)) == 0
        types.append(t.value)
    return types


@pytest.mark.parametrize("op", ["up", "down"])
def test_captured_calls_hold_only_kernel_nodes(op, monkeypatch):
    # Calls captured into a graph take their workspace from a slice allocated
    # outside the graph, so the graph holds kernel nodes only (no allocation,
    # free or memset nodes between them, which would cut the programmatic
    # overlap of consecutive calls); three calls share their capture's slice
    # and replay to the direct calls' bits.
    monkeypatch.setenv("SWIGLU_SK_CLUSTER", "0")     # stream-K: partial sums and counters
    dev = torch.device("cuda", 0)
    if op == "up":
        M, K, N = 4, 1024, 4104
        x, wg, wu = inputs.make_inputs(M, K, N, "bf16", seed=60)
        xs = [inputs.make_inputs(M, K, 8, "bf16", seed=61 + i, x_only=True)[0].to(dev) for i in range(3)]
        wgd, wud = wg.to(dev), wu.to(dev)
        run = lambda i, out: swg.swiglu_up(xs[i], wgd, wud, out=out)
    else:
        M, K, N = 8, 4104, 1032
        _, wd, _ = inputs.make_inputs(1, K, N, "bf16", seed=64)
        xs = [inputs.make_inputs(M, K, 8, "bf16", seed=65 + i, x_only=True)[0].to(dev) for i in range(3)]
        r = inputs.make_inputs(M, N, 8, "bf16", seed=68, x_only=True)[0].to(dev)
        wdd = wd.to(dev)
        run = lambda i, out: swg.swiglu_down(xs[i], wdd, residual=r, out=out)
    assert swg.plan(M, K, N, "bf16", "auto", 0)["workspace"] > 0 if op == "up" else \
        swg.down_plan(M, K, N, "bf16", "auto", 0)["workspace"] > 0
    outs = [torch.empty(M, N, dtype=torch.bfloat16, device=dev) for _ in range(3)]
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(3):
            run(i, outs[i])
    torch.cuda.synchronize()
    direct = [o.clone() for o in outs]
    try:
        g = torch.cuda.CUDAGraph(keep_graph=True)
    except TypeError:
        pytest.skip("this PyTorch cannot keep the captured graph")
    with torch.cuda.graph(g, stream=s):
        for i in range(3):
            run(i, outs[i])
    types = _graph_node_types(g)
    kernel = 0   # CU_GRAPH_NODE_TYPE_KERNEL
    assert types and all(t == kernel for t in types), types
    for o in outs:
        o.fill_(float("nan"))
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for i in range(3):
        assert torch.equal(direct[i].view(torch.int16), outs[i].view(torch.int16)), i
    swg.check_device_status()


def test_forked_capture_gives_each_stream_its_own_workspace(monkeypatch):
    # A capture forked onto two streams runs their calls concurrently on
    # replay; each capturing stream takes its own workspace slice, so the
    # stream-K partial sums of the two never mix: replays equal the direct
    # calls bit for bit.
    monkeypatch.setenv("SWIGLU_SK_CLUSTER", "0")
    dev = torch.device("cuda", 0)
    M, K, N = 8, 1024, 4104
    _, wg, wu = inputs.make_inputs(1, K, N, "bf16", seed=70)
    wgd, wud = wg.to(dev), wu.to(dev)
    xs = [inputs.make_inputs(M, K, 8, "bf16", seed=71 + i, x_only=True)[0].to(dev) for i in range(6)]
    outs = [torch.empty(M, N, dtype=torch.bfloat16, device=dev) for _ in range(6)]
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    for s in (s1, s2):
        s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s1):
        for i in range(6):
            swg.swiglu_up(xs[i], wgd, wud, out=outs[i])
    torch.cuda.synchronize()
    direct = [o.clone() for o in outs]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s1):
        s2.wait_stream(s1)
        for i in range(3):
            swg.swiglu_up(xs[i], wgd, wud, out=outs[i])                 # on s1
            with torch.cuda.stream(s2):
                swg.swiglu_up(xs[3 + i], wgd, wud, out=outs[3 + i])     # on s2, concurrently
        s1.wait_stream(s2)
    for o in outs:
        o.fill_(float("nan"))
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for i in range(6):
        assert torch.equal(direct[i].view(torch.int16), outs[i].view(torch.int16)), i
    swg.check_device_status()
