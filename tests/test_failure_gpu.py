"""Failure detection on the GPU without a fault: a bounded wait that runs out
reports SWIGLU_ERR_TIMEOUT to the host and leaves the context usable."""
import time

import pytest
import torch

import oracle
import swiglu_mlp_projection_gb300 as swg
from swiglu_mlp_projection_gb300 import _lib, inputs
from tests.parity import compare

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(cuda_lib):
    swg.check_device_status()                      # starts clean
    t0 = time.time()
    st = cuda_lib.swiglu_selftest_wait_timeout(50, None)
    assert st == 0
    with pytest.raises(swg.SwiGLUError) as e:
        swg.check_device_status()
    assert e.value.status == 6
    assert time.time() - t0 < 30
    swg.check_device_status()                      # the word was cleared
    # the context still runs the real kernels correctly
    dev = torch.device("cuda", 0)
    for M, path in [(4, "skinny"), (40, "tc")]:
        x, wg, wu = inputs.make_inputs(M, 256, 520, "bf16", seed=3)
        h = swg.swiglu_up(x.to(dev), wg.to(dev), wu.to(dev), path=path)
        torch.cuda.synchronize()
        raw = inputs.raw_bits
        h64, _, s = oracle.swiglu_up(raw(x), raw(wg), raw(wu), oracle.BF16)
        assert compare(h.cpu().double().numpy(), h64, s, "bf16", 256)["ok"]
    swg.check_device_status()


def test_selftest_rejects_bad_limits(cuda_lib):
    assert cuda_lib.swiglu_selftest_wait_timeout(0, None) == 1
    assert cuda_lib.swiglu_selftest_wait_timeout(20000, None) == 1


# ---------------------------------------------------------------------------
# Host-side fault injection: a workspace allocation that fails
# ---------------------------------------------------------------------------

def _check(h, x, wg, wu, d):
    raw = inputs.raw_bits
    h64, _, s = oracle.swiglu_up(raw(x), raw(wg), raw(wu),
                                 oracle.BF16 if x.dtype == torch.bfloat16 else oracle.F32)
    dt = "bf16" if x.dtype == torch.bfloat16 else "f32"
    assert compare(h.cpu().double().numpy(), h64, s, dt, d)["ok"]


@pytest.mark.parametrize("case", [("bf16", "auto", 16, 4096, 14336),   # skinny, stream-K
                                  ("f32", "auto", 5, 512, 2048),       # SIMT split-K (M > 4)
                                  ("bf16", "tc", 64, 4096, 1032)])     # tile, stream-K tail
def test_injected_workspace_oom_enqueues_nothing(case, monkeypatch):
    # SWIGLU_INJECT_OOM=1 makes every library-owned workspace allocation fail:
    # the call returns SWIGLU_ERR_OOM and h keeps its contents (nothing ran)
    dtype, path, M, d, d_ff = case
    dev = torch.device("cuda", 0)
    x, wg, wu = inputs.make_inputs(M, d, d_ff, dtype, seed=M)
    xd, wgd, wud = x.to(dev), wg.to(dev), wu.to(dev)
    assert swg.workspace_bytes(M, d, d_ff, dtype, path) > 0
    monkeypatch.setenv("SWIGLU_INJECT_OOM", "1")
    h = torch.full((M, d_ff), 5.0, dtype=xd.dtype, device=dev)
    with pytest.raises(swg.SwiGLUError) as e:
        swg.swiglu_up(xd, wgd, wud, out=h, path=path)
    assert e.value.status == 4 and "injected" in str(e.value)
    torch.cuda.synchronize()
    assert bool((h == 5.0).all())
    # a caller workspace is not affected by the hook
    ws = torch.empty(swg.workspace_bytes(M, d, d_ff, dtype, path), dtype=torch.uint8, device=dev)
    swg.swiglu_up(xd, wgd, wud, out=h, path=path, workspace=ws)
    torch.cuda.synchronize()
    _check(h, x, wg, wu, d)
    # and without the hook the library workspace works again
    monkeypatch.delenv("SWIGLU_INJECT_OOM")
    h2 = swg.swiglu_up(xd, wgd, wud, path=path)
    torch.cuda.synchronize()
    _check(h2, x, wg, wu, d)
    swg.check_device_status()


def test_injected_oom_spares_calls_without_workspace(monkeypatch):
    # the small model's up projection runs in 2-CTA clusters and needs no
    # workspace, so the hook does not touch it
    dev = torch.device("cuda", 0)
    M, d, d_ff = 1, 896, 4864
    assert swg.workspace_bytes(M, d, d_ff, "bf16", "auto") == 0
    monkeypatch.setenv("SWIGLU_INJECT_OOM", "1")
    x, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=9)
    h = swg.swiglu_up(x.to(dev), wg.to(dev), wu.to(dev))
    torch.cuda.synchronize()
    _check(h, x, wg, wu, d)


# ---------------------------------------------------------------------------
# The per-stream workspace cache gives its buffers back
# ---------------------------------------------------------------------------

def test_stream_workspaces_are_released():
    dev = torch.device("cuda", 0)
    M, d, d_ff = 16, 4096, 14336                   # skinny stream-K: uses the cache
    x, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=21)
    xd, wgd, wud = x.to(dev), wg.to(dev), wu.to(dev)
    swg.release_workspaces()
    assert swg.cached_workspace_bytes() == 0
    streams = [torch.cuda.Stream(dev) for _ in range(3)]
    outs = []
    for s in streams:
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            outs.append(swg.swiglu_up(xd, wgd, wud))
    torch.cuda.synchronize()
    three = swg.cached_workspace_bytes()
    assert three > 0
    # one stream's buffer, stream-ordered
    with torch.cuda.stream(streams[0]):
        swg.release_stream_workspace()
    assert 0 < swg.cached_workspace_bytes() < three
    swg.release_stream_workspace(streams[0])       # nothing left there: a no-op
    # a stream dropped without releasing: release_workspaces frees it as well
    del streams[1]
    swg.release_workspaces()
    assert swg.cached_workspace_bytes() == 0
    for h in outs:
        _check(h, x, wg, wu, d)
    # calls after the release allocate again and still match the oracle
    with torch.cuda.stream(streams[-1]):
        h = swg.swiglu_up(xd, wgd, wud)
    torch.cuda.synchronize()
    _check(h, x, wg, wu, d)
    assert swg.cached_workspace_bytes() > 0
    swg.release_workspaces()
    swg.check_device_status()
