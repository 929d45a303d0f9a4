"""Pins of the down-projection oracle (y = h . W_down + r) and of the
two-operation MLP, against facts independent of the oracle's code."""
import numpy as np
import pytest
import torch

import oracle
from swiglu_mlp_projection_gb300 import inputs


def odt(dtype):
    return oracle.BF16 if dtype == "bf16" else oracle.F32


def ints(shape, seed, dtype):
    rng = np.random.default_rng(seed)
    return torch.from_numpy(rng.integers(-3, 4, shape).astype(np.float32)).to(
        inputs.TORCH_DTYPE[dtype])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", [(1, 1, 1), (2, 5, 3), (3, 17, 9), (4, 70, 33)])
def test_brute_force_small_integers(dtype, shape):
    M, K, N = shape
    h, wd, r = ints((M, K), 1, dtype), ints((K, N), 2, dtype), ints((M, N), 3, dtype)
    raw = inputs.raw_bits
    y64, yr, s = oracle.down_proj(raw(h), raw(wd), odt(dtype), raw(r))
    hi = h.double().numpy().astype(np.int64)
    wi = wd.double().numpy().astype(np.int64)
    ri = r.double().numpy().astype(np.int64)
    for i in range(M):
        for j in range(N):
            exact = sum(int(hi[i, k]) * int(wi[k, j]) for k in range(K)) + int(ri[i, j])
            sabs = sum(abs(int(hi[i, k]) * int(wi[k, j])) for k in range(K)) + abs(int(ri[i, j]))
            assert y64[i, j] == exact and s[i, j] == sabs
    y0, _, _ = oracle.down_proj(raw(h), raw(wd), odt(dtype))
    assert np.array_equal(y64, y0 + ri)           # the residual enters additively
    assert np.array_equal(yr, oracle.round_to_dtype(y64, odt(dtype)))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_one_hot_rows_and_scaling(dtype):
    K, N = 48, 40
    _, wd, _ = inputs.make_inputs(1, K, N, dtype, seed=4)
    h = torch.zeros(3, K, dtype=wd.dtype)
    for r_, k in enumerate([0, 7, K - 1]):
        h[r_, k] = 1.0
    raw = inputs.raw_bits
    y, _, _ = oracle.down_proj(raw(h), raw(wd), odt(dtype))
    w64 = wd.double().numpy()
    assert np.array_equal(y, w64[[0, 7, K - 1]])
    y2, _, _ = oracle.down_proj(raw(h * 2), raw(wd), odt(dtype))
    assert np.array_equal(y2, 2 * y)


@pytest.mark.parametrize("dtype,shape", [("bf16", (4, 2048, 512)), ("f32", (2, 512, 256))])
def test_matches_numpy_fp64(dtype, shape):
    M, K, N = shape
    h, wd, _ = inputs.make_inputs(M, K, N, dtype, seed=5)
    r = inputs.make_inputs(M, N, 8, dtype, seed=6, x_only=True)[0]
    raw = inputs.raw_bits
    y, _, s = oracle.down_proj(raw(h), raw(wd), odt(dtype), raw(r))
    ref = h.double().numpy() @ wd.double().numpy() + r.double().numpy()
    assert np.all(np.abs(y - ref) <= 2 * K * 2.0 ** -53 * s + 4 * np.spacing(np.abs(ref)))


def test_mlp_is_up_then_down_with_bf16_intermediate():
    M, d, d_ff = 3, 64, 96
    x, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=7)
    _, wd, _ = inputs.make_inputs(1, d_ff, d, "bf16", seed=8)
    raw = inputs.raw_bits
    y64, yr, s, h = oracle.mlp(raw(x), raw(wg), raw(wu), raw(wd), oracle.BF16, raw(x))
    _, h_ref, _ = oracle.swiglu_up(raw(x), raw(wg), raw(wu), oracle.BF16)
    assert np.array_equal(h, h_ref)
    # independent evaluation of the second step from the bf16 intermediate
    hv = oracle.to_f64(h, oracle.BF16)
    ref = hv @ wd.double().numpy() + x.double().numpy()
    assert np.allclose(y64, ref, rtol=1e-12, atol=1e-12)


def test_planted_mistakes_fail():
    M, K, N = 3, 9, 7
    h, wd, r = ints((M, K), 11, "f32"), ints((K, N), 12, "f32"), ints((M, N), 13, "f32")
    raw = inputs.raw_bits
    exact = h.double().numpy() @ wd.double().numpy() + r.double().numpy()
    good, _, _ = oracle.down_proj(raw(h), raw(wd), oracle.F32, raw(r))
    assert np.array_equal(good, exact)
    bad, _, _ = oracle.down_proj(raw(h), raw(wd), oracle.F32)            # residual dropped
    assert not np.array_equal(bad, exact)
    bad, _, _ = oracle.down_proj(raw(h[:, 1:]), raw(wd[1:]), oracle.F32, raw(r))   # a term dropped
    assert not np.array_equal(bad, exact)
