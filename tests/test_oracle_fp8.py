"""Pins of the oracle's FP8 (e4m3) arithmetic: the codec against torch's
float8_e4m3fn and worked examples, the per-row / per-column quantizers
against their defining properties, and the FP8 path's definition against the
bf16 oracle on inputs that e4m3 represents exactly."""
import numpy as np
import pytest
import torch

import oracle
from swiglu_mlp_projection_gb300 import inputs


def test_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan) and nan.sum() == 2     # 0x7F, 0xFF
    assert np.array_equal(ours[~nan], ref[~nan])
    assert ours[0x7E] == 448.0 and ours[0x01] == 2.0 ** -9 and ours[0x08] == 2.0 ** -6


def test_encode_matches_torch_in_range():
    rng = np.random.default_rng(0)
    parts = [rng.uniform(-448, 448, 20000), rng.normal(0, 1, 20000),
             rng.uniform(-2 ** -6, 2 ** -6, 5000),                        # subnormal range
             oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8)),       # exact codes
             (oracle.e4m3_decode(np.arange(0, 0x7D, dtype=np.uint8))       # midpoints: ties
              + oracle.e4m3_decode(np.arange(1, 0x7E, dtype=np.uint8))) / 2]
    v = np.concatenate(parts).astype(np.float32)
    v = np.concatenate([v, -v])
    ours = oracle.e4m3_encode(v)
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_encode_worked_examples_and_saturation():
    v = np.array([1.0, 448.0, 2 ** -9, 2 ** -6, 1.0625, 1.1875, 464.0, 470.0, 1e30, -500.0,
                  2 ** -10, 1.5 * 2 ** -10, 0.0, -0.0], np.float32)
    want = [0x38, 0x7E, 0x01, 0x08, 0x38, 0x3A, 0x7E, 0x7E, 0x7E, 0xFE, 0x00, 0x01, 0x00, 0x80]
    assert oracle.e4m3_encode(v).tolist() == want


def test_quantize_rows_properties():
    x, _, _ = inputs.make_inputs(6, 1000, 8, "bf16", seed=4)
    xb = inputs.raw_bits(x)
    xb[5] = 0                                            # an all-zero row
    codes, scales = oracle.quantize_rows_e4m3(xb)
    xf = x.to(torch.float64).numpy()
    xf[5] = 0
    amax = np.abs(xf).max(axis=1)
    assert np.array_equal(scales[:5], (amax[:5].astype(np.float32) / np.float32(448)))
    assert scales[5] == 0 and not codes[5].any()
    deq = oracle.dequant_rows_e4m3(codes, scales)
    for r in range(5):
        k = int(np.argmax(np.abs(xf[r])))
        assert codes[r, k] & 0x7F == 0x7E                # the row's amax becomes +-448
        big = np.abs(xf[r]) >= 2 ** -6 * scales[r]       # normal e4m3 range
        rel = np.abs(deq[r] - xf[r]) / np.abs(xf[r])
        assert rel[big].max() <= 2 ** -4 * (1 + 1e-6)    # half an ulp of a 3-bit mantissa
        if (~big).any():                                 # subnormal range: half of 2^-9
            assert np.abs(deq[r] - xf[r])[~big].max() <= 2 ** -10 * scales[r] * (1 + 1e-6)


def test_quantize_cols_is_rows_of_the_transpose():
    _, w, _ = inputs.make_inputs(1, 264, 136, "bf16", seed=5)
    wb = inputs.raw_bits(w)
    c1, s1 = oracle.quantize_cols_e4m3(wb)
    c2, s2 = oracle.quantize_rows_e4m3(np.ascontiguousarray(wb.T))
    assert np.array_equal(c1, c2) and np.array_equal(s1, s2)


def test_fp8_definition_equals_bf16_oracle_on_exact_inputs():
    # Values e4m3 holds exactly, with every row's (column's) amax 448, so the
    # scales are 1 and quantization changes nothing: the FP8 path's result
    # must then be the bf16 definition's, to the last bit.
    rng = np.random.default_rng(1)
    grid = np.array([0, 1, 2, 3, 4, 6, 8, 12, 16, 24, 448], np.float32)
    M, d, d_ff = 3, 48, 24
    x = rng.choice(grid, (M, d)) * rng.choice([-1, 1], (M, d))
    wg = rng.choice(grid, (d, d_ff)) * rng.choice([-1, 1], (d, d_ff))
    wu = rng.choice(grid, (d, d_ff)) * rng.choice([-1, 1], (d, d_ff))
    x[:, 0] = 448
    wg[0, :] = 448
    wu[0, :] = 448
    to_bits = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    xb, gb, ub = to_bits(x), to_bits(wg), to_bits(wu)
    h8, s8, q = oracle.swiglu_up_fp8(xb, gb, ub)
    assert np.all(q["sx"] == 1) and np.all(q["sg"] == 1) and np.all(q["su"] == 1)
    h64, _, s = oracle.swiglu_up(xb, gb, ub, oracle.BF16)
    assert np.array_equal(h8, h64) and np.array_equal(s8, s)


def test_fp8_down_definition_equals_bf16_oracle_on_exact_inputs():
    # the down projection's FP8 definition, on inputs e4m3 holds exactly with
    # scales 1, is the bf16 down projection to the last bit
    rng = np.random.default_rng(2)
    grid = np.array([0, 1, 2, 3, 4, 6, 8, 12, 16, 24, 448], np.float32)
    M, d_ff, d = 3, 32, 16
    h = rng.choice(grid, (M, d_ff)) * rng.choice([-1, 1], (M, d_ff))
    wd = rng.choice(grid, (d_ff, d)) * rng.choice([-1, 1], (d_ff, d))
    r = rng.choice(grid, (M, d)) * rng.choice([-1, 1], (M, d))
    h[:, 0] = 448
    wd[0, :] = 448
    to_bits = lambda a: torch.from_numpy(a.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    hb, wb, rb = to_bits(h), to_bits(wd), to_bits(r)
    y8, s8 = oracle.down_proj_fp8(hb, wb, rb)
    y64, _, s = oracle.down_proj(hb, wb, oracle.BF16, rb)
    assert np.array_equal(y8, y64) and np.array_equal(s8, s)
