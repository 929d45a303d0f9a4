"""Pins of the oracle's weight packing (step a0, the SwiGLU paper's Kernel-2
interleave of gate and up columns, here in 64-column blocks): a worked
example, unpacking by reshape, zero padding, and the gate/up order."""
import numpy as np
import pytest

import oracle
from swiglu_mlp_projection_gb300 import inputs


def test_worked_example_f32():
    # d = 2, d_ff = 8: one 64-column block, mostly padding
    wg = np.arange(16, dtype=np.float32).reshape(2, 8) + 1
    wu = -np.arange(16, dtype=np.float32).reshape(2, 8) - 1
    p = oracle.pack(wg, wu, oracle.F32)
    assert p.shape == (2, 128)
    want = np.zeros((2, 128), np.float32)
    want[0, 0:8] = [1, 2, 3, 4, 5, 6, 7, 8]
    want[0, 64:72] = [-1, -2, -3, -4, -5, -6, -7, -8]
    want[1, 0:8] = [9, 10, 11, 12, 13, 14, 15, 16]
    want[1, 64:72] = [-9, -10, -11, -12, -13, -14, -15, -16]
    assert np.array_equal(p, want)


@pytest.mark.parametrize("dtype,shape", [("bf16", (5, 200)), ("f32", (3, 64)),
                                         ("bf16", (7, 1032)), ("f32", (1, 8))])
def test_unpack_by_reshape_recovers_the_weights(dtype, shape):
    d, d_ff = shape
    _, wg, wu = inputs.make_inputs(1, d, d_ff, dtype, seed=d_ff)
    od = oracle.BF16 if dtype == "bf16" else oracle.F32
    g, u = inputs.raw_bits(wg), inputs.raw_bits(wu)
    p = oracle.pack(g, u, od)
    tiles = -(-d_ff // 64)
    assert p.shape == (d, 128 * tiles)
    blocks = p.reshape(d, tiles, 2, 64)
    gate = blocks[:, :, 0, :].reshape(d, 64 * tiles)
    up = blocks[:, :, 1, :].reshape(d, 64 * tiles)
    assert np.array_equal(gate[:, :d_ff].view(np.uint8), g.view(np.uint8))
    assert np.array_equal(up[:, :d_ff].view(np.uint8), u.view(np.uint8))
    assert not gate[:, d_ff:].view(np.uint8).any()
    assert not up[:, d_ff:].view(np.uint8).any()


def test_swapping_gate_and_up_swaps_the_halves():
    _, wg, wu = inputs.make_inputs(1, 4, 136, "bf16", seed=3)
    g, u = inputs.raw_bits(wg), inputs.raw_bits(wu)
    a = oracle.pack(g, u, oracle.BF16).reshape(4, 3, 2, 64)
    b = oracle.pack(u, g, oracle.BF16).reshape(4, 3, 2, 64)
    assert np.array_equal(a[:, :, 0], b[:, :, 1]) and np.array_equal(a[:, :, 1], b[:, :, 0])
    assert not np.array_equal(a, b)
