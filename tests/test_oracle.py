"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks the oracle against something independent of its own code:
exact integer arithmetic, high-precision decimal evaluation, a different
closed form of SiLU, algebraic identities of the method, numpy's fp64 matmul,
and torch's bf16 rounding.  The planted-mistake tests at the end show that a
plausible slip (swapped operands, a dropped term, a transposed weight, SiLU on
the wrong product) fails at least one pin.
"""
import decimal
import math

import numpy as np
import pytest
import torch

import oracle
from swiglu_mlp_projection_gb300 import inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

decimal.getcontext().prec = 60


def dec_silu(z):
    """SiLU(z) = z / (1 + e^-z) in 60-digit decimal arithmetic."""
    z = decimal.Decimal(z)
    return z / (1 + (-z).exp())


def tanh_silu(z):
    """SiLU through sigma(z) = (1 + tanh(z/2)) / 2 (a different closed form)."""
    z = np.asarray(z, np.float64)
    return z * (1.0 + np.tanh(z / 2.0)) / 2.0


def as_raw(t):
    return inputs.raw_bits(t)


def odt(dtype):
    return oracle.BF16 if dtype == "bf16" else oracle.F32


# --------------------------------------------------------------------------
# SiLU
# --------------------------------------------------------------------------

def test_silu_closed_forms():
    assert oracle.silu64(0.0) == 0.0
    for z in [1e-300, 1e-8, 0.1, 0.5, 1.0, 2.4, 3.0, 7.5, 20.0, 50.0, 700.0]:
        # sigma(z) + sigma(-z) = 1  =>  silu(z) - silu(-z) = z
        diff = oracle.silu64(z) - oracle.silu64(-z)
        assert abs(diff - z) <= 4e-16 * abs(z), z
    # silu(z) -> z for large z, -> 0 (never NaN) for very negative z
    assert oracle.silu64(800.0) == 800.0
    v = oracle.silu64(-800.0)
    assert v == 0.0 and not math.isnan(v)
    assert oracle.silu64(-745.0) <= 0.0


def test_silu_high_precision_values():
    zs = [-30.0, -10.0, -3.3, -1.0, -0.25, 1e-5, 0.3, 1.0, 2.5, 6.0, 17.0, 40.0]
    for z in zs:
        ref = float(dec_silu(z))
        got = oracle.silu64(z)
        assert abs(got - ref) <= 4 * np.spacing(abs(ref)), (z, got, ref)


def test_silu_matches_tanh_form():
    z = np.linspace(-40, 40, 4001)
    got = np.array([oracle.silu64(v) for v in z])
    ref = tanh_silu(z)
    # the two closed forms agree to a few ulp of the larger of |z|, |silu|
    assert np.all(np.abs(got - ref) <= 8 * np.spacing(np.maximum(np.abs(z), 1e-300)) + 1e-300)


# --------------------------------------------------------------------------
# Number formats
# --------------------------------------------------------------------------

def test_bf16_decode_known_patterns():
    assert oracle.bf16_to_f64(0x3F80) == 1.0
    assert oracle.bf16_to_f64(0xC000) == -2.0
    assert oracle.bf16_to_f64(0x0001) == 2.0 ** -133
    assert oracle.bf16_to_f64(0x7F7F) == (2 - 2 ** -7) * 2.0 ** 127
    assert math.isinf(oracle.bf16_to_f64(0x7F80))
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_to_f64(bits)
    both_nan = np.isnan(t) & np.isnan(got)
    assert np.all((got == t) | both_nan)
    # the vectorised widening helper agrees with the C decoder
    v = oracle.to_f64(bits, oracle.BF16)
    assert np.all((v == got) | both_nan)


def test_bf16_rounding_matches_torch_on_f32_values():
    rng = np.random.default_rng(1)
    e = rng.integers(-140, 128, 20000)
    m = rng.random(20000) + 1.0
    v = (m * np.exp2(e.astype(np.float64))).astype(np.float32)
    v[::3] *= -1
    # exact ties between bf16 neighbours and values one f32 ulp from them
    base = rng.integers(0, 0x7F00, 3000).astype(np.uint32) << 16
    ties = (base | 0x8000).view(np.float32)
    near = np.concatenate([(base | 0x7FFF).view(np.float32), (base | 0x8001).view(np.float32)])
    v = np.concatenate([v, ties, near, np.float32([0.0, -0.0, 1.0, 3.0e38, -3.4e38])])
    v = v[np.isfinite(v)]
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round_to_dtype(v.astype(np.float64), oracle.BF16)
    assert np.array_equal(got, ref)


def test_bf16_rounding_is_single_rounding_from_fp64():
    # 1 + 2^-8 is a tie -> even (1.0); a hair above rounds up.  Rounding via
    # f32 first would turn the second case into a tie and round it down.
    assert oracle.round_to_dtype(np.array([1 + 2 ** -8]), oracle.BF16)[0] == 0x3F80
    assert oracle.round_to_dtype(np.array([1 + 2 ** -8 + 2 ** -40]), oracle.BF16)[0] == 0x3F81
    assert oracle.round_to_dtype(np.array([1 + 3 * 2 ** -8]), oracle.BF16)[0] == 0x3F82
    # subnormal spacing 2^-133; 2^-134 is a tie between 0 and 2^-133
    assert oracle.round_to_dtype(np.array([2.0 ** -133]), oracle.BF16)[0] == 0x0001
    assert oracle.round_to_dtype(np.array([2.0 ** -134]), oracle.BF16)[0] == 0x0000
    assert oracle.round_to_dtype(np.array([1.5 * 2.0 ** -134]), oracle.BF16)[0] == 0x0001
    # largest finite and overflow at the rounding boundary
    mx = (2 - 2 ** -7) * 2.0 ** 127
    mid = (2 - 2 ** -8) * 2.0 ** 127
    assert oracle.round_to_dtype(np.array([mx]), oracle.BF16)[0] == 0x7F7F
    assert oracle.round_to_dtype(np.array([np.nextafter(mid, 0)]), oracle.BF16)[0] == 0x7F7F
    assert oracle.round_to_dtype(np.array([mid]), oracle.BF16)[0] == 0x7F80
    assert oracle.round_to_dtype(np.array([-mid]), oracle.BF16)[0] == 0xFF80


def test_f32_rounding_matches_numpy():
    rng = np.random.default_rng(2)
    v = rng.standard_normal(10000) * np.exp2(rng.integers(-130, 120, 10000))
    got = oracle.round_to_dtype(v, oracle.F32)
    assert np.array_equal(got.view(np.uint32), v.astype(np.float32).view(np.uint32))


# --------------------------------------------------------------------------
# The fused definition
# --------------------------------------------------------------------------

SMALL_SHAPES = [(1, 1, 1), (2, 3, 5), (3, 9, 7), (1, 17, 9), (17, 33, 9), (5, 64, 130)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SMALL_SHAPES)
def test_brute_force_small_integers(dtype, shape):
    M, d, d_ff = shape
    x, wg, wu = inputs.small_int_inputs(M, d, d_ff, dtype, seed=sum(shape))
    xi = x.to(torch.float64).numpy().astype(np.int64)
    wgi = wg.to(torch.float64).numpy().astype(np.int64)
    wui = wu.to(torch.float64).numpy().astype(np.int64)
    h64, hr, sens = oracle.swiglu_up(as_raw(x), as_raw(wg), as_raw(wu), odt(dtype))
    for i in range(M):
        for j in range(d_ff):
            g = int(sum(int(xi[i, k]) * int(wgi[k, j]) for k in range(d)))
            u = int(sum(int(xi[i, k]) * int(wui[k, j]) for k in range(d)))
            G = int(sum(abs(int(xi[i, k]) * int(wgi[k, j])) for k in range(d)))
            U = int(sum(abs(int(xi[i, k]) * int(wui[k, j])) for k in range(d)))
            sg = dec_silu(g)
            ref = float(sg * u)
            assert abs(h64[i, j] - ref) <= 4 * np.spacing(abs(ref)) + 1e-300, (i, j, g, u)
            s_ref = float(decimal.Decimal("1.1") * G * abs(u) + abs(sg) * U)
            assert abs(sens[i, j] - s_ref) <= 1e-14 * s_ref + 1e-300
            assert sens[i, j] >= abs(h64[i, j])
    # the rounded output is the single RNE rounding of h64
    assert np.array_equal(hr, oracle.round_to_dtype(h64, odt(dtype)))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_one_hot_rows_select_weight_rows(dtype):
    d, d_ff = 40, 72
    _, wg, wu = inputs.make_inputs(1, d, d_ff, dtype, seed=3)
    ks = [0, 1, 17, d - 1]
    x = torch.zeros(len(ks), d, dtype=wg.dtype)
    for r, k in enumerate(ks):
        x[r, k] = 1.0
    h64, _, _ = oracle.swiglu_up(as_raw(x), as_raw(wg), as_raw(wu), odt(dtype))
    wg64 = wg.to(torch.float64).numpy()
    wu64 = wu.to(torch.float64).numpy()
    for r, k in enumerate(ks):
        ref = tanh_silu(wg64[k]) * wu64[k]
        assert np.allclose(h64[r], ref, rtol=1e-14, atol=1e-300)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_zeroed_columns_give_exact_zero(dtype):
    M, d, d_ff = 3, 64, 48
    x, wg, wu = inputs.make_inputs(M, d, d_ff, dtype, seed=4)
    wg = wg.clone()
    wu = wu.clone()
    wu[:, 5] = 0
    wg[:, 11] = 0          # silu(0) = 0
    h64, hr, _ = oracle.swiglu_up(as_raw(x), as_raw(wg), as_raw(wu), odt(dtype))
    assert np.all(h64[:, 5] == 0) and np.all(h64[:, 11] == 0)
    assert np.all(np.abs(np.delete(h64, [5, 11], axis=1)) > 0)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_swap_and_permutation(dtype):
    M, d, d_ff = 4, 96, 40
    x, wg, wu = inputs.make_inputs(M, d, d_ff, dtype, seed=5)
    h, _, _ = oracle.swiglu_up(as_raw(x), as_raw(wg), as_raw(wu), odt(dtype))
    hs, _, _ = oracle.swiglu_up(as_raw(x), as_raw(wu), as_raw(wg), odt(dtype))
    assert not np.allclose(h, hs, rtol=1e-2)     # gate and up are not symmetric
    perm = np.random.default_rng(6).permutation(d_ff)
    hp, _, _ = oracle.swiglu_up(as_raw(x), as_raw(wg[:, perm]), as_raw(wu[:, perm]), odt(dtype))
    assert np.array_equal(hp, h[:, perm])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_odd_symmetry_gives_gate_times_up(dtype):
    # silu(g) u + silu(-g)(-u) = (silu(g) - silu(-g)) u = g u
    M, d, d_ff = 5, 256, 64
    x, wg, wu = inputs.make_inputs(M, d, d_ff, dtype, seed=7)
    h, _, sens = oracle.swiglu_up(as_raw(x), as_raw(wg), as_raw(wu), odt(dtype))
    hn, _, _ = oracle.swiglu_up(as_raw(-x), as_raw(wg), as_raw(wu), odt(dtype))
    x64 = x.to(torch.float64).numpy()
    g = x64 @ wg.to(torch.float64).numpy()       # numpy's own fp64 matmul
    u = x64 @ wu.to(torch.float64).numpy()
    scale = np.abs(g * u) + sens
    assert np.all(np.abs((h + hn) - g * u) <= 1e-12 * scale)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_power_of_two_scaling_is_exact(dtype):
    M, d, d_ff = 3, 128, 32
    x, wg, wu = inputs.make_inputs(M, d, d_ff, dtype, seed=8)
    h, _, _ = oracle.swiglu_up(as_raw(x), as_raw(wg), as_raw(wu), odt(dtype))
    h2, _, _ = oracle.swiglu_up(as_raw(x), as_raw(wg), as_raw(wu * 2), odt(dtype))
    assert np.array_equal(h2, 2 * h)


def test_rows_are_independent_and_threads_do_not_matter():
    M, d, d_ff = 6, 200, 56
    x, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=9)
    h, _, _ = oracle.swiglu_up(as_raw(x), as_raw(wg), as_raw(wu), oracle.BF16, nthreads=1)
    h8, _, _ = oracle.swiglu_up(as_raw(x), as_raw(wg), as_raw(wu), oracle.BF16, nthreads=8)
    assert np.array_equal(h, h8)
    for i in range(M):
        hi, _, _ = oracle.swiglu_up(as_raw(x[i:i + 1]), as_raw(wg), as_raw(wu), oracle.BF16)
        assert np.array_equal(hi[0], h[i])


@pytest.mark.parametrize("dtype,shape", [("bf16", (4, 4096, 1024)), ("f32", (2, 512, 2048))])
def test_matches_numpy_fp64_at_realistic_size(dtype, shape):
    M, d, d_ff = shape
    x, wg, wu = inputs.make_inputs(M, d, d_ff, dtype, seed=10)
    h, _, sens = oracle.swiglu_up(as_raw(x), as_raw(wg), as_raw(wu), odt(dtype))
    x64 = x.to(torch.float64).numpy()
    g = x64 @ wg.to(torch.float64).numpy()
    u = x64 @ wu.to(torch.float64).numpy()
    ref = tanh_silu(g) * u
    # two fp64 evaluations with different summation orders: each sum is off by
    # at most ~d * 2^-53 * sum|x||w|, so h by at most that times s.
    bound = 2 * d * 2.0 ** -53 * sens + 16 * np.spacing(np.abs(ref))
    assert np.all(np.abs(h - ref) <= bound)


def test_sampled_outputs_equal_full_evaluation():
    M, d, d_ff = 7, 333, 90
    x, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=11)
    h, _, sens = oracle.swiglu_up(as_raw(x), as_raw(wg), as_raw(wu), oracle.BF16)
    rng = np.random.default_rng(12)
    rows = rng.integers(0, M, 50)
    cols = rng.integers(0, d_ff, 50)
    hs, ss = oracle.swiglu_up_at(as_raw(x), as_raw(wg), as_raw(wu), oracle.BF16, rows, cols)
    assert np.array_equal(hs, h[rows, cols])
    assert np.array_equal(ss, sens[rows, cols])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_fused_equals_unfused_composition(dtype):
    M, d, d_ff = 5, 160, 70
    x, wg, wu = inputs.make_inputs(M, d, d_ff, dtype, seed=13)
    h, _, _ = oracle.swiglu_up(as_raw(x), as_raw(wg), as_raw(wu), odt(dtype))
    hu = oracle.swiglu_up_unfused(as_raw(x), as_raw(wg), as_raw(wu), odt(dtype))
    assert np.allclose(h, hu, rtol=1e-15, atol=0)


def test_empty_shapes():
    x = np.zeros((0, 8), np.float32)
    w = np.zeros((8, 4), np.float32)
    h, hr, s = oracle.swiglu_up(x, w, w, oracle.F32)
    assert h.shape == (0, 4)
    x = np.zeros((3, 0), np.float32)
    w = np.zeros((0, 4), np.float32)
    h, hr, s = oracle.swiglu_up(x, w, w, oracle.F32)
    assert np.all(h == 0)          # empty sums: g = u = 0


# --------------------------------------------------------------------------
# Planted mistakes: each plausible slip must fail a pin above
# --------------------------------------------------------------------------

def _brute_force_ok(h64, x, wg, wu):
    xi = x.to(torch.float64).numpy()
    g = xi @ wg.to(torch.float64).numpy()
    u = xi @ wu.to(torch.float64).numpy()
    ref = np.vectorize(lambda a, b: float(dec_silu(a) * decimal.Decimal(b)))(g, u)
    return np.allclose(h64, ref, rtol=1e-14, atol=0)


def test_planted_mistakes_fail_the_brute_force_pin():
    M, d, d_ff = 3, 9, 7
    x, wg, wu = inputs.small_int_inputs(M, d, d_ff, "f32", seed=14)
    good, _, _ = oracle.swiglu_up(as_raw(x), as_raw(wg), as_raw(wu), oracle.F32)
    assert _brute_force_ok(good, x, wg, wu)
    # gate and up swapped
    bad, _, _ = oracle.swiglu_up(as_raw(x), as_raw(wu), as_raw(wg), oracle.F32)
    assert not _brute_force_ok(bad, x, wg, wu)
    # one term of the sum dropped
    bad, _, _ = oracle.swiglu_up(as_raw(x[:, :-1]), as_raw(wg[:-1]), as_raw(wu[:-1]), oracle.F32)
    assert not _brute_force_ok(bad, x, wg, wu)
    # weight read with the wrong layout (a transposed square block)
    sq = 7
    xs, wgs, wus = inputs.small_int_inputs(2, sq, sq, "f32", seed=15)
    good, _, _ = oracle.swiglu_up(as_raw(xs), as_raw(wgs), as_raw(wus), oracle.F32)
    bad, _, _ = oracle.swiglu_up(as_raw(xs), as_raw(wgs.t()), as_raw(wus.t()), oracle.F32)
    assert _brute_force_ok(good, xs, wgs, wus) and not _brute_force_ok(bad, xs, wgs, wus)
    # SiLU on the up product instead of the gate product
    g = oracle.gemm64(as_raw(x), as_raw(wg), oracle.F32)
    u = oracle.gemm64(as_raw(x), as_raw(wu), oracle.F32)
    assert not _brute_force_ok(oracle.silu_mul64(u, g), x, wg, wu)
