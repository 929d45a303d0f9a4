"""Work counts (FLOP, algorithmic bytes) pinned to the numbers the pages print."""
import os

import pytest

from swiglu_mlp_projection_gb300 import workload

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.txt")


def load_golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            vals[k] = float(v)
    return vals


G = load_golden()


def test_one_512_matrix_is_one_megabyte():
    n = int(G["gemv_matrix"])
    # weight bytes of one f32 matrix = half the weight traffic of the fused op
    w_bytes = workload.algorithmic_bytes(0, n, n, "f32") // 2
    assert w_bytes == G["gemv_weight_mb"] * 2 ** 20


def test_old_gemv_bandwidth_and_full_bandwidth_time():
    w_bytes = int(G["gemv_matrix"]) ** 2 * 4
    gbs = w_bytes / (G["gemv_old_us"] * 1e-6) / 1e9
    assert round(gbs) == G["gemv_old_gbs"]
    t_us = w_bytes / (G["rtx3090_gbs"] * 1e9) * 1e6
    assert round(t_us, 1) == G["gemv_full_bw_us"]


def test_decode_intensity_half_op_per_byte_in_f32():
    # one token (M=1): two operations per f32 weight read
    ai = workload.arithmetic_intensity(1, 4096, 14336, "f32")
    assert ai == pytest.approx(G["decode_ops_per_byte"], rel=1e-3)
    # bf16 weights: ~M operations per byte (the anatomy chapter's I ~ b)
    for M in (1, 2, 4, 8, 16):
        assert workload.arithmetic_intensity(M, 4096, 14336, "bf16") == pytest.approx(M, rel=5e-3)


def test_ridge_and_model_read_time():
    assert round(G["rtx3090_f32_tflops"] * 1e12 / (G["rtx3090_gbs"] * 1e9)) == G["rtx3090_ridge_ops_per_byte"]
    mb = G["model_params_millions"] * 1e6 * 4 / 1e6
    assert round(mb) == G["model_weights_mb"]
    assert round(mb * 1e6 / (G["rtx3090_gbs"] * 1e9) * 1e3, 2) == G["model_read_ms"]


def test_mlp_share_of_gemm_flops():
    # with d_ff = 3.5 d: up-projection (gate + up) + down, in units of bS d^2
    d = 4096
    d_ff = int(G["dff_over_d"] * d)
    up = workload.flops(1, d, d_ff) / d ** 2          # 4 d d_ff / d^2 = 14
    down = 2 * d_ff * d / d ** 2                        # 7
    mlp_units = (up + down) / 2                         # in units of 2 bS d^2
    assert mlp_units == G["mlp_units"]
    share = mlp_units / G["gemm_units"]
    assert round(share * 100) == G["mlp_share_percent"]


def test_prefill_intensity_is_about_bS():
    ai = workload.arithmetic_intensity(int(G["prefill_tokens"]), 4096, 14336, "bf16")
    # the chapter's I ~ bS counts weights only; with x and h traffic it is lower
    assert 0.5 * G["prefill_tokens"] < ai < G["prefill_tokens"]
    assert ai > G["h100_ridge"]


def test_config_work_counts():
    # FLOP of the prefill call: both projections (the "481 GFLOP" figure
    # counts one); bytes of the d=4096 decode sweep
    assert workload.flops(4096, 4096, 14336) == 962_072_674_304
    assert workload.flops(4096, 4096, 14336) // 2 == 481_036_337_152
    assert workload.algorithmic_bytes(16, 4096, 14336, "bf16") == 235_470_848
    assert workload.algorithmic_bytes(1, 512, 2048, "f32") == 8_398_848
    assert workload.algorithmic_bytes(0, 4096, 14336, "bf16") == 234_881_024


def test_down_projection_work_counts():
    # d = 4096, d_ff = 14336, M = 16: W_down 14336 x 4096 (bf16: 2 B, e4m3:
    # 1 B plus 4 B per column scale), h 16 x 14336, residual and y 16 x 4096
    assert workload.down_flops(16, 14336, 4096) == 1_879_048_192
    assert workload.down_bytes(16, 14336, 4096, "bf16") == 118_161_408
    assert workload.fp8_down_bytes(16, 14336, 4096) == 59_457_536
    assert workload.fp8_down_bytes(16, 14336, 4096, residual=False) == 59_326_464
