"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and its host-only logic (slice rule, plans, status strings)
behaves as documented."""
import os
import re

import numpy as np
import pytest
import torch

import oracle
from swiglu_mlp_projection_gb300 import _lib, inputs
import swiglu_mlp_projection_gb300 as swg
from tests.parity import compare, floor_factor, TOL

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "swiglu.h")


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SWIGLU_API\s+[\w\s\*]+?\b(swiglu_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    syms = declared_symbols()
    assert "swiglu_up" in syms and "swiglu_up_ex" in syms
    assert set(syms) == set(_lib.SIGNATURES), "binding and header disagree"


def test_library_exports_every_declared_symbol(cuda_lib):
    for name in declared_symbols():
        assert hasattr(cuda_lib, name), name


def test_status_strings_and_version(cuda_lib):
    for code in range(9):
        s = cuda_lib.swiglu_status_string(code).decode()
        assert s and s != "unknown status"
    assert cuda_lib.swiglu_status_string(99).decode() == "unknown status"
    assert swg.version() >= 100


def test_split_k_rule_reproduces_the_pages_example(cuda_lib):
    # 512 x 512 with 32 columns per block: 16 column blocks; aiming at 256
    # blocks with >= 64 k per slice gives 8 slices and 128 blocks.
    from tests.test_workload_pins import G
    col_blocks = int(G["gemv_matrix"] // G["block_cols"])
    s = swg.split_k_slices(int(G["gemv_matrix"]), col_blocks,
                           int(G["split_target_blocks"]), int(G["split_min_k"]))
    assert s == G["split_example_slices"]
    assert s * col_blocks == G["split_example_blocks"]
    assert s * col_blocks > G["rtx3090_sms"]


def test_split_k_rule_edges(cuda_lib):
    assert swg.split_k_slices(10, 4, 256, 64) == 1          # K below one slice
    assert swg.split_k_slices(4096, 1000, 256, 64) == 1     # enough blocks already
    assert swg.split_k_slices(4096, 1, 608, 64) == 64       # capped by min k
    assert swg.split_k_slices(0, 4, 256, 64) == 1
    assert swg.split_k_slices(64, 0, 256, 64) == -1
    assert swg.split_k_slices(64, 4, 256, 0) == -1


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_plan_covers_all_columns_rows_and_k(cuda_lib, dtype):
    for (M, d, d_ff) in [(1, 512, 2048), (3, 4096, 14336), (16, 896, 4864), (17, 8, 8),
                         (5, 1024, 40)]:
        p = swg.plan(M, d, d_ff, dtype, "simt", 152)
        assert p["path"] == "simt"
        vec = 8 if dtype == "bf16" else 4
        e = 2 if dtype == "bf16" else 4
        if p["cluster"] > 1:
            # the cluster form: 8 K slices per cluster on the host plan,
            # 128-byte column blocks, one launch, no workspace
            assert M == 1 and 8 <= d <= 2048 and 2 * d * d_ff * e <= 32 << 20
            assert p["slices"] == p["cluster"] == 8
            assert p["grid"] == -(-d_ff // (8 * vec)) * 8
            assert p["workspace"] == 0 and p["launches"] == 1
            continue
        cols = 32 * vec
        chunks = -(-M // p["row_chunk"])
        assert p["grid"] == -(-d_ff // cols) * p["slices"] * chunks
        assert 1 <= p["slices"] <= d
        assert p["workspace"] >= p["slices"] * M * 2 * d_ff * 4
        assert p["workspace"] % 256 == 0


def test_simt_cluster_form_selection(cuda_lib, monkeypatch):
    # M = 1, d <= 2048 and weights <= 32 MB take the cluster form of the SIMT
    # path; SWIGLU_SIMT_CLUSTER=0 keeps the split-K kernel with its workspace
    for (M, d, d_ff, dtype, yes) in [(1, 512, 2048, "f32", True), (1, 896, 4864, "bf16", True),
                                     (2, 896, 4864, "bf16", False),
                                     (1, 4096, 14336, "bf16", False),
                                     (1, 2048, 4096, "f32", False),   # 64 MB of weights
                                     (1, 2056, 1024, "bf16", False),  # d above 2048
                                     (1, 8, 8, "f32", True), (1, 0, 8, "f32", False)]:
        p = swg.plan(M, d, d_ff, dtype, "simt", 152)
        assert (p["cluster"] == 8) == yes, (M, d, d_ff, dtype, p)
    monkeypatch.setenv("SWIGLU_SIMT_CLUSTER", "0")
    p = swg.plan(1, 512, 2048, "f32", "simt", 152)
    assert p["cluster"] == 1 and p["workspace"] > 0


@pytest.mark.parametrize("ks", [4, 5, 6, 7, 8])
def test_simt_cluster_sizes(cuda_lib, monkeypatch, ks):
    # SWIGLU_SIMT_CLUSTER=S forces clusters of S K slices.  Fewer than 8 are
    # served only where a slice holds at most 4 rows of W per thread (128 k);
    # 8 slices up to 256 k.  Otherwise the call keeps the split-K kernel.
    monkeypatch.setenv("SWIGLU_SIMT_CLUSTER", str(ks))
    for (d, d_ff, dtype) in [(512, 2048, "f32"), (896, 4864, "bf16"), (520, 264, "bf16"),
                             (2048, 1024, "bf16"), (8, 8, "f32"), (5, 8, "f32")]:
        kn = -(-d // ks)
        fits = d >= ks and (kn <= 256 if ks == 8 else kn <= 128)
        p = swg.plan(1, d, d_ff, dtype, "simt", 152)
        vec = 8 if dtype == "bf16" else 4
        if fits:
            assert p["cluster"] == p["slices"] == ks, (d, d_ff, dtype, p)
            assert p["grid"] == -(-d_ff // (8 * vec)) * ks
            assert p["workspace"] == 0 and p["launches"] == 1
        else:
            assert p["cluster"] == 1 and p["workspace"] > 0, (d, d_ff, dtype, p)


def test_plan_reports_cluster_size(cuda_lib):
    # TC path: CTA pairs above one 128-row block, single CTAs below
    p = swg.plan(4096, 4096, 14336, "bf16", "auto", 152)
    assert p["path"] == "tc" and p["cluster"] == 2 and p["grid"] == 152
    p = swg.plan(64, 896, 4864, "bf16", "tc", 152)
    assert p["cluster"] == 1 and p["grid"] == 38
    p = swg.plan(300, 4096, 14336, "bf16", "tc", 152)
    assert p["cluster"] == 2 and p["grid"] == 152      # 2 x 112 pair tiles > 76 pairs
    p = swg.plan(300, 520, 264, "bf16", "tc", 152)
    assert p["cluster"] == 2 and p["grid"] == 2 * 2 * 3
    # skinny path: split-K clusters for the small down projection only
    assert swg.down_plan(1, 4864, 896, "bf16", "auto", 152)["cluster"] == 8
    assert swg.plan(1, 4096, 14336, "bf16", "auto", 152)["cluster"] == 1
    assert swg.plan(1, 512, 2048, "f32", "auto", 152)["cluster"] == 8   # SIMT cluster form


def test_dispatch_rule(cuda_lib):
    # measured thresholds, weights above 32 MB (stream-K mode): skinny up to
    # M = 32 (up) and every M the skinny kernel serves (down, its sums in a
    # second kernel); smaller weights (cluster mode): 128 (up) and every M
    # the skinny kernel serves (down)
    for M, path in [(1, "skinny"), (16, "skinny"), (32, "skinny"), (33, "tc"), (4096, "tc")]:
        assert swg.plan(M, 4096, 14336, "bf16", "auto", 152)["path"] == path
    # (one row on small weights with d <= 1024: the SIMT path's cluster form)
    for M, path in [(1, "simt"), (2, "skinny"), (64, "skinny"), (128, "skinny"), (129, "tc"),
                    (512, "tc")]:
        assert swg.plan(M, 896, 4864, "bf16", "auto", 152)["path"] == path
    assert swg.plan(1, 2048, 3584, "bf16", "auto", 152)["path"] == "skinny"
    for M, path in [(1, "skinny"), (64, "skinny"), (256, "skinny"), (257, "tc"), (4096, "tc")]:
        assert swg.down_plan(M, 14336, 4096, "bf16", "auto", 152)["path"] == path
    for M, path in [(1, "skinny"), (128, "skinny"), (256, "skinny"), (257, "tc"), (4096, "tc")]:
        assert swg.down_plan(M, 29568, 8192, "bf16", "auto", 152)["path"] == path
    for M, path in [(1, "skinny"), (256, "skinny"), (257, "tc")]:
        assert swg.down_plan(M, 4864, 896, "bf16", "auto", 152)["path"] == path
    assert swg.plan(1, 4096, 14336, "bf16", "auto", 152)["skinny_max_m"] == 32
    assert swg.plan(1, 896, 4864, "bf16", "auto", 152)["skinny_max_m"] == 128
    assert swg.down_plan(1, 14336, 4096, "bf16", "auto", 152)["skinny_max_m"] == 256
    assert swg.down_plan(1, 29568, 8192, "bf16", "auto", 152)["skinny_max_m"] == 256
    assert swg.down_plan(1, 4864, 896, "bf16", "auto", 152)["skinny_max_m"] == 256
    # the bf16 down projection above 32 MB: stream-K with its sums in a
    # second kernel at every M (4-CTA clusters serve FP8 at 16-64 rows)
    for M in (1, 16, 32, 33, 64, 65, 256):
        p = swg.down_plan(M, 14336, 4096, "bf16", "auto", 152)
        assert p["cluster"] == 1 and p["workspace"] > 0 and p["launches"] == 2, (M, p)
    for M in (1, 16, 128, 256):
        p = swg.down_plan(M, 29568, 8192, "bf16", "auto", 152)
        assert p["cluster"] == 1 and p["launches"] == 2, (M, p)
    # the up projection keeps its final sums in one kernel
    assert swg.plan(16, 4096, 14336, "bf16", "auto", 152)["launches"] == 1
    assert swg.plan(1, 512, 2048, "f32", "auto", 152)["path"] == "simt"
    assert swg.plan(3, 0, 64, "bf16", "auto", 152)["path"] == "simt"
    with pytest.raises(swg.SwiGLUError):
        swg.plan(257, 64, 64, "bf16", "skinny", 152)
    with pytest.raises(swg.SwiGLUError):
        swg.plan(4, 64, 64, "f32", "tc", 152)


def test_up_projection_unit_width_rule(cuda_lib):
    # Above 32 MB of weights the up projection's units hold four 64-column
    # blocks up to 8 rows and two from 9 rows on; at d = 4096, d_ff = 14336
    # on 152 SMs that is 4 partial slots per column group against 3, and one
    # launch either way (the final sums stay in the kernel)
    for M in range(1, 17):
        p = swg.plan(M, 4096, 14336, "bf16", "auto", 152)
        assert p["path"] == "skinny" and p["cluster"] == 1 and p["launches"] == 1
        assert p["slices"] == (4 if M <= 8 else 3), (M, p)
    assert [swg.plan(M, 8192, 29568, "bf16", "auto", 152)["slices"] for M in (8, 9)] == [3, 2]
    # small weights keep cluster mode (the SIMT cluster form at one row)
    assert swg.plan(8, 896, 4864, "bf16", "auto", 152)["cluster"] == 2


def test_down_projection_column_groups(cuda_lib, monkeypatch):
    # 256-column groups (11 partial slots at d = 4096) up to 128 rows, then
    # 128-column groups (6 slots); stream-K mode forced at d = 4096
    monkeypatch.setenv("SWIGLU_SK_CLUSTER", "0")
    assert swg.down_plan(16, 14336, 4096, "bf16", "skinny", 152)["slices"] == 11
    assert swg.down_plan(128, 14336, 4096, "bf16", "skinny", 152)["slices"] == 11
    assert swg.down_plan(129, 14336, 4096, "bf16", "skinny", 152)["slices"] == 6
    monkeypatch.delenv("SWIGLU_SK_CLUSTER")
    # above 256 MB of weights, 256-column groups up to 64 rows
    assert swg.down_plan(64, 29568, 8192, "bf16", "skinny", 152)["slices"] == 6
    assert swg.down_plan(65, 29568, 8192, "bf16", "skinny", 152)["slices"] == 4
    # small weights stay in cluster mode; the up projection keeps its groups
    assert swg.down_plan(256, 4864, 896, "bf16", "skinny", 152)["cluster"] == 8
    assert swg.plan(32, 4096, 14336, "bf16", "skinny", 152)["slices"] == 3
    # SWIGLU_SK_NB overrides the rule (and keeps stream-K mode)
    monkeypatch.setenv("SWIGLU_SK_NB", "2")
    assert swg.down_plan(64, 14336, 4096, "bf16", "skinny", 152)["slices"] == 11
    assert swg.down_plan(64, 14336, 4096, "bf16", "skinny", 152)["cluster"] == 1


def test_packed_weight_bytes(cuda_lib):
    # 64-column blocks of gate and up alternate; d_ff is padded to 64
    assert swg.packed_weight_bytes(4096, 14336, "bf16") == 4096 * 2 * 14336 * 2
    assert swg.packed_weight_bytes(8, 200, "bf16") == 8 * 2 * 256 * 2
    assert swg.packed_weight_bytes(4, 1032, "f32") == 4 * 2 * 1088 * 4
    assert swg.packed_weight_bytes(0, 64, "bf16") == 0
    assert cuda_lib.swiglu_packed_weight_bytes(8, 12, _lib.BF16) == 0   # d_ff % 8 != 0


def test_fp8_entry_points_validate_before_touching_the_device(cuda_lib):
    lib = cuda_lib
    # d not a multiple of 16 (e4m3 rows must be 16-byte multiples)
    assert lib.swiglu_up_fp8(16, 32, 48, 64, 80, 96, 1, 24, 8, 0, None, 0, None) == 3
    assert lib.swiglu_quantize_weights_fp8(16, 32, 48, 64, 80, 96, 24, 8, None) == 3
    # null weights
    assert lib.swiglu_up_fp8(16, None, 48, 64, 80, 96, 1, 16, 8, 0, None, 0, None) == 1
    # h overlapping a scale vector
    assert lib.swiglu_up_fp8(4096, 8192, 12288, 16384, 20480, 20480, 1, 16, 8, 0, None, 0,
                             None) == 1


def test_plan_rejects_bad_arguments(cuda_lib):
    with pytest.raises(swg.SwiGLUError):
        swg.plan(-1, 8, 8, "bf16", "auto", 152)
    with pytest.raises(swg.SwiGLUError):
        swg.plan(1, 8, 8, "bf16", 17, 152)
    with pytest.raises(swg.SwiGLUError):
        swg.plan(1, 8, 8, "bf16", "auto", -1)


def test_device_plan_needs_a_device(cuda_lib):
    # num_sms = 0 plans on the current device; without a GPU that is an error
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(swg.SwiGLUError):
        swg.plan(1, 896, 4864, "bf16", "auto", 0)


def test_entry_point_validates_before_touching_the_device(cuda_lib):
    # Invalid arguments are rejected synchronously, before any device query,
    # so these run without a GPU.
    lib = cuda_lib
    st = lib.swiglu_up(None, None, None, None, -1, 8, 8, _lib.BF16, None)
    assert st == 1
    st = lib.swiglu_up(None, None, None, None, 1, 8, 8, 7, None)
    assert st == 1
    st = lib.swiglu_up(None, None, None, None, 1, 8, 8, _lib.BF16, None)
    assert st == 1 and "null" in lib.swiglu_last_error_string().decode()
    st = lib.swiglu_up(16, 32, 48, 65, 1, 8, 8, _lib.BF16, None)
    assert st == 3                       # 65 is not 16-byte aligned
    st = lib.swiglu_up(16, 32, 48, 64, 1, 12, 8, _lib.BF16, None)
    assert st == 3                       # d not a multiple of 8 for bf16
    st = lib.swiglu_up(4096, 8192, 12288, 4096, 2, 8, 8, _lib.BF16, None)
    assert st == 1 and "overlap" in lib.swiglu_last_error_string().decode()
    st = lib.swiglu_up_ex(16, 32, 48, 64, 1, 8, 8, _lib.BF16, 9, None, 0, None)
    assert st == 1


# --------------------------------------------------------------------------
# The comparison rule itself (CPU): f32-accumulation noise passes, a planted
# mistake in the oracle's output fails.
# --------------------------------------------------------------------------

def _f32_emulation(x, wg, wu, dtype):
    """An f32-accumulating evaluation in numpy (another summation order)."""
    x32 = x.to(torch.float32).numpy()
    g = x32 @ wg.to(torch.float32).numpy()
    u = x32 @ wu.to(torch.float32).numpy()
    h = (g / (1 + np.exp(-g.astype(np.float64)))).astype(np.float32) * u
    if dtype == "bf16":
        h = torch.from_numpy(h).to(torch.bfloat16).to(torch.float64).numpy()
    return h


@pytest.mark.parametrize("dtype,shape", [("f32", (1, 512, 2048)), ("bf16", (4, 4096, 512)),
                                         ("bf16", (3, 896, 256))])
def test_comparison_rule_accepts_f32_accumulation(dtype, shape):
    M, d, d_ff = shape
    x, wg, wu = inputs.make_inputs(M, d, d_ff, dtype, seed=21)
    od = oracle.BF16 if dtype == "bf16" else oracle.F32
    h64, _, sens = oracle.swiglu_up(inputs.raw_bits(x), inputs.raw_bits(wg), inputs.raw_bits(wu), od)
    res = compare(_f32_emulation(x, wg, wu, dtype), h64, sens, dtype, d)
    assert res["ok"], res


@pytest.mark.parametrize("dtype,shape", [("f32", (1, 512, 2048)), ("bf16", (4, 4096, 512))])
def test_comparison_rule_rejects_planted_mistakes(dtype, shape):
    M, d, d_ff = shape
    x, wg, wu = inputs.make_inputs(M, d, d_ff, dtype, seed=22)
    od = oracle.BF16 if dtype == "bf16" else oracle.F32
    raw = inputs.raw_bits
    h64, _, sens = oracle.swiglu_up(raw(x), raw(wg), raw(wu), od)
    # (a) one k term dropped (a slice boundary off by one)
    bad, _, _ = oracle.swiglu_up(raw(x[:, 1:]), raw(wg[1:]), raw(wu[1:]), od)
    assert not compare(bad, h64, sens, dtype, d)["ok"]
    # (b) a 64-wide K tile dropped
    bad, _, _ = oracle.swiglu_up(raw(x[:, 64:]), raw(wg[64:]), raw(wu[64:]), od)
    assert not compare(bad, h64, sens, dtype, d)["ok"]
    # (c) gate and up swapped
    bad, _, _ = oracle.swiglu_up(raw(x), raw(wu), raw(wg), od)
    assert not compare(bad, h64, sens, dtype, d)["ok"]
    # (d) two adjacent output columns exchanged
    bad = h64.copy()
    bad[:, [0, 1]] = bad[:, [1, 0]]
    assert not compare(bad, h64, sens, dtype, d)["ok"]
    # (e) output rounded to bf16 where f32 was promised
    if dtype == "f32":
        bad = torch.from_numpy(h64).to(torch.bfloat16).to(torch.float64).numpy()
        assert not compare(bad, h64, sens, dtype, d)["ok"]


def test_floor_factor_values():
    assert floor_factor("bf16", 4096) == pytest.approx(8 * 64 * 2 ** -24 / 2e-2)
    assert floor_factor("f32", 512) == pytest.approx(8 * 512 ** 0.5 * 2 ** -24 / 1e-5)
    assert TOL == {"f32": 1e-5, "bf16": 2e-2}


def test_no_cpu_fallback_for_host_tensors(cuda_lib):
    # Every compute entry point of the binding refuses host tensors instead of
    # computing on the CPU: the only compute path is the CUDA library.
    import torch
    x = torch.randn(2, 64).to(torch.bfloat16)
    w = torch.randn(64, 64).to(torch.bfloat16)
    calls = {
        "swiglu_up": lambda: swg.swiglu_up(x, w, w),
        "swiglu_down": lambda: swg.swiglu_down(x, w),
        "swiglu_mlp": lambda: swg.swiglu_mlp(x, w, w, w),
        "pack_weights": lambda: swg.pack_weights(w, w),
        "quantize_weights_fp8": lambda: swg.quantize_weights_fp8(w, w),
        "quantize_weight_fp8": lambda: swg.quantize_weight_fp8(w),
    }
    for name, call in calls.items():
        with pytest.raises(ValueError, match="CUDA"):
            call()
