"""Host-side logic of bench.py (no GPU): timing statistics, the rows the
oracle leg checks, the torchrun re-launch, the traffic record and the
reference arm's JSON line."""
import hashlib
import json
import os

import pytest

import bench


def test_quantiles():
    q = bench.quantiles(list(range(1, 12)))          # 1..11
    assert q == {"median": 6, "p10": 2, "p90": 10}
    assert bench.quantiles([4.0]) == {"median": 4.0, "p10": 4.0, "p90": 4.0}
    assert bench.quantiles([])["median"] is None


@pytest.mark.parametrize("M,d,d_ff", [(1, 512, 2048), (16, 8192, 29568), (64, 4096, 14336),
                                       (512, 896, 4864), (2048, 8192, 29568),
                                       (4096, 4096, 14336), (8192, 8192, 29568)])
def test_check_rows(M, d, d_ff):
    rows = bench.check_rows(M, d, d_ff)
    assert rows == sorted(set(rows))
    assert all(0 <= r < M for r in rows)
    if M <= 64 or M * d * d_ff <= 4e9:
        assert rows == list(range(M))
    else:
        assert rows[0] == 0 and rows[-1] == M - 1 and len(rows) >= 6
        assert len(set(r // 128 for r in rows)) >= 5


def test_torchrun_argv():
    class A:
        gpus = 4
    argv = bench.torchrun_argv(A, ["--gpus", "4", "--steps", "3"])
    assert argv[1:4] == ["-m", "torch.distributed.run", "--nnodes=1"]
    assert argv[argv.index("--nproc-per-node") + 1] == "4"
    assert argv[argv.index("--master-addr") + 1] == "127.0.0.1"
    assert int(argv[argv.index("--master-port") + 1]) > 0
    assert argv[-4:] == ["--gpus", "4", "--steps", "3"]
    assert argv[-5].endswith("bench.py")


def test_traffic_record_is_tied_to_the_kernel_sources():
    with open(os.path.join(bench.ROOT, bench.TRAFFIC_FILE)) as f:
        rec = json.load(f)
    h = hashlib.sha256()
    for rel in rec["source_files"]:
        with open(os.path.join(bench.ROOT, rel), "rb") as f:
            h.update(f.read())
    expect = int(rec["traffic_bytes_per_launch_mean"]) \
        if h.hexdigest() == rec["source_sha256"] else None
    assert bench.profiled_traffic() == expect
    # the record's traffic is within 1.15x of the algorithmic bytes
    assert 1.0 <= rec["traffic_bytes_per_launch_mean"] / rec["algorithmic_bytes_per_launch_mean"] \
        <= 1.15


def test_reference_arm_line(monkeypatch, capsys):
    # the oracle replaced by a stub that reports a fixed rate: only the line's
    # shape is under test here
    monkeypatch.setattr(bench, "oracle_sweep", lambda cols, budget, threads=None:
                        (2.5, 0.01, 5, 3))
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)

    class A:
        gpus, steps, warmup = 1, 3, 1
    assert bench.run_reference(A) == 0
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] == 2.5
    assert line["config"] == bench.bench_config()
    assert line["n_gpus"] == 1 and line["steps"] == 3 and line["warmup"] == 1
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] == 3
    assert str(bench.ORACLE_COLS) in line["cpu_baseline"]["sample"]
    assert line["e2e"] == {"value": 2.5, "unit": "GB/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_gpus_must_match_world_size(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr("sys.argv", ["bench.py", "--gpus", "3", "--impl", "reference"])
    assert bench.main() == 2
    assert "WORLD_SIZE=2" in capsys.readouterr().err


def test_weight_copies_cover_the_footprint():
    # every timed loop rotates at least 3 L2 capacities and 2 GiB of distinct
    # weights (the headline's 235 MB copies, FP8's 117 MB, d = 8192's 969 MB)
    l2 = 129 << 20
    for nbytes in (8 << 20, 17_432_576, 117_440_512, 234_881_024, 968_884_224, 4 << 30):
        n = bench.copies_for(l2, nbytes)
        assert n >= 2
        assert n * nbytes >= 3 * l2 and n * nbytes >= bench.WEIGHT_FOOTPRINT
        assert (n - 1) * nbytes < max(3 * l2, bench.WEIGHT_FOOTPRINT) or n == 2
