"""World-size-2 checks of the multi-rank logic on CPU (gloo).

The up-projection shards by columns with no exchange step: each rank holds
the same column range of W_gate and W_up and computes its slice of h.  Two
gloo ranks compute their slices with the oracle; the concatenation must equal
the unsharded result bit for bit.  The bench's max-over-ranks timing
reduction is exercised with the same process group.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from swiglu_mlp_projection_gb300 import inputs, sharding

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, M, d, d_ff, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        x, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=11)
        lo, hi = sharding.column_range(d_ff, rank, world)
        raw = inputs.raw_bits
        h64, hr, _ = oracle.swiglu_up(raw(x), raw(wg[:, lo:hi].contiguous()),
                                      raw(wu[:, lo:hi].contiguous()), oracle.BF16, nthreads=2)
        parts = [None] * world
        dist.all_gather_object(parts, (lo, hi, h64, hr))
        import bench
        slowest = bench.max_over_ranks(10.0 * (rank + 1), world)
        if rank == 0:
            np.save(os.path.join(out_dir, "parts.npy"), np.array(parts, dtype=object),
                    allow_pickle=True)
            np.save(os.path.join(out_dir, "slowest.npy"), np.array([slowest]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("shape", [(3, 256, 1000), (1, 512, 2048), (5, 64, 72)])
def test_column_shards_concatenate_to_the_full_result(tmp_path, shape):
    M, d, d_ff = shape
    mp.spawn(_worker, args=(WORLD, _free_port(), M, d, d_ff, str(tmp_path)), nprocs=WORLD,
             join=True)
    parts = list(np.load(tmp_path / "parts.npy", allow_pickle=True))
    parts.sort(key=lambda p: p[0])
    # the ranges tile [0, d_ff)
    assert parts[0][0] == 0 and parts[-1][1] == d_ff
    assert all(parts[i][1] == parts[i + 1][0] for i in range(len(parts) - 1))
    x, wg, wu = inputs.make_inputs(M, d, d_ff, "bf16", seed=11)
    raw = inputs.raw_bits
    h64, hr, _ = oracle.swiglu_up(raw(x), raw(wg), raw(wu), oracle.BF16)
    assert np.array_equal(np.concatenate([p[2] for p in parts], axis=1), h64)
    assert np.array_equal(np.concatenate([p[3] for p in parts], axis=1), hr)
    assert float(np.load(tmp_path / "slowest.npy")[0]) == 10.0 * WORLD


def test_column_range_properties():
    for d_ff in (0, 8, 64, 72, 1000, 14336, 29568):
        for world in (1, 2, 3, 4, 8):
            cov = []
            for r in range(world):
                lo, hi = sharding.column_range(d_ff, r, world)
                assert lo % 64 == 0 and 0 <= lo <= hi <= d_ff
                cov.extend(range(lo, hi))
            assert cov == list(range(d_ff))
    with pytest.raises(ValueError):
        sharding.column_range(64, 2, 2)
