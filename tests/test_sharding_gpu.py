"""The column split of the up projection through the CUDA path, on one GPU:
each "rank" computes swiglu_up on its sharding.column_range share of W_gate
and W_up (its own contiguous tensors, as a rank would hold them), and the
concatenation of the shares is compared element by element with the oracle's
unsharded result.  Every output column depends only on the same column of
both weights, so no exchange is needed (a tensor-parallel split of the MLP's
first GEMM, "1 . Anatomie d'un transformeur sur GPU", worked 70B example)."""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_projection_gb300 as swg
from swiglu_mlp_projection_gb300 import inputs, sharding
from tests.parity import compare, tile_rows

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)
RAW = inputs.raw_bits


@pytest.mark.parametrize("world", [2, 3, 8])
@pytest.mark.parametrize("M,d,d_ff,dtype", [(1, 4096, 14336, "bf16"), (16, 4096, 14336, "bf16"),
                                            (300, 1024, 4104, "bf16"), (2, 520, 1000, "bf16"),
                                            (1, 512, 2048, "f32"), (5, 264, 1032, "f32")])
def test_column_shards_concatenate_to_the_oracle(world, M, d, d_ff, dtype):
    x, wg, wu = inputs.make_inputs(M, d, d_ff, dtype, seed=world + M)
    xd = x.to(DEV)
    parts = []
    for r in range(world):
        lo, hi = sharding.column_range(d_ff, r, world)
        if hi == lo:
            continue
        # a rank holds its share as contiguous tensors of its own
        wg_r = wg[:, lo:hi].contiguous().to(DEV)
        wu_r = wu[:, lo:hi].contiguous().to(DEV)
        parts.append(swg.swiglu_up(xd, wg_r, wu_r))
    torch.cuda.synchronize()
    h = torch.cat(parts, dim=1)
    assert h.shape == (M, d_ff)
    rows = np.arange(M) if M <= 16 else tile_rows(M, seed=world)
    od = oracle.BF16 if dtype == "bf16" else oracle.F32
    h64, _, s = oracle.swiglu_up(RAW(x[rows].contiguous()), RAW(wg), RAW(wu), od)
    res = compare(h.cpu().double().numpy()[rows], h64, s, dtype, d)
    assert res["ok"], (world, M, d, d_ff, dtype, res)
