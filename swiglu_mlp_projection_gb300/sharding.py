"""Column-parallel sharding of the up-projection across ranks.

Every output column j of h = silu(x.W_gate) (.) (x.W_up) depends only on
column j of W_gate and of W_up, so ranks that hold the same column range of
both weights compute their slice of h with no exchange at all; a gathered h,
if wanted, is their concatenation along d_ff.  (The anatomy chapter's
multi-GPU example uses tensor parallelism; this is the column split that
feeds a row-parallel down projection.)
"""


def column_range(d_ff, rank, world, align=64):
    """Columns [lo, hi) of W_gate/W_up held by `rank` of `world`.

    Ranges are contiguous, cover [0, d_ff) exactly once, and start on
    multiples of `align` columns (so each rank's weights stay 16-byte-row
    aligned and map onto whole 64-column kernel units)."""
    if world < 1 or not 0 <= rank < world or align < 1 or d_ff < 0:
        raise ValueError("bad sharding arguments")
    blocks = -(-d_ff // align)
    lo_b = blocks * rank // world
    hi_b = blocks * (rank + 1) // world
    return min(lo_b * align, d_ff), min(hi_b * align, d_ff)
