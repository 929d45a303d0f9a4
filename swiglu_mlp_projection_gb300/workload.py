"""Workloads and their algorithmic work counts.

Work counts follow the pages:
  * FLOP: "1 . Anatomie d'un transformeur sur GPU", section 1.2 -- a
    (bS x d).(d x d') projection costs 2 bS d d' FLOP, and gate and up cost
    2 bS d d_ff *each*, so one up-projection call costs 2 * M * d * 2 d_ff.
    (The element-wise SiLU and product, ~5 M d_ff operations, are not counted.)
  * Bytes: "Ou part le temps d'un token", section "Une borne : la bande
    passante" -- every weight is read once per pass.  Algorithmic bytes of one
    call = e * (2 d d_ff + M d + M d_ff): both weight matrices and x read once,
    h written once, e = bytes per element.  Split-K partial sums are not
    algorithmic traffic.
"""
from dataclasses import dataclass

ELEM_BYTES = {"f32": 4, "bf16": 2}


def flops(M, d, d_ff):
    """FLOP of one call: gate and up GEMMs, 2 M d d_ff each."""
    return 4 * M * d * d_ff


def algorithmic_bytes(M, d, d_ff, dtype):
    """Bytes one call must move at least: Wg, Wu, x read once; h written once."""
    e = ELEM_BYTES[dtype]
    return e * (2 * d * d_ff + M * d + M * d_ff)


def fp8_bytes(M, d, d_ff):
    """Bytes an FP8 call must move at least: the two e4m3 weight matrices and
    their f32 column scales read once, x (bf16) read once, h (bf16) written
    once.  (x's e4m3 codes are an intermediate of M d bytes, not counted.)"""
    return 2 * d * d_ff + 2 * 4 * d_ff + 2 * M * d + 2 * M * d_ff


def down_flops(M, d_ff, d):
    """FLOP of the down projection: 2 M d_ff d (the residual add is not counted)."""
    return 2 * M * d_ff * d


def down_bytes(M, d_ff, d, dtype, residual=True):
    """W_down and h read once, the residual read once, y written once."""
    e = ELEM_BYTES[dtype]
    return e * (d_ff * d + M * d_ff + M * d * (2 if residual else 1))


def fp8_down_bytes(M, d_ff, d, residual=True):
    """Bytes an FP8 down projection must move at least: W_down's e4m3 codes
    and f32 column scales, h (bf16) read once, the residual (bf16) read once,
    y (bf16) written once."""
    return d_ff * d + 4 * d + 2 * M * d_ff + 2 * M * d * (2 if residual else 1)


def arithmetic_intensity(M, d, d_ff, dtype):
    return flops(M, d, d_ff) / algorithmic_bytes(M, d, d_ff, dtype)


@dataclass(frozen=True)
class Config:
    name: str
    dtype: str
    d: int
    d_ff: int
    Ms: tuple

    def shapes(self):
        return [(M, self.d, self.d_ff) for M in self.Ms]


# The five workloads: a tiny f32 decode step, the bf16 decode sweep at
# d=4096 / d_ff=14336, a small model (d=896, d_ff=4864) across the
# skinny/tensor-core crossover, prefill at M=4096, and a large model
# (d=8192, d_ff=29568) in both regimes.
CONFIGS = (
    Config("f32_decode_d512", "f32", 512, 2048, (1,)),
    Config("bf16_decode_d4096", "bf16", 4096, 14336, (1, 2, 4, 8, 16)),
    Config("bf16_small_d896", "bf16", 896, 4864, (1, 64, 512)),
    Config("bf16_prefill_d4096", "bf16", 4096, 14336, (4096,)),
    Config("bf16_large_d8192", "bf16", 8192, 29568, (16, 2048, 8192)),
)

CONFIG_BY_NAME = {c.name: c for c in CONFIGS}
