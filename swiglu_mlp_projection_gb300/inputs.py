"""Seeded synthetic inputs for the SwiGLU up-projection.

This module holds no arithmetic of the method itself: it only draws random
operands.  Both the CUDA path (tests, bench) and the CPU oracle consume what it
returns, bit for bit.

Recipe (the shapes and distributions of the workloads; the pages publish no
data set, so these stand in for the Qwen-2.5 MLP shapes the SwiGLU paper
evaluates on, "Tile-Level Activation Overlap ...", section "Resultats"):
  * one CPU ``torch.Generator`` seeded with ``seed``;
  * draw x [M, d] ~ N(0, 1), then W_gate [d, d_ff], then W_up [d, d_ff], each
    ~ N(0, 1) scaled by 1/sqrt(d) (variance 1/d), all as float32;
  * round each to the operand type (bf16: round-to-nearest-even, done by
    torch's dtype conversion; f32: unchanged).
With variance 1/d, g = x.W_gate and u = x.W_up are ~N(0, 1) for every d.
"""
import math

import numpy as np
import torch

F32 = "f32"
BF16 = "bf16"

TORCH_DTYPE = {F32: torch.float32, BF16: torch.bfloat16}


def make_inputs(M, d, d_ff, dtype, seed=0, x_only=False):
    """Return (x, w_gate, w_up) as CPU torch tensors of ``dtype``.

    With ``x_only`` the weights are None (used to redraw activations while
    keeping the weights of an earlier call with the same seed).
    """
    if dtype not in TORCH_DTYPE:
        raise ValueError("dtype must be 'f32' or 'bf16'")
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed))
    td = TORCH_DTYPE[dtype]
    x = torch.randn(M, d, generator=gen, dtype=torch.float32).to(td)
    if x_only:
        return x, None, None
    scale = 1.0 / math.sqrt(d)
    wg = (torch.randn(d, d_ff, generator=gen, dtype=torch.float32) * scale).to(td)
    wu = (torch.randn(d, d_ff, generator=gen, dtype=torch.float32) * scale).to(td)
    return x, wg, wu


def raw_bits(t):
    """CPU tensor -> numpy array of its raw element bits (uint16 for bf16)."""
    t = t.contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float32:
        return t.numpy()
    raise TypeError("unsupported dtype %s" % t.dtype)


def from_bits(a, dtype):
    """numpy raw bits -> CPU torch tensor of ``dtype`` (inverse of raw_bits)."""
    if dtype == BF16:
        return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a, np.float32))


def small_int_inputs(M, d, d_ff, dtype, seed=0, lo=-3, hi=3):
    """Inputs whose entries are small integers (exact in bf16 and f32), so that
    every sum of products is exact in f32 as well as in fp64."""
    rng = np.random.default_rng(seed)
    td = TORCH_DTYPE[dtype]
    x = torch.from_numpy(rng.integers(lo, hi + 1, (M, d)).astype(np.float32)).to(td)
    wg = torch.from_numpy(rng.integers(lo, hi + 1, (d, d_ff)).astype(np.float32)).to(td)
    wu = torch.from_numpy(rng.integers(lo, hi + 1, (d, d_ff)).astype(np.float32)).to(td)
    return x, wg, wu
