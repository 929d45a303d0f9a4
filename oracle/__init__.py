"""CPU oracle for the fused SwiGLU up-projection h = silu(x.Wg) (.) (x.Wu).

TEST INFRASTRUCTURE ONLY.  Only tests/, ``__graft_entry__.smoke()`` and
``bench.py`` (its cpu_baseline leg and ``--impl reference`` arm) may import
this package.  It shares no code with the CUDA library: the arithmetic lives in
``swiglu_oracle.c`` (fp64, k-ascending sums, its own bf16 codec), this module
only marshals numpy arrays into it.

Definition followed: "Tile-Level Activation Overlap for Efficient LLM
Inference", technical summary, "Enonce du probleme" (Y = SiLU(A W1) (.) (A W2));
layouts per "Ou part le temps d'un token", "Un kernel pour les matrices
etroites" (row-major weights, (k)*cols + col).

The down projection (y = h . W_down + r, the anatomy chapter's kernels #10
and #11) and the two-operation MLP are evaluated the same way.  ``pack``
writes the gate/up-interleaved weight matrix of the SwiGLU paper's Kernel-2
(64-column blocks), a copy of element bits.

Parity pins (tests/test_oracle.py, tests/test_oracle_down.py): exact
small-integer brute force, the silu
identities silu(z) - silu(-z) = z and silu(z) = z (1 + tanh(z/2)) / 2,
high-precision decimal evaluation, one-hot x, zeroed columns, column
permutation, h(x) + h(-x) = g (.) u, power-of-two scaling, row independence,
numpy fp64 matmul at realistic sizes, and torch's bf16 rounding; the packing
against a reshape-based unpacking and a worked example (tests/test_oracle_pack.py).  Every oracle
function is pinned; none is marked "parity unpinned".
"""
import ctypes
import os

import numpy as np

from . import build as _build

F32 = 0
BF16 = 1

_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        i64, vp, ip = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
        lib.oracle_swiglu_up.argtypes = [vp, vp, vp, i64, i64, i64, ip, vp, vp,
                                         vp, ip]
        lib.oracle_swiglu_up.restype = ip
        lib.oracle_swiglu_up_at.argtypes = [vp, vp, vp, i64, i64, i64, ip, vp,
                                            vp, i64, vp, vp]
        lib.oracle_swiglu_up_at.restype = ip
        lib.oracle_gemm64.argtypes = [vp, vp, i64, i64, i64, ip, vp]
        lib.oracle_gemm64.restype = ip
        lib.oracle_silu_mul64.argtypes = [vp, vp, i64, vp]
        lib.oracle_silu_mul64.restype = None
        lib.oracle_silu64.argtypes = [ctypes.c_double]
        lib.oracle_silu64.restype = ctypes.c_double
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
        lib.oracle_round_to_dtype.argtypes = [vp, i64, ip, vp]
        lib.oracle_round_to_dtype.restype = ip
        lib.oracle_down_proj.argtypes = [vp, vp, vp, i64, i64, i64, ip, vp, vp, vp]
        lib.oracle_down_proj.restype = ip
        lib.oracle_pack.argtypes = [vp, vp, i64, i64, ip, vp]
        lib.oracle_pack.restype = ip
        _lib = lib
    return _lib


def _raw(a, dtype):
    """Return a C-contiguous numpy array holding the raw element bits."""
    a = np.ascontiguousarray(a)
    if dtype == BF16:
        if a.dtype != np.uint16:
            raise TypeError("bf16 operands are passed as uint16 bit patterns")
    elif dtype == F32:
        if a.dtype != np.float32:
            raise TypeError("f32 operands are passed as float32")
    else:
        raise ValueError("dtype must be oracle.F32 or oracle.BF16")
    return a


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def default_threads():
    return max(1, os.cpu_count() or 1)


def swiglu_up(x, wg, wu, dtype, nthreads=None, want_rounded=True):
    """Fused definition over all outputs.

    x [M, d], wg/wu [d, d_ff]: uint16 bf16 bit patterns (dtype=BF16) or
    float32 (dtype=F32).  Returns (h64, h_rounded, sens): h64 and sens fp64
    [M, d_ff]; h_rounded in the raw element type (uint16 bits or float32).
    """
    lib = _load()
    x, wg, wu = _raw(x, dtype), _raw(wg, dtype), _raw(wu, dtype)
    M, d = x.shape
    d2, d_ff = wg.shape
    if d2 != d or wu.shape != wg.shape:
        raise ValueError("shape mismatch")
    h64 = np.empty((M, d_ff), np.float64)
    sens = np.empty((M, d_ff), np.float64)
    hr = np.empty((M, d_ff), np.uint16 if dtype == BF16 else np.float32)
    rc = lib.oracle_swiglu_up(_ptr(x), _ptr(wg), _ptr(wu), M, d, d_ff, dtype,
                              _ptr(h64), _ptr(hr) if want_rounded else None,
                              _ptr(sens), nthreads or default_threads())
    if rc != 0:
        raise RuntimeError("oracle_swiglu_up failed (%d)" % rc)
    return h64, (hr if want_rounded else None), sens


def swiglu_up_at(x, wg, wu, dtype, rows, cols):
    """Fused definition at the outputs (rows[t], cols[t]); returns (h64, sens)."""
    lib = _load()
    x, wg, wu = _raw(x, dtype), _raw(wg, dtype), _raw(wu, dtype)
    M, d = x.shape
    d_ff = wg.shape[1]
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    n = rows.size
    if cols.size != n:
        raise ValueError("rows and cols differ in length")
    h64 = np.empty(n, np.float64)
    sens = np.empty(n, np.float64)
    rc = lib.oracle_swiglu_up_at(_ptr(x), _ptr(wg), _ptr(wu), M, d, d_ff, dtype,
                                 _ptr(rows), _ptr(cols), n, _ptr(h64),
                                 _ptr(sens))
    if rc != 0:
        raise RuntimeError("oracle_swiglu_up_at failed (%d)" % rc)
    return h64, sens


def gemm64(a, b, dtype):
    """Plain fp64 product a [m, k] . b [k, n] (k ascending)."""
    lib = _load()
    a, b = _raw(a, dtype), _raw(b, dtype)
    m, kd = a.shape
    k2, n = b.shape
    if k2 != kd:
        raise ValueError("shape mismatch")
    out = np.empty((m, n), np.float64)
    rc = lib.oracle_gemm64(_ptr(a), _ptr(b), m, kd, n, dtype, _ptr(out))
    if rc != 0:
        raise RuntimeError("oracle_gemm64 failed (%d)" % rc)
    return out


def silu_mul64(g, u):
    """silu(g) * u element-wise in fp64."""
    lib = _load()
    g = np.ascontiguousarray(g, np.float64)
    u = np.ascontiguousarray(u, np.float64)
    if g.shape != u.shape:
        raise ValueError("shape mismatch")
    h = np.empty_like(g)
    lib.oracle_silu_mul64(_ptr(g), _ptr(u), g.size, _ptr(h))
    return h


def swiglu_up_unfused(x, wg, wu, dtype):
    """The unfused composition: G = x.Wg, U = x.Wu materialised, then silu(G)*U."""
    g = gemm64(x, wg, dtype)
    u = gemm64(x, wu, dtype)
    return silu_mul64(g, u)


def down_proj(h, wd, dtype, r=None):
    """y = h . wd (+ r): h [M, K], wd [K, N], r [M, N] or None, raw bits.
    Returns (y64, y_rounded, sens)."""
    lib = _load()
    h, wd = _raw(h, dtype), _raw(wd, dtype)
    M, K = h.shape
    K2, N = wd.shape
    if K2 != K:
        raise ValueError("shape mismatch")
    if r is not None:
        r = _raw(r, dtype)
        if r.shape != (M, N):
            raise ValueError("residual shape mismatch")
    y64 = np.empty((M, N), np.float64)
    sens = np.empty((M, N), np.float64)
    yr = np.empty((M, N), np.uint16 if dtype == BF16 else np.float32)
    rc = lib.oracle_down_proj(_ptr(h), _ptr(wd), _ptr(r) if r is not None else None, M, K, N,
                              dtype, _ptr(y64), _ptr(yr), _ptr(sens))
    if rc != 0:
        raise RuntimeError("oracle_down_proj failed (%d)" % rc)
    return y64, yr, sens


def pack(wg, wu, dtype):
    """Step a0: the packed weight matrix [d, 2P] (P = d_ff rounded up to 64),
    64-column blocks of Wg and Wu alternating, zero past d_ff; raw bits."""
    lib = _load()
    wg, wu = _raw(wg, dtype), _raw(wu, dtype)
    if wg.shape != wu.shape:
        raise ValueError("shape mismatch")
    d, d_ff = wg.shape
    width = 2 * 64 * ((d_ff + 63) // 64)
    out = np.empty((d, width), wg.dtype)
    rc = lib.oracle_pack(_ptr(wg), _ptr(wu), d, d_ff, dtype, _ptr(out))
    if rc != 0:
        raise RuntimeError("oracle_pack failed (%d)" % rc)
    return out


def mlp(x, wg, wu, wd, dtype, r=None, nthreads=None):
    """The whole MLP as two operations: h = swiglu_up(x) rounded to the
    operand type (the up-projection's output), then y = h . wd (+ r).
    Returns (y64, y_rounded, sens, h_rounded)."""
    _, h, _ = swiglu_up(x, wg, wu, dtype, nthreads=nthreads)
    y64, yr, sens = down_proj(h, wd, dtype, r)
    return y64, yr, sens, h


def silu64(z):
    return _load().oracle_silu64(float(z))


def bf16_to_f64(bits):
    """Decode bf16 bit patterns (uint16 array or int) to fp64."""
    lib = _load()
    if np.isscalar(bits):
        return lib.oracle_bf16_to_f64(int(bits))
    bits = np.asarray(bits, np.uint16)
    return np.array([lib.oracle_bf16_to_f64(int(b)) for b in bits.ravel()],
                    np.float64).reshape(bits.shape)


def round_to_dtype(v, dtype):
    """Round fp64 values to bf16 bits (uint16) or float32, to nearest even."""
    lib = _load()
    v = np.ascontiguousarray(v, np.float64)
    out = np.empty(v.shape, np.uint16 if dtype == BF16 else np.float32)
    rc = lib.oracle_round_to_dtype(_ptr(v), v.size, dtype, _ptr(out))
    if rc != 0:
        raise RuntimeError("oracle_round_to_dtype failed (%d)" % rc)
    return out


def to_f64(a, dtype):
    """Widen raw operand bits to fp64 with the oracle's own decoder."""
    if dtype == BF16:
        a = np.asarray(a, np.uint16)
        # the decoder is a bit shift; vectorised form of oracle_bf16_to_f64
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return np.asarray(a, np.float32).astype(np.float64)
