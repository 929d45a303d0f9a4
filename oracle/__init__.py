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
(64-column blocks), a copy of element bits.  The FP8 functions (e4m3 codec,
per-row / per-column quantizers, dequantization) define the FP8 path: its
result is the fused definition on the dequantized operands, in fp64.

Parity pins (tests/test_oracle.py, tests/test_oracle_down.py): exact
small-integer brute force, the silu
identities silu(z) - silu(-z) = z and silu(z) = z (1 + tanh(z/2)) / 2,
high-precision decimal evaluation, one-hot x, zeroed columns, column
permutation, h(x) + h(-x) = g (.) u, power-of-two scaling, row independence,
numpy fp64 matmul at realistic sizes, and torch's bf16 rounding; the packing
against a reshape-based unpacking and a worked example (tests/test_oracle_pack.py);
the e4m3 codec against torch's float8_e4m3fn on all codes and 90,000 values,
and the FP8 path against the bf16 definition on exactly representable inputs
(tests/test_oracle_fp8.py).  Every oracle
function is pinned; none is marked "parity unpinned".
"""
import ctypes
import os

import numpy as np

from . import build as _build

F32 = 0
BF16 = 1
F64 = 2   # operands already dequantized to fp64 (the FP8 path)

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
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_quantize_rows_e4m3.argtypes = [vp, i64, i64, vp, vp]
        lib.oracle_quantize_rows_e4m3.restype = ip
        lib.oracle_quantize_cols_e4m3.argtypes = [vp, i64, i64, vp, vp]
        lib.oracle_quantize_cols_e4m3.restype = ip
        lib.oracle_dequant_rows_e4m3.argtypes = [vp, vp, i64, i64, vp]
        lib.oracle_dequant_rows_e4m3.restype = ip
        _lib = lib
    return _lib


def _raw(a, dtype):
    """Return a C-contiguous numpy array holding the raw element bits."""
    a = np.ascontiguousarray(a)
    if dtype == F64:
        if a.dtype != np.float64:
            raise TypeError("dequantized operands are passed as float64")
    elif dtype == BF16:
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
    hr = np.empty((M, d_ff), {BF16: np.uint16, F32: np.float32, F64: np.float64}[dtype])
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
    yr = np.empty((M, N), {BF16: np.uint16, F32: np.float32, F64: np.float64}[dtype])
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


# ---- FP8 (e4m3) ----------------------------------------------------------

def e4m3_decode(codes):
    """Values of e4m3 codes (uint8 array) as float64."""
    lib = _load()
    c = np.ascontiguousarray(codes, np.uint8)
    return np.array([lib.oracle_e4m3_decode(int(v)) for v in c.ravel()]).reshape(c.shape)


def e4m3_encode(values):
    """float32 values -> e4m3 codes (round to nearest even, saturating)."""
    lib = _load()
    v = np.ascontiguousarray(values, np.float32)
    return np.array([lib.oracle_e4m3_encode(float(x)) for x in v.ravel()],
                    np.uint8).reshape(v.shape)


def quantize_rows_e4m3(a):
    """Per-row e4m3 quantization of bf16 bits a [R, K]: (codes [R, K], scales [R] f32)."""
    lib = _load()
    a = _raw(a, BF16)
    R, K = a.shape
    codes = np.empty((R, K), np.uint8)
    scales = np.empty(R, np.float32)
    rc = lib.oracle_quantize_rows_e4m3(_ptr(a), R, K, _ptr(codes), _ptr(scales))
    if rc != 0:
        raise RuntimeError("oracle_quantize_rows_e4m3 failed (%d)" % rc)
    return codes, scales


def quantize_cols_e4m3(w):
    """Per-column e4m3 quantization of bf16 bits w [K, N], codes transposed:
    (codes [N, K], scales [N] f32)."""
    lib = _load()
    w = _raw(w, BF16)
    K, N = w.shape
    codes = np.empty((N, K), np.uint8)
    scales = np.empty(N, np.float32)
    rc = lib.oracle_quantize_cols_e4m3(_ptr(w), K, N, _ptr(codes), _ptr(scales))
    if rc != 0:
        raise RuntimeError("oracle_quantize_cols_e4m3 failed (%d)" % rc)
    return codes, scales


def dequant_rows_e4m3(codes, scales):
    """decode(codes[r, k]) * scales[r] as float64 [R, K]."""
    lib = _load()
    codes = np.ascontiguousarray(codes, np.uint8)
    scales = np.ascontiguousarray(scales, np.float32)
    R, K = codes.shape
    out = np.empty((R, K), np.float64)
    rc = lib.oracle_dequant_rows_e4m3(_ptr(codes), _ptr(scales), R, K, _ptr(out))
    if rc != 0:
        raise RuntimeError("oracle_dequant_rows_e4m3 failed (%d)" % rc)
    return out


def swiglu_up_fp8(x, wg, wu, nthreads=None):
    """The FP8 path's definition: x (bf16 bits [M, d]) quantized per row,
    wg/wu (bf16 bits [d, d_ff]) per column, then the fused definition on the
    dequantized operands in fp64.  Returns (h64, sens, q) with q the dict of
    codes and scales (x8, sx, wg8 [d_ff, d], sg, wu8, su)."""
    x8, sx = quantize_rows_e4m3(x)
    g8, sg = quantize_cols_e4m3(wg)
    u8, su = quantize_cols_e4m3(wu)
    xd = dequant_rows_e4m3(x8, sx)
    gd = np.ascontiguousarray(dequant_rows_e4m3(g8, sg).T)
    ud = np.ascontiguousarray(dequant_rows_e4m3(u8, su).T)
    h64, _, sens = swiglu_up(xd, gd, ud, F64, nthreads=nthreads, want_rounded=False)
    return h64, sens, {"x8": x8, "sx": sx, "wg8": g8, "sg": sg, "wu8": u8, "su": su}


def down_proj_fp8(h, wd, r=None):
    """The FP8 down projection's definition: h (bf16 bits [M, d_ff]) quantized
    per row, wd (bf16 bits [d_ff, d]) per column, then y = h . wd (+ r) in
    fp64 on the dequantized operands (r, bf16 bits, exact).  Returns
    (y64, sens)."""
    h8, sh = quantize_rows_e4m3(h)
    w8, sw = quantize_cols_e4m3(wd)
    hd = dequant_rows_e4m3(h8, sh)
    wdd = np.ascontiguousarray(dequant_rows_e4m3(w8, sw).T)
    rd = bf16_to_f64(_raw(r, BF16)) if r is not None else None
    y64, _, sens = down_proj(hd, wdd, F64, rd)
    return y64, sens

