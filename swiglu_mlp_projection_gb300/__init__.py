"""GB300-native fused SwiGLU up-projection: h = silu(x.W_gate) (.) (x.W_up).

The compute path is the CUDA library built from ``csrc/`` (a C ABI declared in
``include/swiglu.h``); this package only marshals torch tensors (device memory
and the current stream) into it.  The library is loaded on first use and its
absence is an error: there is no CPU fallback.
"""
import ctypes

from . import _lib
from ._lib import (BF16, F32, PATH_AUTO, PATH_SIMT, PATH_SKINNY, PATH_TC,
                   SwiGLUError)

PATHS = {"auto": PATH_AUTO, "simt": PATH_SIMT, "skinny": PATH_SKINNY, "tc": PATH_TC}
PATH_NAMES = {v: k for k, v in PATHS.items()}


def _dtype_code(t):
    import torch
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError("swiglu_up supports bfloat16 and float32 tensors, got %s" % t.dtype)


def _path_code(path):
    if isinstance(path, int):
        return path
    try:
        return PATHS[path]
    except KeyError:
        raise ValueError("path must be one of %s" % sorted(PATHS)) from None


_LIB = None
_TORCH = None            # torch, imported on first use
_RAW_STREAM = None       # torch._C._cuda_getCurrentRawStream, where it exists
_CUR_DEVICE = None       # torch._C._cuda_getDevice, where it exists


def _torch():
    global _TORCH, _RAW_STREAM, _CUR_DEVICE
    if _TORCH is None:
        import torch
        _RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        _CUR_DEVICE = getattr(torch._C, "_cuda_getDevice", None)
        _TORCH = torch
    return _TORCH


def _raw_stream(index):
    """torch's current stream on device `index`, as a raw cudaStream_t value."""
    torch = _TORCH or _torch()
    if _RAW_STREAM is not None:
        return _RAW_STREAM(index)
    return torch.cuda.current_stream(index).cuda_stream


def _current_device():
    torch = _TORCH or _torch()
    return _CUR_DEVICE() if _CUR_DEVICE is not None else torch.cuda.current_device()


def swiglu_up(x, w_gate, w_up, out=None, path="auto", workspace=None, stream=None,
              layout="kn"):
    """h = silu(x @ w_gate) * (x @ w_up) on x's CUDA device.

    x [M, d], w_gate / w_up [d, d_ff] (layout "kn") or [d_ff, d] (layout "nk",
    the torch.nn.Linear.weight layout; then h = silu(x @ w_gate.T) * ...):
    contiguous CUDA tensors of one dtype (bfloat16 or float32).  ``out`` [M, d_ff] is written if given (else
    allocated).  ``path`` forces a kernel path ("simt", "skinny", "tc");
    ``workspace`` is an optional uint8 CUDA tensor for split-K partial sums.
    The call is asynchronous on ``stream`` (a torch.cuda.Stream; default:
    torch's current stream on x's device).
    """
    global _LIB
    torch = _TORCH or _torch()
    index = x.get_device()
    if index < 0 or w_gate.get_device() < 0 or w_up.get_device() < 0:
        raise ValueError("x, w_gate and w_up must be CUDA tensors")
    if not (x.is_contiguous() and w_gate.is_contiguous() and w_up.is_contiguous()):
        raise ValueError("x, w_gate and w_up must be contiguous")
    if x.dim() != 2 or w_gate.dim() != 2 or w_up.shape != w_gate.shape:
        raise ValueError("expected x [M, d] and w_gate, w_up [d, d_ff] or [d_ff, d]")
    if layout not in ("kn", "nk"):
        raise ValueError("layout must be 'kn' or 'nk'")
    M, d = x.shape
    kdim = 0 if layout == "kn" else 1
    if w_gate.shape[kdim] != d:
        raise ValueError("x has d=%d but w_gate is %s (layout %s)" % (d, tuple(w_gate.shape), layout))
    d_ff = w_gate.shape[1 - kdim]
    dt = _dtype_code(x)
    if w_gate.dtype != x.dtype or w_up.dtype != x.dtype:
        raise TypeError("x, w_gate and w_up must share one dtype")
    if out is None:
        out = torch.empty((M, d_ff), dtype=x.dtype, device=x.device)
    elif out.shape != (M, d_ff) or out.dtype != x.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous [M, d_ff] tensor of x's dtype")
    st = stream.cuda_stream if stream is not None else _raw_stream(index)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    if _LIB is None:
        _LIB = _lib.load()
    args = (x.data_ptr(), w_gate.data_ptr(), w_up.data_ptr(), out.data_ptr(), M, d, d_ff, dt,
            _path_code(path), ws_ptr, ws_bytes, st)
    fn = _LIB.swiglu_up_ex if layout == "kn" else _LIB.swiglu_up_nk
    if _current_device() != index:
        with torch.cuda.device(index):
            status = fn(*args)
    else:
        status = fn(*args)
    if status:
        _lib.check(status)
    return out


def _call(index, fn, *args):
    torch = _TORCH or _torch()
    if _current_device() != index:
        with torch.cuda.device(index):
            status = fn(*args)
    else:
        status = fn(*args)
    if status:
        _lib.check(status)


def packed_weight_bytes(d, d_ff, dtype="bf16"):
    """Bytes of the packed gate/up matrix for [d, d_ff] weights (host-only)."""
    dt = BF16 if dtype in ("bf16", BF16) else F32
    n = int(_lib.load().swiglu_packed_weight_bytes(d, d_ff, dt))
    if n == 0 and d * d_ff > 0:
        _lib.check(1)   # invalid sizes (detail in the library's error string)
    return n


def pack_weights(w_gate, w_up, out=None, stream=None):
    """Step a0: pack w_gate and w_up ([d, d_ff], contiguous CUDA tensors of one
    dtype) into one [d, 2 P] matrix (P = d_ff rounded up to 64) whose 64-column
    blocks alternate gate, up (zero past d_ff).  The copy runs on the current
    (or given) stream; returns the packed tensor (``out`` if given)."""
    global _LIB
    import torch
    _check_cuda(w_gate=w_gate, w_up=w_up)
    if w_gate.dim() != 2 or w_up.shape != w_gate.shape or w_up.dtype != w_gate.dtype:
        raise ValueError("expected w_gate and w_up of one shape [d, d_ff] and dtype")
    d, d_ff = w_gate.shape
    width = 128 * ((d_ff + 63) // 64)
    if out is None:
        out = torch.empty((d, width), dtype=w_gate.dtype, device=w_gate.device)
    elif out.shape != (d, width) or out.dtype != w_gate.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous [d, %d] tensor of the weights' dtype" % width)
    index = w_gate.device.index
    st = stream.cuda_stream if stream is not None else _raw_stream(index)
    if _LIB is None:
        _LIB = _lib.load()
    _call(index, _LIB.swiglu_pack_weights, w_gate.data_ptr(), w_up.data_ptr(), out.data_ptr(),
          d, d_ff, _dtype_code(w_gate), st)
    return out


def swiglu_up_packed(x, w_packed, d_ff, out=None, path="auto", workspace=None, stream=None):
    """h = silu(x @ W_gate) * (x @ W_up) with both weights read from the packed
    matrix of ``pack_weights`` (w_packed [d, 2 P]); d_ff is the unpadded
    output width.  Arguments and result otherwise as ``swiglu_up``."""
    global _LIB
    import torch
    _check_cuda(x=x, w_packed=w_packed)
    if x.dim() != 2 or w_packed.dim() != 2 or w_packed.shape[0] != x.shape[1]:
        raise ValueError("expected x [M, d] and w_packed [d, 2P]")
    if w_packed.shape[1] != 128 * ((d_ff + 63) // 64):
        raise ValueError("w_packed has %d columns; d_ff=%d needs %d"
                         % (w_packed.shape[1], d_ff, 128 * ((d_ff + 63) // 64)))
    if w_packed.dtype != x.dtype:
        raise TypeError("x and w_packed must share one dtype")
    M, d = x.shape
    if out is None:
        out = torch.empty((M, d_ff), dtype=x.dtype, device=x.device)
    elif out.shape != (M, d_ff) or out.dtype != x.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous [M, d_ff] tensor of x's dtype")
    index = x.device.index
    st = stream.cuda_stream if stream is not None else _raw_stream(index)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    if _LIB is None:
        _LIB = _lib.load()
    _call(index, _LIB.swiglu_up_packed, x.data_ptr(), w_packed.data_ptr(), out.data_ptr(), M, d,
          d_ff, _dtype_code(x), _path_code(path), ws_ptr, ws_bytes, st)
    return out


class Fp8Weights:
    """W_gate and W_up quantized to e4m3 per output column: codes [d_ff, d]
    (uint8, the shared dimension contiguous) and f32 scales [d_ff]."""

    def __init__(self, w8_gate, w8_up, s_gate, s_up):
        self.w8_gate, self.w8_up, self.s_gate, self.s_up = w8_gate, w8_up, s_gate, s_up
        self.d_ff, self.d = w8_gate.shape


def quantize_weights_fp8(w_gate, w_up, stream=None):
    """Quantize bf16 w_gate, w_up [d, d_ff] to e4m3 per output column (see
    swiglu_quantize_weights_fp8); returns an Fp8Weights."""
    global _LIB
    import torch
    _check_cuda(w_gate=w_gate, w_up=w_up)
    if w_gate.dtype != torch.bfloat16 or w_up.dtype != torch.bfloat16:
        raise TypeError("w_gate and w_up must be bfloat16")
    if w_gate.dim() != 2 or w_up.shape != w_gate.shape:
        raise ValueError("expected w_gate and w_up of one shape [d, d_ff]")
    d, d_ff = w_gate.shape
    dev = w_gate.device
    w8g = torch.empty((d_ff, d), dtype=torch.uint8, device=dev)
    w8u = torch.empty((d_ff, d), dtype=torch.uint8, device=dev)
    sg = torch.empty(d_ff, dtype=torch.float32, device=dev)
    su = torch.empty(d_ff, dtype=torch.float32, device=dev)
    st = stream.cuda_stream if stream is not None else _raw_stream(dev.index)
    if _LIB is None:
        _LIB = _lib.load()
    _call(dev.index, _LIB.swiglu_quantize_weights_fp8, w_gate.data_ptr(), w_up.data_ptr(),
          w8g.data_ptr(), w8u.data_ptr(), sg.data_ptr(), su.data_ptr(), d, d_ff, st)
    return Fp8Weights(w8g, w8u, sg, su)


class Fp8Matrix:
    """One weight matrix quantized to e4m3 per output column: codes [N, K]
    (uint8, K contiguous) and f32 scales [N]."""

    def __init__(self, w8, s):
        self.w8, self.s = w8, s
        self.N, self.K = w8.shape


def quantize_weight_fp8(w, stream=None):
    """Quantize one bf16 matrix w [K, N] (e.g. W_down [d_ff, d]) to e4m3 per
    output column; returns an Fp8Matrix."""
    global _LIB
    import torch
    _check_cuda(w=w)
    if w.dtype != torch.bfloat16 or w.dim() != 2:
        raise ValueError("expected a bfloat16 matrix [K, N]")
    K, N = w.shape
    w8 = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    s = torch.empty(N, dtype=torch.float32, device=w.device)
    st = stream.cuda_stream if stream is not None else _raw_stream(w.device.index)
    if _LIB is None:
        _LIB = _lib.load()
    _call(w.device.index, _LIB.swiglu_quantize_weight_fp8, w.data_ptr(), w8.data_ptr(),
          s.data_ptr(), K, N, st)
    return Fp8Matrix(w8, s)


def swiglu_down_fp8(h, w, residual=None, out=None, path="auto", workspace=None, stream=None):
    """y = h @ W_down (+ residual) with e4m3 weights ``w`` (an Fp8Matrix of
    W_down) and h quantized per row inside the call; h [M, d_ff], residual and
    the result [M, d] are bfloat16."""
    global _LIB
    import torch
    _check_cuda(h=h, residual=residual)
    if h.dtype != torch.bfloat16 or h.dim() != 2 or h.shape[1] != w.K:
        raise ValueError("expected bfloat16 h [M, %d]" % w.K)
    M, d = h.shape[0], w.N
    if residual is not None and (residual.shape != (M, d) or residual.dtype != h.dtype):
        raise ValueError("residual must be a bfloat16 [M, d] tensor")
    if out is None:
        out = torch.empty((M, d), dtype=h.dtype, device=h.device)
    elif out.shape != (M, d) or out.dtype != h.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous bfloat16 [M, d] tensor")
    index = h.device.index
    st = stream.cuda_stream if stream is not None else _raw_stream(index)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    if _LIB is None:
        _LIB = _lib.load()
    _call(index, _LIB.swiglu_down_fp8, h.data_ptr(), w.w8.data_ptr(), w.s.data_ptr(),
          residual.data_ptr() if residual is not None else None, out.data_ptr(), M, w.K, d,
          _path_code(path), ws_ptr, ws_bytes, st)
    return out


def fp8_workspace_bytes(M, d, d_ff, path="auto"):
    """Workspace bytes an FP8 call needs on the current device."""
    n = int(_lib.load().swiglu_fp8_workspace_bytes(M, d, d_ff, _path_code(path)))
    if n == 0 and M > 0 and d > 0:   # a call with rows and a shared dimension needs some
        _lib.check(1)
    return n


def swiglu_up_fp8(x, w, out=None, path="auto", workspace=None, stream=None):
    """h = silu(x @ W_gate) * (x @ W_up) with e4m3 weights ``w`` (an
    Fp8Weights) and x quantized per row to e4m3 inside the call; x [M, d] and
    the result [M, d_ff] are bfloat16."""
    global _LIB
    import torch
    _check_cuda(x=x)
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.shape[1] != w.d:
        raise ValueError("expected bfloat16 x [M, %d]" % w.d)
    M = x.shape[0]
    if out is None:
        out = torch.empty((M, w.d_ff), dtype=x.dtype, device=x.device)
    elif out.shape != (M, w.d_ff) or out.dtype != x.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous bfloat16 [M, d_ff] tensor")
    index = x.device.index
    st = stream.cuda_stream if stream is not None else _raw_stream(index)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    if _LIB is None:
        _LIB = _lib.load()
    _call(index, _LIB.swiglu_up_fp8, x.data_ptr(), w.w8_gate.data_ptr(), w.w8_up.data_ptr(),
          w.s_gate.data_ptr(), w.s_up.data_ptr(), out.data_ptr(), M, w.d, w.d_ff,
          _path_code(path), ws_ptr, ws_bytes, st)
    return out


def _check_cuda(**tensors):
    for name, t in tensors.items():
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("%s must be a CUDA tensor" % name)
        if not t.is_contiguous():
            raise ValueError("%s must be contiguous" % name)


def swiglu_down(h, w_down, residual=None, out=None, path="auto", workspace=None, stream=None,
                layout="kn"):
    """y = h @ w_down (+ residual): the MLP's down projection.

    h [M, d_ff], w_down [d_ff, d] (layout "kn") or [d, d_ff] (layout "nk",
    torch.nn.Linear.weight), residual [M, d] (or None; may be ``out``):
    contiguous bfloat16 CUDA tensors.  Returns y [M, d] (``out`` if given).
    """
    global _LIB
    import torch
    _check_cuda(h=h, w_down=w_down, residual=residual)
    if layout not in ("kn", "nk"):
        raise ValueError("layout must be 'kn' or 'nk'")
    kdim = 0 if layout == "kn" else 1
    if h.dim() != 2 or w_down.dim() != 2 or w_down.shape[kdim] != h.shape[1]:
        raise ValueError("expected h [M, d_ff] and w_down [d_ff, d] (kn) or [d, d_ff] (nk)")
    M, d_ff = h.shape
    d = w_down.shape[1 - kdim]
    dt = _dtype_code(h)
    if w_down.dtype != h.dtype or (residual is not None and residual.dtype != h.dtype):
        raise TypeError("h, w_down and residual must share one dtype")
    if residual is not None and residual.shape != (M, d):
        raise ValueError("residual must be [M, d]")
    if out is None:
        out = torch.empty((M, d), dtype=h.dtype, device=h.device)
    elif out.shape != (M, d) or out.dtype != h.dtype or not out.is_contiguous():
        raise ValueError("out must be a contiguous [M, d] tensor of h's dtype")
    index = h.device.index
    st = stream.cuda_stream if stream is not None else _raw_stream(index)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    if _LIB is None:
        _LIB = _lib.load()
    args = (h.data_ptr(), w_down.data_ptr(), residual.data_ptr() if residual is not None else None,
            out.data_ptr(), M, d_ff, d, dt, _path_code(path), ws_ptr, ws_bytes, st)
    fn = _LIB.swiglu_down_ex if layout == "kn" else _LIB.swiglu_down_nk
    if torch.cuda.current_device() != index:
        with torch.cuda.device(index):
            status = fn(*args)
    else:
        status = fn(*args)
    if status:
        _lib.check(status)
    return out


def swiglu_mlp(x, w_gate, w_up, w_down, residual=None, h=None, out=None, stream=None):
    """y = silu(x @ w_gate) * (x @ w_up) @ w_down (+ residual), as two kernels.

    ``h`` [M, d_ff] receives the intermediate (allocated if None).  Returns
    (y, h).  bfloat16 only.
    """
    global _LIB
    import torch
    _check_cuda(x=x, w_gate=w_gate, w_up=w_up, w_down=w_down, residual=residual)
    M, d = x.shape
    d_ff = w_gate.shape[1]
    if w_down.shape != (d_ff, d) or w_gate.shape != (d, d_ff) or w_up.shape != (d, d_ff):
        raise ValueError("expected x [M, d], w_gate/w_up [d, d_ff], w_down [d_ff, d]")
    dt = _dtype_code(x)
    if h is None:
        h = torch.empty((M, d_ff), dtype=x.dtype, device=x.device)
    if out is None:
        out = torch.empty((M, d), dtype=x.dtype, device=x.device)
    index = x.device.index
    st = stream.cuda_stream if stream is not None else _raw_stream(index)
    if _LIB is None:
        _LIB = _lib.load()
    args = (x.data_ptr(), w_gate.data_ptr(), w_up.data_ptr(), w_down.data_ptr(),
            residual.data_ptr() if residual is not None else None, h.data_ptr(),
            out.data_ptr(), M, d, d_ff, dt, st)
    if torch.cuda.current_device() != index:
        with torch.cuda.device(index):
            status = _LIB.swiglu_mlp(*args)
    else:
        status = _LIB.swiglu_mlp(*args)
    if status:
        _lib.check(status)
    return out, h


def down_workspace_bytes(M, d_ff, d, dtype="bf16", path="auto"):
    lib = _lib.load()
    dt = BF16 if dtype in ("bf16", BF16) else F32
    return int(lib.swiglu_down_workspace_bytes(M, d_ff, d, dt, _path_code(path)))


def down_plan(M, d_ff, d, dtype="bf16", path="auto", num_sms=152):
    """How a down-projection call would be served: host-only for a GPU with
    ``num_sms`` SMs, or on the current device with ``num_sms=0``."""
    lib = _lib.load()
    info = _lib.PlanInfo()
    dt = BF16 if dtype in ("bf16", BF16) else F32
    _lib.check(lib.swiglu_down_plan(M, d_ff, d, dt, _path_code(path), num_sms, ctypes.byref(info)))
    return _plan_dict(info)


def workspace_bytes(M, d, d_ff, dtype="bf16", path="auto"):
    """Workspace bytes a call needs on the current device (0 for TC calls
    whose tiles fill whole waves)."""
    lib = _lib.load()
    dt = BF16 if dtype in ("bf16", BF16) else F32
    return int(lib.swiglu_workspace_bytes(M, d, d_ff, dt, _path_code(path)))


def plan(M, d, d_ff, dtype="bf16", path="auto", num_sms=152):
    """How a call would be served: host-only for a GPU with ``num_sms`` SMs,
    or on the current device with ``num_sms=0``."""
    lib = _lib.load()
    info = _lib.PlanInfo()
    dt = BF16 if dtype in ("bf16", BF16) else F32
    _lib.check(lib.swiglu_plan(M, d, d_ff, dt, _path_code(path), num_sms, ctypes.byref(info)))
    return _plan_dict(info)


def _plan_dict(info):
    return {"path": PATH_NAMES.get(info.path, info.path), "slices": info.slices,
            "grid": info.grid, "row_chunk": info.row_chunk,
            "workspace": info.workspace, "skinny_max_m": info.skinny_max_m,
            "launches": info.launches, "cluster": info.cluster}


def split_k_slices(K, col_blocks, target_blocks, min_k_per_slice):
    """The page's K-slice rule (host-only)."""
    return int(_lib.load().swiglu_split_k_slices(K, col_blocks, target_blocks, min_k_per_slice))


def check_device_status():
    """Synchronise and raise SwiGLUError if a device-side wait timed out."""
    _lib.check(_lib.load().swiglu_check_device_status())


def release_stream_workspace(stream=None):
    """Free the workspace the library caches for ``stream`` (torch's current
    stream by default), stream-ordered; call before dropping a stream."""
    import torch
    dev = torch.cuda.current_device()
    raw = stream.cuda_stream if stream is not None else _raw_stream(dev)
    _call(dev, _lib.load().swiglu_release_stream_workspace, raw)


def release_workspaces():
    """Wait for the current device, then free every workspace the library
    caches on it and trim its pool."""
    _lib.check(_lib.load().swiglu_release_workspaces())


def cached_workspace_bytes():
    """Bytes of workspace the library caches on the current device."""
    return int(_lib.load().swiglu_cached_workspace_bytes())


def version():
    return int(_lib.load().swiglu_version())


__all__ = ["swiglu_up", "swiglu_down", "swiglu_mlp", "workspace_bytes",
           "down_workspace_bytes", "plan", "down_plan", "split_k_slices",
           "check_device_status", "release_stream_workspace", "release_workspaces",
           "cached_workspace_bytes", "version", "SwiGLUError", "PATHS"]
