"""ctypes loader for the CUDA library (_build/libswiglu_gb300.so).

Argument marshalling only.  The library must have been built
(``python -m swiglu_mlp_projection_gb300.build`` or ``__graft_entry__.build()``);
if it is missing, loading raises -- there is no fallback implementation.
"""
import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libswiglu_gb300.so")

# swiglu_dtype / swiglu_path / swiglu_status values of include/swiglu.h
F32, BF16 = 0, 1
PATH_AUTO, PATH_SIMT, PATH_SKINNY, PATH_TC = 0, 1, 2, 3
OK = 0
STATUS_NAMES = {
    0: "SWIGLU_OK", 1: "SWIGLU_ERR_INVALID_ARG", 2: "SWIGLU_ERR_UNSUPPORTED",
    3: "SWIGLU_ERR_ALIGNMENT", 4: "SWIGLU_ERR_OOM", 5: "SWIGLU_ERR_CUDA",
    6: "SWIGLU_ERR_TIMEOUT", 7: "SWIGLU_ERR_ARCH", 8: "SWIGLU_ERR_WORKSPACE",
}

# Every symbol include/swiglu.h declares, with its ctypes signature.
_i64, _vp, _int, _sz = ctypes.c_int64, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t


class PlanInfo(ctypes.Structure):
    _fields_ = [("path", ctypes.c_int), ("slices", ctypes.c_int64),
                ("grid", ctypes.c_int64), ("row_chunk", ctypes.c_int64),
                ("workspace", ctypes.c_int64), ("skinny_max_m", ctypes.c_int64),
                ("launches", ctypes.c_int64), ("cluster", ctypes.c_int64)]


SIGNATURES = {
    "swiglu_up": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp], _int),
    "swiglu_up_ex": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _vp, _sz, _vp], _int),
    "swiglu_up_noalloc": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp], _int),
    "swiglu_down": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp], _int),
    "swiglu_down_ex": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _vp, _sz, _vp], _int),
    "swiglu_down_workspace_bytes": ([_i64, _i64, _i64, _int, _int], _sz),
    "swiglu_up_nk": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _vp, _sz, _vp], _int),
    "swiglu_down_nk": ([_vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _vp, _sz, _vp], _int),
    "swiglu_packed_weight_bytes": ([_i64, _i64, _int], _sz),
    "swiglu_quantize_weights_fp8": ([_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _vp], _int),
    "swiglu_up_fp8": ([_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp, _sz, _vp], _int),
    "swiglu_fp8_workspace_bytes": ([_i64, _i64, _i64, _int], _sz),
    "swiglu_quantize_weight_fp8": ([_vp, _vp, _vp, _i64, _i64, _vp], _int),
    "swiglu_down_fp8": ([_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp, _sz, _vp], _int),
    "swiglu_down_fp8_workspace_bytes": ([_i64, _i64, _i64, _int], _sz),
    "swiglu_pack_weights": ([_vp, _vp, _vp, _i64, _i64, _int, _vp], _int),
    "swiglu_up_packed": ([_vp, _vp, _vp, _i64, _i64, _i64, _int, _int, _vp, _sz, _vp], _int),
    "swiglu_mlp": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _int, _vp], _int),
    "swiglu_down_plan": ([_i64, _i64, _i64, _int, _int, _int, ctypes.POINTER(PlanInfo)], _int),
    "swiglu_workspace_bytes": ([_i64, _i64, _i64, _int, _int], _sz),
    "swiglu_plan": ([_i64, _i64, _i64, _int, _int, _int, ctypes.POINTER(PlanInfo)], _int),
    "swiglu_split_k_slices": ([_i64, _i64, _i64, _i64], _i64),
    "swiglu_check_device_status": ([], _int),
    "swiglu_release_stream_workspace": ([_vp], _int),
    "swiglu_release_workspaces": ([], _int),
    "swiglu_cached_workspace_bytes": ([], _sz),
    "swiglu_selftest_wait_timeout": ([_int, _vp], _int),
    "swiglu_status_string": ([_int], ctypes.c_char_p),
    "swiglu_last_error_string": ([], ctypes.c_char_p),
    "swiglu_version": ([], _int),
}

_lib = None
_lock = threading.Lock()


def load():
    """Load the library once; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    "CUDA library %s is missing: build it with "
                    "`python -m swiglu_mlp_projection_gb300.build`" % LIB_PATH)
            lib = ctypes.CDLL(LIB_PATH)
            for name, (argtypes, restype) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.argtypes = argtypes
                fn.restype = restype
            _lib = lib
    return _lib


class SwiGLUError(RuntimeError):
    def __init__(self, status, detail):
        self.status = status
        name = STATUS_NAMES.get(status, str(status))
        super().__init__("%s: %s" % (name, detail))


def check(status):
    if status != OK:
        lib = load()
        raise SwiGLUError(status, lib.swiglu_last_error_string().decode(errors="replace"))
