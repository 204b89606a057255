"""ctypes loader of libtopkp.so and its C signatures (include/topkp.h).

The library is built in-tree by ``top_logit_filter_gb300.build``; importing
this module never falls back to anything else: a missing or unloadable
library raises immediately.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libtopkp.so")

TOPKP_F32, TOPKP_F16, TOPKP_BF16 = 0, 1, 2
TOPKP_SUCCESS = 0
TOPKP_ERR_PARAM_NULLPTR = 161001
TOPKP_ERR_PARAM_INVALID = 161002
TOPKP_ERR_LAUNCH = 561000
TOPKP_ERR_DEVICE_TIMEOUT = 561001
TOPKP_ERR_NO_MEMORY = 561002
TOPKP_MAX_V = 1 << 23

# every entry point declared in include/topkp.h
EXPORTS = ("topkp_apply", "topkp_apply_sample", "topkp_apply_sorted", "topkp_sample", "topkp_sample_v2", "topkp_sample_v2_workspace_size",
           "topkp_sort", "topkp_sort_workspace_size", "topkp_sort_static", "topkp_last_error_string",
           "topkp_device_status", "topkp_last_launch_count")

_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads (once) and returns the library with argument types declared."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libtopkp.so is not built ({path}); run python -m top_logit_filter_gb300.build")
    lib = ctypes.CDLL(path)
    vp, i64, i32p, c_int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p, ctypes.c_int
    lib.topkp_apply.argtypes = [vp, i64, i64, i64, c_int, vp, i32p, vp, i64, vp]
    lib.topkp_apply.restype = c_int
    lib.topkp_apply_sample.argtypes = [vp, i64, i64, i64, c_int, vp, i32p, vp, vp, i64, ctypes.c_float, vp, i64, vp,
                                       vp]
    lib.topkp_apply_sample.restype = c_int
    lib.topkp_apply_sorted.argtypes = [vp, i32p, i64, i64, c_int, vp, i32p, vp, vp, vp]
    lib.topkp_apply_sorted.restype = c_int
    lib.topkp_sample.argtypes = [vp, i64, i64, i64, c_int, vp, vp, i64, ctypes.c_float, vp, i64, vp, vp]
    lib.topkp_sample.restype = c_int
    lib.topkp_sample_v2_workspace_size.argtypes = [i64, i64, c_int]
    lib.topkp_sample_v2_workspace_size.restype = ctypes.c_size_t
    lib.topkp_sample_v2.argtypes = [vp, i64, i64, i64, c_int, vp, vp, vp, vp, i64, ctypes.c_float, ctypes.c_int32,
                                    ctypes.c_int32, vp, i64, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.topkp_sample_v2.restype = c_int
    lib.topkp_sort_workspace_size.argtypes = [i64, i64, c_int]
    lib.topkp_sort_workspace_size.restype = ctypes.c_size_t
    lib.topkp_sort.argtypes = [vp, i64, i64, i64, c_int, vp, vp, vp, ctypes.c_size_t, vp]
    lib.topkp_sort.restype = c_int
    lib.topkp_sort_static.argtypes = [vp, i64, i64, i64, c_int, vp, vp, vp]
    lib.topkp_sort_static.restype = c_int
    lib.topkp_last_error_string.argtypes = []
    lib.topkp_last_error_string.restype = ctypes.c_char_p
    lib.topkp_device_status.argtypes = [vp]
    lib.topkp_device_status.restype = c_int
    lib.topkp_last_launch_count.argtypes = []
    lib.topkp_last_launch_count.restype = c_int
    _lib = lib
    return lib


def last_error() -> str:
    return load().topkp_last_error_string().decode()
