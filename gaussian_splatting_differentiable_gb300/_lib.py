"""ctypes prototypes of libss.so (the C ABI declared in include/ss.h,
include/ss_project.h and include/ss_ssim.h).

Loading fails with an ImportError when the library has not been built: there
is no fallback implementation behind this package.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libss.so")
# The same library built with device-side bounds checks (build.py
# --debug-bounds); SS_LIBRARY=<path> makes load() take it instead.
DEBUG_LIB_PATH = os.path.join(_HERE, "libss_debug.so")

SS_OK, SS_ERR_INVALID_ARG, SS_ERR_CAPACITY, SS_ERR_CUDA, SS_ERR_TIMEOUT, SS_ERR_UNSUPPORTED, \
    SS_ERR_DEVICE = range(7)
STATUS_NAMES = {0: "SS_OK", 1: "SS_ERR_INVALID_ARG", 2: "SS_ERR_CAPACITY", 3: "SS_ERR_CUDA",
                4: "SS_ERR_TIMEOUT", 5: "SS_ERR_UNSUPPORTED", 6: "SS_ERR_DEVICE"}
SS_ACCUM_WEIGHT = 1
SS_MEDIAN_DEPTH = 2
SS_WEIGHT_STATS = 4
SS_DISTORTION = 8
SS_RECORDS_CLEARED = 16   # bwd: the forward already cleared the gradient records


class SsSplats(ctypes.Structure):
    _fields_ = [("mean2d", ctypes.c_void_p), ("conic", ctypes.c_void_p),
                ("opacity", ctypes.c_void_p), ("rgb", ctypes.c_void_p),
                ("depth", ctypes.c_void_p), ("n", ctypes.c_int32)]


class SsGrads(ctypes.Structure):
    _fields_ = [("dmean2d", ctypes.c_void_p), ("dconic", ctypes.c_void_p),
                ("dopacity", ctypes.c_void_p), ("drgb", ctypes.c_void_p),
                ("ddepth", ctypes.c_void_p)]


class SsSplats3d(ctypes.Structure):
    _fields_ = [("mean3", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("quat", ctypes.c_void_p),
                ("sh", ctypes.c_void_p), ("n", ctypes.c_int32), ("sh_degree", ctypes.c_int32)]


class SsCamera(ctypes.Structure):
    _fields_ = [("R", ctypes.c_float * 9), ("t", ctypes.c_float * 3), ("fx", ctypes.c_float),
                ("fy", ctypes.c_float), ("cx", ctypes.c_float), ("cy", ctypes.c_float),
                ("near_z", ctypes.c_float), ("blur", ctypes.c_float)]


class SsGrads3d(ctypes.Structure):
    _fields_ = [("dmean3", ctypes.c_void_p), ("dscale", ctypes.c_void_p),
                ("dquat", ctypes.c_void_p), ("dsh", ctypes.c_void_p)]


# name -> (restype, argtypes), in the order of include/ss.h, ss_project.h, ss_ssim.h
P = ctypes.c_void_p
I32, I64, U32, SZ = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_size_t
PROTOTYPES = {
    "ss_abi_version": (I32, []),
    "ss_constants": (None, [P]),
    "ss_last_error": (ctypes.c_char_p, []),
    "ss_workspace_bytes": (SZ, [I32, I64, I32, I32]),
    "ss_bin_tiles": (ctypes.c_int, [ctypes.POINTER(SsSplats), I32, I32, P, P, I64, P, P, P]),
    "ss_record_bytes": (SZ, [I32]),
    "ss_pair_count": (ctypes.c_int, [P, I64, ctypes.POINTER(I64), ctypes.POINTER(I64), P]),
    "ss_sort_pairs": (ctypes.c_int, [P, P, I64, I32, I32, P, P, SZ, P]),
    "ss_sort_pairs_dev": (ctypes.c_int, [P, P, P, I64, I32, I32, P, P, SZ, P]),
    "ss_sort_status": (ctypes.c_int, [P, P]),
    "ss_raster_fwd": (ctypes.c_int, [ctypes.POINTER(SsSplats), P, P, I32, I32, P, U32, P, P, P,
                                     P, P]),
    "ss_raster_fwd_records": (ctypes.c_int, [P, I32, P, P, I64, I32, I32, P, U32, P, P, P, P, P,
                                             P, P, P, P, P, SZ, P]),
    "ss_raster_bwd": (ctypes.c_int, [ctypes.POINTER(SsSplats), P, P, I32, I32, P, U32, P, P, P,
                                     ctypes.POINTER(SsGrads), P, P, SZ, P]),
    "ss_raster_bwd_records": (ctypes.c_int, [P, I32, P, P, I64, I32, I32, P, U32, P, P, P, P, P,
                                             P, ctypes.POINTER(SsGrads), P, P, SZ, P]),
    "ss_raster_bwd_noalloc": (ctypes.c_int, [P, I32, P, P, I64, I32, I32, P, U32, P, P, P, P,
                                             ctypes.POINTER(SsGrads), P, P]),
    "ss_profile_enable": (None, [I32]),
    "ss_profile_collect": (I64, [ctypes.c_char_p, SZ]),
    "ss_debug_bounds_enabled": (I32, []),
    "ss_debug_status": (ctypes.c_int, [P]),
    "ss_probe_red_f32": (ctypes.c_int, [P, I64, I32, P]),
    "ss_test_sort_wait_timeout": (ctypes.c_int, [P, SZ, P]),
    "ss_project_fwd": (ctypes.c_int, [ctypes.POINTER(SsSplats3d), ctypes.POINTER(SsCamera), P, P,
                                      P, P, P]),
    "ss_project_bwd": (ctypes.c_int, [ctypes.POINTER(SsSplats3d), ctypes.POINTER(SsCamera), P, P,
                                      P, ctypes.POINTER(SsGrads3d), P]),
    "ss_ssim_workspace_bytes": (SZ, [I32, I32, I32]),
    "ss_ssim_loss": (ctypes.c_int, [P, P, I32, I32, I32, ctypes.c_float, P, P, P, SZ, P]),
}

_lib = None


def load(path: str | None = None):
    """The loaded library with prototypes set; ImportError if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or os.environ.get("SS_LIBRARY") or LIB_PATH
    if not os.path.exists(p):
        raise ImportError("libss.so is not built (%s); run "
                          "`python -c 'import __graft_entry__ as g; g.build()'`" % p)
    lib = ctypes.CDLL(p)
    for name, (res, args) in PROTOTYPES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    if path is None:
        _lib = lib
    return lib
