"""ctypes access to the C oracle in oracle.c.

TEST INFRASTRUCTURE ONLY: imported by tests/, by the smoke check in
__graft_entry__ and by the benchmark's CPU-baseline leg.  The product package
never imports it, and it imports nothing of the product package.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

TILE = 16
AMB_ALPHA, AMB_TERM, AMB_CLAMP, AMB_MEDIAN = 1, 2, 3, 4


def build(force: bool = False, defines: tuple = (), out: str | None = None) -> str:
    """Compile oracle.c with gcc (no FMA contraction) into a shared library."""
    out = out or _LIB_PATH
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= max(os.path.getmtime(_SRC),
                                             os.path.getmtime(os.path.join(_HERE, "oracle.h")))):
        return out
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           *["-D" + d for d in defines], "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class _SplatsF(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int64)] + [(k, ctypes.c_void_p) for k in
                                          ("mean2d", "conic", "opacity", "rgb", "depth")]


class _SplatsD(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int64)] + [(k, ctypes.c_void_p) for k in
                                          ("mean2d", "conic", "opacity", "rgb", "depth")]


class _Frame(ctypes.Structure):
    _fields_ = [("W", ctypes.c_int32), ("H", ctypes.c_int32), ("bg", ctypes.c_double * 3),
                ("vals", ctypes.c_void_p), ("offs", ctypes.c_void_p),
                ("tile_mask", ctypes.c_void_p), ("dL_ddist", ctypes.c_void_p)]


class _FwdOut(ctypes.Structure):
    _fields_ = [(k, ctypes.c_void_p) for k in ("image", "T_final", "last", "median", "n_amb",
                                               "max_w", "count", "splat_amb", "dist",
                                               "dist_err")]


class _Alt(ctypes.Structure):
    _fields_ = [("pixel", ctypes.c_int32), ("kind", ctypes.c_int32), ("list_pos", ctypes.c_int32),
                ("last", ctypes.c_uint32), ("image", ctypes.c_double * 3),
                ("T_final", ctypes.c_double), ("median", ctypes.c_double),
                ("dist", ctypes.c_double)]


class _Grads(ctypes.Structure):
    _fields_ = [(k, ctypes.c_void_p) for k in ("dmean2d", "dconic", "dopacity", "drgb", "accum",
                                               "ddepth")]


ALT_DTYPE = np.dtype([("pixel", "<i4"), ("kind", "<i4"), ("list_pos", "<i4"), ("last", "<u4"),
                      ("image", "<f8", (3,)), ("T_final", "<f8"), ("median", "<f8"),
                      ("dist", "<f8")])
assert ALT_DTYPE.itemsize == ctypes.sizeof(_Alt)


def load(path: str | None = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        # ORACLE_LIB points the tests at a deliberately broken copy of the
        # oracle (planted-mistake tests); unset, the real one is built.
        alt = os.environ.get("ORACLE_LIB")
        _lib = _bind(ctypes.CDLL(alt if alt else build()))
    return _lib


def _bind(lib):
    P = ctypes.POINTER
    lib.orc_constants.argtypes = [P(ctypes.c_double)]
    lib.orc_ln.argtypes = [ctypes.c_float]
    lib.orc_ln.restype = ctypes.c_float
    lib.orc_splat_rect.argtypes = [P(_SplatsF), ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                   P(ctypes.c_int32)]
    lib.orc_splat_rect.restype = ctypes.c_int
    lib.orc_bin.argtypes = [P(_SplatsF), ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p,
                            ctypes.c_void_p, ctypes.c_int64, P(ctypes.c_int64)]
    lib.orc_bin.restype = ctypes.c_int64
    lib.orc_sort.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64]
    lib.orc_offsets.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p]
    lib.orc_offsets.restype = ctypes.c_int
    lib.orc_forward.argtypes = [P(_SplatsD), P(_Frame), P(_FwdOut), ctypes.c_void_p,
                                ctypes.c_int64]
    lib.orc_forward.restype = ctypes.c_int64
    lib.orc_backward.argtypes = [P(_SplatsD), P(_Frame), ctypes.c_void_p, P(_Grads), P(_Grads),
                                 ctypes.c_void_p]
    lib.orc_backward.restype = ctypes.c_int
    return lib


def _p(a):
    return None if a is None else a.ctypes.data


def _splats_f(scene, keep):
    arrs = [np.ascontiguousarray(getattr(scene, k), np.float32)
            for k in ("mean2d", "conic", "opacity", "rgb", "depth")]
    keep.extend(arrs)
    return _SplatsF(scene.n, *[_p(a) for a in arrs])


def _splats_d(scene, params, keep):
    params = params or {}
    arrs = [np.ascontiguousarray(params.get(k, getattr(scene, k)), np.float64)
            for k in ("mean2d", "conic", "opacity", "rgb", "depth")]
    keep.extend(arrs)
    return _SplatsD(scene.n, *[_p(a) for a in arrs])


def constants() -> dict:
    buf = (ctypes.c_double * 4)()
    load().orc_constants(buf)
    return {"alpha_min": buf[0], "alpha_max": buf[1], "T_eps": buf[2], "tile": int(buf[3])}


def ln(x: float) -> float:
    return float(load().orc_ln(ctypes.c_float(x)))


def tiles_xy(W: int, H: int) -> tuple:
    return (W + TILE - 1) // TILE, (H + TILE - 1) // TILE


def splat_rect(scene, i: int):
    """(status, (x0, y0, x1, y1)) of splat i: -1 culled, 0 no tile, 1 rect."""
    keep = []
    s = _splats_f(scene, keep)
    r = (ctypes.c_int32 * 4)()
    v = load().orc_splat_rect(ctypes.byref(s), i, scene.W, scene.H, r)
    return v, tuple(r)


def bin_tiles(scene, capacity: int | None = None):
    """Pairs in emission order (splat, tile row, tile column): (keys, vals, count, culled)."""
    lib = load()
    keep = []
    s = _splats_f(scene, keep)
    culled = ctypes.c_int64(0)
    if capacity is None:
        capacity = lib.orc_bin(ctypes.byref(s), scene.W, scene.H, None, None, 0, None)
    keys = np.zeros(max(capacity, 1), np.uint64)
    vals = np.zeros(max(capacity, 1), np.uint32)
    count = lib.orc_bin(ctypes.byref(s), scene.W, scene.H, _p(keys), _p(vals), capacity,
                        ctypes.byref(culled))
    m = min(count, capacity)
    return keys[:m].copy(), vals[:m].copy(), int(count), int(culled.value)


def sort_pairs(keys, vals):
    k = np.ascontiguousarray(keys, np.uint64).copy()
    v = np.ascontiguousarray(vals, np.uint32).copy()
    load().orc_sort(_p(k), _p(v), k.size)
    return k, v


def offsets(keys, n_tiles: int):
    k = np.ascontiguousarray(keys, np.uint64)
    offs = np.zeros(n_tiles + 1, np.uint32)
    if load().orc_offsets(_p(k), k.size, n_tiles, _p(offs)) != 0:
        raise ValueError("tile id out of range")
    return offs


def tile_lists(scene):
    """bin -> sort -> offsets: dict(keys, vals, offs, count, culled)."""
    keys, vals, count, culled = bin_tiles(scene)
    keys, vals = sort_pairs(keys, vals)
    tx, ty = tiles_xy(scene.W, scene.H)
    return {"keys": keys, "vals": vals, "offs": offsets(keys, tx * ty), "count": count,
            "culled": culled}


def _frame(scene, vals, offs, tile_mask, bg, keep, dL_ddist=None):
    vals = np.ascontiguousarray(vals, np.uint32)
    offs = np.ascontiguousarray(offs, np.uint32)
    keep.extend([vals, offs])
    mask_p = None
    if tile_mask is not None:
        m = np.ascontiguousarray(tile_mask, np.uint8)
        keep.append(m)
        mask_p = _p(m)
    bgv = scene.bg if bg is None else bg
    dd = None
    if dL_ddist is not None:
        dd = np.ascontiguousarray(dL_ddist, np.float64)
        keep.append(dd)
    return _Frame(scene.W, scene.H, (ctypes.c_double * 3)(*[float(x) for x in bgv]),
                  _p(vals) if vals.size else None, _p(offs), mask_p, _p(dd))


def forward(scene, vals, offs, tile_mask=None, params=None, bg=None, alt_capacity=1 << 16):
    """Front-to-back compositing of every pixel of the (masked) tiles.

    Returns image [3][H][W], T_final, last, median, n_amb (knife-edge count per
    pixel), alts (structured array of alternative outcomes) and the per-splat
    max_w (max blend weight), count (blended pixels) and splat_amb (blended at
    a knife-edge pixel in some outcome), dist (the depth distortion per
    pixel) and dist_err (a bound on its float32 evaluation error)."""
    lib = load()
    keep = []
    s = _splats_d(scene, params, keep)
    f = _frame(scene, vals, offs, tile_mask, bg, keep)
    H, W = scene.H, scene.W
    res = {"image": np.zeros((3, H, W)), "T_final": np.ones((H, W)),
           "last": np.zeros((H, W), np.uint32), "median": np.zeros((H, W)),
           "n_amb": np.zeros((H, W), np.uint8), "max_w": np.zeros(scene.n),
           "count": np.zeros(scene.n, np.uint32), "splat_amb": np.zeros(scene.n, np.uint8),
           "dist": np.zeros((H, W)), "dist_err": np.zeros((H, W))}
    out = _FwdOut(*[_p(res[k]) for k in ("image", "T_final", "last", "median", "n_amb",
                                         "max_w", "count", "splat_amb", "dist", "dist_err")])
    alts = np.zeros(max(alt_capacity, 1), ALT_DTYPE)
    n_alt = lib.orc_forward(ctypes.byref(s), ctypes.byref(f), ctypes.byref(out), _p(alts),
                            alt_capacity)
    if n_alt > alt_capacity:
        raise RuntimeError("oracle alternative buffer too small: %d > %d" % (n_alt, alt_capacity))
    res["alts"] = alts[:n_alt].copy()
    return res


_GRAD_KEYS = ("dmean2d", "dconic", "dopacity", "drgb", "accum", "ddepth")


def _grads(n):
    return {"dmean2d": np.zeros((n, 2)), "dconic": np.zeros((n, 3)), "dopacity": np.zeros(n),
            "drgb": np.zeros((n, 3)), "accum": np.zeros(n), "ddepth": np.zeros(n)}


def backward(scene, vals, offs, tile_mask=None, params=None, bg=None, dL_dimage=None,
             slack=True, dL_ddist=None):
    """Per-splat gradients of L = sum dL/dimage * image (+ sum dL/ddist * dist
    when dL_ddist is given) from the masked tiles.

    Returns dict(grads=..., slack=... or None, accum_err=...)."""
    lib = load()
    keep = []
    s = _splats_d(scene, params, keep)
    f = _frame(scene, vals, offs, tile_mask, bg, keep, dL_ddist)
    g = np.ascontiguousarray(scene.dL_dimage if dL_dimage is None else dL_dimage, np.float64)
    keep.append(g)
    gr = _grads(scene.n)
    sl = _grads(scene.n) if slack else None
    aerr = np.zeros(scene.n)
    cg = _Grads(*[_p(gr[k]) for k in _GRAD_KEYS])
    cs = _Grads(*[_p(sl[k]) for k in _GRAD_KEYS]) if slack else None
    lib.orc_backward(ctypes.byref(s), ctypes.byref(f), _p(g), ctypes.byref(cg),
                     ctypes.byref(cs) if slack else None, _p(aerr))
    return {"grads": gr, "slack": sl, "accum_err": aerr}
