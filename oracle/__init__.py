"""ctypes access to the C oracle in oracle.c.

TEST INFRASTRUCTURE ONLY: imported by tests/, by the smoke check in
__graft_entry__ and by the benchmark's CPU-baseline leg.  The product package
never imports it, and it imports nothing of the product package.
"""
from __future__ import annotations

import concurrent.futures
import ctypes
import heapq
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
    lib.orc_margins.argtypes = [ctypes.c_double] * 6 + [P(ctypes.c_double)]
    lib.orc_margins.restype = None
    lib.orc_trace_pixel.argtypes = [P(_SplatsD), ctypes.c_void_p, ctypes.c_int64,
                                    ctypes.c_double, ctypes.c_double, ctypes.c_void_p,
                                    ctypes.c_int64, P(ctypes.c_double), P(ctypes.c_int32)]
    lib.orc_trace_pixel.restype = ctypes.c_int64
    lib.orc_margins_n.argtypes = [ctypes.c_int64] + [ctypes.c_void_p] * 8
    lib.orc_margins_n.restype = None
    return lib


TRACE_DTYPE = np.dtype([("pos", "<i8"), ("alpha", "<f8"), ("G", "<f8"), ("T", "<f8"),
                        ("mrel", "<f8"), ("relT", "<f8"), ("clamped", "<i4"), ("pad", "<i4")])
MAX_AMB = 8


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


def tile_parts(W: int, H: int, offs, tile_mask, parts: int) -> list:
    """The selected tiles split into at most `parts` disjoint tile masks of
    about equal work (a tile's pairs times its pixels, plus its pixels):
    tiles in decreasing order of work, each onto the lightest part so far.
    Only the partition is computed here; each part is an ordinary oracle
    call restricted to its tiles."""
    tx, ty = tiles_xy(W, H)
    T = tx * ty
    sel = np.ones(T, bool) if tile_mask is None else np.asarray(tile_mask).astype(bool)
    idx = np.nonzero(sel)[0]
    parts = max(1, min(int(parts), idx.size))
    per = np.diff(np.asarray(offs, np.int64))[idx]
    px = np.minimum(16, W - 16 * (idx % tx)) * np.minimum(16, H - 16 * (idx // tx))
    cost = (per + 1) * px
    heap = [(0, k) for k in range(parts)]
    masks = np.zeros((parts, T), np.uint8)
    for t in np.argsort(-cost, kind="stable"):
        load_k, k = heapq.heappop(heap)
        masks[k, idx[t]] = 1
        heapq.heappush(heap, (load_k + int(cost[t]), k))
    return [m for m in masks if m.any()] or [masks[0]]


def default_threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def forward(scene, vals, offs, tile_mask=None, params=None, bg=None, alt_capacity=1 << 16,
            threads: int = 1):
    """Front-to-back compositing of every pixel of the (masked) tiles.

    Returns image [3][H][W], T_final, last, median, n_amb (knife-edge count per
    pixel), alts (structured array of alternative outcomes) and the per-splat
    max_w (max blend weight), count (blended pixels) and splat_amb (blended at
    a knife-edge pixel in some outcome), dist (the depth distortion per
    pixel) and dist_err (a bound on its float32 evaluation error).

    threads > 1 splits the tiles into parts (tile_parts) run concurrently,
    one oracle call per part on its own thread (the C call releases the
    interpreter lock).  Pixels are computed by exactly the same code either
    way, so every per-pixel output is identical; the per-splat maximum,
    count and flag are combined exactly (max, integer sum, or); alternatives
    come out grouped by part."""
    lib = load()
    keep = []
    s = _splats_d(scene, params, keep)
    H, W = scene.H, scene.W
    res = {"image": np.zeros((3, H, W)), "T_final": np.ones((H, W)),
           "last": np.zeros((H, W), np.uint32), "median": np.zeros((H, W)),
           "n_amb": np.zeros((H, W), np.uint8), "max_w": np.zeros(scene.n),
           "count": np.zeros(scene.n, np.uint32), "splat_amb": np.zeros(scene.n, np.uint8),
           "dist": np.zeros((H, W)), "dist_err": np.zeros((H, W))}
    masks = [tile_mask] if threads <= 1 else tile_parts(W, H, offs, tile_mask, threads)

    def run(mask):
        # per-pixel arrays are shared (the parts' pixels are disjoint); the
        # per-splat ones are the part's own
        own = {"max_w": np.zeros(scene.n), "count": np.zeros(scene.n, np.uint32),
               "splat_amb": np.zeros(scene.n, np.uint8)}
        mine = []
        f = _frame(scene, vals, offs, mask, bg, mine)
        out = _FwdOut(*[_p(own[k] if k in own else res[k])
                        for k in ("image", "T_final", "last", "median", "n_amb", "max_w",
                                  "count", "splat_amb", "dist", "dist_err")])
        alts = np.zeros(max(alt_capacity, 1), ALT_DTYPE)
        n_alt = lib.orc_forward(ctypes.byref(s), ctypes.byref(f), ctypes.byref(out), _p(alts),
                                alt_capacity)
        if n_alt > alt_capacity:
            raise RuntimeError("oracle alternative buffer too small: %d > %d" %
                               (n_alt, alt_capacity))
        return own, alts[:n_alt].copy()

    if len(masks) == 1:
        outs = [run(masks[0])]
    else:
        with concurrent.futures.ThreadPoolExecutor(len(masks)) as ex:
            outs = list(ex.map(run, masks))
    for own, _ in outs:
        np.maximum(res["max_w"], own["max_w"], out=res["max_w"])
        res["count"] += own["count"]
        np.maximum(res["splat_amb"], own["splat_amb"], out=res["splat_amb"])
    res["alts"] = np.concatenate([a for _, a in outs]) if len(outs) > 1 else outs[0][1]
    return res


_GRAD_KEYS = ("dmean2d", "dconic", "dopacity", "drgb", "accum", "ddepth")


def _grads(n):
    return {"dmean2d": np.zeros((n, 2)), "dconic": np.zeros((n, 3)), "dopacity": np.zeros(n),
            "drgb": np.zeros((n, 3)), "accum": np.zeros(n), "ddepth": np.zeros(n)}


def backward_sums(n: int, parts: int, slack: bool = True) -> list:
    """Zeroed per-part accumulators for backward(..., into=...)."""
    return [(_grads(n), _grads(n) if slack else None, np.zeros(n)) for _ in range(parts)]


def add_backward_sums(sums: list) -> dict:
    """backward()'s result from per-part accumulators: their sum in part order."""
    gr, sl, aerr = (_grads(sums[0][2].size), _grads(sums[0][2].size) if sums[0][1] else None,
                    np.zeros(sums[0][2].size))
    for g2, s2, a2 in sums:
        for k in _GRAD_KEYS:
            gr[k] += g2[k]
            if sl is not None:
                sl[k] += s2[k]
        aerr += a2
    return {"grads": gr, "slack": sl, "accum_err": aerr}


def backward(scene, vals, offs, tile_mask=None, params=None, bg=None, dL_dimage=None,
             slack=True, dL_ddist=None, threads: int = 1, into=None):
    """Per-splat gradients of L = sum dL/dimage * image (+ sum dL/ddist * dist
    when dL_ddist is given) from the masked tiles.

    threads > 1 splits the tiles into parts (tile_parts), one oracle call per
    part on its own thread, each into its own per-splat buffers, which are
    then added in part order (the oracle's per-tile contributions are
    additive; only the order of the double-precision sums differs).
    into: per-part accumulators (backward_sums(n, threads, slack)) that the
    parts add into instead; nothing is returned then (add_backward_sums
    gives the result), so that several calls on disjoint tiles share them.

    Returns dict(grads=..., slack=... or None, accum_err=...)."""
    lib = load()
    keep = []
    s = _splats_d(scene, params, keep)
    g = np.ascontiguousarray(scene.dL_dimage if dL_dimage is None else dL_dimage, np.float64)
    keep.append(g)
    masks = [tile_mask] if threads <= 1 else tile_parts(scene.W, scene.H, offs, tile_mask,
                                                        threads)
    sums = into if into is not None else backward_sums(scene.n, len(masks), slack)
    if len(sums) < len(masks):
        raise ValueError("%d accumulators for %d parts" % (len(sums), len(masks)))

    def run(j):
        mine = []
        f = _frame(scene, vals, offs, masks[j], bg, mine, dL_ddist)
        gr, sl, aerr = sums[j]
        cg = _Grads(*[_p(gr[k]) for k in _GRAD_KEYS])
        cs = _Grads(*[_p(sl[k]) for k in _GRAD_KEYS]) if slack else None
        lib.orc_backward(ctypes.byref(s), ctypes.byref(f), _p(g), ctypes.byref(cg),
                         ctypes.byref(cs) if slack else None, _p(aerr))

    if len(masks) == 1:
        run(0)
    else:
        with concurrent.futures.ThreadPoolExecutor(len(masks)) as ex:
            list(ex.map(run, range(len(masks))))
    if into is not None:
        return None
    if len(sums) == 1:
        gr, sl, aerr = sums[0]
        return {"grads": gr, "slack": sl, "accum_err": aerr}
    return add_backward_sums(sums[:len(masks)])


def margins(a, b, c, dx, dy, o):
    """(skip margin, value margin) of the knife-edge model at one (pixel,
    splat): relative bounds on a float32 evaluation's alpha-floor decision
    and on its alpha."""
    out = (ctypes.c_double * 2)()
    load().orc_margins(float(a), float(b), float(c), float(dx), float(dy), float(o), out)
    return out[0], out[1]


def margins_n(a, b, c, dx, dy, o):
    """margins() over arrays: (skip margins, value margins)."""
    arrs = [np.ascontiguousarray(np.broadcast_to(np.asarray(v, np.float64), np.shape(a)))
            for v in (a, b, c, dx, dy, o)]
    n = arrs[0].size
    skip, val = np.zeros(n), np.zeros(n)
    load().orc_margins_n(n, *[_p(v) for v in arrs], _p(skip), _p(val))
    return skip.reshape(np.shape(a)), val.reshape(np.shape(a))


def trace_pixel(scene, vals, offs, x: int, y: int, params=None):
    """The oracle's compositing of pixel (x, y) over its tile's list, with the
    error bounds of its knife-edge decisions: dict(rec = blended splats
    (TRACE_DTYPE), T_final, relT, last, n_amb, amb = [(list position, kind)])."""
    lib = load()
    keep = []
    s = _splats_d(scene, params, keep)
    tx, _ = tiles_xy(scene.W, scene.H)
    t = (y // TILE) * tx + x // TILE
    offs = np.asarray(offs, np.int64)
    lst = np.ascontiguousarray(np.asarray(vals, np.uint32)[offs[t]:offs[t + 1]])
    rec = np.zeros(max(lst.size, 1), TRACE_DTYPE)
    tail = (ctypes.c_double * 4)()
    amb = (ctypes.c_int32 * (2 * MAX_AMB))()
    n = lib.orc_trace_pixel(ctypes.byref(s), _p(lst) if lst.size else None, lst.size, x + 0.5,
                            y + 0.5, _p(rec), rec.size, tail, amb)
    na = min(int(tail[3]), MAX_AMB)
    return {"rec": rec[:n].copy(), "T_final": tail[0], "relT": tail[1], "last": int(tail[2]),
            "n_amb": int(tail[3]), "amb": [(amb[2 * j], amb[2 * j + 1]) for j in range(na)],
            "list": lst}
