"""Seeded synthetic splat scenes: the inputs both the oracle and the CUDA path consume.

This module only draws random inputs. It holds none of the rasterizer's
arithmetic (no binning, compositing or gradients), so the oracle under
``oracle/`` and the CUDA library can both be fed from it without sharing
any of the method.

Random numbers come from a counter-based generator written here from its
published definition: SplitMix64 (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), applied to
``key + (i + 1) * 0x9E3779B97F4A7C15`` for draw ``i`` of a stream. Every
field of a scene has its own stream key, so the value of splat ``i`` does not
depend on how many splats are drawn, on numpy's version, or on the machine.
Normals use the Box-Muller transform.

Scene recipe (the five workloads of the splat-rasterization benchmark; the
pages describe 2D splats given as mean, conic, opacity, RGB and depth on an
image cut into 16x16 tiles):

* mean2d ~ U[0,W) x U[0,H) (workload 5: 30 % of splats drawn instead from
  one of 4 Gaussian blobs of sigma 60 px whose centres are
  U[0.2W,0.8W] x U[0.2H,0.8H]);
* theta ~ U[0, pi); two scales s1, s2 drawn independently log-uniform over
  the workload's range;
* conic = inverse of R(theta) diag(s1^2, s2^2) R(theta)^T, formed in double
  and stored as float32 (a, b, c) = upper triangle of the symmetric inverse;
* opacity, RGB, depth uniform over the workload's ranges;
* dL/dimage ~ N(0, sigma^2) with sigma the standard deviation;
* dL/ddistortion per pixel ~ N(0, (sigma / dz^2)^2), dz the width of the depth
  range, so that the distortion's gradients have the colour's scale;
* background black.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function (Steele, Lea & Flood 2014)."""
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def stream_key(seed: int, workload: int, field: int) -> np.uint64:
    """Key of one stream: the SplitMix64 mix of (seed, workload, field)."""
    with np.errstate(over="ignore"):
        base = np.array([(seed * 0x100000001B3 + workload * 0x1000193 + field * 0x9E37 + 1)
                         & 0xFFFFFFFFFFFFFFFF], dtype=np.uint64)
        return _mix64(_mix64(base))[0]


def uniform01(key: np.uint64, n: int, offset: int = 0) -> np.ndarray:
    """n float64 draws in [0, 1) from stream ``key``, draws offset..offset+n-1."""
    with np.errstate(over="ignore"):
        i = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
        z = _mix64(key + i * _GOLDEN)
    return (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def normal(key: np.uint64, n: int, std: float) -> np.ndarray:
    """n draws of N(0, std^2) by Box-Muller from two halves of stream ``key``."""
    u1 = 1.0 - uniform01(key, n, 0)          # (0, 1]
    u2 = uniform01(key, n, 1 << 40)
    return std * np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)


@dataclasses.dataclass
class Workload:
    name: str
    W: int
    H: int
    n: int
    scale: tuple          # (lo, hi) px, log-uniform, per axis
    opacity: tuple        # (lo, hi)
    depth: tuple          # (lo, hi)
    grad_std: float       # std of dL/dimage
    accum_weight: bool
    median_depth: bool
    blobs: int = 0        # number of Gaussian position blobs
    blob_frac: float = 0.0
    blob_sigma: float = 0.0
    weight_stats: bool = False   # per-splat max blend weight and blend count
    distortion: bool = False     # per-pixel depth distortion and its gradient


# The six workloads; index 1..6 (6 = workload 4 with the distortion output).
WORKLOADS = {
    1: Workload("tiny-64x64-256", 64, 64, 256, (0.5, 4.0), (0.05, 0.99), (1.0, 10.0), 1.0,
                True, False, weight_stats=True),
    2: Workload("256x256-5207", 256, 256, 5207, (0.5, 6.0), (0.05, 0.99), (1.0, 10.0), 0.1,
                True, False),
    3: Workload("1237x822-76363", 1237, 822, 76363, (0.3, 8.0), (0.05, 0.99), (1.0, 50.0), 0.1,
                True, False, weight_stats=True),
    4: Workload("1237x822-2M", 1237, 822, 2_000_000, (0.3, 3.0), (0.02, 0.9), (1.0, 100.0), 0.1,
                True, False),
    5: Workload("1920x1080-2M-blobs", 1920, 1080, 2_000_000, (0.3, 4.0), (0.02, 0.9),
                (1.0, 100.0), 0.1, True, True, blobs=4, blob_frac=0.3, blob_sigma=60.0,
                weight_stats=True),
    6: Workload("1237x822-2M-dist", 1237, 822, 2_000_000, (0.3, 3.0), (0.02, 0.9), (1.0, 100.0),
                0.1, True, False, distortion=True),
}


@dataclasses.dataclass
class Scene:
    W: int
    H: int
    mean2d: np.ndarray      # f32 [n][2]
    conic: np.ndarray       # f32 [n][3]  (a, b, c) of [[a, b], [b, c]]
    opacity: np.ndarray     # f32 [n]
    rgb: np.ndarray         # f32 [n][3]
    depth: np.ndarray       # f32 [n]
    dL_dimage: np.ndarray   # f32 [3][H][W]
    bg: np.ndarray          # f32 [3]
    accum_weight: bool
    median_depth: bool
    name: str = ""
    weight_stats: bool = False
    distortion: bool = False
    dL_ddist: np.ndarray | None = None   # f32 [H][W]

    @property
    def n(self) -> int:
        return int(self.opacity.shape[0])


def conic_from_scales(theta: np.ndarray, s1: np.ndarray, s2: np.ndarray) -> np.ndarray:
    """(a, b, c) of R diag(1/s1^2, 1/s2^2) R^T, the inverse of R diag(s^2) R^T, in double."""
    ct, st = np.cos(theta), np.sin(theta)
    i1, i2 = 1.0 / (s1 * s1), 1.0 / (s2 * s2)
    a = ct * ct * i1 + st * st * i2
    b = ct * st * (i1 - i2)
    c = st * st * i1 + ct * ct * i2
    return np.stack([a, b, c], axis=1)


def make_scene(workload: int | Workload, seed: int = 0, n: int | None = None,
               W: int | None = None, H: int | None = None) -> Scene:
    """Draw one scene. ``n``, ``W``, ``H`` override the workload's sizes."""
    wl = WORKLOADS[workload] if isinstance(workload, int) else workload
    wid = workload if isinstance(workload, int) else 0
    n = wl.n if n is None else n
    W = wl.W if W is None else W
    H = wl.H if H is None else H
    k = lambda f: stream_key(seed, wid, f)  # noqa: E731

    mx = uniform01(k(1), n) * W
    my = uniform01(k(2), n) * H
    if wl.blobs:
        cx = (0.2 + 0.6 * uniform01(k(20), wl.blobs)) * W
        cy = (0.2 + 0.6 * uniform01(k(21), wl.blobs)) * H
        in_blob = uniform01(k(22), n) < wl.blob_frac
        which = np.minimum((uniform01(k(23), n) * wl.blobs).astype(np.int64), wl.blobs - 1)
        bx = cx[which] + normal(k(24), n, wl.blob_sigma)
        by = cy[which] + normal(k(25), n, wl.blob_sigma)
        mx = np.where(in_blob, bx, mx)
        my = np.where(in_blob, by, my)
    theta = uniform01(k(3), n) * math.pi
    lo, hi = math.log(wl.scale[0]), math.log(wl.scale[1])
    s1 = np.exp(lo + (hi - lo) * uniform01(k(4), n))
    s2 = np.exp(lo + (hi - lo) * uniform01(k(5), n))
    conic = conic_from_scales(theta, s1, s2)
    opacity = wl.opacity[0] + (wl.opacity[1] - wl.opacity[0]) * uniform01(k(6), n)
    rgb = uniform01(k(7), 3 * n).reshape(n, 3)
    depth = wl.depth[0] + (wl.depth[1] - wl.depth[0]) * uniform01(k(8), n)
    dL = normal(k(9), 3 * H * W, wl.grad_std).reshape(3, H, W)
    dz = wl.depth[1] - wl.depth[0]
    dLd = normal(k(14), H * W, wl.grad_std / (dz * dz)).reshape(H, W)
    f32 = lambda x: np.ascontiguousarray(x, dtype=np.float32)  # noqa: E731
    return Scene(W=W, H=H,
                 mean2d=f32(np.stack([mx, my], axis=1)), conic=f32(conic), opacity=f32(opacity),
                 rgb=f32(rgb), depth=f32(depth), dL_dimage=f32(dL),
                 bg=np.zeros(3, np.float32), accum_weight=wl.accum_weight,
                 median_depth=wl.median_depth, name=wl.name, weight_stats=wl.weight_stats,
                 distortion=wl.distortion, dL_ddist=f32(dLd))


def subset(scene: Scene, idx: np.ndarray) -> Scene:
    """The scene restricted to splats ``idx`` (same image and upstream gradient)."""
    return dataclasses.replace(scene, mean2d=scene.mean2d[idx].copy(), conic=scene.conic[idx].copy(),
                               opacity=scene.opacity[idx].copy(), rgb=scene.rgb[idx].copy(),
                               depth=scene.depth[idx].copy())
