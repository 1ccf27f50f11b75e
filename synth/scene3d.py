"""Seeded synthetic 3D splat scenes and pinhole cameras for the projection step.

Like the rest of ``synth`` this only draws inputs: no projection, covariance,
spherical-harmonic or gradient arithmetic lives here. The camera rotation is
built by scipy from a drawn rotation vector; the point cloud is drawn in world
coordinates as a frustum-shaped cloud along +z around the origin, with the
camera near the origin and tilted by a small random rotation, so most splats
land in view and a few fall outside it or behind the camera.

Recipe (per splat, fp32 after drawing in double):

* depth along +z uniform over the workload's range; x and y uniform over
  1.1 x the half extent that a camera of the workload's focal length sees at
  that depth (so about 20 % of the cloud lies outside the image);
  ``behind_frac`` of the splats instead at z in [-3, -1.5] (behind the camera);
* three scales drawn independently so that each projects to a log-uniform
  0.3-3 px at its depth (s = px * z / f);
* rotation: four independent N(0, 1) draws, left unnormalised (the projection
  normalises);
* SH colour coefficients, stored coefficient-major [K][3][n] with
  K = (degree + 1)^2: the constant band U[-1.7, 1.7], the others N(0, 0.2^2);
* opacity U[0.02, 0.9] (passed through to the rasterizer unchanged);
* upstream gradients dL/dmean2d, dL/dconic, dL/drgb ~ N(0, 1);
* camera: fx = fy = W / (2 tan 30 deg), principal point at the image centre,
  world-to-camera rotation from a rotation vector with N(0, 0.06^2) components,
  translation N(0, 0.3^2) per axis, near plane 0.2, 2D blur 0.3.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
from scipy.spatial.transform import Rotation

from . import normal, stream_key, uniform01


@dataclasses.dataclass
class Workload3D:
    name: str
    W: int
    H: int
    n: int
    sh_degree: int
    depth: tuple = (1.0, 100.0)
    px_scale: tuple = (0.3, 3.0)
    behind_frac: float = 0.02


WORKLOADS3D = {
    11: Workload3D("proj-64x64-512", 64, 64, 512, 3),
    12: Workload3D("proj-1237x822-76363", 1237, 822, 76363, 3),
    13: Workload3D("proj-1237x822-2M", 1237, 822, 2_000_000, 3),
}


@dataclasses.dataclass
class Camera:
    R: np.ndarray        # f32 [3][3] world-to-camera rotation
    t: np.ndarray        # f32 [3]
    fx: float
    fy: float
    cx: float
    cy: float
    near: float
    blur: float


@dataclasses.dataclass
class Scene3D:
    W: int
    H: int
    mean3: np.ndarray     # f32 [n][3]
    scale: np.ndarray     # f32 [n][3]
    quat: np.ndarray      # f32 [n][4] (w, x, y, z), unnormalised
    sh: np.ndarray        # f32 [K][3][n]
    opacity: np.ndarray   # f32 [n]
    sh_degree: int
    cam: Camera
    dmean2d: np.ndarray   # f32 [n][2] upstream gradients
    dconic: np.ndarray    # f32 [n][3]
    drgb: np.ndarray      # f32 [n][3]
    name: str = ""

    @property
    def n(self) -> int:
        return int(self.opacity.shape[0])


def make_camera(W: int, H: int, seed: int = 0, wid: int = 0) -> Camera:
    k = lambda f: stream_key(seed, wid, f)  # noqa: E731
    f = W / (2.0 * math.tan(math.radians(30.0)))
    rotvec = normal(k(40), 3, 0.06)
    R = Rotation.from_rotvec(rotvec).as_matrix()
    t = normal(k(41), 3, 0.3)
    return Camera(R=np.ascontiguousarray(R, np.float32), t=np.ascontiguousarray(t, np.float32),
                  fx=float(np.float32(f)), fy=float(np.float32(f)), cx=float(np.float32(W / 2)),
                  cy=float(np.float32(H / 2)), near=0.2, blur=0.3)


def make_scene3d(workload: int | Workload3D, seed: int = 0, n: int | None = None,
                 W: int | None = None, H: int | None = None,
                 sh_degree: int | None = None) -> Scene3D:
    wl = WORKLOADS3D[workload] if isinstance(workload, int) else workload
    wid = workload if isinstance(workload, int) else 0
    n = wl.n if n is None else n
    W = wl.W if W is None else W
    H = wl.H if H is None else H
    deg = wl.sh_degree if sh_degree is None else sh_degree
    k = lambda f: stream_key(seed, wid, f)  # noqa: E731
    cam = make_camera(W, H, seed, wid)

    z = wl.depth[0] + (wl.depth[1] - wl.depth[0]) * uniform01(k(1), n)
    behind = uniform01(k(2), n) < wl.behind_frac
    z = np.where(behind, -3.0 + 1.5 * uniform01(k(3), n), z)
    zz = np.abs(z)
    x = (2.0 * uniform01(k(4), n) - 1.0) * 1.1 * zz * (W / 2) / cam.fx
    y = (2.0 * uniform01(k(5), n) - 1.0) * 1.1 * zz * (H / 2) / cam.fy
    lo, hi = math.log(wl.px_scale[0]), math.log(wl.px_scale[1])
    px = np.exp(lo + (hi - lo) * uniform01(k(6), 3 * n).reshape(n, 3))
    scale = px * (zz / cam.fx)[:, None]
    quat = normal(k(7), 4 * n, 1.0).reshape(n, 4)
    K = (deg + 1) ** 2
    sh = normal(k(8), K * 3 * n, 0.2).reshape(K, 3, n)
    sh[0] = -1.7 + 3.4 * uniform01(k(9), 3 * n).reshape(3, n)
    opacity = 0.02 + 0.88 * uniform01(k(10), n)
    f32 = lambda a: np.ascontiguousarray(a, dtype=np.float32)  # noqa: E731
    return Scene3D(W=W, H=H, mean3=f32(np.stack([x, y, z], axis=1)), scale=f32(scale),
                   quat=f32(quat), sh=f32(sh), opacity=f32(opacity), sh_degree=deg, cam=cam,
                   dmean2d=f32(normal(k(11), 2 * n, 1.0).reshape(n, 2)),
                   dconic=f32(normal(k(12), 3 * n, 1.0).reshape(n, 3)),
                   drgb=f32(normal(k(13), 3 * n, 1.0).reshape(n, 3)), name=wl.name)
