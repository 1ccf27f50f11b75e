"""Pins of the projection oracle (oracle/project.py) to things other than itself.

* the SH basis against scipy's complex spherical harmonics (converted to the
  real, no-Condon-Shortley basis), its orthonormality by exact quadrature and
  the addition theorem;
* the quaternion rotation against the Hamilton product q v q* and scipy;
* the pixel position against homogeneous coordinates K [R | t] p;
* the 2D covariance against the Jacobian of the world-to-pixel map taken by
  central differences, with the 3D covariance built by scipy;
* the colour against the scipy basis with the direction from the camera
  centre; the clamp; culling; the blur term;
* the backward against central differences of L in float64.

A planted-mistake test at the end shows that plausible slips in
oracle/project.py fail at least one pin.
"""
import math
import pathlib
import types

import numpy as np
import pytest

import synth
from synth.scene3d import Camera, make_scene3d

special = pytest.importorskip("scipy.special")
from scipy.spatial.transform import Rotation  # noqa: E402

import oracle.project as OP  # noqa: E402

torch = pytest.importorskip("torch")


def _dirs(n, seed):
    v = np.random.default_rng(seed).normal(size=(n, 3))
    return v / np.linalg.norm(v, axis=1, keepdims=True)


def _real_sh_scipy(deg, d):
    """Real SH from scipy's complex ones (which carry the Condon-Shortley
    phase): sqrt(2) (-1)^m Re Y_l^m for m > 0, sqrt(2) (-1)^m Im Y_l^|m| for
    m < 0, Y_l^0 for m = 0."""
    theta = np.arccos(np.clip(d[:, 2], -1, 1))
    phi = np.arctan2(d[:, 1], d[:, 0])
    out = np.zeros((d.shape[0], (deg + 1) ** 2))
    for l in range(deg + 1):
        for m in range(-l, l + 1):
            Y = special.sph_harm_y(l, abs(m), theta, phi)
            if m > 0:
                v = math.sqrt(2) * (-1) ** m * Y.real
            elif m < 0:
                v = math.sqrt(2) * (-1) ** m * Y.imag
            else:
                v = Y.real
            out[:, l * l + l + m] = v
    return out


def _scene(n=12, deg=3, seed=3, W=64, H=48):
    return make_scene3d(11, seed=seed, n=n, W=W, H=H, sh_degree=deg)


def _cam_simple(R=None, t=(0.0, 0.0, 0.0), f=(50.0, 60.0), c=(32.0, 24.0), blur=0.3):
    return Camera(R=np.eye(3, dtype=np.float32) if R is None else np.asarray(R, np.float32),
                  t=np.asarray(t, np.float32), fx=f[0], fy=f[1], cx=c[0], cy=c[1], near=0.2,
                  blur=blur)


# ------------------------------------------------------------------ pins

def pin_sh_scipy(P):
    d = _dirs(200, 1)
    got = P.sh_basis(3, torch.as_tensor(d)).numpy()
    assert np.allclose(got, _real_sh_scipy(3, d), atol=1e-12, rtol=0), "SH vs scipy"


def pin_sh_orthonormal(P):
    zs, wz = np.polynomial.legendre.leggauss(8)          # exact to degree 15 in z
    phis = 2 * math.pi * np.arange(16) / 16               # exact for trig degree < 16
    Z, PH = np.meshgrid(zs, phis, indexing="ij")
    r = np.sqrt(1 - Z ** 2)
    d = np.stack([r * np.cos(PH), r * np.sin(PH), Z], -1).reshape(-1, 3)
    w = (np.repeat(wz, 16) * (2 * math.pi / 16))
    Y = P.sh_basis(3, torch.as_tensor(d)).numpy()
    G = (Y * w[:, None]).T @ Y
    assert np.allclose(G, np.eye(16), atol=1e-12), "SH Gram matrix"
    for l in range(4):                                      # addition theorem
        s = (Y[:, l * l:(l + 1) ** 2] ** 2).sum(1)
        assert np.allclose(s, (2 * l + 1) / (4 * math.pi), atol=1e-12)


def pin_quaternion(P):
    rng = np.random.default_rng(2)
    q = rng.normal(size=(50, 4))
    R = P.quat_rotmat(torch.as_tensor(q)).numpy()
    u = q / np.linalg.norm(q, axis=1, keepdims=True)

    def ham(a, b):
        w1, x1, y1, z1 = a.T
        w2, x2, y2, z2 = b.T
        return np.stack([w1 * w2 - x1 * x2 - y1 * y2 - z1 * z2,
                         w1 * x2 + x1 * w2 + y1 * z2 - z1 * y2,
                         w1 * y2 - x1 * z2 + y1 * w2 + z1 * x2,
                         w1 * z2 + x1 * y2 - y1 * x2 + z1 * w2], 1)
    v = rng.normal(size=(50, 3))
    conj = u * np.array([1, -1, -1, -1])
    rot = ham(ham(u, np.concatenate([np.zeros((50, 1)), v], 1)), conj)[:, 1:]
    assert np.allclose(np.einsum("nij,nj->ni", R, v), rot, atol=1e-12), "R(q) v != q v q*"
    ref = Rotation.from_quat(u[:, [1, 2, 3, 0]]).as_matrix()   # scipy: scalar last
    assert np.allclose(R, ref, atol=1e-12)
    assert np.allclose(P.quat_rotmat(torch.as_tensor(3.7 * q)).numpy(), R, atol=1e-12)


def _world_to_pixel(cam, p):
    K = np.array([[cam.fx, 0, cam.cx], [0, cam.fy, cam.cy], [0, 0, 1.0]])
    Rt = np.concatenate([np.asarray(cam.R, np.float64), np.asarray(cam.t, np.float64)[:, None]], 1)
    h = (K @ Rt @ np.concatenate([p, np.ones((p.shape[0], 1))], 1).T).T
    return h[:, :2] / h[:, 2:3]


def pin_mean_homogeneous(P):
    sc = _scene(n=40, seed=4)
    f = P.project(sc)
    v = f["valid"]
    ref = _world_to_pixel(sc.cam, sc.mean3.astype(np.float64))
    assert np.allclose(f["mean2d"][v], ref[v], rtol=1e-12, atol=1e-9)
    zc = sc.mean3.astype(np.float64) @ np.asarray(sc.cam.R, np.float64).T + sc.cam.t
    assert np.allclose(f["depth"][v], zc[v, 2], rtol=1e-12)


def pin_cov2_linearised(P):
    sc = _scene(n=40, seed=5)
    sc.cam.fy = 1.25 * sc.cam.fx                   # distinct focal lengths
    f = P.project(sc)
    v = f["valid"]
    p = sc.mean3.astype(np.float64)
    Jw = np.zeros((sc.n, 2, 3))
    for k in range(3):
        h = 1e-5 * np.maximum(1, np.abs(p[:, k]))
        e = np.zeros(3)
        e[k] = 1
        Jw[:, :, k] = (_world_to_pixel(sc.cam, p + h[:, None] * e)
                       - _world_to_pixel(sc.cam, p - h[:, None] * e)) / (2 * h[:, None])
    q = sc.quat.astype(np.float64)
    Rq = Rotation.from_quat(q[:, [1, 2, 3, 0]]).as_matrix()
    s2 = sc.scale.astype(np.float64) ** 2
    cov3 = np.einsum("nij,nj,nkj->nik", Rq, s2, Rq)
    cov2 = np.einsum("nij,njk,nlk->nil", Jw, cov3, Jw) + sc.cam.blur * np.eye(2)
    assert np.allclose(f["cov2"][v], cov2[v], rtol=1e-6, atol=0), "2D covariance"
    inv = np.linalg.inv(cov2)
    conic = np.stack([inv[:, 0, 0], inv[:, 0, 1], inv[:, 1, 1]], 1)
    assert np.allclose(f["conic"][v], conic[v], rtol=1e-5, atol=0), "conic"


def pin_blur(P):
    sc = _scene(n=30, seed=6)
    a = P.project(sc)
    sc.cam.blur = 0.0
    b = P.project(sc)
    v = a["valid"] & b["valid"]
    d = a["cov2"][v] - b["cov2"][v]
    assert np.allclose(d, 0.3 * np.eye(2), atol=1e-9)


def pin_colour(P):
    sc = _scene(n=60, seed=7, deg=3)
    R = Rotation.from_rotvec([0.3, -0.2, 0.5]).as_matrix().astype(np.float32)
    sc.cam = _cam_simple(R=R, t=[0.4, -0.7, 0.2])
    sc.mean3[:, 2] = np.abs(sc.mean3[:, 2]) + 2.0
    f = P.project(sc)
    c = -(R.astype(np.float64).T @ np.float32([0.4, -0.7, 0.2]).astype(np.float64))
    d = sc.mean3.astype(np.float64) - c
    d /= np.linalg.norm(d, axis=1, keepdims=True)
    Y = _real_sh_scipy(3, d)
    raw = np.einsum("kcn,nk->nc", sc.sh.astype(np.float64), Y) + 0.5
    v = f["valid"]
    assert np.allclose(f["rgb"][v], np.maximum(raw[v], 0), atol=1e-12), "colour"
    assert (raw[v] < 0).any(), "no clamped channel in the pin's scene"


def pin_culling(P):
    sc = _scene(n=8, seed=8)
    sc.cam = _cam_simple()
    sc.mean3[:] = np.float32([0.1, 0.1, 5.0])
    sc.mean3[1] = np.float32([0.1, 0.1, 0.19])    # inside the near plane
    sc.mean3[2] = np.float32([0.1, 0.1, -3.0])    # behind
    sc.quat[3] = 0.0                              # no rotation defined
    f = P.project(sc)
    assert f["valid"].tolist() == [True, False, False, False, True, True, True, True]
    for k in ("mean2d", "conic", "depth", "rgb"):
        assert not np.any(f[k][~f["valid"]])
    g = P.project_backward(sc)
    for k in ("dmean3", "dscale", "dquat"):
        assert not np.any(g[k][~f["valid"]])
    assert not np.any(g["dsh"][:, :, ~f["valid"]])


def pin_backward_fd(P):
    sc = _scene(n=10, seed=9)
    sc.mean3[:, 2] = np.abs(sc.mean3[:, 2]) + 1.0
    sc.sh[0, 0, :3] = -2.5                         # clamped red for three splats
    g = P.project_backward(sc)
    names = {"mean3": "dmean3", "scale": "dscale", "quat": "dquat", "sh": "dsh"}
    for field, gname in names.items():
        base = getattr(sc, field).astype(np.float64)
        num = np.zeros_like(base)
        flat = base.reshape(-1)
        for i in range(flat.size):
            h = 1e-6 * max(1.0, abs(flat[i]))
            plus, minus = flat.copy(), flat.copy()
            plus[i] += h
            minus[i] -= h
            lp = P.loss(sc, params={field: plus.reshape(base.shape)})
            lm = P.loss(sc, params={field: minus.reshape(base.shape)})
            num.reshape(-1)[i] = (lp - lm) / (2 * h)
        an = g[gname]
        scale = np.abs(num).max()
        assert np.allclose(an, num, atol=1e-6 * scale + 1e-9, rtol=1e-5), (
            field, np.abs(an - num).max(), scale)


PINS = [pin_sh_scipy, pin_sh_orthonormal, pin_quaternion, pin_mean_homogeneous,
        pin_cov2_linearised, pin_blur, pin_colour, pin_culling, pin_backward_fd]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(OP)


def test_workload_recipe_sane():
    sc = make_scene3d(12, seed=0, n=20000)
    f = OP.project(sc)
    v = f["valid"]
    assert 0.95 < v.mean() < 0.995                  # ~2 % behind the camera
    inside = v & (f["mean2d"][:, 0] >= 0) & (f["mean2d"][:, 0] < sc.W) & \
        (f["mean2d"][:, 1] >= 0) & (f["mean2d"][:, 1] < sc.H)
    assert 0.6 < inside.mean() < 0.95
    sd = 1.0 / np.sqrt(np.abs(f["conic"][v][:, [0, 2]]))
    assert 0.2 < np.median(sd) < 4.0                # a few pixels wide
    assert synth.WORKLOADS[4].W == sc.W


# ------------------------------------------------------------------ planted mistakes

MUTATIONS = [
    ("camera rotation transposed", "pc = mean3 @ R.T + t", "pc = mean3 @ R + t"),
    ("Jacobian x/z^2 sign", "J[:, 0, 2] = -fx * x / (z * z)", "J[:, 0, 2] = fx * x / (z * z)"),
    ("quaternion not normalised", "u = q / q.norm(dim=1, keepdim=True)", "u = q"),
    ("SH m<0 uses the real part", "out[l * l + l - m] = norm * q * powers[m][1]",
     "out[l * l + l - m] = norm * q * powers[m][0]"),
    ("blur dropped", " + float(cam.blur) * torch.eye(2, dtype=_D)", ""),
    ("camera centre = -t", "campos = -(R.T @ t)", "campos = -t"),
    ("clamp dropped", "rgb = torch.clamp(raw, min=0.0)", "rgb = raw"),
    ("conic b sign", "-cov2[:, 0, 1] / det", "cov2[:, 0, 1] / det"),
    ("scales on rows", "M = quat_rotmat(quat) * scale[:, None, :]",
     "M = quat_rotmat(quat) * scale[:, :, None]"),
    ("SH sqrt(2) dropped", "norm *= math.sqrt(2.0)", "norm *= 1.0"),
    ("cy replaced by cx", "fy * y / z + float(cam.cy)", "fy * y / z + float(cam.cx)"),
    ("Jacobian fy", "J[:, 1, 1] = fy / z", "J[:, 1, 1] = fx / z"),
]


def _mutant(old, new):
    src = pathlib.Path(OP.__file__).read_text()
    assert src.count(old) == 1, old
    mod = types.ModuleType("oracle_project_mutant")
    mod.__file__ = OP.__file__
    exec(compile(src.replace(old, new), OP.__file__, "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("label,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(label, old, new):
    M = _mutant(old, new)
    caught = []
    for pin in PINS:
        try:
            pin(M)
        except (AssertionError, FloatingPointError, ValueError, RuntimeError):
            caught.append(pin.__name__)
    assert caught, "planted mistake '%s' passed every pin" % label
