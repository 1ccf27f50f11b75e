"""Plain CPU oracle for the projection of 3D Gaussian splats to the 2D splats
the rasterizer consumes (mean2d, conic, depth, view-dependent RGB), and for
its backward.

TEST INFRASTRUCTURE ONLY: imported by tests/, the smoke check and the
benchmark's CPU legs; the product package never imports it and it imports
nothing of the product package.  It shares no code with the CUDA library;
the two meet only through the seeded inputs of synth.scene3d.

Source: "Phase 5 step 30b -- kernel-by-kernel timing" (otkrickey-splat.pages.dev),
measurement table and hotspot ranking: a forward projection kernel
(project_soa) whose cost the page attributes mostly to spherical-harmonic
colour evaluation, and its backward (project_backwards), on either side of
the rasterizer.  The page prints none of the formulas, so every step below is
the plainest reading of projecting a 3D Gaussian through a pinhole camera:

  P1  camera: p_c = R p + t (R world-to-camera); pixel position
      (fx x/z + cx, fy y/z + cy) in the frame whose pixel centres sit at
      +0.5; depth = z.
  P2  a splat is culled -- every output 0, so the rasterizer culls it on its
      depth, and no gradient -- when z <= near, when the 2D covariance is not
      positive definite, or when an output is not finite.
  P3  3D covariance R(q^) diag(s)^2 R(q^)^T with q^ = q / |q|, q = (w, x, y, z);
      gradients flow through the normalisation.
  P4  2D covariance: the local affine approximation of the perspective map
      at the mean, J R Sigma R^T J^T, J the Jacobian of (fx x/z, fy y/z) at
      p_c (x/z not clamped), plus blur * I (the camera's low-pass term);
      conic = its inverse, stored (a, b, c) = ([0,0], [0,1], [1,1]).
  P5  colour per channel: max(0, sum_k sh[k] Y_k(d) + 0.5), d the unit
      vector from the camera centre -R^T t to the mean; gradient 0 where the
      clamp is active.
  P6  real spherical harmonics, k = l^2 + l + m:
      Y_lm = N_lm P_l^(|m|)(z) Re((x + i y)^|m|) for m >= 0 and
      N_lm P_l^(|m|)(z) Im((x + i y)^|m|) for m < 0, P_l^(m) the m-th
      derivative of the Legendre polynomial, N_lm = sqrt((2l+1)/(4 pi)
      (l-|m|)!/(l+|m|)!) times sqrt(2) when m != 0 (no Condon-Shortley phase).
  P7  backward: the exact partial derivatives of
      L = sum dL/dmean2d . mean2d + dL/dconic . conic + dL/drgb . rgb
      with respect to mean3, scale, quat (unnormalised) and sh; the camera is
      fixed, depth receives no gradient, opacity passes through.

Arithmetic is float64 PyTorch on the CPU; the backward is autograd of that
forward (the exact partials of the composed function).
"""
from __future__ import annotations

import math

import numpy as np
import torch
from numpy.polynomial import legendre as _leg
from numpy.polynomial import polynomial as _poly

_D = torch.float64


def sh_count(degree: int) -> int:
    return (degree + 1) ** 2


def sh_basis(degree: int, d: torch.Tensor) -> torch.Tensor:
    """Real spherical harmonics (P6) of unit vectors d [n][3] -> [n][K]."""
    x, y, z = d[:, 0], d[:, 1], d[:, 2]
    out = [None] * sh_count(degree)
    re, im = torch.ones_like(x), torch.zeros_like(x)     # (x + i y)^0
    powers = []
    for m in range(degree + 1):
        powers.append((re, im))
        re, im = re * x - im * y, re * y + im * x
    for l in range(degree + 1):
        pl = _leg.leg2poly([0] * l + [1])                # power-series coefficients of P_l
        for m in range(l + 1):
            coef = _poly.polyder(pl, m) if m else pl
            q = torch.zeros_like(z)
            for c in coef[::-1]:                         # Horner in z
                q = q * z + float(c)
            norm = math.sqrt((2 * l + 1) / (4 * math.pi) * math.factorial(l - m)
                             / math.factorial(l + m))
            if m:
                norm *= math.sqrt(2.0)
            out[l * l + l + m] = norm * q * powers[m][0]
            if m:
                out[l * l + l - m] = norm * q * powers[m][1]
    return torch.stack(out, dim=1)


def quat_rotmat(q: torch.Tensor) -> torch.Tensor:
    """Rotation matrix [n][3][3] of the normalised quaternions q [n][4] = (w, x, y, z)."""
    u = q / q.norm(dim=1, keepdim=True)
    w, x, y, z = u.unbind(1)
    return torch.stack([
        torch.stack([1 - 2 * (y * y + z * z), 2 * (x * y - w * z), 2 * (x * z + w * y)], 1),
        torch.stack([2 * (x * y + w * z), 1 - 2 * (x * x + z * z), 2 * (y * z - w * x)], 1),
        torch.stack([2 * (x * z - w * y), 2 * (y * z + w * x), 1 - 2 * (x * x + y * y)], 1),
    ], 1)


def _camera(cam):
    R = torch.as_tensor(np.asarray(cam.R, np.float64), dtype=_D)
    t = torch.as_tensor(np.asarray(cam.t, np.float64), dtype=_D)
    return R, t


def _project(mean3, scale, quat, sh, cam, degree):
    """P1-P6 on float64 tensors; returns every output and intermediate."""
    R, t = _camera(cam)
    pc = mean3 @ R.T + t
    x, y, z = pc[:, 0], pc[:, 1], pc[:, 2]
    fx, fy = float(cam.fx), float(cam.fy)
    n = mean3.shape[0]
    J = torch.zeros(n, 2, 3, dtype=_D)
    J[:, 0, 0] = fx / z
    J[:, 0, 2] = -fx * x / (z * z)
    J[:, 1, 1] = fy / z
    J[:, 1, 2] = -fy * y / (z * z)
    Tm = J @ R
    M = quat_rotmat(quat) * scale[:, None, :]
    cov3 = M @ M.transpose(1, 2)
    cov2 = Tm @ cov3 @ Tm.transpose(1, 2) + float(cam.blur) * torch.eye(2, dtype=_D)
    det = cov2[:, 0, 0] * cov2[:, 1, 1] - cov2[:, 0, 1] * cov2[:, 1, 0]
    conic = torch.stack([cov2[:, 1, 1] / det, -cov2[:, 0, 1] / det, cov2[:, 0, 0] / det], 1)
    mean2d = torch.stack([fx * x / z + float(cam.cx), fy * y / z + float(cam.cy)], 1)
    campos = -(R.T @ t)
    v = mean3 - campos
    d = v / v.norm(dim=1, keepdim=True)
    Y = sh_basis(degree, d)                                      # [n][K]
    terms = sh.permute(2, 1, 0) * Y[:, None, :]                  # [n][3][K]
    raw = terms.sum(dim=2) + 0.5
    rgb = torch.clamp(raw, min=0.0)
    return {"mean2d": mean2d, "conic": conic, "depth": z, "rgb": rgb, "raw": raw,
            "cov2": cov2, "det": det, "rgb_scale": terms.abs().sum(dim=2) + 0.5, "pc": pc}


def _inputs(scene, idx, params):
    params = params or {}
    g = lambda k: torch.as_tensor(np.asarray(params.get(k, getattr(scene, k)),  # noqa: E731
                                             np.float64), dtype=_D)
    sh = g("sh")
    return g("mean3")[idx], g("scale")[idx], g("quat")[idx], sh[:, :, idx]


def project(scene, idx=None, params=None) -> dict:
    """Forward of the splats ``idx`` (all when None): numpy dict with mean2d,
    conic, depth, rgb (culled splats all 0), valid, and the intermediates
    cov2, det, raw (unclamped colour) and rgb_scale (sum of |terms| + 0.5)."""
    n = scene.n if idx is None else len(idx)
    idx = np.arange(scene.n) if idx is None else np.asarray(idx)
    with torch.no_grad():
        r = _project(*_inputs(scene, idx, params), scene.cam, scene.sh_degree)
        fin = torch.ones(n, dtype=torch.bool)
        for k in ("mean2d", "conic", "rgb"):
            fin &= torch.isfinite(r[k]).all(dim=1)
        valid = (r["depth"] > scene.cam.near) & (r["det"] > 0) & fin
    out = {k: r[k].numpy().copy() for k in r}
    v = valid.numpy()
    for k in ("mean2d", "conic", "depth", "rgb"):
        out[k][~v] = 0.0
    out["valid"] = v
    return out


def project_backward(scene, idx=None, params=None, upstream=None) -> dict:
    """P7 for the splats ``idx``: dmean3 [n][3], dscale [n][3], dquat [n][4],
    dsh [K][3][n] (0 for culled splats), plus valid."""
    idx = np.arange(scene.n) if idx is None else np.asarray(idx)
    fw = project(scene, idx, params)
    v = np.nonzero(fw["valid"])[0]
    up = upstream or {}
    gm = torch.as_tensor(np.asarray(up.get("dmean2d", scene.dmean2d), np.float64)[idx][v])
    gc = torch.as_tensor(np.asarray(up.get("dconic", scene.dconic), np.float64)[idx][v])
    gr = torch.as_tensor(np.asarray(up.get("drgb", scene.drgb), np.float64)[idx][v])
    mean3, scale, quat, sh = [a.clone().requires_grad_(True)
                              for a in _inputs(scene, idx[v], params)]
    r = _project(mean3, scale, quat, sh, scene.cam, scene.sh_degree)
    L = (gm * r["mean2d"]).sum() + (gc * r["conic"]).sum() + (gr * r["rgb"]).sum()
    gs = torch.autograd.grad(L, [mean3, scale, quat, sh])
    n, K = len(idx), sh_count(scene.sh_degree)
    out = {"dmean3": np.zeros((n, 3)), "dscale": np.zeros((n, 3)), "dquat": np.zeros((n, 4)),
           "dsh": np.zeros((K, 3, n)), "valid": fw["valid"]}
    out["dmean3"][v] = gs[0].numpy()
    out["dscale"][v] = gs[1].numpy()
    out["dquat"][v] = gs[2].numpy()
    out["dsh"][:, :, v] = gs[3].numpy()
    return out


def loss(scene, params=None, upstream=None) -> float:
    """L of P7 over all splats, in float64 (for finite-difference pins)."""
    fw = project(scene, None, params)
    up = upstream or {}
    return float((np.asarray(up.get("dmean2d", scene.dmean2d), np.float64) * fw["mean2d"]).sum()
                 + (np.asarray(up.get("dconic", scene.dconic), np.float64) * fw["conic"]).sum()
                 + (np.asarray(up.get("drgb", scene.drgb), np.float64) * fw["rgb"]).sum())
