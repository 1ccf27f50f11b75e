"""Parity of the CUDA projection (through the C ABI) against the projection oracle.

Tolerances, from float32 evaluation of each output (u = 2^-24):
  * mean2d: 32 u E, E = fx (sum_j |R_0j p_j| + |t_0| + |x/z| (sum_j |R_2j p_j| + |t_2|)) / z
    + |cx| (likewise for y), the magnitude of the terms the pixel position is
    summed from;
  * depth: 32 u (sum_j |R_2j p_j| + |t_2|);
  * conic: 64 u kappa max|conic|, kappa = the condition number of the 2D
    covariance (its inverse amplifies the covariance's rounding by kappa);
  * rgb: 32 u (sum_k |sh_k Y_k| + 0.5);
  * culled flags: exact;
  * gradients: max(1e-4, 1e-3 max|field|) per element, field = dmean3, dscale,
    dquat, dsh (the rasterizer's gradient bar); splats whose colour clamp is
    within the rgb tolerance of 0 are skipped (either side of the clamp is
    correct there).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle.project as OP
import gaussian_splatting_differentiable_gb300 as ss

U = 2.0 ** -24
FIELDS3 = ("dmean3", "dscale", "dquat", "dsh")


def cam_struct(cam):
    return ss.camera(cam.R, cam.t, cam.fx, cam.fy, cam.cx, cam.cy, cam.near, cam.blur)


def run_gpu(sc, stream=None):
    dev = torch.device("cuda")
    sp = ss.Splats3D.from_numpy(sc, dev)
    pr = ss.Projector(sc.n, sc.sh_degree, dev)
    cam = cam_struct(sc.cam)
    pr.forward(sp, cam, stream)
    f = lambda a: torch.from_numpy(a).to(dev).contiguous()  # noqa: E731
    pr.backward(sp, cam, f(sc.dmean2d), f(sc.dconic), f(sc.drgb), stream)
    torch.cuda.synchronize()
    out = {k: getattr(pr, k).cpu().numpy() for k in ("mean2d", "conic", "depth", "rgb")}
    out.update({k: v.cpu().numpy() for k, v in pr.grads.items()})
    return out


def _tolerances(sc, ofw, idx):
    p = sc.mean3[idx].astype(np.float64)
    R = np.asarray(sc.cam.R, np.float64)
    t = np.asarray(sc.cam.t, np.float64)
    a = np.abs(p[:, None, :] * R[None, :, :]).sum(2) + np.abs(t)      # [n][3]
    z = np.where(ofw["valid"], ofw["depth"], 1.0)
    pc = ofw["pc"]
    pz = np.where(ofw["valid"], pc[:, 2], 1.0)   # culled splats (z may be 0) are not compared
    xz, yz = np.abs(pc[:, 0] / pz), np.abs(pc[:, 1] / pz)
    Eu = sc.cam.fx * (a[:, 0] + xz * a[:, 2]) / np.abs(z) + abs(sc.cam.cx)
    Ev = sc.cam.fy * (a[:, 1] + yz * a[:, 2]) / np.abs(z) + abs(sc.cam.cy)
    cov2 = np.where(ofw["valid"][:, None, None], np.nan_to_num(ofw["cov2"]), np.eye(2))
    ev = np.linalg.eigvalsh(cov2)
    kappa = np.abs(ev[:, 1]) / np.maximum(np.abs(ev[:, 0]), 1e-300)
    return {"mean2d": 32 * U * np.stack([Eu, Ev], 1), "depth": 32 * U * a[:, 2],
            "conic": 64 * U * (kappa * np.abs(ofw["conic"]).max(1))[:, None],
            "rgb": 32 * U * ofw["rgb_scale"]}


def check(sc, gpu, idx=None):
    """Compare the splats ``idx`` (all when None); returns a report."""
    idx = np.arange(sc.n) if idx is None else np.asarray(idx)
    ofw = OP.project(sc, idx)
    v = ofw["valid"]
    gv = gpu["depth"][idx] > 0
    assert np.array_equal(gv, v), "culled flags differ at %s" % np.nonzero(gv != v)[0][:8]
    tol = _tolerances(sc, ofw, idx)
    rep = {"splats": int(len(idx)), "culled": int((~v).sum())}
    for k in ("mean2d", "depth", "conic", "rgb"):
        got = gpu[k][idx].astype(np.float64)
        ref = ofw[k]
        err = np.abs(got - ref)
        t = np.broadcast_to(tol[k] if tol[k].ndim == ref.ndim else tol[k][:, None], ref.shape)
        bad = err > t
        bad[~v] = got[~v] != 0
        assert not bad.any(), "%s: %d off; worst err %.3g tol %.3g" % (
            k, bad.sum(), err[bad].max(), t[bad][np.argmax(err[bad])])
        rep[k] = float((err[v] / np.maximum(t[v], 1e-300)).max(initial=0.0))
    # backward
    amb = (np.abs(ofw["raw"]) <= tol["rgb"]).any(1) & v
    obw = OP.project_backward(sc, idx)
    keep = ~amb
    for k in FIELDS3:
        got = gpu[k][:, :, idx] if k == "dsh" else gpu[k][idx]
        ref = obw[k]
        if k == "dsh":
            got, ref = got.transpose(2, 0, 1), ref.transpose(2, 0, 1)
        got = got.reshape(len(idx), -1).astype(np.float64)
        ref = ref.reshape(len(idx), -1)
        t = max(1e-4, 1e-3 * np.abs(ref[keep]).max(initial=0.0))
        err = np.abs(got - ref)
        bad = (err > t) & keep[:, None]
        assert not bad.any(), "%s: %d elements off; worst %.3g tol %.3g" % (
            k, bad.sum(), err[bad].max(), t)
        assert not np.any(got[~v]), "%s: nonzero gradient for a culled splat" % k
        rep[k] = float(err[keep].max(initial=0.0) / t)
    rep["clamp_knife_edge"] = int(amb.sum())
    return rep


def full_parity(sc):
    return check(sc, run_gpu(sc))


def sampled_parity(sc, n_sample=20000, seed=0):
    gpu = run_gpu(sc)
    idx = np.sort(np.random.default_rng(seed).choice(sc.n, min(n_sample, sc.n), replace=False))
    return check(sc, gpu, idx)
