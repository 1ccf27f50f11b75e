"""Pins of the L1 + SSIM oracle (oracle/ssim.py) to things other than itself.

* the window against scipy's normal density;
* the SSIM map against a brute force of the definition written with explicit
  loops and explicit zero padding, on small images;
* closed forms: identical images give SSIM 1 and zero gradient; constant
  images give (2ab + C1) / (a^2 + b^2 + C1) away from the border; symmetry in
  the two images; lambda = 0 reduces to the mean absolute error;
* the gradient against central differences of the loss.

A planted-mistake test shows that plausible slips in oracle/ssim.py fail at
least one pin.
"""
import math
import pathlib
import types

import numpy as np
import pytest

from synth.images import make_image_pair

torch = pytest.importorskip("torch")
stats = pytest.importorskip("scipy.stats")

import oracle.ssim as OS  # noqa: E402


def _pair(C=2, H=9, W=11, seed=1):
    return make_image_pair(21, seed=seed, C=C, H=H, W=W)


def pin_window(P):
    g = P.window1d().numpy()
    ref = stats.norm.pdf(np.arange(7) - 3, scale=1.5)
    assert np.allclose(g, ref / ref.sum(), rtol=1e-14, atol=0), "window"


def _brute_map(x, y):
    C, H, W = x.shape
    i = np.arange(7) - 3
    g = np.exp(-(i * i) / (2 * 1.5 ** 2))
    g /= g.sum()
    c1, c2 = 0.01 ** 2, 0.03 ** 2
    out = np.zeros((C, H, W))
    for c in range(C):
        for py in range(H):
            for px in range(W):
                s = np.zeros(5)
                for dy in range(-3, 4):
                    for dx in range(-3, 4):
                        yy, xx = py + dy, px + dx
                        if 0 <= yy < H and 0 <= xx < W:
                            a, b = float(x[c, yy, xx]), float(y[c, yy, xx])
                        else:
                            a = b = 0.0
                        w = g[dy + 3] * g[dx + 3]
                        s += w * np.array([a, b, a * a, b * b, a * b])
                mx, my = s[0], s[1]
                vx, vy, cxy = s[2] - mx * mx, s[3] - my * my, s[4] - mx * my
                out[c, py, px] = ((2 * mx * my + c1) * (2 * cxy + c2)) / (
                    (mx * mx + my * my + c1) * (vx + vy + c2))
    return out


def pin_brute_force_map(P):
    x, y = _pair()
    got = P.loss_and_grad(x, y)["map"]
    assert np.allclose(got, _brute_map(x, y), rtol=0, atol=1e-12), "SSIM map vs brute force"


def pin_identical_images(P):
    x, _ = _pair(seed=2)
    r = P.loss_and_grad(x, x)
    assert np.allclose(r["map"], 1.0, atol=1e-12)
    assert abs(r["loss"]) < 1e-12
    assert np.abs(r["grad"]).max() < 1e-12


def pin_constant_images(P):
    a, b = 0.3, 0.7
    x = np.full((1, 20, 20), a, np.float32)
    y = np.full((1, 20, 20), b, np.float32)
    S = P.loss_and_grad(x, y)["map"]
    a, b = float(np.float32(a)), float(np.float32(b))
    ref = (2 * a * b + 0.01 ** 2) / (a * a + b * b + 0.01 ** 2)
    assert np.allclose(S[0, 3:-3, 3:-3], ref, atol=1e-12), "constant images"


def pin_symmetry(P):
    x, y = _pair(seed=3)
    assert np.allclose(P.loss_and_grad(x, y)["map"], P.loss_and_grad(y, x)["map"], atol=1e-14)


def pin_l1_only(P):
    x, y = _pair(seed=4)
    r = P.loss_and_grad(x, y, lam=0.0)
    d = x.astype(np.float64) - y.astype(np.float64)
    assert abs(r["loss"] - np.abs(d).mean()) < 1e-14
    assert np.allclose(r["grad"], np.sign(d) / d.size, atol=1e-18)


def pin_ssim_weight(P):
    """lambda = 1: the loss is 1 - mean SSIM, the brute-force map's mean."""
    x, y = _pair(C=1, H=8, W=8, seed=6)
    r = P.loss_and_grad(x, y, lam=1.0)
    assert abs(r["loss"] - (1 - _brute_map(x, y).mean())) < 1e-12


def pin_gradient_fd(P):
    x, y = _pair(C=2, H=8, W=9, seed=5)
    x = x.astype(np.float64)
    x[x == y] += 1e-3                            # keep |x - y| differentiable
    g = P.loss_and_grad(x, y, lam=0.2)["grad"]
    num = np.zeros_like(x)
    for idx in np.ndindex(x.shape):
        h = 1e-6
        xp, xm = x.copy(), x.copy()
        xp[idx] += h
        xm[idx] -= h
        num[idx] = (P.loss_value(xp, y) - P.loss_value(xm, y)) / (2 * h)
    assert np.allclose(g, num, atol=1e-9 * np.abs(num).max() + 1e-12, rtol=1e-5), \
        np.abs(g - num).max()


PINS = [pin_window, pin_brute_force_map, pin_identical_images, pin_constant_images, pin_symmetry,
        pin_l1_only, pin_ssim_weight, pin_gradient_fd]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(OS)


MUTATIONS = [
    ("C1 and C2 swapped", "C1 = 0.01 ** 2\nC2 = 0.03 ** 2", "C1 = 0.03 ** 2\nC2 = 0.01 ** 2"),
    ("covariance without the mean product", "sxy = _corr(x * y, w2) - mx * my",
     "sxy = _corr(x * y, w2)"),
    ("sigma 1.0", "SIGMA = 1.5", "SIGMA = 1.0"),
    ("reflect padding", "return F.conv2d(a[None], w2.expand(C, 1, k, k), padding=k // 2, groups=C)[0]",
     "return F.conv2d(F.pad(a[None], (k // 2,) * 4, mode='reflect'), w2.expand(C, 1, k, k), "
     "groups=C)[0]"),
    ("lambda on the L1 term", "L = (1 - lam) * l1 + lam * (1 - S.mean())",
     "L = lam * l1 + (1 - lam) * (1 - S.mean())"),
    ("variance of y from x", "syy = _corr(y * y, w2) - my * my", "syy = _corr(y * y, w2) - mx * my"),
    ("window not normalised", "return g / g.sum()", "return g"),
    ("sum instead of mean", "l1 = (x - y).abs().mean()", "l1 = (x - y).abs().sum()"),
]


def _mutant(old, new):
    src = pathlib.Path(OS.__file__).read_text()
    assert src.count(old) == 1, old
    mod = types.ModuleType("oracle_ssim_mutant")
    mod.__file__ = OS.__file__
    exec(compile(src.replace(old, new), OS.__file__, "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("label,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(label, old, new):
    M = _mutant(old, new)
    caught = []
    for pin in PINS:
        try:
            pin(M)
        except (AssertionError, ValueError, RuntimeError):
            caught.append(pin.__name__)
    assert caught, "planted mistake '%s' passed every pin" % label
