"""Seeded synthetic image pairs (rendered, target) for the L1 + SSIM loss.

Only draws inputs. Each channel of the target is 0.5 plus eight random plane
waves (wavelengths log-uniform 4-200 px, amplitudes U[0.02, 0.12], random
direction and phase) plus N(0, 0.02^2) pixel noise, clipped to [0, 1]; the
rendered image is the target plus four more plane waves of amplitude
U[0, 0.05] plus N(0, 0.05^2) noise, clipped to [0, 1] -- a rendering that is
close to its target with both smooth and pixel-level differences, and flat
clipped regions where the two agree exactly.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

from . import normal, stream_key, uniform01


@dataclasses.dataclass
class ImageWorkload:
    name: str
    C: int
    H: int
    W: int


IMAGE_WORKLOADS = {
    21: ImageWorkload("ssim-3x48x64", 3, 48, 64),
    22: ImageWorkload("ssim-3x822x1237", 3, 822, 1237),
    23: ImageWorkload("ssim-3x1080x1920", 3, 1080, 1920),
}


def _waves(key_base, n_waves, C, H, W, amp_lo, amp_hi):
    ys, xs = np.mgrid[0:H, 0:W].astype(np.float64)
    out = np.zeros((C, H, W))
    for c in range(C):
        k = lambda f: stream_key(key_base, c, f)  # noqa: E731
        lam = np.exp(math.log(4) + (math.log(200) - math.log(4)) * uniform01(k(1), n_waves))
        th = 2 * math.pi * uniform01(k(2), n_waves)
        ph = 2 * math.pi * uniform01(k(3), n_waves)
        amp = amp_lo + (amp_hi - amp_lo) * uniform01(k(4), n_waves)
        for j in range(n_waves):
            w = 2 * math.pi / lam[j]
            out[c] += amp[j] * np.sin(w * (math.cos(th[j]) * xs + math.sin(th[j]) * ys) + ph[j])
    return out


def make_image_pair(workload: int | ImageWorkload, seed: int = 0, C=None, H=None, W=None):
    """(rendered, target), float32 [C][H][W] each."""
    wl = IMAGE_WORKLOADS[workload] if isinstance(workload, int) else workload
    wid = workload if isinstance(workload, int) else 0
    C = wl.C if C is None else C
    H = wl.H if H is None else H
    W = wl.W if W is None else W
    base = int(stream_key(seed, wid, 60)) & 0xFFFFFFFF
    tgt = 0.5 + _waves(base, 8, C, H, W, 0.02, 0.12)
    tgt += normal(stream_key(seed, wid, 61), C * H * W, 0.02).reshape(C, H, W)
    tgt = np.clip(tgt, 0.0, 1.0)
    ren = tgt + _waves(base + 1, 4, C, H, W, 0.0, 0.05)
    ren += normal(stream_key(seed, wid, 62), C * H * W, 0.05).reshape(C, H, W)
    ren = np.clip(ren, 0.0, 1.0)
    return np.ascontiguousarray(ren, np.float32), np.ascontiguousarray(tgt, np.float32)
