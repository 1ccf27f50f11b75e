"""Plain CPU oracle for the training loss L1 + SSIM and its gradient with
respect to the rendered image.

TEST INFRASTRUCTURE ONLY: imported by tests/, the smoke check and the
benchmark's CPU legs; the product package never imports it and it imports
nothing of the product package.

Source: "Phase 5 step 30b -- kernel-by-kernel timing" (otkrickey-splat.pages.dev):
the measured configuration trains with an L1 + SSIM loss, lambda = 0.20 and
a K = 7 window (setup section), and times "ssim_fwd_bwd", the SSIM forward
and backward in one command buffer (measurement table, hotspot ranking).
The page prints no formula; the readings are the plainest ones of the
structural-similarity index of Wang et al. (2004) used as a loss:

  S1  window: the 7 x 7 Gaussian, the outer product of the 1D window
      g_i = exp(-(i - 3)^2 / (2 sigma^2)) / sum, sigma = 1.5;
  S2  local statistics per channel by "same"-size correlation with zero
      padding outside the image: mu_x = w * x, sigma_x^2 = w * x^2 - mu_x^2,
      sigma_xy = w * (x y) - mu_x mu_y (likewise for y);
  S3  SSIM(p) = (2 mu_x mu_y + C1)(2 sigma_xy + C2) /
                ((mu_x^2 + mu_y^2 + C1)(sigma_x^2 + sigma_y^2 + C2)),
      C1 = 0.01^2, C2 = 0.03^2 (dynamic range 1);
  S4  loss = (1 - lambda) mean |x - y| + lambda (1 - mean SSIM), means over
      every channel and pixel; x is the rendered image, y the target;
  S5  the gradient is with respect to x only; |x - y| has derivative
      sign(x - y) (0 where x = y).

Arithmetic is float64 PyTorch on the CPU (conv2d as the correlation), the
gradient by autograd of that forward.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F

_D = torch.float64
K = 7
SIGMA = 1.5
C1 = 0.01 ** 2
C2 = 0.03 ** 2


def window1d(k: int = K, sigma: float = SIGMA) -> torch.Tensor:
    i = torch.arange(k, dtype=_D) - (k - 1) / 2
    g = torch.exp(-(i * i) / (2 * sigma * sigma))
    return g / g.sum()


def _corr(a: torch.Tensor, w2: torch.Tensor) -> torch.Tensor:
    """'same' correlation of every channel of a [C][H][W] with w2 [k][k], zero padded."""
    C = a.shape[0]
    k = w2.shape[0]
    return F.conv2d(a[None], w2.expand(C, 1, k, k), padding=k // 2, groups=C)[0]


def ssim_map(x: torch.Tensor, y: torch.Tensor) -> torch.Tensor:
    g = window1d()
    w2 = torch.outer(g, g)
    mx, my = _corr(x, w2), _corr(y, w2)
    sxx = _corr(x * x, w2) - mx * mx
    syy = _corr(y * y, w2) - my * my
    sxy = _corr(x * y, w2) - mx * my
    return ((2 * mx * my + C1) * (2 * sxy + C2)) / ((mx * mx + my * my + C1) * (sxx + syy + C2))


def _loss(x, y, lam):
    return (1 - lam) * (x - y).abs().mean() + lam * (1 - ssim_map(x, y).mean())


def loss_and_grad(img, target, lam: float = 0.2) -> dict:
    """img, target: [C][H][W] arrays.  Returns loss, ssim (mean), l1 (mean),
    the SSIM map and dL/dimg, all float64 numpy."""
    x = torch.as_tensor(np.asarray(img, np.float64)).clone().requires_grad_(True)
    y = torch.as_tensor(np.asarray(target, np.float64))
    S = ssim_map(x, y)
    l1 = (x - y).abs().mean()
    L = (1 - lam) * l1 + lam * (1 - S.mean())
    (g,) = torch.autograd.grad(L, [x])
    return {"loss": float(L.detach()), "ssim": float(S.detach().mean()), "l1": float(l1.detach()),
            "map": S.detach().numpy(), "grad": g.numpy()}


def loss_value(img, target, lam: float = 0.2) -> float:
    with torch.no_grad():
        return float(_loss(torch.as_tensor(np.asarray(img, np.float64)),
                           torch.as_tensor(np.asarray(target, np.float64)), lam))
