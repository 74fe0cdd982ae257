"""Float64 oracle of GroupNorm, forward and backward.

Test infrastructure only, like the rest of ``oracle/``: imported by
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py``; the CUDA path never imports it and shares no code with it.

Source: Liger-Kernel PR #1608 "fix(group_norm): keep the backward
statistics and reductions in fp32" (summary and commit message): the input
is (batch, channels, spatial...) with the channels split into groups; the
forward stores Mean and RSTD per (sample, group), in fp32; the backward
upcasts X, the upstream gradient and the weight W to fp32 before every
reduction.  No formula is printed; the plain definition is used:

  per (n, g): mean = mean of x over the group's channels and positions,
  var = mean of (x - mean)**2 (biased), rstd = 1 / sqrt(var + eps),
  x_hat = (x - mean) * rstd,  y = x_hat * W[c] + B[c];
  backward with g = dy * W[c]:
  dx = rstd * (g - mean_group(g) - x_hat * mean_group(g * x_hat)),
  dW[c] = sum over samples and positions of dy * x_hat,
  dB[c] = sum over samples and positions of dy.

Arrays are [n, channels, spatial] (spatial positions flattened); mean and
rstd are [n, groups]; eps is a float32 value widened to float64; outputs
are the float64 values rounded once to the storage format (mean, rstd, dW,
dB to float32).
"""
from __future__ import annotations

import numpy as np

from .rounding import round_to


def _grouped(a, groups: int):
    n, c, s = a.shape
    return a.reshape(n, groups, (c // groups) * s)


def stats_exact(x, groups: int, eps):
    """(mean, rstd), each [n, groups], float64."""
    xg = _grouped(np.asarray(x, dtype=np.float64), groups)
    mean = xg.mean(axis=-1)
    var = np.mean((xg - mean[..., None]) ** 2, axis=-1)
    return mean, 1.0 / np.sqrt(var + float(np.float32(eps)))


def _x_hat(x, mean, rstd, groups: int):
    x = np.asarray(x, dtype=np.float64)
    xg = _grouped(x, groups)
    xh = (xg - np.asarray(mean, float)[..., None]) * np.asarray(rstd, float)[..., None]
    return xh.reshape(x.shape)


def forward_exact(x, gamma, beta, groups: int, eps):
    """Unrounded (y, mean, rstd); beta may be None."""
    mean, rstd = stats_exact(x, groups, eps)
    xh = _x_hat(x, mean, rstd, groups)
    y = xh * np.asarray(gamma, float)[None, :, None]
    if beta is not None:
        y = y + np.asarray(beta, float)[None, :, None]
    return y, mean, rstd


def forward(x, gamma, beta, groups: int, eps, fmt: str):
    """(y in ``fmt``, mean and rstd in float32)."""
    y, mean, rstd = forward_exact(x, gamma, beta, groups, eps)
    return round_to(y, fmt), round_to(mean, "f32"), round_to(rstd, "f32")


def backward_exact(dy, x, gamma, mean, rstd, groups: int):
    """Unrounded (dx, dgamma, dbeta) given the cached mean and rstd."""
    dy = np.asarray(dy, dtype=np.float64)
    xh = _x_hat(x, mean, rstd, groups)
    g = dy * np.asarray(gamma, float)[None, :, None]
    gg, xhg = _grouped(g, groups), _grouped(xh, groups)
    c1 = gg.mean(axis=-1, keepdims=True)
    c2 = (gg * xhg).mean(axis=-1, keepdims=True)
    dx = np.asarray(rstd, float)[..., None] * (gg - c1 - xhg * c2)
    dgamma = np.sum(dy * xh, axis=(0, 2))
    dbeta = np.sum(dy, axis=(0, 2))
    return dx.reshape(dy.shape), dgamma, dbeta


def backward(dy, x, gamma, mean, rstd, groups: int, fmt: str):
    """(dx in ``fmt``, dgamma and dbeta in float32)."""
    dx, dg, db = backward_exact(dy, x, gamma, mean, rstd, groups)
    return round_to(dx, fmt), round_to(dg, "f32"), round_to(db, "f32")
