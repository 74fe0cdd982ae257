"""Plain float64 LayerNorm forward and backward, the oracle of the fused
LayerNorm path.

Test infrastructure only (see the package docstring): nothing on the CUDA
path imports it and it shares no code with the CUDA sources.

The pages treat LayerNorm as the sibling of RMSNorm: Liger-Kernel PR #1608
("fix(group_norm): keep the backward statistics and reductions in fp32",
the commit message after the timing table) notes that layer_norm stores its
Mean and RSTD in fp32, and candle PR #4059 ("Add backward passes to the
fused rms_norm, layer_norm and softmax_last_dim ops", description) adds the
layer_norm backward with statistics in f32 for half types.  Neither page
writes the formulas out; this module uses the standard definition (biased
variance, eps under the root) and its exact derivative:

    mean  = sum_j x_j / N
    var   = sum_j (x_j - mean)**2 / N
    rstd  = 1 / sqrt(var + eps)
    x_hat = (x - mean) * rstd
    y     = x_hat * gamma + beta          (stored with one rounding)

    g     = dy * gamma
    dx    = rstd * (g - mean_j(g) - x_hat * mean_j(g * x_hat))
    dgamma = sum over rows of dy * x_hat,  dbeta = sum over rows of dy

The store rounds once, after the gain and the bias, following the rounding
lesson of "Den dolda avrundningen i RMSNorm" (section "Två ställen att
avrunda"); mean and rstd are returned rounded once to float32.
"""
from __future__ import annotations

import numpy as np

from .rms_norm import eps_value
from .rounding import round_to


def stats_exact(x, eps):
    """(mean, rstd) per row in float64."""
    x = np.asarray(x, dtype=np.float64)
    n = x.shape[-1]
    mean = np.sum(x, axis=-1) / n
    d = x - mean[..., None]
    var = np.sum(d * d, axis=-1) / n
    return mean, 1.0 / np.sqrt(var + eps_value(eps))


def forward_exact(x, gamma, beta, eps):
    """Unrounded forward: (y, mean, rstd), float64.  ``beta`` may be None."""
    x = np.asarray(x, dtype=np.float64)
    mean, rstd = stats_exact(x, eps)
    x_hat = (x - mean[..., None]) * rstd[..., None]
    y = x_hat * np.asarray(gamma, dtype=np.float64)
    if beta is not None:
        y = y + np.asarray(beta, dtype=np.float64)
    return y, mean, rstd


def forward(x, gamma, beta, eps, fmt: str):
    """Forward as stored: (y in ``fmt``, mean in float32, rstd in float32)."""
    y, mean, rstd = forward_exact(x, gamma, beta, eps)
    return round_to(y, fmt), round_to(mean, "f32"), round_to(rstd, "f32")


def backward_exact(dy, x, gamma, mean, rstd):
    """Unrounded backward given the cached statistics: (dx, dgamma, dbeta)."""
    dy = np.asarray(dy, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    mean = np.asarray(mean, dtype=np.float64)
    rstd = np.asarray(rstd, dtype=np.float64)
    n = x.shape[-1]
    x_hat = (x - mean[..., None]) * rstd[..., None]
    g = dy * np.asarray(gamma, dtype=np.float64)
    c1 = np.sum(g, axis=-1) / n
    c2 = np.sum(g * x_hat, axis=-1) / n
    dx = rstd[..., None] * (g - c1[..., None] - x_hat * c2[..., None])
    dgamma = np.sum(dy * x_hat, axis=0)
    dbeta = np.sum(dy, axis=0)
    return dx, dgamma, dbeta


def backward(dy, x, gamma, mean, rstd, fmt: str):
    """Backward as stored: (dx in ``fmt``, dgamma and dbeta in float32)."""
    dx, dgamma, dbeta = backward_exact(dy, x, gamma, mean, rstd)
    return round_to(dx, fmt), round_to(dgamma, "f32"), round_to(dbeta, "f32")
