"""Plain float64 RMSNorm forward and backward, the oracle of the fused path.

Test infrastructure only: the oracle is imported by ``tests/``, by the
``smoke()`` check in ``__graft_entry__`` and by the CPU-baseline leg of
``bench.py``; nothing on the CUDA path may import it, and it shares no code,
header, table or constant with the CUDA sources.

Every array argument holds the input *values* as float64 (a bf16 or fp16
input widens to float64 exactly).  All arithmetic is float64; the only other
roundings are the explicit stores to the output format, made with
``oracle.rounding.round_to``.

Sources, by page and section:

* normalisation and gain -- "Den dolda avrundningen i RMSNorm"
  (precisit.com), section "En välbekant operation", the two displayed
  equations: x_hat_i = x_i / sqrt(mean_j x_j**2 + eps), y_i = x_hat_i * gamma_i.
* where the result is rounded -- same page, section "Två ställen att
  avrunda": "round once" stores bf16(x_hat * gamma) after a wide multiply;
  "round twice" stores bf16(bf16(x_hat) * gamma).
* the Gemma gain 1 + gamma, multiplied wide and stored last -- same page,
  section "Vilken konvention hör till modellen?".
* statistics and the cached inverse RMS kept in fp32 for half inputs, weight
  gradients in fp32 -- Liger-Kernel PR #92 "feat: correct casts in RMSNorm to
  match references" (the author's comment after the benchmark tables).
* the backward with its statistics in f32 for half types -- candle PR #4059
  "Add backward passes to the fused rms_norm, layer_norm and
  softmax_last_dim ops" (description).  No page writes the backward out; the
  formula used here is the exact derivative of the forward above:
  g = dy * gain, c = mean_j(g_j * x_hat_j), dx = rstd * (g - x_hat * c),
  dgamma = sum over rows of dy * x_hat.

Readings where the pages leave a step open (each one is listed with the
design notes):

* eps is a float32 argument; it enters the float64 sum as its exact float32
  value, under the root, added to the mean of squares.
* the rstd output is the float64 value rounded once to float32.
* round once rounds the float64 product x_hat * gain straight to the output
  format (one rounding, no float32 step in between).
* round twice rounds x_hat to the output format first; the product of that
  value and the gain is exact in float64 and is then rounded once more.
* the backward takes rstd as an input (the cached float32 value in normal
  use) and ignores the cast mode: it differentiates the unrounded forward.
* the Gemma gain 1 + gamma is formed exactly in float64.
"""
from __future__ import annotations

import numpy as np

from .rounding import round_to

# Storage formats of x, gamma, y, dy and dx.
F32 = "f32"
BF16 = "bf16"
F16 = "f16"

ROUND_ONCE = "round_once"
ROUND_TWICE = "round_twice"


def eps_value(eps) -> float:
    """The float32 value of eps, widened to float64."""
    return float(np.float32(eps))


def gain(gamma, offset: int) -> np.ndarray:
    """gamma (offset 0) or the Gemma gain 1 + gamma (offset 1), in float64."""
    gamma = np.asarray(gamma, dtype=np.float64)
    return gamma + 1.0 if offset else gamma


def rstd_exact(x, eps) -> np.ndarray:
    """1 / sqrt(mean(x**2) + eps) per row, in float64 (no rounding)."""
    x = np.asarray(x, dtype=np.float64)
    n = x.shape[-1]
    mean_sq = np.sum(x * x, axis=-1) / n
    return 1.0 / np.sqrt(mean_sq + eps_value(eps))


def forward_exact(x, gamma, eps, offset: int = 0):
    """Unrounded forward: (y, rstd), both float64."""
    x = np.asarray(x, dtype=np.float64)
    rstd = rstd_exact(x, eps)
    x_hat = x * rstd[..., None]
    return x_hat * gain(gamma, offset), rstd


def store_y(x_hat, g, fmt: str, cast_mode: str) -> np.ndarray:
    """The output store: one rounding (round once) or two (round twice)."""
    if cast_mode == ROUND_ONCE:
        return round_to(x_hat * g, fmt)
    if cast_mode == ROUND_TWICE:
        return round_to(round_to(x_hat, fmt) * g, fmt)
    raise ValueError(f"unknown cast mode {cast_mode!r}")


def forward(x, gamma, eps, offset: int, fmt: str, cast_mode: str = ROUND_ONCE):
    """Forward as stored by the path: (y in ``fmt``, rstd in float32).

    Both returned arrays hold float64 values that are exactly representable
    in their storage format.
    """
    x = np.asarray(x, dtype=np.float64)
    rstd = rstd_exact(x, eps)
    x_hat = x * rstd[..., None]
    y = store_y(x_hat, gain(gamma, offset), fmt, cast_mode)
    return y, round_to(rstd, F32)


def backward_exact(dy, x, gamma, rstd, offset: int = 0):
    """Unrounded backward given the cached rstd: (dx, dgamma), float64."""
    dy = np.asarray(dy, dtype=np.float64)
    x = np.asarray(x, dtype=np.float64)
    rstd = np.asarray(rstd, dtype=np.float64)
    n = x.shape[-1]
    x_hat = x * rstd[..., None]
    g = dy * gain(gamma, offset)
    c = np.sum(g * x_hat, axis=-1) / n
    dx = rstd[..., None] * (g - x_hat * c[..., None])
    dgamma = np.sum(dy * x_hat, axis=0)
    return dx, dgamma


def backward(dy, x, gamma, rstd, offset: int, fmt: str):
    """Backward as stored by the path: (dx in ``fmt``, dgamma in float32)."""
    dx, dgamma = backward_exact(dy, x, gamma, rstd, offset)
    return round_to(dx, fmt), round_to(dgamma, F32)
