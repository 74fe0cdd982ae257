"""Float64 oracle of softmax over the last dimension, forward and backward.

Test infrastructure only, like the rest of ``oracle/``: imported by
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py``; the CUDA path never imports it and shares no code with it.

Source: candle PR #4059 "Add backward passes to the fused rms_norm,
layer_norm and softmax_last_dim ops" (its description):

* forward: per row, y_j = exp(x_j - max_k x_k) / sum_k exp(x_k - max_k x_k);
  for bf16/f16 inputs the arithmetic is done wide and the result is rounded
  once at the store (the PR replaces a path that stored exp in bf16 and then
  scaled it, rounding twice);
* backward: dx = y * (dy - sum_j dy_j * y_j), from the forward's output y,
  with the reduction done wide (f32 for the half types).

Readings where the PR leaves a step open (each is listed with the design
notes):

* subtracting the row maximum changes nothing in exact arithmetic; the
  oracle does it too so that float64 exp never overflows;
* the forward result is the float64 value rounded once to the storage
  format;
* the backward takes y as stored (already rounded), as a fused backward
  that reads the forward's output does, and differentiates the exact
  softmax at that y; dx is rounded once.
"""
from __future__ import annotations

import numpy as np

from .rounding import round_to


def forward_exact(x) -> np.ndarray:
    """Unrounded softmax over the last axis, float64."""
    x = np.asarray(x, dtype=np.float64)
    z = x - np.max(x, axis=-1, keepdims=True)
    e = np.exp(z)
    return e / np.sum(e, axis=-1, keepdims=True)


def forward(x, fmt: str) -> np.ndarray:
    """Softmax as stored by the path: one rounding to ``fmt``."""
    return round_to(forward_exact(x), fmt)


def backward_exact(dy, y) -> np.ndarray:
    """Unrounded dx = y * (dy - sum(dy * y)) per row, float64."""
    dy = np.asarray(dy, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    s = np.sum(dy * y, axis=-1, keepdims=True)
    return y * (dy - s)


def backward(dy, y, fmt: str) -> np.ndarray:
    """Backward as stored by the path: dx rounded once to ``fmt``."""
    return round_to(backward_exact(dy, y), fmt)
