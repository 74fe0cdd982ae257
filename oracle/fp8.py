"""Float64 oracle of the RMSNorm forward with an FP8 (E4M3) output and a
per-tensor scale.

Test infrastructure only, like the rest of ``oracle/``: imported by
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py``; the CUDA path never imports it and shares no code with it.

Source: "Den dolda avrundningen i RMSNorm" (precisit.com), section "Var
implementationerna skiljer sig", the paragraph on Transformer Engine and its
footnote 3: in the FP8 output path with one scale factor per tensor the
normalisation, the multiplication by the weight and the output scaling are
all done in float32, and only the final conversion to FP8 rounds; no bf16
intermediate is rounded on the way.

Per row:  y8 = e4m3( x_hat * gain * scale ),  x_hat = x * rstd, with the
rstd of the RMSNorm forward (stored in float32 as usual).

Readings where the page leaves a step open (each one is listed with the
design notes):

* the FP8 format is E4M3 (the "fn" variant, largest finite value 448), the
  format of forward activations in FP8 training;
* the conversion rounds to nearest, ties to even, and saturates: a value
  beyond +-448 becomes +-448 (the page names no overflow rule; saturation is
  the conversion whose result stays finite);
* ``scale`` multiplies after the gain, as the page orders the steps; the
  oracle forms the product exactly in float64 and rounds once;
* the backward is the RMSNorm backward unchanged (it reads x, dy and the
  float32 rstd, not y).
"""
from __future__ import annotations

import numpy as np

from .rms_norm import forward_exact
from .rounding import round_to, round_to_saturating

E4M3 = "e4m3"


def store_e4m3(v) -> np.ndarray:
    """Saturating round-to-nearest-even of float64 values to E4M3."""
    return round_to_saturating(v, E4M3)


def forward_fp8(x, gamma, eps, offset: int, scale: float):
    """(y8, rstd): y8 the E4M3 values (as float64) of x_hat * gain * scale,
    rstd rounded once to float32."""
    y, rstd = forward_exact(x, gamma, eps, offset)
    y8 = store_e4m3(y * float(scale))
    return y8, round_to(rstd, "f32")
