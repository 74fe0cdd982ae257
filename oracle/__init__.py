"""Float64 CPU oracle for fused RMSNorm forward and backward.

TEST INFRASTRUCTURE ONLY.  ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it; the library under
``bwd_rms_norm_gb300/`` never does, and the two share no code.

Parity status of each function (what pins it is in ``tests/test_oracle.py``):

* ``rounding.round_to`` -- pinned: the worked example and the two-million
  sample count of "Den dolda avrundningen i RMSNorm", exhaustive checks of
  every bf16 and fp16 value and midpoint, numpy's float64-to-float16 cast and
  torch's float32-to-bfloat16 cast.
* ``rms_norm.forward`` / ``forward_exact`` -- pinned: torch's CPU ``rms_norm``
  in float64 (the plain definition), torch's CPU bf16 ``rms_norm`` (single
  rounding after a float32 multiply), closed forms for one-element and
  constant rows, scale invariance, the Gemma gain identity.
* ``rms_norm.backward`` / ``backward_exact`` -- pinned: central finite
  differences of sum(dy * y) in float64, torch autograd through CPU
  ``rms_norm`` in float64, the orthogonality of dx to x at eps = 0.
* ``layer_norm.forward`` / ``backward`` (and the ``_exact`` forms) -- pinned
  in ``tests/test_oracle_layer_norm.py``: torch's CPU ``layer_norm`` in
  float64 and its autograd, finite differences, shift invariance of dx,
  zero mean and the variance identity of x_hat, torch's CPU bf16
  ``layer_norm``.
* ``fp8.forward_fp8`` / ``store_e4m3`` (and ``rounding.round_to_saturating``)
  -- pinned in ``tests/test_oracle_fp8.py``: every E4M3 code, every midpoint
  and the points beside it against torch's float8_e4m3fn cast, the format's
  value set, torch's float64 ``rms_norm`` times the scale cast by torch, a
  hand-worked Gemma case; saturation beyond 448 is a reading of the page
  (torch turns those values into NaN, so nothing outside pins it).
* ``softmax.forward`` / ``backward`` (and the ``_exact`` forms) -- pinned in
  ``tests/test_oracle_softmax.py``: torch's CPU softmax in float64 (with a
  row whose exp overflows unshifted) and its autograd, finite differences,
  rows summing to 1, dx rows summing to 0, shift invariance, closed forms
  for one, two and constant elements, torch's CPU bf16 softmax.
* ``group_norm.forward`` / ``backward`` (and the ``_exact`` forms) -- pinned
  in ``tests/test_oracle_group_norm.py``: torch's CPU ``group_norm`` in
  float64 and its autograd, finite differences (x, W, B), per-group sums of
  dx and x_hat, the upstream-of-ones case of Liger-Kernel PR #1608 (dx = 0),
  G = 1 against the LayerNorm oracle, G = C against torch's
  ``instance_norm``, torch's CPU bf16 ``group_norm``.
"""
from . import fp8, group_norm, layer_norm, softmax  # noqa: F401
from .rounding import FORMATS, max_finite, round_to, ulp_distance  # noqa: F401
from .rms_norm import (  # noqa: F401
    BF16,
    F16,
    F32,
    ROUND_ONCE,
    ROUND_TWICE,
    backward,
    backward_exact,
    eps_value,
    forward,
    forward_exact,
    gain,
    rstd_exact,
    store_y,
)
