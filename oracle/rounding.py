"""Round-to-nearest-even from float64 to the storage formats of the path.

Test infrastructure only: the oracle is imported by ``tests/``, by the
``smoke()`` check in ``__graft_entry__`` and by the CPU-baseline leg of
``bench.py``; nothing on the CUDA path may import it.

The rounding rule is the one "Den dolda avrundningen i RMSNorm"
(precisit.com, section "En skillnad du kan återskapa") uses for its bf16
helper: round to nearest, ties to even.  That page's helper works on the bit
pattern of a finite float32 and leaves NaN undefined; this module instead
rounds a float64 value straight to a format given by its significand width
and exponent range, so that one routine serves bf16, fp16, fp32 and FP8
E4M3, covers
gradual underflow (fp16 subnormals occur in small gradients), overflow to
infinity, signed zero and NaN, and never rounds twice.

Method: write |v| = m * 2**e with the leading bit of m at 2**e.  The spacing
of representable values next to v is 2**q with q = max(e, emin) - (p - 1).
Scaling v by 2**-q is exact in float64 for every input the path produces,
``numpy.rint`` rounds the scaled value to an integer with ties to even, and
scaling back is exact again.  A result beyond the largest finite value of the
format becomes an infinity of the same sign.
"""
from __future__ import annotations

import numpy as np

# (significand bits including the implicit one, smallest normal exponent,
#  largest exponent) of each storage format.
FORMATS = {
    "f32": (24, -126, 127),
    "bf16": (8, -126, 127),
    "f16": (11, -14, 15),
    # FP8 E4M3 (the "fn" variant: no infinities, and the all-ones code of the
    # top binade is NaN, so the largest finite value is 1.75 * 2**8 = 448
    # rather than the 480 of the full grid)
    "e4m3": (4, -6, 8),
}

# Formats whose largest finite value is below the top of their grid.
_MAX_FINITE = {"e4m3": 448.0}


def max_finite(fmt: str) -> float:
    """Largest finite value of ``fmt``: (2 - 2**(1-p)) * 2**emax, except for
    e4m3, whose top code is NaN (448)."""
    if fmt in _MAX_FINITE:
        return _MAX_FINITE[fmt]
    p, _, emax = FORMATS[fmt]
    return float(np.ldexp(2.0 - 2.0 ** (1 - p), emax))


def round_to_saturating(v, fmt: str) -> np.ndarray:
    """``round_to`` followed by clamping to +-max_finite(fmt): a value that
    rounds past the largest finite value becomes that value with its sign
    (NaN stays NaN).  The FP8 store of the path converts this way."""
    r = round_to(v, fmt)
    m = max_finite(fmt)
    return np.clip(r, -m, m)


def round_to(v, fmt: str) -> np.ndarray:
    """Round float64 values ``v`` to the nearest value of ``fmt`` (ties to even).

    Returns float64 values that are exactly representable in ``fmt``.
    Zeros keep their sign, infinities stay, NaN stays NaN.
    """
    p, emin, emax = FORMATS[fmt]
    v = np.asarray(v, dtype=np.float64)
    out = v.copy()
    finite = np.isfinite(v) & (v != 0.0)
    if not np.any(finite):
        return out
    vf = v[finite]
    _, e_frexp = np.frexp(vf)            # |vf| = m * 2**e_frexp, 0.5 <= m < 1
    lead = e_frexp - 1                   # exponent of the leading bit
    q = np.maximum(lead, emin) - (p - 1)  # exponent of the spacing at vf
    r = np.rint(np.ldexp(vf, -q))        # integer multiple of 2**q, ties to even
    res = np.ldexp(r, q)
    # Keep the sign of a result that rounded to zero (rint keeps it already,
    # ldexp of -0.0 stays -0.0).
    overflow = np.abs(res) > max_finite(fmt)
    res[overflow] = np.copysign(np.inf, vf[overflow])
    out[finite] = res
    return out


def ulp_distance(a, b, fmt: str) -> np.ndarray:
    """Number of representable ``fmt`` values between ``a`` and ``b``.

    Both inputs must already be values of ``fmt``.  The distance is taken on
    the monotone integer order of the format (negative values mirrored below
    zero, +0 and -0 at the same place); an infinity counts as the value one
    step past the largest finite value.  A NaN on either side gives a huge
    distance.
    """
    return np.abs(_ordinal(a, fmt) - _ordinal(b, fmt))


def _ordinal(v, fmt: str) -> np.ndarray:
    """Signed position of each value in the ordered list of ``fmt`` values."""
    p, emin, emax = FORMATS[fmt]
    v = np.asarray(v, dtype=np.float64)
    mag = np.abs(v)
    out = np.zeros(v.shape, dtype=np.int64)
    nan = np.isnan(v)
    inf = np.isinf(v)
    fin = ~(nan | inf)
    m = mag[fin]
    _, e_frexp = np.frexp(m)
    lead = np.where(m > 0, e_frexp - 1, emin)
    sub = lead < emin
    lead = np.maximum(lead, emin)
    # Values in binade ``lead`` occupy positions
    #   (lead - emin + 1) * 2**(p-1) + (m / 2**(lead-p+1) - 2**(p-1)).
    # Subnormals (and zero) sit at positions 0 .. 2**(p-1)-1.
    steps = np.ldexp(m, -(lead - (p - 1))).astype(np.int64)
    pos = np.where(sub, steps, (lead - emin) * (1 << (p - 1)) + steps)
    out[fin] = pos
    top = ((emax - emin) + 2) * (1 << (p - 1))   # one past the largest finite
    out[inf] = top
    out = np.where(v < 0, -out, out)
    out[nan] = np.iinfo(np.int64).max // 4
    return out
