"""Tolerance checks of GPU results against the oracle (test helper).

The numbers come with the hot path's specification: fp32 outputs within a
relative 1e-5, bf16/fp16 y and dx within one ulp of the output format with
at least 99.9% of elements bit-identical, rstd within a relative 1e-6, dw
within a relative 1e-3.  The readings of these numbers used here:

* an output formed without cancellation -- the RMSNorm forward
  y = (x * rstd) * gain, its FP8 store, the softmax forward -- is held to
  the rule as written, element by element: fp32 within 1e-5 of |ref|
  itself, half and FP8 outputs within one ulp everywhere, and the 99.9%
  bit-identical rate counted over every compared element.  Its fp32
  arithmetic is good to a few fp32 rounding errors of the element itself,
  so nothing looser is needed;
* an output that cancels (``cancels=True``) -- dx = rstd * (g - x_hat * c),
  and the LayerNorm / GroupNorm y = x_hat * gamma + beta with its centring
  and bias -- can be far smaller than the terms it is formed from, and fp32
  arithmetic cannot resolve it below the size of those terms.  There the
  relative errors are taken against max(|ref|, s), with s the rms over the
  row of the terms (``terms``); a half element passes with at most one ulp
  OR with |got - ref| <= 1e-5 * s; and the rate counts only elements with
  |ref| > 2**-10 * s: below that the value left after cancellation is
  within a few hundred fp32 rounding errors of the terms, and no fp32
  computation decides its half-precision rounding (GroupNorm's dx for an
  upstream of ones is such a case throughout).  A one-element RMSNorm row
  cancels completely: dx = rstd * g * eps / (x**2 + eps);
* the rate allows ceil(0.1% of n) of the n counted elements to differ
  (99.9% identical as a rate, which a sample under 1000 elements cannot
  show otherwise);
* round twice rounds x_hat to the storage type, a decision the kernel takes
  on its fp32 x_hat.  Where the exact x_hat lies so close to a rounding
  midpoint that an fp32 x_hat (relative error well under 4e-6) may fall on
  either side, the output built from either neighbour is correct;
* rstd: |got - ref| <= 1e-6 * ref elementwise; dw: |got - ref| <= 1e-3 *
  max(|ref_j|, rms(ref)).
"""
from __future__ import annotations

import numpy as np

from oracle import rounding

REL_F32 = 1e-5
REL_RSTD = 1e-6
REL_DW = 1e-3
MIN_BIT_IDENTICAL = 0.999
FLOOR_REL = 1e-5
MIDPOINT_WINDOW = 4e-6
RESOLVABLE_REL = 2.0 ** -10


def _row_rms(ref: np.ndarray) -> np.ndarray:
    r = np.sqrt(np.mean(np.square(ref, dtype=np.float64), axis=-1, keepdims=True))
    return np.broadcast_to(r, ref.shape)


def check_rows(got: np.ndarray, ref: np.ndarray, fmt: str, alt=None, what="y", terms=None,
               cancels: bool = False):
    """Compare a [rows, hidden] output.  ``alt`` (optional) is a list of
    (mask, values) pairs of other correct results.  ``cancels`` marks an
    output that cancels; ``terms`` (same shape, only with ``cancels``) holds
    the terms it is formed from, whose row rms sets the floor (default: the
    reference itself).  Returns a dict of stats and raises AssertionError
    with a description when the check fails."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert cancels or terms is None, f"{what}: terms only apply to an output that cancels"
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    diff = np.abs(got - ref)
    if cancels:
        scale = _row_rms(ref if terms is None else np.asarray(terms, dtype=np.float64))
    else:
        scale = np.zeros_like(ref)
    if fmt == "f32":
        ok = diff <= REL_F32 * np.maximum(np.abs(ref), scale)
        same = float(np.mean(got == ref)) if got.size else 1.0
        worst_ulp = None
    else:
        ulps = rounding.ulp_distance(got, ref, fmt)
        ok = ulps <= 1
        if cancels:
            ok |= diff <= FLOOR_REL * scale
        if alt is not None:
            for mask, vals in alt:
                ok |= mask & (got == vals)
        counted = np.abs(ref) > RESOLVABLE_REL * scale if cancels else np.ones(ref.shape, bool)
        same = float(np.mean(ulps[counted] == 0)) if np.any(counted) else 1.0
        worst_ulp = int(ulps.max()) if ulps.size else 0
    bad = np.argwhere(~ok)
    if bad.size:
        i = tuple(bad[0])
        raise AssertionError(
            f"{what}: {bad.shape[0]} elements out of tolerance; first at {i}: "
            f"got {got[i]!r} ref {ref[i]!r}")
    n = int(np.count_nonzero(counted)) if fmt != "f32" else int(got.size)
    if fmt != "f32":
        # the fraction is a rate: below 1000 compared elements one element
        # that rounds the other way is already 0.1%, so allow ceil(0.1% n)
        allowed = int(np.ceil((1.0 - MIN_BIT_IDENTICAL) * n - 1e-9))
        differ = int(round((1.0 - same) * n))
        assert differ <= allowed, f"{what}: only {same:.5f} bit-identical ({differ} of {n})"
    return {"bit_identical": same, "max_ulp": worst_ulp, "counted": n}


def check_rstd(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rel = np.abs(got - ref) / np.abs(ref)
    worst = float(rel.max()) if rel.size else 0.0
    assert worst <= REL_RSTD, f"rstd: worst relative error {worst:.3e}"
    return {"rstd_max_rel": worst}


def check_dw(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.maximum(np.abs(ref), np.sqrt(np.mean(ref * ref)))
    diff = np.abs(got - ref)
    # an all-zero reference (a one-element LayerNorm row has x_hat = 0) must
    # be met exactly
    rel = np.where(scale > 0, diff / np.where(scale > 0, scale, 1.0), np.where(diff == 0, 0.0, np.inf))
    worst = float(rel.max()) if rel.size else 0.0
    assert worst <= REL_DW, f"dw: worst relative error {worst:.3e}"
    return {"dw_max_rel": worst}


def spacing_exponent(v: np.ndarray, fmt: str) -> np.ndarray:
    p, emin, _ = rounding.FORMATS[fmt]
    _, e = np.frexp(v)
    return np.maximum(e - 1, emin) - (p - 1)


def round_twice_alternatives(x_hat: np.ndarray, gain: np.ndarray, fmt: str):
    """(mask, lower, upper): where x_hat is within the fp32 window of a
    rounding midpoint of ``fmt``, the stores built from the neighbour below
    and above x_hat."""
    q = spacing_exponent(x_hat, fmt)
    scaled = np.ldexp(x_hat, -q)
    lo = np.ldexp(np.floor(scaled), q)
    hi = np.ldexp(np.ceil(scaled), q)
    mid = (lo + hi) / 2.0
    mask = np.abs(x_hat - mid) <= MIDPOINT_WINDOW * np.abs(x_hat)
    y_lo = rounding.round_to(lo * gain, fmt)
    y_hi = rounding.round_to(hi * gain, fmt)
    return mask, y_lo, y_hi
