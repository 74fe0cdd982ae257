"""Pins of the E4M3 rounding and of the FP8-output forward of the oracle
against facts fixed outside it (torch's own float8_e4m3fn conversion, the
format's definition, torch's float64 rms_norm), and planted mistakes that
those pins catch.  Host only."""
import types

import numpy as np
import pytest
import torch

from oracle import fp8 as of8
from oracle import rms_norm as orm
from oracle import rounding

E4M3 = torch.float8_e4m3fn


def _codes():
    """Every E4M3 code decoded by torch (float64), NaN codes dropped."""
    v = torch.arange(256, dtype=torch.uint8).view(E4M3).float().double().numpy()
    return v[np.isfinite(v)]


def test_format_has_the_expected_values():
    """254 finite codes (+-0 and 126 magnitudes a sign), largest 448,
    smallest subnormal 2**-9, smallest normal 2**-6."""
    v = _codes()
    assert v.size == 254
    pos = np.unique(v[v > 0])
    assert pos.size == 126
    assert pos.max() == 448.0 and pos.min() == 2.0 ** -9
    assert np.min(pos[pos >= 2.0 ** -6]) == 2.0 ** -6
    assert rounding.max_finite("e4m3") == 448.0


def check_rounding_vs_torch(store=of8.store_e4m3):
    """Fixed points, midpoints and points just beside the midpoints, against
    torch's float32 -> float8_e4m3fn cast (round to nearest even).  Returns
    the number of disagreements."""
    v = np.unique(_codes())
    bad = int(np.sum(store(v) != v))
    mids = (v[:-1] + v[1:]) / 2.0
    gaps = v[1:] - v[:-1]
    probes = np.concatenate([mids, mids + gaps * 2.0 ** -12, mids - gaps * 2.0 ** -12])
    probes = probes[np.abs(probes) <= 464.0]    # torch turns larger values into NaN
    assert np.array_equal(probes.astype(np.float32).astype(np.float64), probes)
    ref = torch.from_numpy(probes.astype(np.float32)).to(E4M3).float().double().numpy()
    bad += int(np.sum(store(probes) != ref))
    return bad


def test_rounding_matches_torch_cast():
    assert check_rounding_vs_torch() == 0


def test_saturation():
    """Reading: the store saturates -- everything past +-448 becomes +-448;
    the 464 tie rounds to the even code 448 in any case; NaN stays NaN."""
    v = np.array([448.0, 463.9, 464.0, 464.1, 480.0, 1e6, np.inf, -500.0, -np.inf])
    got = of8.store_e4m3(v)
    assert np.array_equal(got, [448, 448, 448, 448, 448, 448, 448, -448, -448])
    assert np.isnan(of8.store_e4m3(np.array([np.nan])))[0]
    # without saturation the same values overflow
    assert np.isinf(rounding.round_to(np.array([470.0]), "e4m3"))[0]


def test_subnormals_and_signed_zero():
    t = 2.0 ** -9
    v = np.array([t, 0.5 * t, 0.50001 * t, 1.5 * t, 2.5 * t, -0.25 * t])
    got = of8.store_e4m3(v)
    assert np.array_equal(got, [t, 0.0, t, 2 * t, 2 * t, -0.0])
    assert np.signbit(got[-1])


def check_forward_vs_torch(mod=of8, seed=3):
    """forward_fp8 against torch's float64 CPU rms_norm times the scale,
    converted by torch's own float8 cast (in-range elements: the scale keeps
    |y| under 448 for this draw).  Returns (mismatches, elements)."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(64, 256, generator=g, dtype=torch.float64)
    w = torch.rand(256, generator=g, dtype=torch.float64) * 0.2 + 0.9
    scale = 37.5
    eps = 1e-5
    ref = torch.nn.functional.rms_norm(x, (256,), weight=w, eps=float(np.float32(eps)))
    ref = (ref * scale).float()
    assert ref.abs().max().item() < 448.0
    ref8 = ref.to(E4M3).float().double().numpy()
    y8, rstd = mod.forward_fp8(x.numpy(), w.numpy(), eps, 0, scale)
    return int(np.sum(y8 != ref8)), ref8.size


def test_forward_matches_torch_composition():
    """The float64 -> float32 step of the torch composition is a second
    rounding; it can only move a value that sits within 2**-24 of an E4M3
    midpoint, which this draw does not hit."""
    bad, n = check_forward_vs_torch()
    assert bad == 0, f"{bad} of {n}"


def test_forward_gemma_gain_and_rstd():
    x = np.array([[3.0, -4.0]])
    y8, rstd = of8.forward_fp8(x, np.array([0.5, 0.25]), 0.0, 1, 2.0)
    # rstd = 1/sqrt(12.5); gains 1.5, 1.25; y = x * rstd * gain * 2
    r = 1.0 / np.sqrt(12.5)
    assert rstd[0] == np.float32(r)
    want = rounding.round_to(np.array([3 * r * 1.5 * 2, -4 * r * 1.25 * 2]), "e4m3")
    assert np.array_equal(y8[0], want)
    # 2.5456 -> 2.5 and -2.8284 -> -2.75 on the E4M3 grid (spacing 0.25 in [2, 4))
    assert np.array_equal(y8[0], [2.5, -2.75])


def test_scale_is_applied_before_rounding():
    """Scaling by a power of two commutes with the rounding only inside the
    normal range; a scale of 3 does not (a single rounding at the end)."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((8, 64))
    w = rng.uniform(0.9, 1.1, 64)
    a, _ = of8.forward_fp8(x, w, 1e-6, 0, 4.0)
    b, _ = of8.forward_fp8(x, w, 1e-6, 0, 1.0)
    y, _ = orm.forward_exact(x, w, 1e-6, 0)
    norm = np.abs(y) >= 2.0 ** -6        # the exact value, not the rounded one
    assert np.array_equal(a[norm], 4.0 * b[norm])
    assert not np.array_equal(a[~norm], 4.0 * b[~norm])   # subnormals do not commute
    c, _ = of8.forward_fp8(x, w, 1e-6, 0, 3.0)
    assert np.array_equal(c, of8.store_e4m3(3.0 * y))


# --- planted mistakes -------------------------------------------------------

def _mutant_store(kind):
    def f(v):
        v = np.asarray(v, float)
        if kind == "truncate":
            p, emin, _ = rounding.FORMATS["e4m3"]
            _, e = np.frexp(v)
            q = np.maximum(e - 1, emin) - (p - 1)
            r = np.ldexp(np.trunc(np.ldexp(v, -q)), q)
            return np.clip(r, -448, 448)
        if kind == "ties_away":
            p, emin, _ = rounding.FORMATS["e4m3"]
            _, e = np.frexp(v)
            q = np.maximum(e - 1, emin) - (p - 1)
            s = np.ldexp(v, -q)
            r = np.ldexp(np.sign(s) * np.floor(np.abs(s) + 0.5), q)
            return np.clip(r, -448, 448)
        if kind == "no_subnormals":
            r = of8.store_e4m3(v)
            return np.where(np.abs(v) < 2.0 ** -6, 0.0, r)
        if kind == "e5m2_grid":
            r = rounding.round_to(v, "f16")
            p, emin = 3, -14
            _, e = np.frexp(r)
            q = np.maximum(e - 1, emin) - (p - 1)
            return np.clip(np.ldexp(np.rint(np.ldexp(v, -q)), q), -448, 448)
        raise ValueError(kind)
    return f


@pytest.mark.parametrize("kind", ["truncate", "ties_away", "no_subnormals", "e5m2_grid"])
def test_rounding_mutant_is_caught(kind):
    assert check_rounding_vs_torch(_mutant_store(kind)) > 0


def _forward_mutant(kind):
    def forward_fp8(x, gamma, eps, offset, scale):
        y, rstd = orm.forward_exact(x, gamma, eps, offset)
        if kind == "scale_dropped":
            y8 = of8.store_e4m3(y)
        elif kind == "round_before_scale":
            y8 = of8.store_e4m3(of8.store_e4m3(y) * scale)
        elif kind == "divide_by_scale":
            y8 = of8.store_e4m3(y / scale)
        else:
            raise ValueError(kind)
        return y8, rounding.round_to(rstd, "f32")
    return types.SimpleNamespace(forward_fp8=forward_fp8)


@pytest.mark.parametrize("kind", ["scale_dropped", "round_before_scale", "divide_by_scale"])
def test_forward_mutant_is_caught(kind):
    bad, _ = check_forward_vs_torch(_forward_mutant(kind))
    assert bad > 0
