"""Plant plausible mistakes in copies of the oracle and check that the pins
catch each one.  Host only; the real oracle is never modified."""
import types

import numpy as np
import pytest

from oracle import rounding
from oracle import rms_norm as orm

import test_oracle as pins


def _copy(**overrides):
    m = types.SimpleNamespace(**{k: getattr(orm, k) for k in dir(orm) if not k.startswith("__")})
    for k, v in overrides.items():
        setattr(m, k, v)
    # forward_exact / forward / backward call through the copy's helpers
    m.forward_exact = lambda x, gamma, eps, offset=0: _fwd_exact(m, x, gamma, eps, offset)
    if "backward_exact" not in overrides:
        m.backward_exact = lambda dy, x, gamma, rstd, offset=0: orm.backward_exact(dy, x, gamma, rstd, offset)
    m.forward = lambda x, gamma, eps, offset, fmt, cast_mode=orm.ROUND_ONCE: _fwd(m, x, gamma, eps, offset, fmt, cast_mode)
    return m


def _fwd_exact(m, x, gamma, eps, offset):
    x = np.asarray(x, dtype=np.float64)
    rstd = m.rstd_exact(x, eps)
    return x * rstd[..., None] * m.gain(gamma, offset), rstd


def _fwd(m, x, gamma, eps, offset, fmt, cast_mode):
    x = np.asarray(x, dtype=np.float64)
    rstd = m.rstd_exact(x, eps)
    y = m.store_y(x * rstd[..., None], m.gain(gamma, offset), fmt, cast_mode)
    return y, rounding.round_to(rstd, "f32")


def _all_pins(m):
    """True when every pin still passes on module ``m``."""
    ok = pins.check_worked_example(m) == 0
    for off in (0, 1):
        ok &= pins.check_forward_vs_torch_f64(m, offset=off) < 1e-13
        ok &= pins.check_backward_finite_differences(m, offset=off) < 1e-7
        ok &= pins.check_backward_vs_torch_autograd(m, offset=off) < 1e-12
    ok &= pins.check_dx_orthogonal_to_x(m) < 1e-13
    ok &= pins.check_sum_of_squares_identity(m) < 1e-13
    same, worst = pins.check_bf16_vs_torch_cpu(m)
    ok &= same >= 0.999 and worst <= 1
    return bool(ok)


def _eps_outside_root(x, eps):
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / (np.sqrt(np.mean(x * x, axis=-1)) + orm.eps_value(eps))


def _sum_not_mean(x, eps):
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / np.sqrt(np.sum(x * x, axis=-1) + orm.eps_value(eps))


def _eps_as_float64_squared(x, eps):
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / np.sqrt(np.mean(x * x, axis=-1) + orm.eps_value(eps) ** 2)


def _bwd_factory(kind):
    def bwd(dy, x, gamma, rstd, offset=0):
        dy = np.asarray(dy, float); x = np.asarray(x, float); rstd = np.asarray(rstd, float)
        n = x.shape[-1]
        xh = x * rstd[..., None]
        g = dy * (gamma if kind == "offset_ignored" else orm.gain(gamma, offset))
        c = np.sum(g * xh, axis=-1) / n
        if kind == "drop_c":
            dx = rstd[..., None] * g
        elif kind == "sign":
            dx = rstd[..., None] * (g + xh * c[..., None])
        elif kind == "c_sum_not_mean":
            dx = rstd[..., None] * (g - xh * (c * n)[..., None])
        elif kind == "no_rstd":
            dx = g - xh * c[..., None]
        else:
            dx = rstd[..., None] * (g - xh * c[..., None])
        if kind == "dw_uses_x":
            dw = np.sum(dy * x, axis=0)
        elif kind == "dw_uses_g":
            dw = np.sum(g * xh, axis=0)
        else:
            dw = np.sum(dy * xh, axis=0)
        return dx, dw
    return bwd


def _store_round_once_always(x_hat, g, fmt, cast_mode):
    return rounding.round_to(x_hat * g, fmt)


def _store_twice_rounds_gain(x_hat, g, fmt, cast_mode):
    if cast_mode == orm.ROUND_ONCE:
        return rounding.round_to(x_hat * g, fmt)
    return rounding.round_to(x_hat * rounding.round_to(g, fmt), fmt)


def _store_truncating(x_hat, g, fmt, cast_mode):
    # chop toward zero instead of rounding to nearest
    p = rounding.FORMATS[fmt][0]
    v = x_hat * g
    _, e = np.frexp(v)
    q = e - p
    return np.trunc(np.ldexp(v, -q)) * np.ldexp(1.0, q)


def _gain_ignores_offset(gamma, offset):
    return np.asarray(gamma, dtype=np.float64)


MUTANTS = {
    "eps_outside_root": dict(rstd_exact=_eps_outside_root),
    "sum_not_mean": dict(rstd_exact=_sum_not_mean),
    "eps_squared": dict(rstd_exact=_eps_as_float64_squared),
    "bwd_drop_c": dict(backward_exact=_bwd_factory("drop_c")),
    "bwd_sign": dict(backward_exact=_bwd_factory("sign")),
    "bwd_c_sum_not_mean": dict(backward_exact=_bwd_factory("c_sum_not_mean")),
    "bwd_no_rstd": dict(backward_exact=_bwd_factory("no_rstd")),
    "bwd_offset_ignored": dict(backward_exact=_bwd_factory("offset_ignored")),
    "bwd_dw_uses_x": dict(backward_exact=_bwd_factory("dw_uses_x")),
    "bwd_dw_uses_g": dict(backward_exact=_bwd_factory("dw_uses_g")),
    "store_once_always": dict(store_y=_store_round_once_always),
    "store_twice_rounds_gain": dict(store_y=_store_twice_rounds_gain),
    "store_truncates": dict(store_y=_store_truncating),
    "gain_ignores_offset": dict(gain=_gain_ignores_offset),
}


def test_unmutated_copy_passes():
    assert _all_pins(_copy())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    assert not _all_pins(_copy(**MUTANTS[name]))


def _round_half_away(v, fmt):
    p, emin, _ = rounding.FORMATS[fmt]
    v = np.asarray(v, dtype=np.float64)
    _, e = np.frexp(v)
    q = np.maximum(e - 1, emin) - (p - 1)
    s = np.ldexp(v, -q)
    return np.ldexp(np.sign(s) * np.floor(np.abs(s) + 0.5), q)


def _round_wrong_width(v, fmt):
    p, emin, emax = rounding.FORMATS[fmt]
    v = np.asarray(v, dtype=np.float64)
    _, e = np.frexp(v)
    q = np.maximum(e - 1, emin) - p          # one bit too many
    return np.ldexp(np.rint(np.ldexp(v, -q)), q)


@pytest.mark.parametrize("bad", [_round_half_away, _round_wrong_width])
def test_rounding_mutants_are_caught(bad):
    """The page's example and the 2M count reject a rounding routine with the
    wrong tie rule or the wrong significand width."""
    caught = pins.check_worked_example(orm, rnd=bad) != 0
    rng = np.random.default_rng(42)
    x_hat = rng.standard_normal(2_000_000).astype(np.float32)
    gamma = rng.uniform(0.9, 1.1, x_hat.size).astype(np.float32)
    gb = bad(gamma, "bf16").astype(np.float32)
    once = bad((x_hat * gb).astype(np.float32), "bf16")
    twice = bad((bad(x_hat, "bf16").astype(np.float32) * gb).astype(np.float32), "bf16")
    caught |= int(np.count_nonzero(once != twice)) != 495539
    assert caught
