"""Pins of the float64 oracle against facts fixed outside the oracle itself.

Host only.  Each pin is written as a check that returns its worst error, so
that ``test_oracle_mutations.py`` can run the same checks on deliberately
broken copies of the oracle and show that every plausible mistake fails at
least one of them.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import rounding
from oracle import rms_norm as orm

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ----------------------------------------------------------------------------
# checks (shared with the mutation tests)
# ----------------------------------------------------------------------------

def check_worked_example(mod=orm, rnd=rounding.round_to):
    """Worked bf16 example of the precision page: returns the number of
    printed values the oracle misses (0 when it matches)."""
    g = _golden("worked_example.json")
    gamma = float(rnd(g["gamma_requested"], "bf16"))
    x_hat = float(np.float32(g["x_hat_float32_of"]))
    once = float(mod.store_y(np.array(x_hat), np.array(gamma), "bf16", mod.ROUND_ONCE))
    twice = float(mod.store_y(np.array(x_hat), np.array(gamma), "bf16", mod.ROUND_TWICE))
    return sum([gamma != g["gamma_bf16"], once != g["round_once"], twice != g["round_twice"]])


def check_forward_vs_torch_f64(mod=orm, offset=0, seed=1):
    """Relative error of the unrounded forward against torch's CPU rms_norm
    run in float64 (the plain definition, computed by the library)."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((7, 37)) * 3.0
    gamma = rng.uniform(0.5, 1.5, 37)
    eps = 1e-3
    y, rstd = mod.forward_exact(x, gamma, eps, offset)
    w = torch.from_numpy(gamma + (1.0 if offset else 0.0))
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (37,), weight=w,
                                       eps=float(np.float32(eps))).numpy()
    return float(np.max(np.abs(y - ref) / np.maximum(np.abs(ref), 1e-300)))


def check_backward_vs_torch_autograd(mod=orm, offset=0, seed=2):
    """Relative error of the unrounded backward against torch autograd
    through CPU rms_norm in float64."""
    rng = np.random.default_rng(seed)
    r, n = 5, 29
    x = rng.standard_normal((r, n)) * 2.0
    gamma = rng.uniform(0.5, 1.5, n)
    dy = rng.standard_normal((r, n))
    eps = 1e-2
    xt = torch.from_numpy(x.copy()).requires_grad_(True)
    wt = torch.from_numpy(gamma + (1.0 if offset else 0.0)).requires_grad_(True)
    yt = torch.nn.functional.rms_norm(xt, (n,), weight=wt, eps=float(np.float32(eps)))
    yt.backward(torch.from_numpy(dy))
    rstd = mod.rstd_exact(x, eps)
    dx, dw = mod.backward_exact(dy, x, gamma, rstd, offset)
    ex = np.max(np.abs(dx - xt.grad.numpy())) / np.max(np.abs(xt.grad.numpy()))
    ew = np.max(np.abs(dw - wt.grad.numpy())) / np.max(np.abs(wt.grad.numpy()))
    return float(max(ex, ew))


def check_backward_finite_differences(mod=orm, offset=0, seed=3):
    """Relative error of the backward against central differences of
    L = sum(dy * y) with y the unrounded forward."""
    rng = np.random.default_rng(seed)
    r, n = 3, 11
    x = rng.standard_normal((r, n))
    gamma = rng.uniform(0.5, 1.5, n)
    dy = rng.standard_normal((r, n))
    eps = 0.05

    def loss(xv, gv):
        y, _ = mod.forward_exact(xv, gv, eps, offset)
        return float(np.sum(dy * y))

    h = 1e-6
    fd_x = np.zeros_like(x)
    for i in range(r):
        for j in range(n):
            xp = x.copy(); xp[i, j] += h
            xm = x.copy(); xm[i, j] -= h
            fd_x[i, j] = (loss(xp, gamma) - loss(xm, gamma)) / (2 * h)
    fd_g = np.zeros_like(gamma)
    for j in range(n):
        gp = gamma.copy(); gp[j] += h
        gm = gamma.copy(); gm[j] -= h
        fd_g[j] = (loss(x, gp) - loss(x, gm)) / (2 * h)
    rstd = mod.rstd_exact(x, eps)
    dx, dw = mod.backward_exact(dy, x, gamma, rstd, offset)
    ex = np.max(np.abs(dx - fd_x)) / np.max(np.abs(fd_x))
    ew = np.max(np.abs(dw - fd_g)) / np.max(np.abs(fd_g))
    return float(max(ex, ew))


def check_dx_orthogonal_to_x(mod=orm, seed=4):
    """At eps = 0 the forward is invariant to scaling x, so sum_j x_j dx_j = 0
    in every row.  Returns the largest |<x, dx>| relative to |x| |dx|."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((6, 19))
    gamma = rng.uniform(0.5, 1.5, 19)
    dy = rng.standard_normal((6, 19))
    rstd = mod.rstd_exact(x, 0.0)
    dx, _ = mod.backward_exact(dy, x, gamma, rstd, 0)
    dots = np.abs(np.sum(x * dx, axis=1))
    scale = np.linalg.norm(x, axis=1) * np.linalg.norm(dx, axis=1)
    return float(np.max(dots / scale))


def check_sum_of_squares_identity(mod=orm, seed=5):
    """sum_j x_hat_j**2 = n * ms / (ms + eps) for every row; returns the
    worst relative error."""
    rng = np.random.default_rng(seed)
    n = 23
    x = rng.standard_normal((4, n)) * 0.1
    eps = 3e-3
    y, _ = mod.forward_exact(x, np.ones(n), eps, 0)
    ms = np.mean(x * x, axis=1)
    want = n * ms / (ms + float(np.float32(eps)))
    return float(np.max(np.abs(np.sum(y * y, axis=1) - want) / want))


def check_bf16_vs_torch_cpu(mod=orm, seed=6):
    """Share of bf16 outputs equal to torch's CPU bf16 rms_norm and the worst
    ulp distance, at the page's 4096 x 512 shape (footnote 2 of the precision
    page: that routine multiplies in float32 and converts last)."""
    g = torch.Generator().manual_seed(seed)
    xb = torch.randn(4096, 512, generator=g).to(torch.bfloat16)
    wb = (torch.rand(512, generator=g) * 0.2 + 0.9).to(torch.bfloat16)
    eps = 1e-6
    ref = torch.nn.functional.rms_norm(xb, (512,), weight=wb, eps=eps).to(torch.float64).numpy()
    y, _ = mod.forward(xb.to(torch.float64).numpy(), wb.to(torch.float64).numpy(),
                       eps, 0, "bf16", mod.ROUND_ONCE)
    d = rounding.ulp_distance(y, ref, "bf16")
    return float(np.mean(d == 0)), int(d.max())


# ----------------------------------------------------------------------------
# rounding pins
# ----------------------------------------------------------------------------

def test_worked_example():
    assert check_worked_example() == 0


def _page_bit_trick_bf16(v32):
    """The page's bf16 helper restated: add 0x7FFF plus the lowest kept bit
    to the float32 pattern, then clear the low 16 bits.  Finite inputs only."""
    bits = np.asarray(v32, dtype=np.float32).view(np.uint32)
    rounded = bits + np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))
    return (rounded & np.uint32(0xFFFF0000)).view(np.float32)


def test_two_million_sample_count():
    """The page's 2M-sample experiment, with the page's float32 product:
    the count of differing outputs and the largest relative difference."""
    g = _golden("two_million_samples.json")
    rng = np.random.default_rng(42)
    x_hat = rng.standard_normal(g["samples"]).astype(np.float32)
    gamma = rng.uniform(0.9, 1.1, x_hat.size).astype(np.float32)
    gb = rounding.round_to(gamma, "bf16").astype(np.float32)
    once = rounding.round_to((x_hat * gb).astype(np.float32), "bf16")
    t = rounding.round_to(x_hat, "bf16").astype(np.float32)
    twice = rounding.round_to((t * gb).astype(np.float32), "bf16")
    different = int(np.count_nonzero(once != twice))
    assert different == g["different"]
    assert round(100.0 * different / x_hat.size, 2) == g["share_percent_2dp"]
    nz = once != 0
    rel = np.abs(once[nz] - twice[nz]) / np.abs(once[nz])
    assert 100.0 * rel.max() == g["largest_relative_difference_percent"]
    # The oracle's own store rounds the exact product once.  It differs from
    # the page's float32-then-bf16 rounding only where the float32 product
    # lands exactly on a bf16 midpoint, i.e. a handful of the 2M samples.
    once64 = orm.store_y(x_hat.astype(np.float64), gb.astype(np.float64), "bf16", orm.ROUND_ONCE)
    twice64 = orm.store_y(x_hat.astype(np.float64), gb.astype(np.float64), "bf16", orm.ROUND_TWICE)
    assert np.count_nonzero(once64 != once) < 100
    assert np.count_nonzero(twice64 != twice) < 100
    assert abs(int(np.count_nonzero(once64 != twice64)) - g["different"]) < 100


def _all_bf16_values():
    bits = (np.arange(1 << 16, dtype=np.uint32) << np.uint32(16))
    return bits.view(np.float32).astype(np.float64)


def _all_f16_values():
    return np.arange(1 << 16, dtype=np.uint16).view(np.float16).astype(np.float64)


@pytest.mark.parametrize("fmt,values", [("bf16", _all_bf16_values), ("f16", _all_f16_values)])
def test_every_value_and_midpoint(fmt, values):
    """Every finite value of the format is a fixed point; every midpoint
    between neighbours rounds to the neighbour with the even last bit; a hair
    either side of a midpoint rounds to the nearer neighbour."""
    v = values()
    fin = v[np.isfinite(v)]
    assert np.array_equal(rounding.round_to(fin, fmt), fin)
    pos = np.unique(fin[fin >= 0])            # ascending, 0 .. max
    lo, hi = pos[:-1], pos[1:]
    mid = (lo + hi) / 2.0                     # exact in float64
    r = rounding.round_to(mid, fmt)
    # position of lo in the ordered list of values is its index; even index
    # means an even last significand bit.
    idx = np.arange(lo.size)
    want = np.where(idx % 2 == 0, lo, hi)
    assert np.array_equal(r, want)
    tiny = (hi - lo) * 1e-6
    assert np.array_equal(rounding.round_to(mid - tiny, fmt), lo)
    assert np.array_equal(rounding.round_to(mid + tiny, fmt), hi)
    # negative side mirrors the positive side
    assert np.array_equal(rounding.round_to(-mid, fmt), -want)
    # overflow: half a step past the largest finite value goes to infinity
    top = rounding.max_finite(fmt)
    step = top - pos[-2]
    assert rounding.round_to(top + step / 2, fmt) == np.inf
    assert rounding.round_to(top + step / 2 * (1 - 1e-9), fmt) == top
    assert rounding.round_to(-(top + step), fmt) == -np.inf


def test_f16_against_numpy_cast():
    """numpy's float64 -> float16 cast rounds once to nearest even, including
    subnormals and overflow."""
    rng = np.random.default_rng(7)
    m = rng.uniform(1.0, 2.0, 400_000)
    e = rng.integers(-30, 18, m.size)
    s = rng.choice([-1.0, 1.0], m.size)
    v = s * np.ldexp(m, e)
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).astype(np.float64)
    got = rounding.round_to(v, "f16")
    assert np.array_equal(got, ref)
    assert np.array_equal(np.signbit(got), np.signbit(ref))


def test_f32_against_numpy_cast():
    rng = np.random.default_rng(8)
    m = rng.uniform(1.0, 2.0, 400_000)
    e = rng.integers(-155, 130, m.size)
    v = rng.choice([-1.0, 1.0], m.size) * np.ldexp(m, e)
    with np.errstate(over="ignore"):
        ref = v.astype(np.float32).astype(np.float64)
    assert np.array_equal(rounding.round_to(v, "f32"), ref)


def test_bf16_against_torch_and_page_helper():
    """float32 patterns (a strided sweep over all 2**32, NaN excluded) rounded
    to bf16 by the oracle, by torch's CPU cast and by the page's bit helper."""
    bits = np.arange(0, 1 << 32, 4099, dtype=np.uint64).astype(np.uint32)
    # add the patterns right around every rounding boundary of a few binades
    extra = np.array([0x3F808000, 0x3F818000, 0x3F807FFF, 0x3F808001, 0x7F7FFFFF,
                      0x7F7F7FFF, 0x7F7F8000, 0x00008000, 0x00018000, 0x80008000],
                     dtype=np.uint32)
    bits = np.concatenate([bits, extra])
    v32 = bits.view(np.float32)
    v32 = v32[~np.isnan(v32)]
    ours = rounding.round_to(v32.astype(np.float64), "bf16")
    theirs = torch.from_numpy(v32.copy()).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(ours, theirs)
    fin = np.isfinite(v32)
    page = _page_bit_trick_bf16(v32[fin]).astype(np.float64)
    assert np.array_equal(ours[fin], page)


def test_ulp_distance():
    a = np.array([1.0, 1.0, 0.0, 2.0 ** -24, rounding.max_finite("f16"), -1.0])
    b = np.array([1.0 + 2 ** -10, 1.0 + 2 ** -9, -0.0, -(2.0 ** -24), np.inf, 1.0])
    d = rounding.ulp_distance(a, b, "f16")
    assert list(d) == [1, 2, 0, 2, 1, 2 * 15 * 1024]


# ----------------------------------------------------------------------------
# forward pins
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("offset", [0, 1])
def test_forward_matches_torch_float64(offset):
    assert check_forward_vs_torch_f64(offset=offset) < 1e-13


def test_forward_bf16_matches_torch_cpu_bf16():
    same, worst = check_bf16_vs_torch_cpu()
    assert same >= 0.999 and worst <= 1


def test_forward_closed_forms():
    # one element, eps = 0: x_hat = sign(x)
    x = np.array([[3.5], [-0.25], [1e-30]])
    y, rstd = orm.forward_exact(x, np.array([1.0]), 0.0)
    assert np.array_equal(y[:, 0], np.sign(x[:, 0]))
    # constant row a, eps = 0: every x_hat is sign(a)
    x = np.full((2, 9), -7.0)
    y, _ = orm.forward_exact(x, np.ones(9), 0.0)
    assert np.array_equal(y, -np.ones((2, 9)))
    # zero row with eps > 0: rstd = 1/sqrt(eps) and y = 0
    y, rstd = orm.forward_exact(np.zeros((1, 4)), np.ones(4), 0.25)
    assert rstd[0] == 2.0 and not np.any(y)


def test_forward_scale_invariance():
    """eps = 0: multiplying x by a power of two leaves y bit-identical."""
    rng = np.random.default_rng(9)
    x = rng.standard_normal((5, 33))
    gamma = rng.uniform(0.5, 1.5, 33)
    y0, _ = orm.forward_exact(x, gamma, 0.0)
    for k in (-40, -3, 5, 60):
        yk, _ = orm.forward_exact(np.ldexp(x, k), gamma, 0.0)
        assert np.array_equal(yk, y0)


def test_forward_sum_of_squares_identity():
    assert check_sum_of_squares_identity() < 1e-13


def test_gemma_gain_zero_gamma_is_plain_round():
    """offset 1 with gamma = 0 stores round(x_hat); so does offset 0 with
    gamma = 1."""
    rng = np.random.default_rng(10)
    x = rng.standard_normal((4, 16))
    for fmt in ("bf16", "f16", "f32"):
        ya, ra = orm.forward(x, np.zeros(16), 1e-5, 1, fmt)
        yb, rb = orm.forward(x, np.ones(16), 1e-5, 0, fmt)
        assert np.array_equal(ya, yb) and np.array_equal(ra, rb)


def test_round_twice_equals_round_once_in_f32():
    """In float32 the intermediate of round twice is x_hat rounded to float32,
    and float32 times float32 is exact in float64, so the two modes differ at
    most where round once would land on a different float32 neighbour:
    never by more than one ulp."""
    rng = np.random.default_rng(11)
    x = rng.standard_normal((8, 64))
    g = rounding.round_to(rng.uniform(0.9, 1.1, 64), "f32")
    a, _ = orm.forward(x, g, 1e-6, 0, "f32", orm.ROUND_ONCE)
    b, _ = orm.forward(x, g, 1e-6, 0, "f32", orm.ROUND_TWICE)
    assert rounding.ulp_distance(a, b, "f32").max() <= 1


def test_rstd_output_is_float32():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((16, 40))
    _, rstd = orm.forward(x, np.ones(40), 1e-5, 0, "bf16")
    assert np.array_equal(rstd.astype(np.float32).astype(np.float64), rstd)


# ----------------------------------------------------------------------------
# backward pins
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("offset", [0, 1])
def test_backward_finite_differences(offset):
    assert check_backward_finite_differences(offset=offset) < 1e-7


@pytest.mark.parametrize("offset", [0, 1])
def test_backward_matches_torch_autograd(offset):
    assert check_backward_vs_torch_autograd(offset=offset) < 1e-12


def test_backward_dx_orthogonal_to_x_at_zero_eps():
    assert check_dx_orthogonal_to_x() < 1e-13


def test_backward_dgamma_brute_force():
    """dgamma_j = sum over rows of dy * x_hat, by explicit loops."""
    rng = np.random.default_rng(13)
    r, n = 4, 6
    x = rng.standard_normal((r, n))
    dy = rng.standard_normal((r, n))
    rstd = orm.rstd_exact(x, 1e-5)
    _, dw = orm.backward_exact(dy, x, rng.uniform(size=n), rstd, 0)
    for j in range(n):
        acc = 0.0
        for i in range(r):
            acc += dy[i, j] * x[i, j] * rstd[i]
        assert abs(acc - dw[j]) <= 1e-14 * max(1.0, abs(acc))


def test_backward_rounding_formats():
    rng = np.random.default_rng(14)
    x = rng.standard_normal((3, 10))
    dy = rng.standard_normal((3, 10))
    rstd = orm.rstd_exact(x, 1e-5)
    for fmt in ("bf16", "f16", "f32"):
        dx, dw = orm.backward(dy, x, np.ones(10), rstd, 0, fmt)
        assert np.array_equal(rounding.round_to(dx, fmt), dx)
        assert np.array_equal(rounding.round_to(dw, "f32"), dw)


def test_oracle_package_exports():
    for name in ("forward", "backward", "round_to", "ulp_distance", "rstd_exact"):
        assert hasattr(oracle, name)
