"""Pins of the float64 LayerNorm oracle against facts fixed outside it, and
planted mistakes that those pins catch.  Host only."""
import types

import numpy as np
import pytest
import torch

from oracle import layer_norm as oln
from oracle import rounding


def _data(seed, r=5, n=29, scale=2.0, shift=0.7):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((r, n)) * scale + shift
    gamma = rng.uniform(0.5, 1.5, n)
    beta = rng.standard_normal(n) * 0.3
    dy = rng.standard_normal((r, n))
    return x, gamma, beta, dy


def check_forward_vs_torch(mod=oln, seed=1):
    x, gamma, beta, _ = _data(seed)
    eps = 1e-3
    y, mean, rstd = mod.forward_exact(x, gamma, beta, eps)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (x.shape[1],),
                                         weight=torch.from_numpy(gamma),
                                         bias=torch.from_numpy(beta),
                                         eps=float(np.float32(eps))).numpy()
    return float(np.max(np.abs(y - ref)) / np.max(np.abs(ref)))


def check_backward_vs_autograd(mod=oln, seed=2):
    x, gamma, beta, dy = _data(seed)
    eps = 1e-2
    xt = torch.from_numpy(x.copy()).requires_grad_(True)
    gt = torch.from_numpy(gamma.copy()).requires_grad_(True)
    bt = torch.from_numpy(beta.copy()).requires_grad_(True)
    torch.nn.functional.layer_norm(xt, (x.shape[1],), weight=gt, bias=bt,
                                   eps=float(np.float32(eps))).backward(torch.from_numpy(dy))
    mean, rstd = mod.stats_exact(x, eps)
    dx, dg, db = mod.backward_exact(dy, x, gamma, mean, rstd)
    errs = [np.max(np.abs(a - b.numpy())) / np.max(np.abs(b.numpy()))
            for a, b in ((dx, xt.grad), (dg, gt.grad), (db, bt.grad))]
    return float(max(errs))


def check_finite_differences(mod=oln, seed=3):
    x, gamma, beta, dy = _data(seed, r=3, n=9)
    eps = 0.05

    def loss(xv, gv, bv):
        y, _, _ = mod.forward_exact(xv, gv, bv, eps)
        return float(np.sum(dy * y))

    h = 1e-6

    def fd(arr, f):
        out = np.zeros_like(arr)
        it = np.nditer(arr, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            p = arr.copy(); p[i] += h
            m = arr.copy(); m[i] -= h
            out[i] = (f(p) - f(m)) / (2 * h)
        return out

    fx = fd(x, lambda v: loss(v, gamma, beta))
    fg = fd(gamma, lambda v: loss(x, v, beta))
    fb = fd(beta, lambda v: loss(x, gamma, v))
    mean, rstd = mod.stats_exact(x, eps)
    dx, dg, db = mod.backward_exact(dy, x, gamma, mean, rstd)
    return float(max(np.max(np.abs(a - b)) / np.max(np.abs(b))
                     for a, b in ((dx, fx), (dg, fg), (db, fb))))


def check_invariants(mod=oln, seed=4):
    """sum_j dx_j = 0 (y is invariant to shifting x); sum_j x_hat_j = 0;
    sum_j x_hat_j**2 = N var / (var + eps)."""
    x, gamma, beta, dy = _data(seed, r=6, n=21)
    eps = 3e-3
    mean, rstd = mod.stats_exact(x, eps)
    dx, _, _ = mod.backward_exact(dy, x, gamma, mean, rstd)
    y, _, _ = mod.forward_exact(x, np.ones(21), None, eps)
    var = np.var(x, axis=1)
    e1 = np.max(np.abs(dx.sum(axis=1))) / np.max(np.abs(dx))
    e2 = np.max(np.abs(y.sum(axis=1))) / np.max(np.abs(y))
    want = 21 * var / (var + float(np.float32(eps)))
    e3 = np.max(np.abs((y * y).sum(axis=1) - want) / want)
    return float(max(e1, e2, e3))


def _all_pins(m):
    return (check_forward_vs_torch(m) < 1e-13 and check_backward_vs_autograd(m) < 1e-12
            and check_finite_differences(m) < 1e-7 and check_invariants(m) < 1e-12)


def test_forward_matches_torch_float64():
    assert check_forward_vs_torch() < 1e-13


def test_backward_matches_torch_autograd():
    assert check_backward_vs_autograd() < 1e-12


def test_backward_finite_differences():
    assert check_finite_differences() < 1e-7


def test_invariants():
    assert check_invariants() < 1e-12


def test_bf16_store_matches_torch_cpu_bf16():
    """torch's CPU bf16 layer_norm (fp32 compute, one rounding): at least
    99.99% of outputs identical; the rest within one ulp or within the fp32
    noise of the terms x_hat*gamma and beta that cancel."""
    g = torch.Generator().manual_seed(6)
    xb = torch.randn(4096, 512, generator=g).to(torch.bfloat16)
    wb = (torch.rand(512, generator=g) * 0.2 + 0.9).to(torch.bfloat16)
    bb = (torch.randn(512, generator=g) * 0.1).to(torch.bfloat16)
    ref = torch.nn.functional.layer_norm(xb, (512,), weight=wb, bias=bb,
                                         eps=1e-5).double().numpy()
    y, _, _ = oln.forward(xb.double().numpy(), wb.double().numpy(), bb.double().numpy(), 1e-5,
                          "bf16")
    d = rounding.ulp_distance(y, ref, "bf16")
    assert np.mean(d == 0) >= 0.9999
    scale = np.sqrt(np.mean(ref * ref, axis=1, keepdims=True))
    assert np.all((d <= 1) | (np.abs(y - ref) <= 1e-2 * scale))


def test_outputs_are_stored_values():
    x, gamma, beta, dy = _data(7)
    for fmt in ("f32", "bf16", "f16"):
        y, mean, rstd = oln.forward(x, gamma, beta, 1e-5, fmt)
        assert np.array_equal(rounding.round_to(y, fmt), y)
        assert np.array_equal(rounding.round_to(mean, "f32"), mean)
        assert np.array_equal(rounding.round_to(rstd, "f32"), rstd)
        dx, dg, db = oln.backward(dy, x, gamma, mean, rstd, fmt)
        assert np.array_equal(rounding.round_to(dx, fmt), dx)
        assert np.array_equal(rounding.round_to(db, "f32"), db)


def test_no_bias_is_zero_bias():
    x, gamma, beta, _ = _data(8)
    a = oln.forward(x, gamma, None, 1e-5, "bf16")
    b = oln.forward(x, gamma, np.zeros_like(beta), 1e-5, "bf16")
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


# --- planted mistakes -------------------------------------------------------

def _copy(**kw):
    m = types.SimpleNamespace(stats_exact=oln.stats_exact, backward_exact=oln.backward_exact)
    for k, v in kw.items():
        setattr(m, k, v)

    def forward_exact(x, gamma, beta, eps):
        x = np.asarray(x, float)
        mean, rstd = m.stats_exact(x, eps)
        y = (x - mean[..., None]) * rstd[..., None] * gamma
        return (y if beta is None else y + beta), mean, rstd
    m.forward_exact = forward_exact
    return m


def _stats_sum_var(x, eps):
    x = np.asarray(x, float)
    mean = x.mean(axis=-1)
    return mean, 1 / np.sqrt(((x - mean[..., None]) ** 2).sum(axis=-1) + np.float32(eps))


def _stats_eps_outside(x, eps):
    x = np.asarray(x, float)
    mean = x.mean(axis=-1)
    return mean, 1 / (np.sqrt(((x - mean[..., None]) ** 2).mean(axis=-1)) + np.float32(eps))


def _stats_no_centering(x, eps):
    x = np.asarray(x, float)
    mean = x.mean(axis=-1)
    return mean, 1 / np.sqrt((x * x).mean(axis=-1) + np.float32(eps))


def _bwd(kind):
    def f(dy, x, gamma, mean, rstd):
        n = x.shape[-1]
        xh = (x - mean[..., None]) * rstd[..., None]
        g = dy * gamma
        c1 = g.sum(-1) / n
        c2 = (g * xh).sum(-1) / n
        if kind == "drop_c1":
            dx = rstd[..., None] * (g - xh * c2[..., None])
        elif kind == "drop_c2":
            dx = rstd[..., None] * (g - c1[..., None])
        elif kind == "sign":
            dx = rstd[..., None] * (g + c1[..., None] - xh * c2[..., None])
        else:
            dx = rstd[..., None] * (g - c1[..., None] - xh * c2[..., None])
        dg = (dy * (x if kind == "dg_uses_x" else xh)).sum(0)
        db = (g if kind == "db_uses_g" else dy).sum(0)
        return dx, dg, db
    return f


MUTANTS = {
    "sum_not_mean_var": dict(stats_exact=_stats_sum_var),
    "eps_outside": dict(stats_exact=_stats_eps_outside),
    "no_centering": dict(stats_exact=_stats_no_centering),
    "drop_c1": dict(backward_exact=_bwd("drop_c1")),
    "drop_c2": dict(backward_exact=_bwd("drop_c2")),
    "sign": dict(backward_exact=_bwd("sign")),
    "dg_uses_x": dict(backward_exact=_bwd("dg_uses_x")),
    "db_uses_g": dict(backward_exact=_bwd("db_uses_g")),
}


def test_unmutated_copy_passes():
    assert _all_pins(_copy())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    assert not _all_pins(_copy(**MUTANTS[name]))
