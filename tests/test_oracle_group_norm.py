"""Pins of the float64 GroupNorm oracle against facts fixed outside it
(torch's CPU group_norm in float64 and its autograd, finite differences,
invariants, the special cases G = 1 and G = C, the upstream-of-ones case of
Liger-Kernel PR #1608, torch's CPU bf16 group_norm), and planted mistakes
those pins catch.  Host only."""
import types

import numpy as np
import pytest
import torch

from oracle import group_norm as ogn
from oracle import layer_norm as oln
from oracle import rounding


def _data(seed, n=2, c=6, s=10, shift=0.8, scale=1.7):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, c, s)) * scale + shift
    gamma = rng.uniform(0.5, 1.5, c)
    beta = rng.standard_normal(c) * 0.3
    dy = rng.standard_normal((n, c, s))
    return x, gamma, beta, dy


def check_forward_vs_torch(mod=ogn, seed=1, groups=3):
    x, gamma, beta, _ = _data(seed)
    eps = 1e-3
    y, mean, rstd = mod.forward_exact(x, gamma, beta, groups, eps)
    ref = torch.nn.functional.group_norm(torch.from_numpy(x), groups, torch.from_numpy(gamma),
                                         torch.from_numpy(beta), float(np.float32(eps))).numpy()
    return float(np.max(np.abs(y - ref)) / np.max(np.abs(ref)))


def check_backward_vs_autograd(mod=ogn, seed=2, groups=2):
    x, gamma, beta, dy = _data(seed)
    eps = 1e-2
    xt = torch.from_numpy(x.copy()).requires_grad_(True)
    gt = torch.from_numpy(gamma.copy()).requires_grad_(True)
    bt = torch.from_numpy(beta.copy()).requires_grad_(True)
    torch.nn.functional.group_norm(xt, groups, gt, bt, float(np.float32(eps))).backward(
        torch.from_numpy(dy))
    mean, rstd = mod.stats_exact(x, groups, eps)
    dx, dg, db = mod.backward_exact(dy, x, gamma, mean, rstd, groups)
    return float(max(np.max(np.abs(a - b.numpy())) / np.max(np.abs(b.numpy()))
                     for a, b in ((dx, xt.grad), (dg, gt.grad), (db, bt.grad))))


def check_finite_differences(mod=ogn, seed=3, groups=2):
    x, gamma, beta, dy = _data(seed, n=2, c=4, s=3)
    eps = 0.05
    h = 1e-6

    def loss(xv, gv, bv):
        return float(np.sum(dy * mod.forward_exact(xv, gv, bv, groups, eps)[0]))

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
    mean, rstd = mod.stats_exact(x, groups, eps)
    dx, dg, db = mod.backward_exact(dy, x, gamma, mean, rstd, groups)
    return float(max(np.max(np.abs(a - b)) / np.max(np.abs(b))
                     for a, b in ((dx, fx), (dg, fg), (db, fb))))


def check_invariants(mod=ogn, seed=4, groups=3):
    """Per group: sum of dx = 0 and sum of x_hat = 0; the upstream-of-ones
    case of Liger-Kernel PR #1608 (W = 1, dy = 1): dx = 0 and dB = n * S."""
    x, gamma, beta, dy = _data(seed)
    n, c, s = x.shape
    eps = 1e-4
    mean, rstd = mod.stats_exact(x, groups, eps)
    dx, _, _ = mod.backward_exact(dy, x, gamma, mean, rstd, groups)
    e1 = np.max(np.abs(dx.reshape(n, groups, -1).sum(-1))) / np.max(np.abs(dx))
    y, _, _ = mod.forward_exact(x, np.ones(c), None, groups, eps)
    e2 = np.max(np.abs(y.reshape(n, groups, -1).sum(-1))) / np.max(np.abs(y))
    ones = np.ones_like(x)
    dx1, _, db1 = mod.backward_exact(ones, x, np.ones(c), mean, rstd, groups)
    e3 = np.max(np.abs(dx1)) + np.max(np.abs(db1 - n * s))
    return float(max(e1, e2, e3))


def check_special_groups(mod=ogn, seed=5):
    """G = 1 is a LayerNorm over channels x positions with a per-channel
    gain (the LayerNorm oracle, pinned on its own); G = C normalises each
    channel alone (torch's instance_norm)."""
    x, gamma, beta, dy = _data(seed)
    n, c, s = x.shape
    eps = 1e-3
    y1, m1, r1 = mod.forward_exact(x, gamma, beta, 1, eps)
    g_full = np.repeat(gamma, s)
    b_full = np.repeat(beta, s)
    yl, ml, rl = oln.forward_exact(x.reshape(n, c * s), g_full, b_full, eps)
    e1 = np.max(np.abs(y1.reshape(n, -1) - yl))
    dx1, dg1, db1 = mod.backward_exact(dy, x, gamma, m1, r1, 1)
    dxl, dgl, dbl = oln.backward_exact(dy.reshape(n, -1), x.reshape(n, -1), g_full, ml, rl)
    e2 = np.max(np.abs(dx1.reshape(n, -1) - dxl))
    e3 = np.max(np.abs(dg1 - dgl.reshape(c, s).sum(-1))) + np.max(np.abs(db1 - dbl.reshape(c, s).sum(-1)))
    yc, _, _ = mod.forward_exact(x, gamma, beta, c, eps)
    ref = torch.nn.functional.instance_norm(torch.from_numpy(x), weight=torch.from_numpy(gamma),
                                            bias=torch.from_numpy(beta),
                                            eps=float(np.float32(eps))).numpy()
    e4 = np.max(np.abs(yc - ref))
    return float(max(e1, e2, e3, e4))


def _all_pins(m):
    return (check_forward_vs_torch(m) < 1e-13 and check_backward_vs_autograd(m) < 1e-12
            and check_finite_differences(m) < 1e-7 and check_invariants(m) < 1e-12
            and check_special_groups(m) < 1e-12)


def test_forward_matches_torch_float64():
    assert check_forward_vs_torch() < 1e-13


def test_backward_matches_torch_autograd():
    assert check_backward_vs_autograd() < 1e-12


def test_backward_finite_differences():
    assert check_finite_differences() < 1e-7


def test_invariants_and_upstream_of_ones():
    assert check_invariants() < 1e-12


def test_one_group_and_one_group_per_channel():
    assert check_special_groups() < 1e-12


def test_bf16_store_matches_torch_cpu_bf16():
    """torch's CPU bf16 group_norm (fp32 statistics, one rounding): at least
    99.9% identical; the rest one ulp apart or within the fp32 noise of the
    terms x_hat * W and B."""
    g = torch.Generator().manual_seed(6)
    xb = (torch.randn(4, 32, 256, generator=g) + 0.5).to(torch.bfloat16)
    wb = (torch.rand(32, generator=g) * 0.2 + 0.9).to(torch.bfloat16)
    bb = (torch.randn(32, generator=g) * 0.1).to(torch.bfloat16)
    ref = torch.nn.functional.group_norm(xb, 8, wb, bb, 1e-5).double().numpy()
    y, _, _ = ogn.forward(xb.double().numpy(), wb.double().numpy(), bb.double().numpy(), 8,
                          1e-5, "bf16")
    d = rounding.ulp_distance(y, ref, "bf16")
    assert np.mean(d == 0) >= 0.999
    assert np.all((d <= 1) | (np.abs(y - ref) <= 1e-2))


def test_outputs_are_stored_values():
    x, gamma, beta, dy = _data(7)
    for fmt in ("f32", "bf16", "f16"):
        y, mean, rstd = ogn.forward(x, gamma, beta, 2, 1e-5, fmt)
        assert np.array_equal(rounding.round_to(y, fmt), y)
        assert np.array_equal(rounding.round_to(rstd, "f32"), rstd)
        dx, dg, db = ogn.backward(dy, x, gamma, mean, rstd, 2, fmt)
        assert np.array_equal(rounding.round_to(dx, fmt), dx)
        assert np.array_equal(rounding.round_to(dg, "f32"), dg)


# --- planted mistakes -------------------------------------------------------

def _stats(kind):
    def stats_exact(x, groups, eps):
        x = np.asarray(x, float)
        n, c, s = x.shape
        if kind == "per_channel":
            xg = x.reshape(n, c, s)
            mean = xg.mean(-1)
            var = xg.var(-1)
            # collapse to groups by taking the first channel of each group
            idx = np.arange(groups) * (c // groups)
            return mean[:, idx], 1 / np.sqrt(var[:, idx] + np.float32(eps))
        xg = x.reshape(n, groups, -1)
        mean = xg.mean(-1)
        if kind == "unbiased":
            var = xg.var(-1, ddof=1)
        elif kind == "interleaved":
            # group g taken as the strided channels g, g + G, g + 2G, ...
            xi = x.reshape(n, c // groups, groups, s).transpose(0, 2, 1, 3).reshape(n, groups, -1)
            mean = xi.mean(-1)
            var = xi.var(-1)
        else:
            var = xg.var(-1)
        return mean, 1 / np.sqrt(var + np.float32(eps))
    return stats_exact


def _bwd(kind):
    def backward_exact(dy, x, gamma, mean, rstd, groups):
        dy = np.asarray(dy, float)
        n, c, s = dy.shape
        xh = ((np.asarray(x, float).reshape(n, groups, -1) - mean[..., None])
              * rstd[..., None]).reshape(n, c, s)
        w = gamma[None, :, None] if kind != "gain_by_group" else \
            np.repeat(gamma[:groups], c // groups)[None, :, None]
        g = dy * w
        gg, xhg = g.reshape(n, groups, -1), xh.reshape(n, groups, -1)
        c1 = gg.mean(-1, keepdims=True)
        c2 = (gg * xhg).mean(-1, keepdims=True)
        if kind == "drop_c1":
            c1 = 0 * c1
        dx = rstd[..., None] * (gg - c1 - xhg * c2)
        dgamma = np.sum(dy * (np.asarray(x, float) if kind == "dg_uses_x" else xh), axis=(0, 2))
        dbeta = np.sum(dy, axis=(0, 2)) if kind != "db_over_batch_only" else np.sum(dy[:, :, 0], 0)
        return dx.reshape(n, c, s), dgamma, dbeta
    return backward_exact


MUTANTS = {
    "unbiased_variance": dict(stats_exact=_stats("unbiased")),
    "per_channel_stats": dict(stats_exact=_stats("per_channel")),
    "interleaved_groups": dict(stats_exact=_stats("interleaved")),
    "gain_by_group": dict(backward_exact=_bwd("gain_by_group")),
    "drop_c1": dict(backward_exact=_bwd("drop_c1")),
    "dg_uses_x": dict(backward_exact=_bwd("dg_uses_x")),
    "db_over_batch_only": dict(backward_exact=_bwd("db_over_batch_only")),
}


def _copy(**kw):
    m = types.SimpleNamespace(stats_exact=ogn.stats_exact, backward_exact=ogn.backward_exact)
    for k, v in kw.items():
        setattr(m, k, v)

    def forward_exact(x, gamma, beta, groups, eps):
        x = np.asarray(x, float)
        mean, rstd = m.stats_exact(x, groups, eps)
        n, c, s = x.shape
        xh = ((x.reshape(n, groups, -1) - mean[..., None]) * rstd[..., None]).reshape(n, c, s)
        y = xh * gamma[None, :, None]
        return (y if beta is None else y + beta[None, :, None]), mean, rstd
    m.forward_exact = forward_exact
    return m


def test_unmutated_copy_passes():
    assert _all_pins(_copy())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    assert not _all_pins(_copy(**MUTANTS[name]))
