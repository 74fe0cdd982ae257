"""Pins of the float64 softmax oracle against facts fixed outside it (torch's
CPU softmax and autograd in float64, finite differences, closed forms,
invariants, torch's bf16 softmax), and planted mistakes those pins catch.
Host only."""
import types

import numpy as np
import pytest
import torch

from oracle import rounding
from oracle import softmax as osm


def _data(seed, r=6, n=33, scale=3.0):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((r, n)) * scale, rng.standard_normal((r, n))


def check_forward_vs_torch(mod=osm, seed=1):
    x, _ = _data(seed)
    x[0] += 800.0       # a row whose exp overflows without the max shift
    ref = torch.softmax(torch.from_numpy(x), dim=-1).numpy()
    y = mod.forward_exact(x)
    if not np.all(np.isfinite(y)):
        return np.inf
    return float(np.max(np.abs(y - ref) / np.maximum(np.abs(ref), 1e-300)))


def check_backward_vs_autograd(mod=osm, seed=2):
    x, dy = _data(seed)
    xt = torch.from_numpy(x.copy()).requires_grad_(True)
    torch.softmax(xt, dim=-1).backward(torch.from_numpy(dy))
    y = torch.softmax(torch.from_numpy(x), dim=-1).numpy()
    dx = mod.backward_exact(dy, y)
    g = xt.grad.numpy()
    return float(np.max(np.abs(dx - g)) / np.max(np.abs(g)))


def check_finite_differences(mod=osm, seed=3):
    x, dy = _data(seed, r=3, n=7, scale=1.5)
    h = 1e-6
    fd = np.zeros_like(x)
    for i in range(x.shape[0]):
        for j in range(x.shape[1]):
            p = x.copy(); p[i, j] += h
            m = x.copy(); m[i, j] -= h
            fd[i, j] = (np.sum(dy * mod.forward_exact(p)) - np.sum(dy * mod.forward_exact(m))) / (2 * h)
    dx = mod.backward_exact(dy, mod.forward_exact(x))
    return float(np.max(np.abs(dx - fd)) / np.max(np.abs(fd)))


def check_invariants(mod=osm, seed=4):
    """Rows sum to 1; dx rows sum to 0; shift invariance; closed forms."""
    x, dy = _data(seed)
    y = mod.forward_exact(x)
    e1 = np.max(np.abs(y.sum(axis=-1) - 1.0))
    e2 = np.max(np.abs(mod.backward_exact(dy, y).sum(axis=-1))) / np.max(np.abs(dy))
    e3 = np.max(np.abs(mod.forward_exact(x + 17.25) - y))
    # one element: y = 1 and dx = 0; a constant row: y = 1/n;
    # two elements: y_0 = 1 / (1 + exp(x_1 - x_0))
    one = mod.forward_exact(np.array([[3.5]]))
    e4 = abs(one[0, 0] - 1.0) + abs(mod.backward_exact(np.array([[2.0]]), one)[0, 0])
    e5 = np.max(np.abs(mod.forward_exact(np.full((2, 9), -4.0)) - 1.0 / 9.0))
    two = mod.forward_exact(np.array([[0.3, -1.2]]))
    e6 = abs(two[0, 0] - 1.0 / (1.0 + np.exp(-1.5)))
    return float(max(e1, e2, e3, e4, e5, e6))


def _all_pins(m):
    return (check_forward_vs_torch(m) < 1e-13 and check_backward_vs_autograd(m) < 1e-13
            and check_finite_differences(m) < 1e-7 and check_invariants(m) < 1e-14)


def test_forward_matches_torch_float64():
    assert check_forward_vs_torch() < 1e-13


def test_backward_matches_torch_autograd():
    assert check_backward_vs_autograd() < 1e-13


def test_backward_finite_differences():
    assert check_finite_differences() < 1e-7


def test_invariants_and_closed_forms():
    assert check_invariants() < 1e-14


def test_bf16_store_matches_torch_cpu_bf16():
    """torch's CPU bf16 softmax computes in fp32 and rounds once: at least
    99.9% identical to the oracle's single rounding from float64, the rest
    one ulp apart."""
    g = torch.Generator().manual_seed(6)
    xb = (torch.randn(2048, 1024, generator=g) * 2.0).to(torch.bfloat16)
    ref = torch.softmax(xb, dim=-1).double().numpy()
    y = osm.forward(xb.double().numpy(), "bf16")
    d = rounding.ulp_distance(y, ref, "bf16")
    assert np.mean(d == 0) >= 0.999 and d.max() <= 1


def test_outputs_are_stored_values():
    x, dy = _data(7)
    for fmt in ("f32", "bf16", "f16"):
        y = osm.forward(x, fmt)
        assert np.array_equal(rounding.round_to(y, fmt), y)
        dx = osm.backward(dy, y, fmt)
        assert np.array_equal(rounding.round_to(dx, fmt), dx)


# --- planted mistakes -------------------------------------------------------

def _fwd(kind):
    def forward_exact(x):
        x = np.asarray(x, float)
        if kind == "no_max_shift":
            with np.errstate(over="ignore", invalid="ignore"):
                e = np.exp(x)
        elif kind == "global_max_shift":
            # one maximum for the whole tensor: rows far below it underflow
            e = np.exp(x - np.max(x))
        elif kind == "divide_by_n":
            e = np.exp(x - np.max(x, axis=-1, keepdims=True))
            return e / x.shape[-1]
        else:
            e = np.exp(x - np.max(x, axis=-1, keepdims=True))
        with np.errstate(invalid="ignore"):
            return e / np.sum(e, axis=-1, keepdims=True)
    return forward_exact


def _bwd(kind):
    def backward_exact(dy, y):
        dy = np.asarray(dy, float)
        y = np.asarray(y, float)
        if kind == "sum_of_dy":
            s = np.sum(dy, axis=-1, keepdims=True)
        elif kind == "mean_not_sum":
            s = np.mean(dy * y, axis=-1, keepdims=True)
        else:
            s = np.sum(dy * y, axis=-1, keepdims=True)
        if kind == "sign":
            return y * (dy + s)
        if kind == "no_y_factor":
            return dy - s
        return y * (dy - s)
    return backward_exact


MUTANTS = {
    "no_max_shift": dict(forward_exact=_fwd("no_max_shift")),
    "global_max_shift": dict(forward_exact=_fwd("global_max_shift")),
    "divide_by_n": dict(forward_exact=_fwd("divide_by_n")),
    "sum_of_dy": dict(backward_exact=_bwd("sum_of_dy")),
    "mean_not_sum": dict(backward_exact=_bwd("mean_not_sum")),
    "sign": dict(backward_exact=_bwd("sign")),
    "no_y_factor": dict(backward_exact=_bwd("no_y_factor")),
}


def _copy(**kw):
    m = types.SimpleNamespace(forward_exact=osm.forward_exact, backward_exact=osm.backward_exact)
    for k, v in kw.items():
        setattr(m, k, v)
    return m


def test_unmutated_copy_passes():
    assert _all_pins(_copy())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name):
    assert not _all_pins(_copy(**MUTANTS[name]))
