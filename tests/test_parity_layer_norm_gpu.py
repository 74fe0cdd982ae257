"""LayerNorm on the GPU against the float64 oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import layer_norm as oln
from oracle import rounding

import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import bwd_rms_norm_gb300 as lib
    lib.load_library()
    return lib


def _sample_rows(rows, limit):
    if rows <= limit:
        return np.arange(rows)
    rng = np.random.default_rng(4321)
    pick = rng.choice(rows, size=limit - 4, replace=False)
    return np.unique(np.concatenate([pick, [0, 1, rows - 2, rows - 1]]))


def run_and_check(L, w, sample_limit=1024, bias=True, to_dev=None):
    inp = W.make_inputs(w)
    to_dev = to_dev or (lambda t: t.cuda())
    x, g, dy = inp["x"], inp["gamma"], inp["dy"]
    b = inp.get("beta") if bias else None
    xd, gd, dyd = W.as_float64(x), W.as_float64(g), W.as_float64(dy)
    bd = W.as_float64(b) if b is not None else None
    fmt = w.dtype
    xc, gc, dyc = to_dev(x), to_dev(g), to_dev(dy)
    bc = to_dev(b) if b is not None else None

    y, mean, rstd = L.layer_norm_fwd(xc, gc, bc, w.eps)
    torch.cuda.synchronize()
    rows = _sample_rows(w.rows, sample_limit)
    mean_ex, rstd_ex = oln.stats_exact(xd, w.eps)
    mean_ref, rstd_ref = rounding.round_to(mean_ex, "f32"), rounding.round_to(rstd_ex, "f32")
    P.check_rstd(rstd.cpu().numpy(), rstd_ref)
    # mean: relative to the row's rms (a mean near zero has no relative scale)
    scale = np.sqrt(np.mean(xd * xd, axis=1))
    assert np.max(np.abs(mean.cpu().numpy() - mean_ref) / scale) <= 1e-6
    y_ref, _, _ = oln.forward(xd[rows], gd, bd, w.eps, fmt)
    x_hat = (xd[rows] - mean_ex[rows, None]) * rstd_ex[rows, None]
    terms = np.abs(x_hat * gd) + (np.abs(bd) if bd is not None else 0.0)
    P.check_rows(W.as_float64(y.cpu())[rows], y_ref, fmt, None, "y", terms, cancels=True)

    m_in = to_dev(torch.from_numpy(mean_ref.astype(np.float32)))
    r_in = to_dev(torch.from_numpy(rstd_ref.astype(np.float32)))
    dx, dgam, dbet = L.layer_norm_bwd(dyc, xc, gc, m_in, r_in)
    torch.cuda.synchronize()
    dx_ex, dg_ex, db_ex = oln.backward_exact(dyd, xd, gd, mean_ref, rstd_ref)
    dterms = rstd_ref[rows, None] * dyd[rows] * gd[None, :]
    P.check_rows(W.as_float64(dx.cpu())[rows], rounding.round_to(dx_ex[rows], fmt), fmt, None,
                 "dx", dterms, cancels=True)
    P.check_dw(dgam.cpu().numpy(), rounding.round_to(dg_ex, "f32"))
    P.check_dw(dbet.cpu().numpy(), rounding.round_to(db_ex, "f32"))


@pytest.mark.parametrize("name", sorted(W.layer_norm_workloads()))
def test_named_layer_norm_workload(L, name):
    w = W.layer_norm_workloads()[name]
    run_and_check(L, w, sample_limit=2048 if w.rows * w.hidden > (1 << 25) else w.rows)


SHAPES = [(1, 1, "f32"), (3, 8, "bf16"), (17, 24, "f16"), (5, 1001, "bf16"), (9, 1024, "bf16"),
          (7, 1032, "f16"), (300, 4096, "bf16"), (4, 16384, "bf16"), (2, 32768, "f32"),
          (2, 65536, "bf16"), (33, 3072, "f16"), (3, 16392, "bf16"),
          # the TMA-staged kernels: one and two vectors per applier, ragged
          # row counts over the 152-CTA grid, the forward above 16 KB rows
          (1000, 8192, "bf16"), (157, 6144, "f16"), (301, 4096, "f32"), (611, 12288, "bf16"),
          (5, 20000, "bf16"), (153, 7168, "bf16"), (1, 1024, "bf16")]


@pytest.mark.parametrize("rows,hidden,dtype", SHAPES)
def test_layer_norm_shapes(L, rows, hidden, dtype):
    w = W.Workload("ln_shape", rows, hidden, dtype, 1e-5, 0, "round_once", ("normal", 0.5, 1.0),
                   ("uniform", 0.9, 1.1), ("normal", 0.0, 1.0), seed=rows + hidden, kind="ln",
                   beta_dist=("normal", 0.0, 0.01))
    run_and_check(L, w)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_layer_norm_without_bias(L, dtype):
    w = W.layer_norm_workloads()["ln_bf16_4096x4096"].with_(rows=64, dtype=dtype)
    run_and_check(L, w, bias=False)


def _misaligned_copy(t):
    buf = torch.empty(t.numel() + 1, dtype=t.dtype, device="cuda")
    v = buf[1:].view(t.shape)
    v.copy_(t.cuda())
    return v


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_layer_norm_unaligned(L, dtype):
    w = W.layer_norm_workloads()["ln_bf16_4096x4096"].with_(rows=40, hidden=1024, dtype=dtype)
    run_and_check(L, w, to_dev=_misaligned_copy)


def test_layer_norm_backward_deterministic(L):
    w = W.layer_norm_workloads()["ln_bf16_4096x4096"].with_(rows=777)
    inp = {k: v.cuda() for k, v in W.make_inputs(w).items()}
    _, m, r = L.layer_norm_fwd(inp["x"], inp["gamma"], inp["beta"], w.eps)
    first = L.layer_norm_bwd(inp["dy"], inp["x"], inp["gamma"], m, r)
    for _ in range(3):
        again = L.layer_norm_bwd(inp["dy"], inp["x"], inp["gamma"], m, r)
        for a, b in zip(first, again):
            assert torch.equal(a, b)


def test_layer_norm_zero_rows(L):
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    y, m, r = L.layer_norm_fwd(x, g, None, 1e-5)
    assert y.shape == (0, 64)
    dg = torch.full((64,), 3.0, device="cuda")
    db = torch.full((64,), 3.0, device="cuda")
    L.layer_norm_bwd(x, x, g, m, r, dgamma=dg, dbeta=db)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dg).item() == 0 and torch.count_nonzero(db).item() == 0


def test_layer_norm_without_dbeta(L):
    """dbeta NULL: dx and dgamma are the same as with it."""
    w = W.layer_norm_workloads()["ln_bf16_4096x4096"].with_(rows=300)
    inp = {k: v.cuda() for k, v in W.make_inputs(w).items()}
    _, m, r = L.layer_norm_fwd(inp["x"], inp["gamma"], inp["beta"], w.eps)
    dx1, dg1, db1 = L.layer_norm_bwd(inp["dy"], inp["x"], inp["gamma"], m, r)
    dx2, dg2, db2 = L.layer_norm_bwd(inp["dy"], inp["x"], inp["gamma"], m, r, with_dbeta=False)
    assert db2 is None and db1 is not None
    assert torch.equal(dx1, dx2) and torch.equal(dg1, dg2)


def test_layer_norm_no_wait_timeouts(L):
    assert L.wait_timeouts() == 0
