"""GroupNorm on the GPU against the float64 oracle (oracle.group_norm),
through the C ABI."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import group_norm as ogn
from oracle import rounding

import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import bwd_rms_norm_gb300 as lib
    lib.load_library()
    return lib


def _rows(a, n, groups):
    """[n, C, S] -> [n * groups, group length]: one row per group."""
    return np.asarray(a).reshape(n * groups, -1)


def run_and_check(L, w, to_dev=None, bias=True, sample_limit=4):
    inp = W.make_inputs(w)
    to_dev = to_dev or (lambda t: t.cuda())
    n, G, fmt = w.rows, w.groups, w.dtype
    x, g, dy = inp["x"], inp["gamma"], inp["dy"]
    b = inp.get("beta") if bias else None
    xd, gd, dyd = W.as_float64(x), W.as_float64(g), W.as_float64(dy)
    bd = W.as_float64(b) if b is not None else None

    y, mean, rstd = L.group_norm_fwd(to_dev(x), to_dev(g), to_dev(b) if b is not None else None,
                                     G, w.eps)
    torch.cuda.synchronize()
    mean_ex, rstd_ex = ogn.stats_exact(xd, G, w.eps)
    P.check_rstd(rstd.cpu().numpy().ravel(), rounding.round_to(rstd_ex, "f32").ravel())
    scale = np.sqrt(np.mean(_rows(xd, n, G) ** 2, axis=1))
    mean_err = np.abs(mean.cpu().numpy().ravel() - rounding.round_to(mean_ex, "f32").ravel())
    assert np.max(mean_err / scale) <= 1e-6
    # y and dx on the first samples (the statistics are per sample)
    k = min(n, sample_limit)
    y_ref, _, _ = ogn.forward(xd[:k], gd, bd, G, w.eps, fmt)
    xh = ((_rows(xd[:k], k, G) - mean_ex[:k].reshape(-1, 1)) * rstd_ex[:k].reshape(-1, 1))
    xh = xh.reshape(xd[:k].shape)
    terms = np.abs(xh * gd[None, :, None])
    if bd is not None:
        terms = terms + np.abs(bd)[None, :, None]
    terms = _rows(terms, k, G)
    P.check_rows(_rows(W.as_float64(y[:k].cpu()), k, G), _rows(y_ref, k, G), fmt, None, "y",
                 terms, cancels=True)

    m_in = rounding.round_to(mean_ex, "f32")
    r_in = rounding.round_to(rstd_ex, "f32")
    dx, dgam, dbet = L.group_norm_bwd(to_dev(dy), to_dev(x), to_dev(g),
                                      torch.from_numpy(m_in.astype(np.float32)).cuda(),
                                      torch.from_numpy(r_in.astype(np.float32)).cuda(), G)
    torch.cuda.synchronize()
    dx_ex, dg_ex, db_ex = ogn.backward_exact(dyd, xd, gd, m_in, r_in, G)
    dterms = (np.abs(dyd[:k]) * gd[None, :, None]) * np.repeat(r_in[:k], dyd.shape[1] // G,
                                                              axis=1)[:, :, None]
    P.check_rows(_rows(W.as_float64(dx[:k].cpu()), k, G),
                 _rows(rounding.round_to(dx_ex[:k], fmt), k, G), fmt, None, "dx",
                 _rows(dterms, k, G), cancels=True)
    P.check_dw(dgam.cpu().numpy(), rounding.round_to(dg_ex, "f32"))
    P.check_dw(dbet.cpu().numpy(), rounding.round_to(db_ex, "f32"))
    return dx, dgam, dbet


@pytest.mark.parametrize("name", sorted(W.group_norm_workloads()))
def test_named_group_norm_workload(L, name):
    run_and_check(L, W.group_norm_workloads()[name])


# (n, channels, spatial, groups, dtype): one CTA per group and clusters of 2
# to 16, odd spatial sizes (scalar kernels), one group, one group per channel
SHAPES = [(1, 1, 1, 1, "f32"), (2, 4, 8, 2, "bf16"), (3, 6, 7, 3, "f16"), (2, 8, 24, 4, "bf16"),
          (5, 32, 256, 8, "bf16"), (2, 16, 4096, 4, "f16"), (3, 64, 1024, 1, "bf16"),
          (2, 12, 512, 12, "f32"), (1, 8, 32768, 2, "bf16"), (2, 4, 65536, 4, "f32"),
          (1, 32, 65536, 2, "bf16"), (3, 10, 100, 5, "bf16"), (2, 6, 1000, 2, "f16")]


@pytest.mark.parametrize("n,c,s,g,dtype", SHAPES)
def test_group_norm_shapes(L, n, c, s, g, dtype):
    w = W.group_norm("gn_shape", n, c, s, g, dtype, x_dist=("normal", 0.3, 1.0), seed=n + c + s)
    run_and_check(L, w)


def test_group_norm_without_bias(L):
    w = W.group_norm("gn_nobias", 2, 16, 1024, 4, "bf16", beta_dist=None)
    run_and_check(L, w, bias=False)


def _misaligned_copy(t):
    buf = torch.empty(t.numel() + 1, dtype=t.dtype, device="cuda")
    v = buf[1:].view(t.shape)
    v.copy_(t.cuda())
    return v


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_group_norm_unaligned(L, dtype):
    w = W.group_norm("gn_unaligned", 2, 8, 256, 4, dtype)
    run_and_check(L, w, to_dev=_misaligned_copy)


def test_upstream_of_ones_in_fp16(L):
    """Liger-Kernel PR #1608's case: fp16 (1, 16, 256, 256), 4 groups, unit
    weights, dy = 1.  A channel sum of 65536 ones does not fit fp16; with
    fp32 reductions dx is 0 up to fp32 rounding and dB = 65536 exactly."""
    w = W.group_norm_workloads()["gn_f16_1x16x256x256_g4_ones"]
    dx, _, db = run_and_check(L, w)
    assert torch.all(torch.isfinite(dx.float()))
    assert dx.float().abs().max().item() < 1e-3
    assert torch.all(db == 65536.0)


def test_group_norm_backward_deterministic(L):
    w = W.group_norm_workloads()["gn_bf16_2x64x32x32_g8_offset16"]
    inp = {k: v.cuda() for k, v in W.make_inputs(w).items()}
    _, m, r = L.group_norm_fwd(inp["x"], inp["gamma"], inp["beta"], w.groups, w.eps)
    first = L.group_norm_bwd(inp["dy"], inp["x"], inp["gamma"], m, r, w.groups)
    for _ in range(3):
        again = L.group_norm_bwd(inp["dy"], inp["x"], inp["gamma"], m, r, w.groups)
        for a, b in zip(first, again):
            assert torch.equal(a, b)


def test_group_norm_without_dbeta(L):
    w = W.group_norm("gn_nodb", 2, 32, 2048, 8, "bf16")
    inp = {k: v.cuda() for k, v in W.make_inputs(w).items()}
    _, m, r = L.group_norm_fwd(inp["x"], inp["gamma"], inp["beta"], w.groups, w.eps)
    a = L.group_norm_bwd(inp["dy"], inp["x"], inp["gamma"], m, r, w.groups)
    b = L.group_norm_bwd(inp["dy"], inp["x"], inp["gamma"], m, r, w.groups, with_dbeta=False)
    assert b[2] is None and torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_group_norm_zero_samples(L):
    x = torch.empty(0, 8, 16, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(8, dtype=torch.bfloat16, device="cuda")
    y, m, r = L.group_norm_fwd(x, g, None, 4, 1e-5)
    assert y.shape == x.shape
    dg = torch.full((8,), 5.0, device="cuda")
    db = torch.full((8,), 5.0, device="cuda")
    L.group_norm_bwd(x, x, g, m, r, 4, dgamma=dg, dbeta=db)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dg).item() == 0 and torch.count_nonzero(db).item() == 0


def test_group_norm_no_wait_timeouts(L):
    assert L.wait_timeouts() == 0
