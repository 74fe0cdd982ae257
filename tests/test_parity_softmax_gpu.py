"""Softmax over the last dimension on the GPU against the float64 oracle
(oracle.softmax), through the C ABI."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import rounding
from oracle import softmax as osm

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
    rng = np.random.default_rng(7)
    pick = rng.choice(rows, size=limit - 4, replace=False)
    return np.unique(np.concatenate([pick, [0, 1, rows - 2, rows - 1]]))


def check_forward(L, x_cpu, fmt, rows, to_dev=None):
    to_dev = to_dev or (lambda t: t.cuda())
    y = L.softmax_fwd(to_dev(x_cpu))
    torch.cuda.synchronize()
    xd = W.as_float64(x_cpu)[rows]
    y_exact = osm.forward_exact(xd)
    P.check_rows(W.as_float64(y.cpu())[rows], rounding.round_to(y_exact, fmt), fmt, None, "y")
    return y


def check_backward(L, dy_cpu, y_cpu, fmt, rows, to_dev=None):
    """Both sides start from the same stored y."""
    to_dev = to_dev or (lambda t: t.cuda())
    dx = L.softmax_bwd(to_dev(dy_cpu), to_dev(y_cpu))
    torch.cuda.synchronize()
    dyd, yd = W.as_float64(dy_cpu)[rows], W.as_float64(y_cpu)[rows]
    s = np.sum(dyd * yd, axis=-1, keepdims=True)
    terms = yd * (np.abs(dyd) + np.abs(s))
    P.check_rows(W.as_float64(dx.cpu())[rows], osm.backward(dyd, yd, fmt), fmt, None, "dx",
                 terms, cancels=True)


def run_and_check(L, w, sample_limit=1024, to_dev=None):
    inp = W.make_inputs(w)
    rows = _sample_rows(w.rows, sample_limit)
    check_forward(L, inp["x"], w.dtype, rows, to_dev)
    # the stored y the backward reads: the oracle's forward, in the storage type
    y_store = torch.from_numpy(osm.forward(W.as_float64(inp["x"]), w.dtype)).to(
        W.DTYPES[w.dtype])
    check_backward(L, inp["dy"], y_store, w.dtype, rows, to_dev)


@pytest.mark.parametrize("name", sorted(W.softmax_workloads()))
def test_named_softmax_workload(L, name):
    w = W.softmax_workloads()[name]
    run_and_check(L, w, sample_limit=2048)


SHAPES = [(1, 1, "f32"), (3, 8, "bf16"), (17, 24, "f16"), (5, 1001, "bf16"), (9, 1024, "bf16"),
          (7, 1032, "f16"), (300, 4096, "bf16"), (40, 3072, "f32"), (4, 16384, "bf16"),
          (3, 16392, "f16"), (6, 24576, "bf16"), (2, 32768, "bf16"), (2, 32768, "f32"),
          (2, 65536, "bf16"), (1000, 256, "f16"), (129, 8192, "f32")]


@pytest.mark.parametrize("rows,cols,dtype", SHAPES)
def test_softmax_shapes(L, rows, cols, dtype):
    w = W.softmax_workloads()["softmax_bf16_4096x4096"].with_(rows=rows, hidden=cols,
                                                              dtype=dtype, seed=rows + cols)
    run_and_check(L, w)


def _misaligned_copy(t):
    buf = torch.empty(t.numel() + 1, dtype=t.dtype, device="cuda")
    v = buf[1:].view(t.shape)
    v.copy_(t.cuda())
    return v


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_softmax_unaligned(L, dtype):
    w = W.softmax_workloads()["softmax_bf16_4096x4096"].with_(rows=33, hidden=2048, dtype=dtype)
    run_and_check(L, w, to_dev=_misaligned_copy)


@pytest.mark.parametrize("cols", [512, 4096])
def test_softmax_large_logits_and_masking(L, cols):
    """Logits near 1e4 (exp overflows without the max shift), rows with -inf
    entries (masked positions give exactly 0), and a fully masked row (NaN,
    as the formula gives); rows for one warp (512) and one CTA (4096), whose
    16-bit maxima are taken on packed pairs."""
    g = torch.Generator().manual_seed(11)
    x = torch.randn(6, cols, generator=g) * 3.0
    x[0] += 1.0e4
    x[1, ::3] = float("-inf")
    x[2, 100:] = float("-inf")
    x[3, :] = float("-inf")
    x[4, 7] = 60.0
    y = L.softmax_fwd(x.cuda()).cpu()
    ok = [0, 1, 2, 4, 5]
    check_forward(L, x, "f32", np.array(ok))
    assert torch.all(y[1, ::3] == 0) and torch.all(y[2, 100:] == 0)
    assert torch.all(torch.isnan(y[3]))
    for dt, fmt in ((torch.bfloat16, "bf16"), (torch.float16, "f16")):
        xh = x.to(dt)
        check_forward(L, xh, fmt, np.array(ok))
        yh = L.softmax_fwd(xh.cuda()).cpu()
        assert torch.all(yh[1, ::3] == 0) and torch.all(torch.isnan(yh[3]))


def test_softmax_rows_sum_to_one(L):
    w = W.softmax_workloads()["softmax_f16_65536x1024"]
    x = W.make_inputs(w)["x"].cuda()
    y = L.softmax_fwd(x).float()
    s = y.sum(dim=-1)
    # each of 1024 fp16 outputs is within half an ulp of its exact value
    assert torch.max(torch.abs(s - 1.0)).item() < 1024 * 2.0 ** -11


def test_softmax_zero_rows(L):
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    assert L.softmax_fwd(x).shape == (0, 64)
    assert L.softmax_bwd(x, x).shape == (0, 64)
