"""The backward entry point that allocates nothing: rms_norm_bwd_noalloc.

Some callers cannot allocate device memory at the point where they run the
backward -- a plugin whose enqueue hook must not call cudaMalloc, or a
service held to a fixed, pre-reserved memory budget -- so they cannot hand
rms_norm_bwd the workspace it asks for.  rms_norm_bwd_noalloc keeps the
weight-gradient partials in a fixed 16 MiB array inside the library instead.

These tests call it through the C ABI on two calls in a row (every call
reuses the same array) and check each result against the float64 oracle
with the parity tolerances, and bit for bit against rms_norm_bwd, which runs
the same kernels with the same number of partials.  One case goes through
the Python wrapper.  The refusal of sizes the array cannot hold, and the
wrapper's host-side argument checks, need no GPU.

This file is named so that pytest collects it last.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

import workloads as W
from oracle import rms_norm as orm
from oracle import rounding

import parity as P


@pytest.fixture(scope="module")
def L():
    import bwd_rms_norm_gb300 as lib
    if not os.path.exists(lib.LIB_PATH):
        from bwd_rms_norm_gb300 import build
        build.build()
    lib.load_library()
    return lib


def _f64(t):
    return t.detach().cpu().to(torch.float64).numpy()


CASES = [
    # rows, hidden, dtype, offset -- vector kernels at the 4096 x 4096 bf16
    # size, the scalar kernels (hidden not a multiple of the vector), fp32
    (4096, 4096, "bf16", 0),
    (777, 1001, "f16", 1),
    (300, 2048, "f32", 0),
]


def _inputs(rows, hidden, dtype, offset):
    w = W.Workload("noalloc", rows, hidden, dtype, 1e-5, offset, "round_once",
                   ("normal", 0.0, 1.0),
                   ("normal", 0.0, 0.1) if offset else ("uniform", 0.9, 1.1),
                   ("normal", 0.0, 1.0), seed=rows + hidden)
    return w, W.make_inputs(w)


def _check_against_oracle(w, inp, rstd_ref, dx, dw, sample):
    xd, gd, dyd = (W.as_float64(inp[k]) for k in ("x", "gamma", "dy"))
    dx_exact, dw_exact = orm.backward_exact(dyd, xd, gd, rstd_ref, w.offset)
    terms = rstd_ref[sample, None] * dyd[sample] * orm.gain(gd, w.offset)[None, :]
    P.check_rows(_f64(dx)[sample], rounding.round_to(dx_exact[sample], w.dtype), w.dtype, None,
                 "dx", terms, cancels=True)
    P.check_dw(dw.cpu().numpy(), rounding.round_to(dw_exact, "f32"))


@pytest.mark.gpu
@pytest.mark.parametrize("rows,hidden,dtype,offset", CASES)
def test_noalloc_matches_oracle_and_workspace_backward(L, rows, hidden, dtype, offset):
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    lib = L.load_library()
    w, inp = _inputs(rows, hidden, dtype, offset)
    rstd_ref = rounding.round_to(orm.rstd_exact(W.as_float64(inp["x"]), w.eps), "f32")
    x, g, dy = (inp[k].cuda() for k in ("x", "gamma", "dy"))
    rstd = torch.from_numpy(rstd_ref.astype(np.float32)).cuda()
    dx_ref, dw_ref = L.rms_norm_bwd(dy, x, g, rstd, offset)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream().cuda_stream
    sample = np.unique(np.concatenate([np.arange(0, rows, max(1, rows // 256)), [rows - 1]]))
    for _ in range(2):
        dx = torch.full_like(x, 5.0)
        dw = torch.full((hidden,), 5.0, dtype=torch.float32, device="cuda")
        st = lib.rms_norm_bwd_noalloc(
            ctypes.c_void_p(dy.data_ptr()), ctypes.c_void_p(x.data_ptr()),
            ctypes.c_void_p(g.data_ptr()), ctypes.c_void_p(rstd.data_ptr()),
            ctypes.c_void_p(dx.data_ptr()), ctypes.c_void_p(dw.data_ptr()),
            rows, hidden, offset, L.DTYPE_CODES[x.dtype], ctypes.c_void_p(stream))
        assert st == L.RMSN_OK, lib.rms_norm_status_string(st)
        assert L.last_launch_count() == 2
        torch.cuda.synchronize()
        _check_against_oracle(w, inp, rstd_ref, dx, dw, sample)
        assert torch.equal(dx, dx_ref)
        assert torch.equal(dw, dw_ref)


@pytest.mark.gpu
def test_noalloc_python_wrapper(L):
    w, inp = _inputs(512, 4096, "bf16", 0)
    x, g, dy = (inp[k].cuda() for k in ("x", "gamma", "dy"))
    _, rstd = L.rms_norm_fwd(x, g, w.eps)
    dx_ref, dw_ref = L.rms_norm_bwd(dy, x, g, rstd)
    dx = torch.empty_like(x)
    dw = torch.empty(4096, dtype=torch.float32, device="cuda")
    for _ in range(2):
        out = L.rms_norm_bwd_noalloc(dy, x, g, rstd, dx=dx, dw=dw)
        assert out[0] is dx and out[1] is dw
        torch.cuda.synchronize()
        assert torch.equal(dx, dx_ref) and torch.equal(dw, dw_ref)
    assert L.wait_timeouts() == 0


def test_noalloc_refuses_sizes_beyond_its_array(L):
    """16384 x 8192 would need 32 MiB of partials: refused on the host,
    before any CUDA call, so this runs without a GPU."""
    lib = L.load_library()
    fake = ctypes.c_void_p(0x1000)   # never dereferenced: the size check fails first
    st = lib.rms_norm_bwd_noalloc(fake, fake, fake, fake, fake, fake, 16384, 8192, 0,
                                  L.RMSN_BF16, None)
    assert st == 2  # RMSN_ERR_SHAPE
    assert lib.rms_norm_bwd_workspace_size(16384, 8192, L.RMSN_BF16) > (16 << 20)
    assert lib.rms_norm_bwd_workspace_size(4096, 4096, L.RMSN_BF16) <= (16 << 20)


@pytest.mark.parametrize("bad", ["gamma", "dy", "rstd", "dx", "dw", "dtype"])
def test_noalloc_wrapper_checks_sizes_before_any_launch(L, bad):
    """A short gamma or rstd, a dy or dx of another shape, a dw of the wrong
    length or type: refused on the host before the library is called (CPU
    tensors, so nothing could have reached a device)."""
    rows, hidden = 8, 64
    x = torch.zeros(rows, hidden, dtype=torch.bfloat16)
    args = {"dy": torch.zeros(rows, hidden, dtype=torch.bfloat16),
            "gamma": torch.ones(hidden, dtype=torch.bfloat16),
            "rstd": torch.ones(rows, dtype=torch.float32),
            "dx": torch.empty(rows, hidden, dtype=torch.bfloat16),
            "dw": torch.empty(hidden, dtype=torch.float32)}
    if bad == "gamma":
        args["gamma"] = torch.ones(hidden - 8, dtype=torch.bfloat16)
    elif bad == "dy":
        args["dy"] = torch.zeros(rows, hidden + 8, dtype=torch.bfloat16)
    elif bad == "rstd":
        args["rstd"] = torch.ones(rows - 1, dtype=torch.float32)
    elif bad == "dx":
        args["dx"] = torch.empty(rows - 1, hidden, dtype=torch.bfloat16)
    elif bad == "dw":
        args["dw"] = torch.empty(hidden, dtype=torch.bfloat16)
    else:
        args["dy"] = torch.zeros(rows, hidden, dtype=torch.float16)
    with pytest.raises(RuntimeError, match=f"^{bad if bad != 'dtype' else 'dy'} must"):
        L.rms_norm_bwd_noalloc(args["dy"], x, args["gamma"], args["rstd"], dx=args["dx"],
                               dw=args["dw"])
    with pytest.raises(RuntimeError, match=f"^{bad if bad != 'dtype' else 'dy'} must"):
        L.rms_norm_bwd(args["dy"], x, args["gamma"], args["rstd"], dx=args["dx"], dw=args["dw"])
