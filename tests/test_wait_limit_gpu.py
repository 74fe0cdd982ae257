"""The bounded waits of the staged kernels, made to run out on purpose.

Every wait on a shared-memory barrier in the staged kernels is bounded
(about one second); a wait that runs out counts on the device and the CTA
returns.  Correct runs never get there, so rms_norm_selftest_wait_limit
makes one: a single thread waits, through the same bounded wait, on a
barrier nothing completes.  Nothing faults, traps or hangs: the wait gives
up after its limit, the kernel returns, and the library keeps working.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import rms_norm as orm
from oracle import rounding

import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import bwd_rms_norm_gb300 as lib
    lib.load_library()
    return lib


def test_a_wait_nothing_completes_runs_out_and_returns(L):
    before = L.wait_timeouts()
    n, seconds = L.selftest_wait_limit()
    assert n == 1
    assert 0.9 < seconds < 30, seconds
    # its counter is its own: the library's stays as it was
    assert L.wait_timeouts() == before


def test_the_library_works_after_a_wait_ran_out(L):
    L.selftest_wait_limit()
    w = W.Workload("after_timeout", 300, 4096, "bf16", 1e-5, 0, "round_once",
                   ("normal", 0.0, 1.0), ("uniform", 0.9, 1.1), ("normal", 0.0, 1.0), seed=9)
    inp = W.make_inputs(w)
    x, g, dy = (inp[k].cuda() for k in ("x", "gamma", "dy"))
    y, rstd = L.rms_norm_fwd(x, g, w.eps)
    dx, dw = L.rms_norm_bwd(dy, x, g, rstd)
    torch.cuda.synchronize()
    xd, gd, dyd = (W.as_float64(inp[k]) for k in ("x", "gamma", "dy"))
    rstd_ref = rounding.round_to(orm.rstd_exact(xd, w.eps), "f32")
    P.check_rstd(rstd.cpu().numpy(), rstd_ref)
    y_ref, _ = orm.forward(xd, gd, w.eps, 0, "bf16", "round_once")
    P.check_rows(W.as_float64(y.cpu()), y_ref, "bf16", None, "y")
    _, dw_exact = orm.backward_exact(dyd, xd, gd, rstd.cpu().numpy().astype(np.float64), 0)
    P.check_dw(dw.cpu().numpy(), rounding.round_to(dw_exact, "f32"))
