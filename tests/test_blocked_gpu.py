"""The weight gradient over fixed row blocks (rms_norm_bwd_blocked and
rms_norm_dw_sum), on the GPU, through the C ABI.

Its point is a summation order that does not depend on how the rows are
shared out: block partials (sequential over a block's rows), chunks of 32
blocks each summed on its own in a fixed order, chunk sums added in
order.  These tests check, for every backward kernel family:

* dx and dw against the float64 oracle with the parity tolerances;
* that splitting the rows over several calls along whole chunks (the ranks
  of a data-parallel job, here run one after the other on one GPU) and
  adding all their chunk sums gives bit-identical dw and dx;
* that an SM budget, which changes how many CTAs share the blocks, changes
  no bit.
The default rms_norm_bwd, whose blocks are one per CTA, is checked against
the oracle under an SM budget as well.
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
    yield lib
    lib.rms_norm_set_sm_budget(0)


# rows, hidden, dtype, the kernel the backward runs (for narrow rows: with
# blocks of 3 rows, and with blocks of 16, whose stages hold several rows)
CASES = [
    (600, 4096, "bf16", "bwd_tma"),
    (300, 8192, "bf16", "bwd_tma"),
    (500, 256, "f32", ("bwd_tma", "bwd_tma_rows")),
    (600, 1024, "bf16", ("bwd_tma", "bwd_tma_rows")),
    (300, 2048, "f16", ("bwd_tma", "bwd_tma_rows")),
    (200, 16384, "f16", "bwd_tma_wide"),
    (100, 32768, "f16", "bwd_tma_split"),
    (90, 16384, "f32", "bwd_tma_split"),
    (40, 12292, "f32", "bwd_cta_rows"),
    (20, 65536, "f32", "bwd_cluster"),
    (77, 1001, "f16", "bwd_scalar"),
]


def _setup(rows, hidden, dtype, offset=0):
    w = W.Workload("blocked", rows, hidden, dtype, 1e-5, offset, "round_once",
                   ("normal", 0.0, 1.0),
                   ("normal", 0.0, 0.1) if offset else ("uniform", 0.9, 1.1),
                   ("normal", 0.0, 1.0), seed=rows * 3 + hidden)
    inp = W.make_inputs(w)
    xd, gd, dyd = (W.as_float64(inp[k]) for k in ("x", "gamma", "dy"))
    rstd_ref = rounding.round_to(orm.rstd_exact(xd, w.eps), "f32")
    dev = {k: inp[k].cuda() for k in ("x", "gamma", "dy")}
    dev["rstd"] = torch.from_numpy(rstd_ref.astype(np.float32)).cuda()
    return w, (xd, gd, dyd, rstd_ref), dev


def _ran(L, kernel):
    """The last call launched `kernel` (mangled or demangled symbol name)."""
    names = L.last_kernels()
    return any(f"{len(kernel)}{kernel}I" in n or f"{kernel}<" in n for n in names), names


def _blocked(L, dev, brows, offset, rows=None):
    sl = slice(None) if rows is None else slice(*rows)
    dx, chunks = L.rms_norm_bwd_blocked(dev["dy"][sl], dev["x"][sl], dev["gamma"],
                                        dev["rstd"][sl], brows, offset)
    return dx, chunks


@pytest.mark.parametrize("rows,hidden,dtype,kernel", CASES)
@pytest.mark.parametrize("brows", [3, 16])
def test_blocked_matches_oracle(L, rows, hidden, dtype, kernel, brows):
    offset = 1 if brows == 3 else 0
    w, (xd, gd, dyd, rstd_ref), dev = _setup(rows, hidden, dtype, offset)
    dx, chunks = _blocked(L, dev, brows, offset)
    if isinstance(kernel, tuple):
        kernel = kernel[0] if brows == 3 else kernel[1]
    ok, names = _ran(L, kernel)
    assert ok, names
    assert chunks.shape == (L.rms_norm_dw_chunk_count(rows, brows), hidden)
    dw = L.rms_norm_dw_sum(chunks)
    torch.cuda.synchronize()
    dx_exact, dw_exact = orm.backward_exact(dyd, xd, gd, rstd_ref, offset)
    terms = rstd_ref[:, None] * dyd * orm.gain(gd, offset)[None, :]
    P.check_rows(W.as_float64(dx.cpu()), rounding.round_to(dx_exact, dtype), dtype, None, "dx",
                 terms, cancels=True)
    P.check_dw(dw.cpu().numpy(), rounding.round_to(dw_exact, "f32"))


@pytest.mark.parametrize("rows,hidden,dtype,kernel", CASES)
@pytest.mark.parametrize("world", [2, 3])
def test_split_over_ranks_gives_the_same_bits(L, rows, hidden, dtype, kernel, world):
    """The rows split along whole chunks (rms_norm_rank_rows), one call per
    slab, the slabs' chunk sums laid end to end: the same dx and dw, bit for
    bit, as one call over all rows."""
    rows = max(rows, 128)
    brows = 1 if rows < 400 else 2
    _, _, dev = _setup(rows, hidden, dtype)
    dx_all, chunks_all = _blocked(L, dev, brows, 0)
    dw_all = L.rms_norm_dw_sum(chunks_all)
    spans = [L.rms_norm_rank_rows(rows, brows, world, r) for r in range(world)]
    assert sum(1 for a, b in spans if b > a) >= 2, spans   # a real split
    parts = [(a, b, _blocked(L, dev, brows, 0, (a, b))) for a, b in spans if b > a]
    chunks = torch.cat([c for _, _, (_, c) in parts])
    dw = L.rms_norm_dw_sum(chunks)
    torch.cuda.synchronize()
    assert torch.equal(chunks, chunks_all)
    assert torch.equal(dw, dw_all)
    for a, b, (dx, _) in parts:
        assert torch.equal(dx, dx_all[a:b])


@pytest.mark.parametrize("rows,hidden,dtype,kernel", CASES)
def test_sm_budget_changes_no_bit(L, rows, hidden, dtype, kernel):
    """Fewer CTAs (an SM budget) deal the same blocks differently: same bits."""
    _, _, dev = _setup(rows, hidden, dtype)
    brows = 2
    L.rms_norm_set_sm_budget(0)
    dx0, c0 = _blocked(L, dev, brows, 0)
    try:
        for sms in (37, 8):
            L.rms_norm_set_sm_budget(sms)
            dx1, c1 = _blocked(L, dev, brows, 0)
            torch.cuda.synchronize()
            assert torch.equal(dx0, dx1) and torch.equal(c0, c1), sms
    finally:
        L.rms_norm_set_sm_budget(0)


def test_default_backward_under_a_budget_meets_the_oracle(L):
    w, (xd, gd, dyd, rstd_ref), dev = _setup(777, 4096, "bf16")
    L.rms_norm_set_sm_budget(19)
    try:
        dx, dw = L.rms_norm_bwd(dev["dy"], dev["x"], dev["gamma"], dev["rstd"])
        torch.cuda.synchronize()
    finally:
        L.rms_norm_set_sm_budget(0)
    _, dw_exact = orm.backward_exact(dyd, xd, gd, rstd_ref, 0)
    P.check_dw(dw.cpu().numpy(), rounding.round_to(dw_exact, "f32"))


def test_empty_and_zero_chunk_calls(L):
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    r = torch.empty(0, dtype=torch.float32, device="cuda")
    dx, chunks = L.rms_norm_bwd_blocked(x, x, g, r, 4)
    assert chunks.shape == (0, 64) and L.last_launch_count() == 0
    dw = L.rms_norm_dw_sum(chunks, dw=torch.full((64,), 3.0, device="cuda"))
    torch.cuda.synchronize()
    assert torch.count_nonzero(dw).item() == 0


def test_no_bounded_wait_ran_out(L):
    assert L.wait_timeouts() == 0


@pytest.mark.parametrize("rows,hidden,dtype", [(600, 1024, "bf16"), (300, 2048, "f16"),
                                               (500, 256, "f32"), (97, 512, "f16")])
def test_multi_row_stages_give_the_one_row_kernels_dx(L, rows, hidden, dtype):
    """Narrow rows are staged several to a ring slot (bwd_tma_rows) unless the
    caller's blocks are not a multiple of the stage: blocks of 3 rows run the
    one-row-a-stage kernel (bwd_tma).  dx does not depend on the blocks, so
    the two kernels' dx must agree bit for bit, and with the default call."""
    _, _, dev = _setup(rows, hidden, dtype)
    dx3, _ = _blocked(L, dev, 3, 0)
    assert _ran(L, "bwd_tma")[0]
    dx16, _ = _blocked(L, dev, 16, 0)
    assert _ran(L, "bwd_tma_rows")[0]
    dx, _ = L.rms_norm_bwd(dev["dy"], dev["x"], dev["gamma"], dev["rstd"])
    assert _ran(L, "bwd_tma_rows")[0]
    torch.cuda.synchronize()
    assert torch.equal(dx3, dx16)
    assert torch.equal(dx3, dx)
