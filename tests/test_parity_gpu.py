"""GPU results against the float64 oracle on the same seeded inputs.

Every call goes through the C ABI (via the ctypes binding).  The named
workloads run at their full sizes in the launch configuration the benchmark
times; where the oracle would need minutes for every row, y and dx are
compared on a fixed sample of rows (rows are independent), while rstd and dw
are always compared in full.
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


def _sample_rows(rows: int, limit: int) -> np.ndarray:
    if rows <= limit:
        return np.arange(rows)
    rng = np.random.default_rng(1234)
    pick = rng.choice(rows, size=limit - 4, replace=False)
    return np.unique(np.concatenate([pick, [0, 1, rows - 2, rows - 1]]))


def run_and_check(L, w: W.Workload, sample_limit: int = 1024, inputs=None, to_dev=None):
    inp = inputs if inputs is not None else W.make_inputs(w)
    x, g, dy = inp["x"], inp["gamma"], inp["dy"]
    xd, gd, dyd = W.as_float64(x), W.as_float64(g), W.as_float64(dy)
    fmt = w.dtype
    to_dev = to_dev or (lambda t: t.cuda())
    xc, gc, dyc = to_dev(x), to_dev(g), to_dev(dy)

    y, rstd = L.rms_norm_fwd(xc, gc, w.eps, w.offset, w.cast_mode)
    torch.cuda.synchronize()
    rows = _sample_rows(w.rows, sample_limit)

    # rstd over every row, y on the sampled rows
    rstd_ref = rounding.round_to(orm.rstd_exact(xd, w.eps), "f32")
    stats = P.check_rstd(rstd.cpu().numpy(), rstd_ref)
    y_ref, _ = orm.forward(xd[rows], gd, w.eps, w.offset, fmt, w.cast_mode)
    alt = None
    if w.cast_mode == orm.ROUND_TWICE and fmt != "f32":
        x_hat = xd[rows] * orm.rstd_exact(xd[rows], w.eps)[:, None]
        mask, y_lo, y_hi = P.round_twice_alternatives(x_hat, orm.gain(gd, w.offset)[None, :], fmt)
        alt = [(mask, y_lo), (mask, y_hi)]
    y_got = W.as_float64(y.cpu())[rows]
    stats.update({"y_" + k: v for k, v in P.check_rows(y_got, y_ref, fmt, alt, "y").items()})

    # backward from the oracle's rstd
    rstd_in = to_dev(torch.from_numpy(rstd_ref.astype(np.float32)))
    dx, dw = L.rms_norm_bwd(dyc, xc, gc, rstd_in, w.offset)
    torch.cuda.synchronize()
    # dw needs every row; dx is rounded (the slow step) on the sampled rows only
    dx_exact, dw_exact = orm.backward_exact(dyd, xd, gd, rstd_ref, w.offset)
    dx_ref = rounding.round_to(dx_exact[rows], fmt)
    dw_ref = rounding.round_to(dw_exact, "f32")
    dx_got = W.as_float64(dx.cpu())[rows]
    terms = rstd_ref[rows, None] * dyd[rows] * orm.gain(gd, w.offset)[None, :]
    stats.update({"dx_" + k: v for k, v in
                  P.check_rows(dx_got, dx_ref, fmt, None, "dx", terms,
                                cancels=True).items()})
    stats.update(P.check_dw(dw.cpu().numpy(), dw_ref))
    return stats


NAMED = sorted(W.all_workloads())


@pytest.mark.parametrize("name", NAMED)
def test_named_workload(L, name):
    w = W.all_workloads()[name]
    stats = run_and_check(L, w, sample_limit=2048 if w.rows * w.hidden > (1 << 25) else w.rows)
    print(name, stats)


def test_fp16_overflow_stress(L):
    """x with standard deviation 64: a sum of squares in fp16 would overflow
    for every row at every width; fp32 statistics keep every output finite."""
    for hidden in (1024, 8192):
        w = W.fp16_sweep(hidden, x_var=4096.0).with_(rows=512)
        run_and_check(L, w)


@pytest.mark.parametrize("rows,hidden,dtype", [
    (64, 1024, "bf16"), (40, 2048, "f32"), (24, 4096, "bf16"), (16, 8192, "f32"),
    (12, 16384, "bf16"), (6, 65536, "f32"), (10, 1001, "bf16"), (8, 3, "f32"),
    (8, 32768, "bf16"), (6, 16384, "f32")])
def test_sum_of_squares_past_fp32(L, rows, hidden, dtype):
    """Rows of bf16/fp32 values so large that an fp32 sum of squares
    overflows (every square past 2**128 for the 2**70 rows; only the sum for
    the 2**60 rows), beside ordinary rows and rows near 2**100: the kernels
    sum those rows again scaled by a power of two, so rstd, y and the
    backward match the float64 oracle, whose squares never overflow."""
    w = W.Workload("overflow", rows, hidden, dtype, 1e-5, 0, "round_once",
                   ("normal", 0.0, 1.0), ("uniform", 0.9, 1.1), ("normal", 0.0, 1.0),
                   seed=rows + hidden)
    inp = W.make_inputs(w)
    scale = torch.tensor([2.0 ** (70, 60, 0, 100)[r % 4] for r in range(rows)])
    inp["x"] = (inp["x"].double() * scale[:, None]).to(inp["x"].dtype)
    assert torch.isfinite(inp["x"]).all()
    x32 = inp["x"].float()
    assert torch.isinf((x32 * x32).sum(dim=1)[0])      # the fp32 sum does overflow
    run_and_check(L, w, inputs=inp)


SHAPES = [
    # rows, hidden, dtype -- covers warp-per-row, CTA-per-row, 16-vector
    # rows, the scalar path (hidden not a multiple of the vector), widths
    # one past a vector, tiny rows and the maximum width
    (1, 1, "f32"), (3, 8, "bf16"), (17, 24, "f16"), (5, 1001, "bf16"), (7, 1032, "f16"),
    (9, 1024, "bf16"), (6, 1028, "f32"), (3, 4104, "bf16"), (4, 16384, "bf16"),
    (3, 16392, "bf16"), (2, 32768, "f32"), (2, 65536, "bf16"), (2, 65536, "f32"),
    (2, 65536, "f16"), (300, 4096, "bf16"), (151, 2048, "f16"), (153, 512, "f32"),
    (1, 32768, "f16"), (33, 3072, "bf16"), (2, 7, "f16"),
    # the staged backward for 2048-vector rows (a packed gain copy in shared
    # memory, four vectors per applier): ragged row counts over the 152-CTA
    # grid
    (1000, 16384, "f16"), (157, 16384, "bf16"), (301, 8192, "f32"),
    # the cluster-split forward and backward for 4096-vector rows (each CTA
    # of a cluster stages its part of every row): ragged row counts over the
    # clusters, fewer rows than clusters, and a width between 2048 and 4096
    # vectors
    (300, 32768, "f16"), (157, 16384, "f32"), (5, 32768, "bf16"), (77, 24576, "bf16"),
]


@pytest.mark.parametrize("rows,hidden,dtype", SHAPES)
def test_shapes(L, rows, hidden, dtype):
    w = W.Workload(f"shape_{rows}x{hidden}_{dtype}", rows, hidden, dtype, 1e-5, 0,
                   "round_once", ("normal", 0.0, 1.0), ("uniform", 0.9, 1.1),
                   ("normal", 0.0, 1.0), seed=rows * 7 + hidden)
    run_and_check(L, w)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("offset", [0, 1])
@pytest.mark.parametrize("cast_mode", ["round_once", "round_twice"])
@pytest.mark.parametrize("hidden", [256, 2560])
def test_modes(L, dtype, offset, cast_mode, hidden):
    gamma_dist = ("normal", 0.0, 0.1) if offset else ("uniform", 0.9, 1.1)
    w = W.Workload("modes", 64, hidden, dtype, 1e-6, offset, cast_mode,
                   ("normal", 0.0, 2.0), gamma_dist, ("normal", 0.0, 1.0), seed=11)
    run_and_check(L, w)


@pytest.mark.parametrize("rows,hidden,dtype", [(40, 32768, "bf16"), (33, 32768, "f16"),
                                               (20, 16384, "f32")])
@pytest.mark.parametrize("offset", [0, 1])
@pytest.mark.parametrize("cast_mode", ["round_once", "round_twice"])
def test_split_forward_modes(L, rows, hidden, dtype, offset, cast_mode):
    """Rows split over a cluster in the forward (fwd_tma_split): both cast
    modes and the Gemma offset, against the oracle."""
    gamma_dist = ("normal", 0.0, 0.1) if offset else ("uniform", 0.9, 1.1)
    w = W.Workload("split_modes", rows, hidden, dtype, 1e-6, offset, cast_mode,
                   ("normal", 0.0, 2.0), gamma_dist, ("normal", 0.0, 1.0), seed=rows + offset)
    inp = W.make_inputs(w)
    L.rms_norm_fwd(inp["x"].cuda(), inp["gamma"].cuda(), w.eps, w.offset, w.cast_mode)
    assert any("fwd_tma_split" in k for k in L.last_kernels()), L.last_kernels()
    run_and_check(L, w, inputs=inp)


def _misaligned_copy(t: torch.Tensor, shift_elems: int = 1) -> torch.Tensor:
    """A contiguous CUDA copy of ``t`` whose data pointer is not 16-byte
    aligned (it starts ``shift_elems`` elements into a larger buffer)."""
    buf = torch.empty(t.numel() + shift_elems, dtype=t.dtype, device="cuda")
    v = buf[shift_elems:].view(t.shape)
    v.copy_(t.cuda())
    assert v.data_ptr() % 16 != 0
    return v


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
@pytest.mark.parametrize("cast_mode", ["round_once", "round_twice"])
def test_unaligned_pointers(L, dtype, cast_mode):
    """Data that is not 16-byte aligned runs the scalar kernels; they meet the
    same tolerances against the oracle."""
    w = W.Workload("unaligned", 40, 1024, dtype, 1e-5, 1, cast_mode,
                   ("normal", 0.0, 1.0), ("normal", 0.0, 0.1), ("normal", 0.0, 1.0), seed=5)
    run_and_check(L, w, to_dev=_misaligned_copy)


def test_zero_rows(L):
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    y, rstd = L.rms_norm_fwd(x, g, 1e-5)
    assert y.shape == (0, 64) and rstd.shape == (0,)
    assert L.last_launch_count() == 0
    dw = torch.full((64,), 7.0, device="cuda")
    dx, dw = L.rms_norm_bwd(x, x, g, rstd, dw=dw)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dw).item() == 0


def test_zero_input_rows(L):
    """x = 0 with eps > 0: rstd = 1/sqrt(eps), y = 0, dx = rstd * dy * gain."""
    for dtype in (torch.float32, torch.bfloat16):
        x = torch.zeros(8, 512, dtype=dtype, device="cuda")
        g = torch.full((512,), 0.5, dtype=dtype, device="cuda")
        y, rstd = L.rms_norm_fwd(x, g, 0.25)
        assert torch.all(rstd == 2.0) and torch.count_nonzero(y).item() == 0
        dy = torch.ones(8, 512, dtype=dtype, device="cuda")
        dx, dw = L.rms_norm_bwd(dy, x, g, rstd)
        assert torch.all(dx.float() == 1.0) and torch.count_nonzero(dw).item() == 0


@pytest.mark.parametrize("hidden,dtype", [(4096, torch.bfloat16), (1001, torch.float16),
                                          (1024, torch.float32)])
def test_backward_deterministic(L, hidden, dtype):
    gen = torch.Generator().manual_seed(3)
    x = torch.randn(777, hidden, generator=gen).to(dtype).cuda()
    dy = torch.randn(777, hidden, generator=gen).to(dtype).cuda()
    g = (torch.rand(hidden, generator=gen) + 0.5).to(dtype).cuda()
    _, rstd = L.rms_norm_fwd(x, g, 1e-5)
    first = L.rms_norm_bwd(dy, x, g, rstd)
    for _ in range(3):
        again = L.rms_norm_bwd(dy, x, g, rstd)
        assert torch.equal(first[0], again[0])
        assert torch.equal(first[1], again[1])


@pytest.mark.parametrize("rows,hidden,dtype", [(5, 4096, torch.bfloat16), (3, 1001, torch.float16),
                                               (9, 24, torch.float32), (2, 65536, torch.bfloat16)])
def test_outputs_stay_in_bounds(L, rows, hidden, dtype):
    """Canary elements around every output stay untouched."""
    pad = 64
    gen = torch.Generator().manual_seed(9)
    x = torch.randn(rows, hidden, generator=gen).to(dtype).cuda()
    dy = torch.randn(rows, hidden, generator=gen).to(dtype).cuda()
    g = torch.rand(hidden, generator=gen).to(dtype).cuda()

    def guarded(n, dt, fill):
        buf = torch.full((n + 2 * pad,), fill, dtype=dt, device="cuda")
        return buf, buf[pad:pad + n]

    ybuf, y = guarded(rows * hidden, dtype, 3.0)
    rbuf, r = guarded(rows, torch.float32, 3.0)
    L.rms_norm_fwd(x, g, 1e-5, y=y.view(rows, hidden), rstd=r)
    dxbuf, dxv = guarded(rows * hidden, dtype, 3.0)
    dwbuf, dwv = guarded(hidden, torch.float32, 3.0)
    L.rms_norm_bwd(dy, x, g, r, dx=dxv.view(rows, hidden), dw=dwv)
    torch.cuda.synchronize()
    for buf in (ybuf, rbuf, dxbuf, dwbuf):
        assert torch.all(buf[:pad] == 3.0) and torch.all(buf[-pad:] == 3.0)


def test_launch_counts(L):
    x = torch.randn(64, 4096, device="cuda").to(torch.bfloat16)
    g = torch.ones(4096, device="cuda", dtype=torch.bfloat16)
    _, rstd = L.rms_norm_fwd(x, g, 1e-5)
    assert L.last_launch_count() == 1
    L.rms_norm_bwd(x, x, g, rstd)
    assert L.last_launch_count() == 2


def test_no_bounded_wait_ran_out(L):
    """No bounded wait of the staged kernels timed out during this file."""
    assert L.wait_timeouts() == 0
