"""RMSNorm forward with an FP8 E4M3 output, on the GPU, against the float64
oracle (oracle.fp8), through the C ABI."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import fp8 as of8

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
    rng = np.random.default_rng(99)
    pick = rng.choice(rows, size=limit - 4, replace=False)
    return np.unique(np.concatenate([pick, [0, 1, rows - 2, rows - 1]]))


def _y8_values(y):
    return y.float().cpu().double().numpy()


def run_and_check(L, w, scale, sample_limit=1024, to_dev=None):
    inp = W.make_inputs(w)
    to_dev = to_dev or (lambda t: t.cuda())
    x, g = to_dev(inp["x"]), to_dev(inp["gamma"])
    sc = torch.tensor([scale], dtype=torch.float32, device="cuda")
    y8, rstd = L.rms_norm_fwd_fp8(x, g, sc, w.eps, w.offset)
    torch.cuda.synchronize()
    assert y8.dtype == torch.float8_e4m3fn and y8.shape == x.shape
    xd, gd = W.as_float64(inp["x"]), W.as_float64(inp["gamma"])
    rows = _sample_rows(w.rows, sample_limit)
    ref, rstd_ref = of8.forward_fp8(xd[rows], gd, w.eps, w.offset, scale)
    P.check_rstd(rstd.cpu().numpy()[rows], rstd_ref)
    P.check_rows(_y8_values(y8)[rows], ref, "e4m3", None, "y8")
    # the rstd of the storage-type forward: bit-identical where the same
    # kernel runs (every width but the fp32 rows that only a cluster holds,
    # where the FP8 store takes the scalar kernel and sums in another order)
    _, rstd_plain = L.rms_norm_fwd(x, g, w.eps, w.offset)
    if w.dtype == "f32" and w.hidden > 32768:
        P.check_rstd(rstd.cpu().numpy(), rstd_plain.cpu().double().numpy())
    else:
        assert torch.equal(rstd, rstd_plain)
    return y8, rstd


@pytest.mark.parametrize("name", sorted(W.fp8_workloads()))
def test_named_fp8_workload(L, name):
    w = W.fp8_workloads()[name]
    run_and_check(L, w, w.scale, sample_limit=2048)


SHAPES = [(1, 1, "f32"), (3, 8, "bf16"), (17, 24, "f16"), (5, 1001, "bf16"), (9, 1024, "bf16"),
          (7, 1032, "f16"), (300, 4096, "bf16"), (40, 3072, "f32"), (4, 16384, "bf16"),
          (3, 16392, "f16"), (2, 32768, "f32"), (2, 65536, "bf16"), (2, 65536, "f32"),
          (611, 12288, "bf16"), (1000, 8192, "f16"), (40, 32768, "bf16"), (9, 16384, "f32")]


@pytest.mark.parametrize("rows,hidden,dtype", SHAPES)
def test_fp8_shapes(L, rows, hidden, dtype):
    w = W.Workload("fp8_shape", rows, hidden, dtype, 1e-5, 0, "round_once", ("normal", 0.0, 1.0),
                   ("uniform", 0.9, 1.1), ("normal", 0.0, 1.0), seed=rows * 7 + hidden)
    run_and_check(L, w, 24.0)


@pytest.mark.parametrize("scale", [1.0, 0.01, 200.0, 1.0e4])
def test_fp8_scales_subnormals_and_saturation(L, scale):
    """Small scales put many outputs in the E4M3 subnormal range; large
    ones saturate most of them at +-448."""
    w = W.LLAMA_BF16_4096x4096.with_(rows=96)
    y8, _ = run_and_check(L, w, scale)
    v = _y8_values(y8)
    if scale >= 200.0:
        assert np.mean(np.abs(v) == 448.0) > 0.01
    if scale <= 0.01:
        assert np.mean((np.abs(v) < 2.0 ** -6) & (v != 0)) > 0.01


def test_fp8_gemma_offset(L):
    w = W.GEMMA_BF16_8192x3072.with_(rows=128)
    run_and_check(L, w, 16.0)


def _misaligned_copy(t):
    buf = torch.empty(t.numel() + 1, dtype=t.dtype, device="cuda")
    v = buf[1:].view(t.shape)
    v.copy_(t.cuda())
    return v


@pytest.mark.parametrize("dtype", ["f32", "bf16", "f16"])
def test_fp8_unaligned(L, dtype):
    w = W.LLAMA_BF16_4096x4096.with_(rows=33, hidden=2048, dtype=dtype)
    run_and_check(L, w, 8.0, to_dev=_misaligned_copy)


def test_fp8_scale_is_read_on_the_device(L):
    """The scale is a device value: a captured CUDA graph picks up a new
    value on replay."""
    w = W.LLAMA_BF16_4096x4096.with_(rows=64)
    inp = W.make_inputs(w)
    x, g = inp["x"].cuda(), inp["gamma"].cuda()
    sc = torch.tensor([4.0], dtype=torch.float32, device="cuda")
    y8 = torch.empty(x.shape, dtype=torch.float8_e4m3fn, device="cuda")
    rstd = torch.empty(w.rows, dtype=torch.float32, device="cuda")
    L.rms_norm_fwd_fp8(x, g, sc, w.eps, y=y8, rstd=rstd)   # set-up outside capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            L.rms_norm_fwd_fp8(x, g, sc, w.eps, y=y8, rstd=rstd)
    for scale in (4.0, 64.0):
        sc.fill_(scale)
        graph.replay()
        torch.cuda.synchronize()
        ref, _ = of8.forward_fp8(W.as_float64(inp["x"]), W.as_float64(inp["gamma"]), w.eps, 0,
                                 scale)
        P.check_rows(_y8_values(y8), ref, "e4m3", None, "y8")


def test_fp8_backward_runs_on_its_rstd(L):
    """The backward needs only x, dy, gamma and rstd: the FP8 forward's rstd
    gives the same dx and dw as the storage-type forward's."""
    w = W.LLAMA_BF16_4096x4096.with_(rows=256)
    inp = {k: v.cuda() for k, v in W.make_inputs(w).items()}
    sc = torch.tensor([32.0], dtype=torch.float32, device="cuda")
    _, r8 = L.rms_norm_fwd_fp8(inp["x"], inp["gamma"], sc, w.eps)
    _, r = L.rms_norm_fwd(inp["x"], inp["gamma"], w.eps)
    a = L.rms_norm_bwd(inp["dy"], inp["x"], inp["gamma"], r8)
    b = L.rms_norm_bwd(inp["dy"], inp["x"], inp["gamma"], r)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_fp8_no_wait_timeouts(L):
    assert L.wait_timeouts() == 0
