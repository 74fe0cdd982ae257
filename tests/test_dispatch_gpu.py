"""Which kernel each call runs, on the shapes the benchmarks time: a change
that silently routes a shape to a slower kernel (for instance to the scalar
fallback) keeps every parity test green, so the dispatch is pinned here
through rms_norm_last_kernels()."""
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import bwd_rms_norm_gb300 as lib
    lib.load_library()
    return lib


def _dev(w, rows=None):
    return {k: v.cuda() for k, v in W.make_inputs(w, rows).items()}


def _kernels(L):
    return L.last_kernels()


def _expect(names, *parts):
    assert len(names) == len(parts), names
    for n, p in zip(names, parts):
        assert p in n, (p, names)


# workload, forward kernel, backward row kernel (a part of the mangled name:
# "7bwd_tmaI" is bwd_tma itself, not bwd_tma_rows or bwd_tma_wide)
RMS = [
    ("llama_bf16_4096x4096", "fwd_tma", "7bwd_tmaI"),
    ("gemma_bf16_8192x3072", "fwd_tma", "7bwd_tmaI"),
    ("fp16_4096x1024", "fwd_warp_rows", "bwd_tma_rowsI6__halfLi4E"),
    ("fp16_4096x2048", "fwd_cta_row", "bwd_tma_rowsI6__halfLi2E"),
    ("fp16_4096x8192", "fwd_tma", "7bwd_tmaI"),
    ("fp16_4096x16384", "fwd_tma", "bwd_tma_wide"),
    ("fp16_4096x32768", "fwd_tma_split", "bwd_tma_split"),
    ("large_bf16_16384x8192_once", "fwd_tma", "7bwd_tmaI"),
    ("fp32_256x1024", "fwd_cta_row", "bwd_tma_rowsIfLi2E"),
]


@pytest.mark.parametrize("name,fwd,bwd", RMS)
def test_rms_norm_dispatch(L, name, fwd, bwd):
    w = W.all_workloads()[name]
    t = _dev(w, rows=min(w.rows, 512))
    y, r = L.rms_norm_fwd(t["x"], t["gamma"], w.eps, w.offset, w.cast_mode)
    _expect(_kernels(L), fwd)
    L.rms_norm_bwd(t["dy"], t["x"], t["gamma"], r, w.offset)
    _expect(_kernels(L), bwd, "dw_finalize")
    sc = torch.tensor([8.0], device="cuda")
    L.rms_norm_fwd_fp8(t["x"], t["gamma"], sc, w.eps, w.offset)
    _expect(_kernels(L), fwd)


def test_staged_forwards_deal_wide_rows_round_robin(L):
    """The staged forwards take the CTA's rows round-robin for rows of 16 KB
    and more (the last template argument, RR; the one before it is F8, the
    FP8 store), contiguous ranges for narrower rows."""
    sc = torch.tensor([8.0], device="cuda")
    for name, plain, fp8 in (("large_bf16_16384x8192_once", "Lb0ELb1EE", "Lb1ELb1EE"),
                             ("fp16_4096x16384", "Lb0ELb1EE", "Lb1ELb1EE"),
                             ("llama_bf16_4096x4096", "Lb0ELb0EE", "Lb1ELb0EE"),
                             ("gemma_bf16_8192x3072", "Lb0ELb0EE", "Lb1ELb0EE")):
        w = W.all_workloads()[name]
        t = _dev(w, rows=300)
        L.rms_norm_fwd(t["x"], t["gamma"], w.eps, w.offset, w.cast_mode)
        _expect(_kernels(L), plain)
        L.rms_norm_fwd_fp8(t["x"], t["gamma"], sc, w.eps, w.offset)
        _expect(_kernels(L), fp8)
    for name, part in (("ln_bf16_16384x8192", "ln_fwd_tmaI13__nv_bfloat16Li2ELb1EE"),
                       ("ln_bf16_4096x4096", "ln_fwd_tmaI13__nv_bfloat16Li1ELb0EE")):
        w = W.layer_norm_workloads()[name]
        t = _dev(w, rows=300)
        L.layer_norm_fwd(t["x"], t["gamma"], t["beta"], w.eps)
        _expect(_kernels(L), part)


def test_unaligned_rows_take_the_scalar_kernels(L):
    x = torch.randn(8, 1001, device="cuda").to(torch.bfloat16)
    g = torch.ones(1001, device="cuda", dtype=torch.bfloat16)
    y, r = L.rms_norm_fwd(x, g, 1e-5)
    _expect(_kernels(L), "fwd_scalar")
    L.rms_norm_bwd(x, x, g, r)
    _expect(_kernels(L), "bwd_scalar", "dw_finalize")
    L.softmax_fwd(x)
    _expect(_kernels(L), "sm_fwd_scalar")


def test_layer_norm_dispatch(L):
    for name, fwd, bwd in (("ln_bf16_4096x4096", "ln_fwd_tma", "ln_bwd_tma"),
                           ("ln_fp32_256x1024", "ln_fwd_cta_row", "ln_bwd_tma"),
                           ("ln_bf16_16384x8192", "ln_fwd_tma", "ln_bwd_tma")):
        w = W.layer_norm_workloads()[name]
        t = _dev(w, rows=min(w.rows, 512))
        _, m, r = L.layer_norm_fwd(t["x"], t["gamma"], t["beta"], w.eps)
        _expect(_kernels(L), fwd)
        L.layer_norm_bwd(t["dy"], t["x"], t["gamma"], m, r)
        _expect(_kernels(L), bwd, "dw_finalize")


def test_softmax_dispatch(L):
    for name, fwd, bwd in (("softmax_bf16_4096x4096", "sm_fwd_cta_row", "sm_bwd_cta_row"),
                           ("softmax_bf16_16384x8192", "sm_fwd_cta_row", "sm_bwd_rows"),
                           ("softmax_f16_65536x1024", "sm_fwd_warp_rows", "sm_bwd_warp_rows")):
        w = W.softmax_workloads()[name]
        t = _dev(w, rows=512)
        y = L.softmax_fwd(t["x"])
        _expect(_kernels(L), fwd)
        L.softmax_bwd(t["dy"], y)
        _expect(_kernels(L), bwd)


def test_group_norm_dispatch(L):
    for name, fwd, bwd in (("gn_bf16_16x32x256x256_g8", "gn_fwd_pipe", "gn_bwd_l2"),
                           ("gn_bf16_16x512x64x64_g32", "gn_fwd_pipe", "gn_bwd_l2"),
                           ("gn_fp32_16x32x256x256_g8", "gn_fwd_pipe", "gn_bwd_l2")):
        w = W.group_norm_workloads()[name]
        t = _dev(w, rows=2)
        _, m, r = L.group_norm_fwd(t["x"], t["gamma"], t["beta"], w.groups, w.eps)
        _expect(_kernels(L), fwd)
        L.group_norm_bwd(t["dy"], t["x"], t["gamma"], m, r, w.groups)
        _expect(_kernels(L), bwd, "dw_finalize")


def test_nothing_launched_reports_nothing(L):
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    L.rms_norm_fwd(x, g, 1e-5)
    assert _kernels(L) == []
