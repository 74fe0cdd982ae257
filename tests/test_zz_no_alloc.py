"""The backward entry point that allocates nothing: rms_norm_bwd_noalloc.

Some callers cannot allocate device memory at the point where they run the
backward -- a plugin whose enqueue hook must not call cudaMalloc, or a
service held to a fixed, pre-reserved memory budget -- so they cannot hand
rms_norm_bwd the workspace it asks for.  rms_norm_bwd_noalloc keeps the
weight-gradient partials in a fixed 16 MiB array inside the library instead.
These tests call it through the C ABI and check it against rms_norm_bwd, on
two calls in a row because every call reuses the same array, and check that
it refuses sizes the array cannot hold.

This file is named so that pytest collects it last.
"""
import ctypes
import os

import numpy as np
import pytest
import torch

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
    # rows, hidden, dtype, offset -- vector kernels at the benchmark size, the
    # scalar kernels (hidden not a multiple of the vector), fp32
    (4096, 4096, torch.bfloat16, 0),
    (777, 1001, torch.float16, 1),
    (300, 2048, torch.float32, 0),
]


@pytest.mark.gpu
@pytest.mark.parametrize("rows,hidden,dtype,offset", CASES)
def test_noalloc_matches_workspace_backward(L, rows, hidden, dtype, offset):
    assert torch.cuda.is_available(), "GPU test needs a CUDA device"
    lib = L.load_library()
    fmt = {torch.float32: "f32", torch.bfloat16: "bf16", torch.float16: "f16"}[dtype]
    gen = torch.Generator().manual_seed(rows + hidden)
    x = torch.randn(rows, hidden, generator=gen).to(dtype).cuda()
    dy = torch.randn(rows, hidden, generator=gen).to(dtype).cuda()
    g = (torch.rand(hidden, generator=gen) * 0.2 + 0.9).to(dtype).cuda()
    _, rstd = L.rms_norm_fwd(x, g, 1e-5, offset)
    dx_ref, dw_ref = L.rms_norm_bwd(dy, x, g, rstd, offset)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream().cuda_stream
    for _ in range(2):
        dx = torch.full_like(x, 5.0)
        dw = torch.full((hidden,), 5.0, dtype=torch.float32, device="cuda")
        st = lib.rms_norm_bwd_noalloc(
            ctypes.c_void_p(dy.data_ptr()), ctypes.c_void_p(x.data_ptr()),
            ctypes.c_void_p(g.data_ptr()), ctypes.c_void_p(rstd.data_ptr()),
            ctypes.c_void_p(dx.data_ptr()), ctypes.c_void_p(dw.data_ptr()),
            rows, hidden, offset, L.DTYPE_CODES[dtype], ctypes.c_void_p(stream))
        assert st == L.RMSN_OK, lib.rms_norm_status_string(st)
        torch.cuda.synchronize()
        P.check_rows(_f64(dx), _f64(dx_ref), fmt, None, "dx")
        P.check_dw(dw.cpu().numpy(), dw_ref.cpu().numpy())


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
