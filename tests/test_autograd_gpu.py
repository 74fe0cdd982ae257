"""The autograd layer (``rms_norm`` / ``RMSNorm``) runs the library's
forward and backward: its outputs and gradients are bit-identical to direct
calls of rms_norm_fwd / rms_norm_bwd, whose parity with the oracle the other
GPU tests establish."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    import bwd_rms_norm_gb300 as lib
    lib.load_library()
    return lib


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
@pytest.mark.parametrize("offset", [0, 1])
def test_module_matches_direct_calls(L, dtype, offset):
    gen = torch.Generator().manual_seed(5)
    x0 = torch.randn(3, 40, 1024, generator=gen).to(dtype).cuda()
    dy = torch.randn(3, 40, 1024, generator=gen).to(dtype).cuda()
    m = L.RMSNorm(1024, eps=1e-5, offset=offset, device="cuda", dtype=dtype)
    with torch.no_grad():
        m.weight.copy_((torch.rand(1024, generator=gen) * 0.2 + (0.0 if offset else 0.9))
                       .to(dtype))
    x = x0.clone().requires_grad_(True)
    y = m(x)
    y.backward(dy)
    torch.cuda.synchronize()
    y_ref, rstd = L.rms_norm_fwd(x0, m.weight.detach(), 1e-5, offset)
    dx_ref, dw_ref = L.rms_norm_bwd(dy, x0, m.weight.detach(), rstd, offset)
    torch.cuda.synchronize()
    assert y.dtype == dtype and y.shape == x0.shape
    assert torch.equal(y.detach(), y_ref)
    assert torch.equal(x.grad, dx_ref)
    assert m.weight.grad.dtype == dtype
    assert torch.equal(m.weight.grad, dw_ref.to(dtype))


def test_non_contiguous_input_and_round_twice(L):
    gen = torch.Generator().manual_seed(6)
    base = torch.randn(256, 64, generator=gen).to(torch.bfloat16).cuda()
    xt = base.t()                      # [64, 256], not contiguous
    w = (torch.rand(256, generator=gen) + 0.5).to(torch.bfloat16).cuda().requires_grad_(True)
    x = xt.clone().requires_grad_(True)
    assert not x.is_contiguous()
    y = L.rms_norm(x, w, 1e-6, 0, "round_twice")
    dy = torch.randn(y.shape, generator=gen).to(torch.bfloat16).cuda()
    y.backward(dy)
    torch.cuda.synchronize()
    xc = xt.contiguous()
    y_ref, rstd = L.rms_norm_fwd(xc, w.detach(), 1e-6, 0, "round_twice")
    dx_ref, dw_ref = L.rms_norm_bwd(dy, xc, w.detach(), rstd, 0)
    torch.cuda.synchronize()
    assert torch.equal(y.detach(), y_ref)
    assert torch.equal(x.grad, dx_ref)
    assert torch.equal(w.grad, dw_ref.to(torch.bfloat16))
