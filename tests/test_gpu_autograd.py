"""The autograd wrapper on the GPU: forward outputs and input / weight
gradients against the oracle (and against a plain PyTorch FP32 autograd of
the same formula), on the plain and residual routes, N-D inputs, expanded
gradients and both weight types."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
from normalization_rmsnorm_fwd_gb300 import synth
import normalization_rmsnorm_fwd_gb300 as crm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


def _bf16_rows(seed, T, H):
    return synth.random_rows(seed, T, H)[0]


def _torch_reference(x, w, eps, bias, residual=None):
    """Plain FP32 PyTorch autograd of the same formula (no kernels)."""
    xf = x.detach().float().requires_grad_(True)
    wf = w.detach().float().requires_grad_(True)
    rf = None
    if residual is not None:
        rf = residual.detach().float().requires_grad_(True)
        h = xf + rf
    else:
        h = xf
    y = h * torch.rsqrt(h.pow(2).mean(-1, keepdim=True) + eps) * (wf + bias)
    return xf, wf, rf, h, y


def _grad_check_dw(orc_dw, orc_abs, got, dtype):
    if dtype == torch.float32:
        gu.check_dw(got.cpu().numpy().astype(np.float64), orc_dw, orc_abs)
    else:
        gu.check_bf16(gu.host_bits(got), orc_dw, allowance=1e-5 * orc_abs, what="dw (bf16)")


@pytest.mark.parametrize("wtype", ["bf16", "f32"])
def test_plain_route(orc, wtype):
    B, S, H = 3, 41, 512
    xb = _bf16_rows(1, B * S, H)
    wb = synth.random_weight(1, H, f32=wtype == "f32")
    bias = 1.0 if wtype == "f32" else 0.0
    gb = _bf16_rows(2, B * S, H)
    x = gu.dev_bf16(xb).reshape(B, S, H).requires_grad_(True)
    w = (gu.dev_f32(wb) if wtype == "f32" else gu.dev_bf16(wb)).requires_grad_(True)
    y = crm.rmsnorm(x, w, 1e-6, weight_bias=bias)
    assert y.shape == (B, S, H) and y.dtype == torch.bfloat16
    y.backward(gu.dev_bf16(gb).reshape(B, S, H))
    torch.cuda.synchronize()
    f = orc.rmsnorm_fwd(xb, wb, 1e-6, weight_bias=bias)
    gu.check_bf16(gu.host_bits(y.detach().reshape(-1, H)), f["y_exact"], what="y")
    ref = orc.rmsnorm_bwd(gb, xb, wb, f["rstd"], weight_bias=bias)
    allow = gu.dx_allowance(gb, xb, orc.weight_eff(wb, bias), f["rstd"], ref["m"])
    gu.check_bf16(gu.host_bits(x.grad.reshape(-1, H)), ref["dx_exact"], allowance=allow, what="dx")
    assert w.grad.dtype == w.dtype
    _grad_check_dw(ref["dw"], ref["dw_abs"], w.grad, w.dtype)
    # The same gradients from plain FP32 PyTorch autograd, loosely (BF16 I/O).
    xf, wf, _, _, yr = _torch_reference(x, w, 1e-6, bias)
    yr.backward(gu.dev_bf16(gb).reshape(B, S, H).float())
    scale = xf.grad.abs().max()
    assert (x.grad.float() - xf.grad).abs().max() <= 2e-2 * scale
    assert torch.allclose(w.grad.float(), wf.grad, rtol=2e-2, atol=2e-2 * wf.grad.abs().max().item())


def test_residual_route(orc):
    T, H = 96, 1024
    xb, ub = _bf16_rows(3, T, H), _bf16_rows(4, T, H)
    wb = synth.random_weight(3, H)
    gyb, ghb = _bf16_rows(5, T, H), _bf16_rows(6, T, H)
    x = gu.dev_bf16(xb).requires_grad_(True)
    u = gu.dev_bf16(ub).requires_grad_(True)
    w = gu.dev_bf16(wb).requires_grad_(True)
    y, h_new = crm.rmsnorm(x, w, 1e-6, residual=u)
    torch.autograd.backward([y, h_new], [gu.dev_bf16(gyb), gu.dev_bf16(ghb)])
    torch.cuda.synchronize()
    f = orc.rmsnorm_fwd(xb, wb, 1e-6, residual=ub)
    assert np.array_equal(gu.host_bits(h_new.detach()), f["h_new"])
    ref = orc.rmsnorm_bwd(gyb, f["h_new"], wb, f["rstd"], g_res=ghb)
    allow = gu.dx_allowance(gyb, f["h_new"], orc.weight_eff(wb), f["rstd"], ref["m"])
    gu.check_bf16(gu.host_bits(x.grad), ref["dx_exact"], allowance=allow, what="dx")
    assert torch.equal(x.grad, u.grad), "x and residual get the same gradient"
    _grad_check_dw(ref["dw"], ref["dw_abs"], w.grad, w.dtype)


def test_only_h_new_used(orc):
    # No gradient reaches y: dx is the gradient of h_new exactly, dw is 0.
    T, H = 32, 256
    x = gu.dev_bf16(_bf16_rows(7, T, H)).requires_grad_(True)
    u = gu.dev_bf16(_bf16_rows(8, T, H)).requires_grad_(True)
    w = gu.dev_bf16(synth.random_weight(7, H)).requires_grad_(True)
    gh = gu.dev_bf16(_bf16_rows(9, T, H))
    _, h_new = crm.rmsnorm(x, w, 1e-6, residual=u)
    h_new.backward(gh)
    torch.cuda.synchronize()
    assert torch.equal(x.grad, gh) and torch.equal(u.grad, gh)
    assert torch.count_nonzero(w.grad) == 0


def test_expanded_gradient(orc):
    # loss = y.sum(): the incoming gradient is an expanded tensor of ones
    # (row stride 0), which the wrapper materialises once.
    T, H = 50, 768
    xb, wb = _bf16_rows(10, T, H), synth.random_weight(10, H)
    x = gu.dev_bf16(xb).requires_grad_(True)
    w = gu.dev_bf16(wb).requires_grad_(True)
    crm.rmsnorm(x, w, 1e-6).sum().backward()
    torch.cuda.synchronize()
    ones = synth.bf16_bits(torch.ones(T, H))
    f = orc.rmsnorm_fwd(xb, wb, 1e-6)
    ref = orc.rmsnorm_bwd(ones, xb, wb, f["rstd"])
    allow = gu.dx_allowance(ones, xb, orc.weight_eff(wb), f["rstd"], ref["m"])
    gu.check_bf16(gu.host_bits(x.grad), ref["dx_exact"], allowance=allow, what="dx")


def test_transposed_input_is_materialised(orc):
    H, T = 256, 64
    base = gu.dev_bf16(_bf16_rows(11, H, T))          # [H, T]
    x = base.t().requires_grad_(False)                # [T, H], features strided
    xb = gu.host_bits(x.contiguous())
    wb = synth.random_weight(11, H)
    y = crm.rmsnorm(x, gu.dev_bf16(wb), 1e-6)
    torch.cuda.synchronize()
    gu.check_bf16(gu.host_bits(y), orc.rmsnorm_fwd(xb, wb, 1e-6)["y_exact"], what="y")
