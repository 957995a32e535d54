"""PyTorch-facing binding of the C ABI: argument marshalling only.

Each function has the name of the C entry point it calls, takes CUDA tensors,
turns them into pointers, row counts and row strides, allocates outputs the
caller did not pass (``torch.empty``), and enqueues the call on the current
stream of the tensors' device.  Every step of the computation runs in the
CUDA library; a failing status raises :class:`CrmsnError`.

Row tensors are ``[..., H]`` with a contiguous feature dimension.  Leading
dimensions collapse into rows when each is contiguous with the next in
row-major order (``stride(i) == stride(i+1) * size(i+1)``), so a
``[T, heads, H]`` slice of a wider ``[T, heads, W]`` buffer is read in place
as ``T*heads`` rows of stride ``W`` ("cake_rmsnorm_det_train_forward"
Parameters/x); any other layout raises ``ValueError``.
"""
from __future__ import annotations

import contextlib
import math

import torch

from . import _abi
from ._abi import BF16, E4M3, E5M2, F32, CrmsnError, check  # noqa: F401

_FP8 = {torch.float8_e4m3fn: E4M3, torch.float8_e5m2: E5M2}


def _lib():
    return _abi.load()


# The raw handle of the current stream without building a Stream object
# (a few microseconds a call); the public query where it is missing.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(t: torch.Tensor) -> int:
    if _raw_stream is not None:
        return _raw_stream(t.get_device())
    return torch.cuda.current_stream(t.device).cuda_stream


_SAME_DEVICE = contextlib.nullcontext()


def _on_device(t: torch.Tensor):
    """A context making t's device current; nothing to do when it already is."""
    idx = t.get_device()
    if idx == torch.cuda.current_device():
        return _SAME_DEVICE
    return torch.cuda.device(idx)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _need_cuda(t: torch.Tensor, name: str):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")


def as_rows(t: torch.Tensor, name: str = "x") -> tuple[int, int, int]:
    """(rows, H, row stride in elements) of a row-collapsible tensor."""
    shape = t.shape
    nd = len(shape)
    if nd < 1:
        raise ValueError(f"{name}: needs at least one dimension")
    st = t.stride()
    H = shape[-1]
    if H > 1 and st[-1] != 1:
        raise ValueError(f"{name}: the feature dimension must be contiguous")
    if nd == 1:
        return 1, H, H
    for i in range(nd - 2):
        if shape[i] > 1 and st[i] != st[i + 1] * shape[i + 1]:
            raise ValueError(
                f"{name}: leading dimensions must be contiguous with one another "
                "(stride(i) == stride(i+1) * size(i+1)) to collapse into rows")
    rows = shape[0] if nd == 2 else math.prod(shape[:-1])
    ld = st[-2] if shape[-2] > 1 else max(H, st[-2])
    return rows, H, ld


def _bf16(t, name):
    _need_cuda(t, name)
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")


def _weight(w):
    _need_cuda(w, "w")
    if w.dtype == torch.bfloat16:
        kind = BF16
    elif w.dtype == torch.float32:
        kind = F32
    else:
        raise TypeError(f"w must be bfloat16 or float32, got {w.dtype}")
    if w.dim() != 1 or (w.numel() > 1 and w.stride(0) != 1):
        raise ValueError("w must be a contiguous 1-D tensor")
    return kind


def _scale_tensor(scale, device):
    if isinstance(scale, torch.Tensor):
        s = scale.to(device=device, dtype=torch.float32)
        return s.reshape(1).contiguous()
    return torch.tensor([float(scale)], dtype=torch.float32, device=device)


# ---------------------------------------------------------------- forward --

def rmsnorm_fwd(x, w, eps: float = 1e-6, residual=None, weight_bias: float = 0.0,
                y=None, rstd=None, h_new=None, want_rstd: bool = True):
    """y = bf16((h * rstd) * f32(w + weight_bias)) with h = x or
    h_new = bf16(x + residual).  Returns (y, rstd, h_new)."""
    _bf16(x, "x")
    kind = _weight(w)
    T, H, ldx = as_rows(x, "x")
    ldr = 0
    if residual is not None:
        _bf16(residual, "residual")
        if residual.shape != x.shape:
            raise ValueError("residual must have x's shape")
        _, _, ldr = as_rows(residual, "residual")
        if h_new is None:
            h_new = torch.empty_like(x, memory_format=torch.contiguous_format)
    if y is None:
        y = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
    if rstd is None and want_rstd:
        rstd = torch.empty(x.shape[:-1], dtype=torch.float32, device=x.device)
    _, _, ldy = as_rows(y, "y")
    ldh = as_rows(h_new, "h_new")[2] if h_new is not None else 0
    with _on_device(x):
        st = _lib().rmsnorm_fwd(_ptr(x), ldx, _ptr(residual), ldr, _ptr(w), kind,
                                float(weight_bias), float(eps), T, H, _ptr(y), ldy, _ptr(rstd),
                                _ptr(h_new), ldh, _stream(x))
    check("rmsnorm_fwd", st)
    return y, rstd, h_new


def rmsnorm_quant(out, x, w, scale, eps: float = 1e-6, weight_bias: float = 0.0, rstd=None):
    """out = fp8(RMSNorm(x) * w / scale) (no residual)."""
    return fused_add_rmsnorm_quant(out, x, None, w, scale, eps, weight_bias, rstd)


def fused_add_rmsnorm_quant(out, x, residual, w, scale, eps: float = 1e-6,
                            weight_bias: float = 0.0, rstd=None):
    """residual <- bf16(x + residual) in place (when given); out = fp8 of the
    normalised value divided by the static FP32 scale."""
    _bf16(x, "x")
    _need_cuda(out, "out")
    if out.dtype not in _FP8:
        raise TypeError("out must be float8_e4m3fn or float8_e5m2")
    kind = _weight(w)
    T, H, ldx = as_rows(x, "x")
    ldr = 0
    if residual is not None:
        _bf16(residual, "residual")
        _, _, ldr = as_rows(residual, "residual")
    _, _, ldo = as_rows(out, "out")
    s = _scale_tensor(scale, x.device)
    with _on_device(x):
        st = _lib().fused_add_rmsnorm_quant(_ptr(out), ldo, _FP8[out.dtype], _ptr(x), ldx,
                                            _ptr(residual), ldr, _ptr(w), kind,
                                            float(weight_bias), _ptr(s), float(eps), T, H,
                                            _ptr(rstd), _stream(x))
    check("fused_add_rmsnorm_quant", st)
    return out


def fused_add_rmsnorm_fp8_block_quant(out, block_scale, normed_out, x, residual, w,
                                      eps: float = 1e-6):
    """residual <- bf16(x + residual); normed_out = bf16(RMSNorm * w);
    out / block_scale = its 1x128 E4M3 quantisation, block_scale being
    (H/128, ldT) column-major with ldT = block_scale.shape[1] >= T."""
    for t, n in ((x, "x"), (residual, "residual"), (normed_out, "normed_out")):
        _bf16(t, n)
    _need_cuda(out, "out")
    if out.dtype != torch.float8_e4m3fn:
        raise TypeError("out must be float8_e4m3fn")
    if block_scale.dtype != torch.float32 or not block_scale.is_contiguous():
        raise TypeError("block_scale must be a contiguous float32 tensor")
    if _weight(w) != BF16:
        raise TypeError("w must be bfloat16")
    T, H, ldx = as_rows(x, "x")
    _, _, ldr = as_rows(residual, "residual")
    if not (out.is_contiguous() and normed_out.is_contiguous()):
        raise ValueError("out and normed_out must be contiguous")
    if block_scale.dim() != 2 or block_scale.shape[0] != H // 128:
        raise ValueError("block_scale must be (H/128, ldT)")
    ldT = block_scale.shape[1]
    with _on_device(x):
        st = _lib().fused_add_rmsnorm_fp8_block_quant(_ptr(out), _ptr(block_scale), ldT,
                                                      _ptr(normed_out), _ptr(x), ldx,
                                                      _ptr(residual), ldr, _ptr(w), float(eps),
                                                      T, H, _stream(x))
    check("fused_add_rmsnorm_fp8_block_quant", st)
    return out, block_scale, normed_out


def ada_rms_norm_style(x, w, style, eps: float = 1e-6, out=None, gate_out=None):
    """AdaRMSNorm: bf16(RMSNorm(x, w) * (1 + scale) + shift); gate_out is the
    style's last third.  style is (rows, 3*dim) or (1, 3*dim)."""
    _bf16(x, "x")
    _bf16(style, "style")
    if _weight(w) != BF16:
        raise TypeError("w must be bfloat16")
    if not (x.is_contiguous() and style.is_contiguous()):
        raise ValueError("x and style must be contiguous")
    T, D = x.shape
    if out is None:
        out = torch.empty_like(x)
    if gate_out is None:
        gate_out = torch.empty_like(x)
    with _on_device(x):
        st = _lib().ada_rms_norm_style(_ptr(x), _ptr(w), _ptr(style), style.shape[0],
                                       float(eps), T, D, _ptr(out), _ptr(gate_out), _stream(x))
    check("ada_rms_norm_style", st)
    return out, gate_out


def gate_residual_ada_norm_fp8(residual, x, gate, w, style, scale, eps: float = 1e-6,
                               out=None, gate_out=None):
    """residual <- bf16(residual + bf16(x * gate)); out = e4m3 of the
    AdaRMSNorm of the new residual divided by scale.  Returns
    (residual, out, gate_out)."""
    for t, n in ((residual, "residual"), (x, "x"), (gate, "gate"), (style, "style")):
        _bf16(t, n)
        if not t.is_contiguous():
            raise ValueError(f"{n} must be contiguous")
    if _weight(w) != BF16:
        raise TypeError("w must be bfloat16")
    T, D = x.shape
    if out is None:
        out = torch.empty((T, D), dtype=torch.float8_e4m3fn, device=x.device)
    if gate_out is None:
        gate_out = torch.empty_like(x)
    s = _scale_tensor(scale, x.device)
    with _on_device(x):
        st = _lib().gate_residual_ada_norm_fp8(_ptr(residual), _ptr(x), _ptr(gate), _ptr(w),
                                               _ptr(style), style.shape[0], _ptr(s),
                                               float(eps), T, D, _ptr(out), _ptr(gate_out),
                                               _stream(x))
    check("gate_residual_ada_norm_fp8", st)
    return residual, out, gate_out



def fused_rmsnorm_silu(x, w, eps: float = 1e-6, weight_bias: float = 0.0, out=None,
                       scale=None, rstd=None):
    """SiLU(RMSNorm(x) * w_eff): out is BF16 (default, allocated when None) or
    a float8_e4m3fn tensor, which receives e4m3(silu / scale) (scale None:
    no scale).  Returns out."""
    _bf16(x, "x")
    kind = _weight(w)
    T, H, ldx = as_rows(x, "x")
    if out is None:
        out = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
    _need_cuda(out, "out")
    if out.dtype == torch.bfloat16:
        fmt = _abi.OUT_BF16
    elif out.dtype == torch.float8_e4m3fn:
        fmt = _abi.OUT_E4M3
    else:
        raise TypeError("out must be bfloat16 or float8_e4m3fn")
    _, _, ldo = as_rows(out, "out")
    s = _scale_tensor(scale, x.device) if (scale is not None and fmt == _abi.OUT_E4M3) else None
    with _on_device(x):
        st = _lib().fused_rmsnorm_silu(_ptr(out), ldo, fmt, _ptr(x), ldx, _ptr(w), kind,
                                       float(weight_bias), _ptr(s), float(eps), T, H,
                                       _ptr(rstd), _stream(x))
    check("fused_rmsnorm_silu", st)
    return out


def _ln_params(x, gamma, beta):
    _bf16(x, "x")
    for t, name in ((gamma, "gamma"), (beta, "beta")):
        _need_cuda(t, name)
        if t.dtype != torch.float32 or t.dim() != 1 or (t.numel() > 1 and t.stride(0) != 1):
            raise TypeError(f"{name} must be a contiguous 1-D float32 tensor")
    return as_rows(x, "x")


def layernorm(x, gamma, beta, eps: float = 1e-5, out=None, mean=None, rstd=None):
    """bf16((x - E[x]) / sqrt(Var[x] + eps) * gamma + beta) with the
    population variance; gamma and beta FP32.  Returns out."""
    T, H, ldx = _ln_params(x, gamma, beta)
    if out is None:
        out = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
    _bf16(out, "out")
    _, _, ldo = as_rows(out, "out")
    with _on_device(x):
        st = _lib().layernorm(_ptr(out), ldo, _ptr(x), ldx, _ptr(gamma), _ptr(beta), float(eps),
                              T, H, _ptr(mean), _ptr(rstd), _stream(x))
    check("layernorm", st)
    return out


def layernorm_quant(out, x, gamma, beta, scale, eps: float = 1e-5, mean=None, rstd=None):
    """out = fp8(layernorm(x) / scale) with out float8_e4m3fn or
    float8_e5m2.  Returns out."""
    T, H, ldx = _ln_params(x, gamma, beta)
    _need_cuda(out, "out")
    if out.dtype not in _FP8:
        raise TypeError("out must be float8_e4m3fn or float8_e5m2")
    _, _, ldo = as_rows(out, "out")
    s = _scale_tensor(scale, x.device)
    with _on_device(x):
        st = _lib().layernorm_quant(_ptr(out), ldo, _FP8[out.dtype], _ptr(x), ldx, _ptr(gamma),
                                    _ptr(beta), _ptr(s), float(eps), T, H, _ptr(mean), _ptr(rstd),
                                    _stream(x))
    check("layernorm_quant", st)
    return out

# --------------------------------------------------------------- backward --

def rmsnorm_bwd_workspace_bytes(rows: int, hidden: int, device=None, residual: bool = False) -> int:
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    idx = dev.index if dev.index is not None else torch.cuda.current_device()
    n = _lib().rmsnorm_bwd_workspace_bytes(int(rows), int(hidden), idx, int(bool(residual)))
    if n == 0:
        raise CrmsnError("rmsnorm_bwd_workspace_bytes", 3, "invalid hidden size or device")
    return n


def rmsnorm_bwd_workspace(rows: int, hidden: int, device=None) -> torch.Tensor:
    """A zero-filled uint8 workspace of rmsnorm_bwd_workspace_bytes() bytes
    (the caching allocator returns 512-byte aligned blocks)."""
    dev = torch.device(device) if device is not None else torch.device("cuda")
    return torch.zeros(rmsnorm_bwd_workspace_bytes(rows, hidden, dev), dtype=torch.uint8,
                       device=dev)


def rmsnorm_bwd(g, x, w, rstd, weight_bias: float = 0.0, g_residual=None, workspace=None,
                dx=None, dw=None):
    """dx = bf16(rstd*g*w_eff - x*rstd^3*mean(g*w_eff*x) (+ g_residual)) and the
    deterministic FP32 dw = sum_t g*x*rstd.  Returns (dx, dw)."""
    _bf16(g, "g")
    _bf16(x, "x")
    kind = _weight(w)
    T, H, ldx = as_rows(x, "x")
    if g.shape != x.shape:
        raise ValueError("g must have x's shape")
    _, _, ldg = as_rows(g, "g")
    ldgr = 0
    if g_residual is not None:
        _bf16(g_residual, "g_residual")
        _, _, ldgr = as_rows(g_residual, "g_residual")
    if rstd.dtype != torch.float32 or not rstd.is_contiguous() or rstd.numel() != T:
        raise ValueError("rstd must be a contiguous float32 tensor with one value per row")
    if dx is None:
        dx = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
    _, _, lddx = as_rows(dx, "dx")
    if dw is None:
        dw = torch.empty(H, dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = torch.empty(rmsnorm_bwd_workspace_bytes(T, H, x.device), dtype=torch.uint8,
                                device=x.device)
    with _on_device(x):
        st = _lib().rmsnorm_bwd(_ptr(g), ldg, _ptr(x), ldx, _ptr(w), kind, float(weight_bias),
                                _ptr(rstd), _ptr(g_residual), ldgr, T, H, _ptr(dx), lddx,
                                _ptr(dw), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                _stream(x))
    check("rmsnorm_bwd", st)
    return dx, dw


def rmsnorm_bwd_noalloc(g, x, w, rstd, weight_bias: float = 0.0, g_residual=None, dx=None,
                        dw=None):
    """rmsnorm_bwd for callers that cannot provide a workspace: the library's
    built-in 16 MiB scratch is used instead, shared by every call on the
    device (overlapping calls race).  Returns (dx, dw)."""
    _bf16(g, "g")
    _bf16(x, "x")
    kind = _weight(w)
    T, H, ldx = as_rows(x, "x")
    _, _, ldg = as_rows(g, "g")
    ldgr = 0
    if g_residual is not None:
        _bf16(g_residual, "g_residual")
        _, _, ldgr = as_rows(g_residual, "g_residual")
    if dx is None:
        dx = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device)
    _, _, lddx = as_rows(dx, "dx")
    if dw is None:
        dw = torch.empty(H, dtype=torch.float32, device=x.device)
    with _on_device(x):
        st = _lib().rmsnorm_bwd_noalloc(_ptr(g), ldg, _ptr(x), ldx, _ptr(w), kind,
                                        float(weight_bias), _ptr(rstd), _ptr(g_residual), ldgr, T,
                                        H, _ptr(dx), lddx, _ptr(dw), _stream(x))
    check("rmsnorm_bwd_noalloc", st)
    return dx, dw


def rmsnorm_supports(H: int, w_dtype: int = BF16, op: int = _abi.OP_FWD) -> int:
    return _lib().rmsnorm_supports(int(H), int(w_dtype), int(op))
