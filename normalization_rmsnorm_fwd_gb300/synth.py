"""Seeded synthetic inputs for the RMSNorm workloads.

This module only draws random numbers and stores them in the formats the
operations consume; it holds none of the normalisation arithmetic.  The same
host bits feed the CPU oracle and the CUDA library.

Recipe: a CPU ``torch.Generator`` seeded with ``seed`` draws FP32 standard
normals in a fixed tensor order (x, residual, gate, style, g, weight noise),
each affinely mapped in FP32 (``shift + scale * N(0, 1)``) and rounded to BF16
with round-to-nearest-even (``Tensor.to(torch.bfloat16)``).  FP32 weights stay
FP32.  BF16 tensors are returned as numpy ``uint16`` bit patterns.

Workloads (shapes and distributions of the pages' own examples):

* ``plain_small``     T=64, H=256: x, g ~ N(0,1); w = 1 + 0.1 N(0,1).
* ``residual_large``  T=16384, H=4096: x, residual, g ~ N(0,1); w = 1 + 0.1 N.
* ``zero_centred``    H=5120, T given: x ~ 4 N(0,1); g ~ N(0,1); FP32
                      w ~ 0.02 N(0,1) (effective weight 1 + w).
* ``strided_heads``   a [2048, 32, 256] BF16 buffer whose [..., :128] slice is
                      normalised row by row (65536 rows, H=128, row stride 256);
                      the gradient lives in a second buffer of the same shape;
                      FP32 w ~ 0.02 N(0,1) [128].
* ``fp8``             T=H=8192: x, residual ~ N(0,1); w = 1 + 0.1 N; scale 0.04.
* ``ada``             rows=2520, dim=3072: x, residual, gate ~ N(0,1); w = 1;
                      style ~ N(0,1) as (rows, 3*dim) and (1, 3*dim);
                      scale 0.04.
"""
from __future__ import annotations

import numpy as np
import torch

EPS = 1e-6
FP8_SCALE = 0.04


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """FP32 tensor -> BF16 (round to nearest even) bit patterns as uint16."""
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


class Draw:
    """Fixed-order normal draws from one seeded CPU generator."""

    def __init__(self, seed: int = 0):
        self.g = torch.Generator().manual_seed(int(seed))

    def normal_f32(self, shape, scale: float = 1.0, shift: float = 0.0) -> torch.Tensor:
        t = torch.randn(tuple(shape), generator=self.g, dtype=torch.float32)
        if scale != 1.0:
            t.mul_(scale)
        if shift != 0.0:
            t.add_(shift)
        return t

    def bf16(self, shape, scale: float = 1.0, shift: float = 0.0) -> np.ndarray:
        return bf16_bits(self.normal_f32(shape, scale, shift))

    def f32(self, shape, scale: float = 1.0, shift: float = 0.0) -> np.ndarray:
        return self.normal_f32(shape, scale, shift).numpy()


def plain_small(seed: int = 0, T: int = 64, H: int = 256) -> dict:
    d = Draw(seed)
    x = d.bf16((T, H))
    g = d.bf16((T, H))
    w = d.bf16((H,), 0.1, 1.0)
    return dict(x=x, g=g, w=w, eps=EPS, T=T, H=H)


def residual_large(seed: int = 0, T: int = 16384, H: int = 4096) -> dict:
    d = Draw(seed)
    x = d.bf16((T, H))
    residual = d.bf16((T, H))
    g = d.bf16((T, H))
    w = d.bf16((H,), 0.1, 1.0)
    return dict(x=x, residual=residual, g=g, w=w, eps=EPS, T=T, H=H)


def zero_centred(T: int, seed: int = 0, H: int = 5120) -> dict:
    d = Draw(seed)
    x = d.bf16((T, H), 4.0)
    g = d.bf16((T, H))
    w32 = d.f32((H,), 0.02)
    return dict(x=x, g=g, w=w32, eps=EPS, T=T, H=H)


def strided_heads(seed: int = 0, T: int = 2048, heads: int = 32, W: int = 256,
                  H: int = 128) -> dict:
    d = Draw(seed)
    buf = d.bf16((T, heads, W))
    gbuf = d.bf16((T, heads, W))
    w32 = d.f32((H,), 0.02)
    return dict(buf=buf, gbuf=gbuf, w=w32, eps=EPS, T=T, heads=heads, W=W, H=H)


def fp8(seed: int = 0, T: int = 8192, H: int = 8192) -> dict:
    d = Draw(seed)
    x = d.bf16((T, H))
    residual = d.bf16((T, H))
    w = d.bf16((H,), 0.1, 1.0)
    return dict(x=x, residual=residual, w=w, scale=FP8_SCALE, eps=EPS, T=T, H=H)


def ada(seed: int = 0, T: int = 2520, D: int = 3072) -> dict:
    d = Draw(seed)
    x = d.bf16((T, D))
    residual = d.bf16((T, D))
    gate = d.bf16((T, D))
    style = d.bf16((T, 3 * D))
    style1 = d.bf16((1, 3 * D))
    w = bf16_bits(torch.ones(D, dtype=torch.float32))
    return dict(x=x, residual=residual, gate=gate, style=style, style1=style1, w=w,
                scale=FP8_SCALE, eps=EPS, T=T, D=D)


def random_rows(seed: int, T: int, H: int, scale: float = 1.0, n: int = 1) -> list:
    """n independent BF16 [T, H] tensors ~ scale * N(0, 1) (edge-case tests)."""
    d = Draw(seed)
    return [d.bf16((T, H), scale) for _ in range(n)]


def bf16_codes(seed: int, shape, lo: int, hi: int, signed: bool = True) -> np.ndarray:
    """BF16 bit patterns whose magnitude codes are drawn uniformly from
    [lo, hi) (0x0001..0x007F are the subnormals, 0x0080 is 2^-126) with, when
    `signed`, a random sign bit (edge-case tests near the bottom of the
    range)."""
    g = torch.Generator().manual_seed(int(seed))
    mag = torch.randint(int(lo), int(hi), tuple(shape), generator=g, dtype=torch.int32)
    if signed:
        mag |= torch.randint(0, 2, tuple(shape), generator=g, dtype=torch.int32) << 15
    return mag.numpy().astype(np.uint16)


def random_weight(seed: int, H: int, f32: bool = False) -> np.ndarray:
    """BF16 w = 1 + 0.1 N(0,1), or FP32 zero-centred w = 0.02 N(0,1)."""
    d = Draw(seed)
    return d.f32((H,), 0.02) if f32 else d.bf16((H,), 0.1, 1.0)
