"""Brute-force number-format tables for the tests, independent of the oracle.

Values of every finite code come from the bit-level definitions (BF16 is the
upper half of an IEEE binary32) or from PyTorch's own FP8 dtypes, and the
nearest-code searches run over those sorted tables.  Nothing here is shared
with ``oracle/`` or with the CUDA library.
"""
from __future__ import annotations

import functools

import numpy as np
import torch


@functools.lru_cache(None)
def bf16_table():
    """(codes, values) of the non-negative finite BF16 values in increasing
    order, with +inf appended as the value 2^128 (the next step of the
    sequence), so that round-to-nearest overflows exactly as IEEE does."""
    codes = np.arange(0, 0x7F80, dtype=np.uint32)
    vals = (codes << 16).view(np.float32).astype(np.float64)
    return (np.append(codes, 0x7F80).astype(np.uint16), np.append(vals, 2.0 ** 128))


@functools.lru_cache(None)
def fp8_table(kind: int):
    """(codes, values) of the non-negative finite FP8 values (0 = E4M3FN,
    1 = E5M2), decoded by PyTorch's float8 dtypes."""
    dt = torch.float8_e4m3fn if kind == 0 else torch.float8_e5m2
    top = 0x7E if kind == 0 else 0x7B
    codes = np.arange(0, top + 1, dtype=np.uint8)
    vals = torch.from_numpy(codes.copy()).view(dt).to(torch.float64).numpy()
    assert np.all(np.diff(vals) > 0)
    return codes, vals


def decode_bf16(bits) -> np.ndarray:
    bits = np.asarray(bits, np.uint16)
    with np.errstate(invalid="ignore"):
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def decode_fp8(codes, kind: int) -> np.ndarray:
    dt = torch.float8_e4m3fn if kind == 0 else torch.float8_e5m2
    c = np.ascontiguousarray(codes, np.uint8)
    return torch.from_numpy(c.copy()).view(dt).to(torch.float64).numpy()


def _nearest(a: np.ndarray, codes: np.ndarray, vals: np.ndarray) -> np.ndarray:
    """Index of the nearest table value to each a >= 0, ties to the even code."""
    i = np.searchsorted(vals, a)            # vals[i-1] < a <= vals[i]
    hi = np.clip(i, 0, len(vals) - 1)
    lo = np.clip(i - 1, 0, len(vals) - 1)
    d_lo = a - vals[lo]
    d_hi = vals[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (codes[hi] % 2 == 0))
    return np.where(vals[hi] == a, hi, np.where(pick_hi, hi, lo))


def nearest_bf16(v) -> np.ndarray:
    """Round doubles to BF16 bit patterns, nearest with ties to even."""
    v = np.asarray(v, np.float64)
    codes, vals = bf16_table()
    a = np.abs(v)
    idx = _nearest(np.minimum(a, 2.0 ** 128), codes, vals)
    out = codes[idx]
    out = np.where(np.signbit(v), out | 0x8000, out).astype(np.uint16)
    return np.where(np.isnan(v), np.uint16(0x7FC0), out).astype(np.uint16)


def nearest_fp8(v, kind: int) -> np.ndarray:
    """Round to FP8 codes, nearest with ties to even, magnitudes beyond the
    largest finite value saturating to it; NaN -> 0x7F."""
    v = np.asarray(v, np.float64)
    codes, vals = fp8_table(kind)
    a = np.minimum(np.abs(v), vals[-1])
    out = codes[_nearest(a, codes, vals)]
    out = np.where(np.signbit(v), out | 0x80, out).astype(np.uint8)
    return np.where(np.isnan(v), np.uint8(0x7F), out).astype(np.uint8)


def bf16_ulp(v) -> np.ndarray:
    """Spacing of BF16 values at |v| (2^(floor(log2|v|) - 7), at least the
    subnormal quantum 2^-133)."""
    a = np.abs(np.asarray(v, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -126)
    return np.where(a > 0, np.exp2(e - 7), 2.0 ** -133)


def fp8_midpoint_distance(v, kind: int) -> np.ndarray:
    """Relative distance of each |v| to the nearest rounding midpoint between
    two adjacent FP8 values (inf where |v| is beyond the largest value)."""
    _, vals = fp8_table(kind)
    mids = (vals[1:] + vals[:-1]) / 2
    a = np.abs(np.asarray(v, np.float64))
    i = np.clip(np.searchsorted(mids, a), 1, len(mids) - 1)
    d = np.minimum(np.abs(a - mids[i - 1]), np.abs(a - mids[i]))
    return np.where(a > vals[-1], np.inf, d / np.maximum(a, 1e-300))


def to_bits_bf16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
