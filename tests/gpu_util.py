"""Helpers for the GPU parity tests: host<->device transfer of BF16 bit
patterns and the tolerance checks.

Tolerances (the pages' accuracy contract as restated for this library):
* rstd: |gpu - exact| <= 4e-7 * exact.
* BF16 outputs (y, normed, Ada out, dx): |gpu - exact| <= one BF16 ulp of
  the exact value, i.e. either neighbour of the exact value.  Where the value
  is a difference of larger FP32 terms (dx, Ada's shift) an FP32 evaluation
  cannot be closer than the rounding of those terms, so 2^-20 * (|term1| +
  |term2|) is added (a few FP32 ulps of the terms); for dx also the FP32
  rounding of m = mean(g*w*x), 2^-18 * |x| * rstd^3 * mean|g*w*x|.
* h_new, residual updates, gate_out: bit-exact.
* FP8 codes: equal, except one code step where the exact pre-quantisation
  value lies within a relative 2^-18 of a rounding midpoint (the FP32 value
  either side decides can fall on either side there), widened by the same
  cancellation allowance where the value is a difference of larger terms
  (the Ada shift).
* dw: relative L2 error <= 1e-5 and |error_j| <= 1e-5 * sum_t |g x rstd|_j.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import numfmt

DEV = torch.device("cuda:0")
RSTD_TOL = 4e-7
FP8_TIE_WINDOW = 2.0 ** -18


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(DEV)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def host_u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().view(torch.uint8).numpy()


def check_rstd(got, exact, what="rstd"):
    got = np.asarray(got, np.float64)
    err = np.abs(got - exact) / exact
    bad = ~(err <= RSTD_TOL)
    assert not bad.any(), f"{what}: {bad.sum()} rows, max rel err {np.nanmax(err):.3g}"


def check_bf16(got_bits, exact, allowance=None, what="y"):
    got = numfmt.decode_bf16(got_bits)
    tol = numfmt.bf16_ulp(exact)
    if allowance is not None:
        tol = tol + allowance
    err = np.abs(got - exact)
    bad = ~(err <= tol)
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; "
                           f"e.g. got {got[bad][:4]} exact {exact[bad][:4]}")
    return int((got_bits != numfmt.nearest_bf16(exact)).sum())


def check_exact(got, want, what):
    bad = got != want
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} differ (must be bit-exact)"


def check_fp8(got, want, v_exact, kind, what="fp8", allowance=None):
    diff = got != want
    if not diff.any():
        return 0
    window = FP8_TIE_WINDOW
    if allowance is not None:
        window = window + np.asarray(allowance)[diff] / np.maximum(np.abs(v_exact[diff]), 1e-300)
    near_tie = numfmt.fp8_midpoint_distance(v_exact[diff], kind) <= window
    g = got[diff].astype(np.int32)
    w = want[diff].astype(np.int32)
    adjacent = ((g & 0x80) == (w & 0x80)) & (np.abs((g & 0x7F) - (w & 0x7F)) == 1)
    ok = near_tie & adjacent
    assert ok.all(), (f"{what}: {(~ok).sum()} codes differ away from a rounding tie; e.g. "
                      f"got {got[diff][~ok][:4]} want {want[diff][~ok][:4]} "
                      f"exact {v_exact[diff][~ok][:4]}")
    return int(diff.sum())


def check_dw(got, ref, ref_abs, what="dw"):
    got = np.asarray(got, np.float64)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    assert rel <= 1e-5, f"{what}: relative L2 error {rel:.3g}"
    bad = ~(np.abs(got - ref) <= 1e-5 * ref_abs + 1e-30)
    assert not bad.any(), f"{what}: {bad.sum()} columns beyond 1e-5 * sum|terms|"


def dx_allowance(g_bits, x_bits, w_eff, rstd, m):
    """Per element: 2^-20 * (|rstd*g*w| + |x*rstd^3*m|), the FP32 evaluation
    of dx's two terms, plus 2^-18 * |x| * rstd^3 * mean_j |g_j w_j x_j|, the
    rounding of m itself.  m is an FP32 sum of H products (the statistics are
    FP32), whose error is bounded by a few tens of FP32 ulps of the sum of the
    products' magnitudes (each thread adds its at most 32 products in turn,
    then a tree of depth <= 9 adds the threads), not of |m|: where the
    row's products cancel, that is many times |m|."""
    g = numfmt.decode_bf16(g_bits)
    x = numfmt.decode_bf16(x_bits)
    r = np.asarray(rstd, np.float64)[:, None]
    w = np.asarray(w_eff, np.float64)[None, :]
    mabs = np.abs(g * w * x).mean(axis=1, keepdims=True)
    return (2.0 ** -20 * (np.abs(r * g * w) + np.abs(x * r ** 3 * np.asarray(m)[:, None]))
            + 2.0 ** -18 * np.abs(x) * r ** 3 * mabs)


def row_blocks(T: int, H: int, budget: int = 1 << 20) -> list:
    """Consecutive row ranges [lo, hi) of about `budget` elements each."""
    rows = max(1, budget // max(int(H), 1))
    return [(lo, min(T, lo + rows)) for lo in range(0, T, rows)]


def each_block(T: int, H: int, fn, budget: int = 1 << 20):
    """Call fn(lo, hi) for every row block of a [T, H] problem on the host's
    cores and return the results in block order.  The oracle's C calls and
    numpy's whole-array operations release the interpreter lock, so the
    blocks run in parallel; the oracle itself stays single-threaded, each
    call seeing only its own rows.  The first failing block's error is
    raised."""
    blocks = row_blocks(T, H, budget)
    n = min(len(blocks), os.cpu_count() or 1, 16)
    if n <= 1:
        return [fn(lo, hi) for lo, hi in blocks]
    with ThreadPoolExecutor(max_workers=n) as ex:
        futs = [ex.submit(fn, lo, hi) for lo, hi in blocks]
        return [f.result() for f in futs]
