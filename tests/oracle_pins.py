"""Pins that tie the CPU oracle to what the pages and the mathematics fix.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with an independent fact: a closed form, an invariant, a
finite-difference gradient, a library routine (PyTorch's BF16/FP8 casts,
numpy's norm and FP32 add) or a brute-force search over a format's code table.
``test_oracle_pins.py`` runs them on the oracle; ``test_oracle_mutants.py``
runs them on copies of the oracle with planted mistakes and expects each
mistake to be caught.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

import numfmt
from normalization_rmsnorm_fwd_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "closed_forms.json")


def _close(a, b, rel, what=""):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    scale = np.maximum(np.abs(b), 1e-300)
    bad = ~(np.abs(a - b) <= rel * scale)
    bad &= ~((a == 0) & (b == 0))
    assert not bad.any(), f"{what}: {a[bad][:5]} vs {b[bad][:5]}"


def _bits(vals) -> np.ndarray:
    return synth.bf16_bits(torch.tensor(vals, dtype=torch.float32))


def _eval(expr: str, eps32: float = 0.0) -> float:
    env = {"sqrt": math.sqrt, "log": math.log, "e": math.e, "eps32": eps32, "nan": math.nan,
           "inf": math.inf, "f32": lambda v: float(np.float32(v))}
    return float(eval(expr.replace("^", "**"), {"__builtins__": {}}, env))


# ---------------------------------------------------------------- formats --

def pin_bf16_from_float(o):
    """BF16 rounding of every float matches PyTorch's float->bfloat16 cast
    (round to nearest even) on random bit patterns and constructed ties."""
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2 ** 32, 200_000, dtype=np.uint64).astype(np.uint32)
    hi = rng.integers(0, 2 ** 16, 20_000, dtype=np.uint64).astype(np.uint32) << 16
    special = np.concatenate([
        hi | 0x8000, hi | 0x7FFF, hi | 0x8001,              # ties and near-ties
        np.array([0, 0x80000000, 0x00008000, 0x00018000, 0x7F7FFFFF,
                  0x7F7F8000, 0x7F7F7FFF, 0x7F800000, 0xFF800000, 0x00000001],
                 np.uint32)])
    bits = np.concatenate([bits, special])
    f = bits.view(np.float32)
    f = f[~np.isnan(f)]
    ref = numfmt.to_bits_bf16(torch.from_numpy(f.copy()).to(torch.bfloat16))
    got = o.bf16_from_f64(f.astype(np.float64))
    assert np.array_equal(got, ref), np.flatnonzero(got != ref)[:5]
    assert o.bf16_from_f64(np.array([np.nan]))[0] & 0x7FFF > 0x7F80


def pin_bf16_from_double(o):
    """Doubles between BF16 values round to the nearest table entry, ties to
    even (brute force over all finite BF16 values)."""
    rng = np.random.default_rng(2)
    base = numfmt.decode_bf16(rng.integers(0, 0x7F7F, 50_000).astype(np.uint16))
    ulp = numfmt.bf16_ulp(base)
    frac = rng.choice([0.5, 0.25, 0.75, 0.5 + 2 ** -30, 0.5 - 2 ** -30, 0.999], base.size)
    frac = np.where(rng.random(base.size) < 0.3, rng.random(base.size), frac)
    v = (base + frac * ulp) * rng.choice([-1.0, 1.0], base.size)
    v = np.concatenate([v, [2.0 ** -140, 3 * 2.0 ** -134, 2.0 ** 128 * (1 - 2 ** -9),
                            2.0 ** 128 * (1 - 2 ** -10), 1e300, -1e300]])
    got = o.bf16_from_f64(v)
    ref = numfmt.nearest_bf16(v)
    assert np.array_equal(got, ref), (v[got != ref][:5], got[got != ref][:5], ref[got != ref][:5])


def pin_bf16_decode(o):
    """All 65536 BF16 patterns decode to the upper half of a binary32."""
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = o.bf16_to_f64(codes)
    ref = numfmt.decode_bf16(codes)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all(), codes[~same][:5]
    assert np.array_equal(np.signbit(got[~np.isnan(got)]), np.signbit(ref[~np.isnan(ref)]))


def pin_fp8_decode(o):
    """All 256 codes of E4M3FN and E5M2 decode as PyTorch's float8 dtypes do."""
    codes = np.arange(256, dtype=np.uint16).astype(np.uint8)
    for kind in (0, 1):
        got = o.fp8_to_f64(codes, kind)
        ref = numfmt.decode_fp8(codes, kind)
        same = (got == ref) | (np.isnan(got) & np.isnan(ref))
        assert same.all(), (kind, codes[~same][:5])


def pin_fp8_encode(o):
    """FP8 encoding is round-to-nearest-even with saturation: exact on every
    code value, ties at every midpoint go to the even code, random values go
    to the nearest code, out-of-range values saturate, NaN -> 0x7F."""
    rng = np.random.default_rng(3)
    for kind in (0, 1):
        codes, vals = numfmt.fp8_table(kind)
        mids = (vals[1:] + vals[:-1]) / 2
        rand = np.exp(rng.uniform(np.log(2.0 ** -18), np.log(vals[-1] * 1.2), 20_000))
        v = np.concatenate([vals, mids, rand, [vals[-1] * 1.03, vals[-1] * 4, 1e30, np.inf]])
        v = np.concatenate([v, -v]).astype(np.float32)
        got = o.fp8_from_f32(v, kind)
        ref = numfmt.nearest_fp8(v.astype(np.float64), kind)
        assert np.array_equal(got, ref), (kind, v[got != ref][:5], got[got != ref][:5])
        assert np.array_equal(o.fp8_from_f32(vals.astype(np.float32), kind), codes)
        assert o.fp8_from_f32(np.array([np.nan], np.float32), kind)[0] == 0x7F


def pin_golden_formats(o):
    g = json.load(open(GOLDEN))
    for kind, key in ((0, "e4m3"), (1, "e5m2")):
        for code, expr in g[key].items():
            v = o.fp8_to_f64(np.array([int(code, 16)], np.uint8), kind)[0]
            want = _eval(expr)
            if math.isnan(want):
                assert math.isnan(v), (key, code)
            else:
                assert v == want and math.copysign(1, v) == math.copysign(1, want), (key, code, v)


# ---------------------------------------------------------------- forward --

def pin_golden_forward(o):
    """Hand-derived closed forms of rstd and y (and h_new)."""
    g = json.load(open(GOLDEN))
    for c in g["fwd"]:
        eps32 = float(np.float32(c["eps"]))
        x = _bits([c["x"]])
        w = _bits(c["w"])
        res = _bits([c["residual"]]) if "residual" in c else None
        r = o.rmsnorm_fwd(x, w, c["eps"], residual=res, weight_bias=c["bias"])
        _close(r["rstd_exact"][0], _eval(c["rstd"], eps32), 4e-16, c["name"] + " rstd")
        _close(r["y_exact"][0], [_eval(e, eps32) for e in c["y"]], 4e-16, c["name"] + " y")
        if res is not None:
            _close(numfmt.decode_bf16(r["h_new"][0]), [_eval(e) for e in c["h_new"]], 0,
                   c["name"] + " h_new")


def pin_constant_row(o):
    """A constant row c has mean(h^2) = c^2: rstd = 1/sqrt(c^2 + eps) and
    y = c * rstd * w_eff, for several widths and eps."""
    for c in (0.5, 1.0, -3.0, 100.0, 2.0 ** -20):
        for H in (1, 7, 256):
            for eps in (0.0, 1e-6):
                x = _bits(np.full((1, H), c))
                w = synth.random_weight(5, H)
                r = o.rmsnorm_fwd(x, w, eps)
                e32 = float(np.float32(eps))
                rstd = 1.0 / math.sqrt(c * c + e32) if (c * c + e32) > 0 else math.inf
                _close(r["rstd_exact"][0], rstd, 4e-16, f"rstd c={c} H={H}")
                w_eff = numfmt.decode_bf16(w)
                _close(r["y_exact"][0], c * rstd * w_eff, 1e-15, f"y c={c} H={H}")


def pin_scale_invariance(o):
    """With eps = 0, scaling the input by 2^k leaves y bit-identical and
    scales rstd by exactly 2^-k."""
    x = synth.random_rows(6, 5, 96)[0]
    w = synth.random_weight(6, 96)
    base = o.rmsnorm_fwd(x, w, 0.0)
    for k in (-5, 3):
        xs = synth.bf16_bits(torch.from_numpy(numfmt.decode_bf16(x) * 2.0 ** k).float())
        r = o.rmsnorm_fwd(xs, w, 0.0)
        assert np.array_equal(r["y"], base["y"]) and np.array_equal(r["y_exact"], base["y_exact"])
        assert np.array_equal(r["rstd_exact"] * 2.0 ** k, base["rstd_exact"])


def pin_gemma_equivalence(o):
    """Gemma (BF16 w, bias 1) equals the FP32-weight route fed the same
    values with bias 1, bitwise; the effective weight is the IEEE FP32 sum."""
    x = synth.random_rows(7, 6, 64)[0]
    w = synth.random_weight(7, 64)
    w32 = numfmt.decode_bf16(w).astype(np.float32)
    a = o.rmsnorm_fwd(x, w, 1e-6, weight_bias=1.0)
    b = o.rmsnorm_fwd(x, w32, 1e-6, weight_bias=1.0)
    for k in ("y", "y_exact", "rstd", "rstd_exact"):
        assert np.array_equal(a[k], b[k]), k
    assert np.array_equal(o.weight_eff(w, 1.0), (w32 + np.float32(1.0)).astype(np.float64))
    wz = synth.random_weight(8, 64, f32=True)
    assert np.array_equal(o.weight_eff(wz, 1.0), (wz + np.float32(1.0)).astype(np.float64))
    assert np.array_equal(o.weight_eff(w, 0.0), numfmt.decode_bf16(w))


def pin_textbook_norm(o):
    """With w = 1 and eps = 0, RMSNorm of one row is x * sqrt(H) / ||x||_2."""
    for H in (3, 64, 1000):
        x = synth.random_rows(9, 1, H)[0]
        r = o.rmsnorm_fwd(x, _bits(np.ones(H)), 0.0)
        xd = numfmt.decode_bf16(x[0])
        _close(r["y_exact"][0], xd * math.sqrt(H) / np.linalg.norm(xd), 2e-15, "textbook")


def pin_residual(o):
    """h_new is the nearest BF16 of the exact sum x + residual (brute force),
    including operands whose exponents differ widely; a zero residual gives
    the plain route's outputs."""
    rng = np.random.default_rng(10)
    T, H = 8, 128
    x = synth.random_rows(10, T, H)[0]
    u = synth.bf16_bits(torch.from_numpy(
        numfmt.decode_bf16(synth.random_rows(11, T, H)[0]) *
        np.exp2(rng.integers(-24, 24, (T, H)))).float())
    w = synth.random_weight(10, H)
    r = o.rmsnorm_fwd(x, w, 1e-6, residual=u)
    ref = numfmt.nearest_bf16(numfmt.decode_bf16(x) + numfmt.decode_bf16(u))
    assert np.array_equal(r["h_new"], ref)
    plain = o.rmsnorm_fwd(ref, w, 1e-6)
    for k in ("y", "y_exact", "rstd_exact"):
        assert np.array_equal(r[k], plain[k]), k
    z = o.rmsnorm_fwd(x, w, 1e-6, residual=np.zeros_like(x))
    p = o.rmsnorm_fwd(x, w, 1e-6)
    assert np.array_equal(z["h_new"], x)
    for k in ("y", "y_exact", "rstd_exact"):
        assert np.array_equal(z[k], p[k]), k


def pin_strided(o):
    """A row-strided view gives the results of its contiguous copy."""
    buf = synth.random_rows(12, 9, 160, n=3)
    x = buf[0][:, 16:96]
    g = buf[1][:, 32:112]
    w = synth.random_weight(12, 80, f32=True)
    a = o.rmsnorm_fwd(x, w, 1e-6, weight_bias=1.0)
    b = o.rmsnorm_fwd(np.ascontiguousarray(x), w, 1e-6, weight_bias=1.0)
    for k in ("y", "y_exact", "rstd_exact"):
        assert np.array_equal(a[k], b[k]), k
    ga = o.rmsnorm_bwd(g, x, w, a["rstd"], weight_bias=1.0)
    gb = o.rmsnorm_bwd(np.ascontiguousarray(g), np.ascontiguousarray(x), w, a["rstd"],
                       weight_bias=1.0)
    for k in ("dx", "dx_exact", "dw"):
        assert np.array_equal(ga[k], gb[k]), k


def pin_rstd32(o):
    """The stored FP32 rstd is the nearest float of the exact value."""
    x = synth.random_rows(13, 16, 200, scale=3.0)[0]
    r = o.rmsnorm_fwd(x, synth.random_weight(13, 200), 1e-6)
    assert np.array_equal(r["rstd"], r["rstd_exact"].astype(np.float32))
    assert np.array_equal(r["y"], numfmt.nearest_bf16(r["y_exact"]))


# --------------------------------------------------------------- backward --

def pin_golden_backward(o):
    g = json.load(open(GOLDEN))
    for c in g["bwd"]:
        x = _bits([c["x"]])
        r = o.rmsnorm_bwd(_bits([c["g"]]), x, _bits(c["w"]), np.array([c["rstd"]], np.float32),
                          weight_bias=c["bias"])
        _close(r["m"][0], _eval(c["m"]), 1e-15, c["name"] + " m")
        _close(r["dx_exact"][0], [_eval(e) for e in c["dx"]], 1e-15, c["name"] + " dx")
        _close(r["dw"], [_eval(e) for e in c["dw"]], 1e-15, c["name"] + " dw")


def _loss(o, h, w_eff, eps, g):
    yv, _ = o.row_fwd_f64(h, w_eff, eps)
    return float(np.dot(g, yv))


def pin_finite_differences(o):
    """dx and dw of the double-precision row math match central finite
    differences of L = sum_j g_j * y_j, with and without eps."""
    rng = np.random.default_rng(14)
    for H in (1, 3, 16):
        for eps in (0.0, 0.3):
            h = rng.normal(size=H)
            w_eff = 1 + 0.3 * rng.normal(size=H)
            g = rng.normal(size=H)
            _, rstd = o.row_fwd_f64(h, w_eff, eps)
            dxv, dwr, _ = o.row_bwd_f64(g, h, w_eff, rstd)
            fd_x = np.empty(H)
            fd_w = np.empty(H)
            for j in range(H):
                d = 1e-6 * max(1.0, abs(h[j]))
                hp, hm = h.copy(), h.copy()
                hp[j] += d
                hm[j] -= d
                fd_x[j] = (_loss(o, hp, w_eff, eps, g) - _loss(o, hm, w_eff, eps, g)) / (2 * d)
                wp, wm = w_eff.copy(), w_eff.copy()
                wp[j] += 1e-6
                wm[j] -= 1e-6
                fd_w[j] = (_loss(o, h, wp, eps, g) - _loss(o, h, wm, eps, g)) / 2e-6
            scale = np.max(np.abs(dxv)) + 1e-3
            assert np.max(np.abs(fd_x - dxv)) <= 1e-6 * scale, (H, eps, fd_x, dxv)
            assert np.max(np.abs(fd_w - dwr)) <= 1e-6 * (np.max(np.abs(dwr)) + 1e-3), (H, eps)
            gr = rng.normal(size=H)
            dx2, _, _ = o.row_bwd_f64(g, h, w_eff, rstd, gr)
            _close(dx2 - dxv, gr, 1e-12, "g_res adds")


def pin_dx_invariant(o):
    """sum_j h_j * dx_j = rstd^3 * H * m * eps (zero when eps = 0): the
    gradient is orthogonal to the input up to the eps term."""
    rng = np.random.default_rng(15)
    for eps in (0.0, 0.25):
        H = 50
        h = rng.normal(size=H)
        w_eff = 1 + 0.2 * rng.normal(size=H)
        g = rng.normal(size=H)
        _, rstd = o.row_fwd_f64(h, w_eff, eps)
        dxv, _, m = o.row_bwd_f64(g, h, w_eff, rstd)
        lhs = float(np.dot(h, dxv))
        rhs = rstd ** 3 * H * m * eps
        assert abs(lhs - rhs) <= 1e-13 * float(np.sum(np.abs(h * dxv))) + 1e-300, (eps, lhs, rhs)


def pin_dw(o):
    """dw: for one row it is g * x * rstd elementwise; over rows it is the sum
    of the one-row results; dw and dx are linear in g."""
    T, H = 6, 40
    x = synth.random_rows(16, T, H)[0]
    g = synth.random_rows(17, T, H)[0]
    w = synth.random_weight(16, H)
    rstd = o.rmsnorm_fwd(x, w, 1e-6)["rstd"]
    full = o.rmsnorm_bwd(g, x, w, rstd)
    rows = [o.rmsnorm_bwd(g[t:t + 1], x[t:t + 1], w, rstd[t:t + 1]) for t in range(T)]
    for t in range(T):
        want = numfmt.decode_bf16(g[t]) * numfmt.decode_bf16(x[t]) * float(rstd[t])
        _close(rows[t]["dw"], want, 1e-15, "dw one row")
        assert np.array_equal(rows[t]["dx"], full["dx"][t:t + 1])
    _close(full["dw"], np.sum([r["dw"] for r in rows], axis=0), 1e-13, "dw sum of rows")
    g2 = synth.bf16_bits(torch.from_numpy(numfmt.decode_bf16(g) * 2).float())
    twice = o.rmsnorm_bwd(g2, x, w, rstd)
    assert np.array_equal(twice["dw"], 2 * full["dw"])
    assert np.array_equal(twice["dx_exact"], 2 * full["dx_exact"])
    assert np.all(full["dw_abs"] >= np.abs(full["dw"]))
    assert np.array_equal(full["dx"], numfmt.nearest_bf16(full["dx_exact"]))


def pin_dx_residual_gradient(o):
    """With g_residual the BF16 inputs' gradient is the normalisation gradient
    plus g_residual."""
    T, H = 4, 32
    x = synth.random_rows(18, T, H)[0]
    g, gr = synth.random_rows(19, T, H, n=2)
    w = synth.random_weight(18, H)
    rstd = o.rmsnorm_fwd(x, w, 1e-6)["rstd"]
    a = o.rmsnorm_bwd(g, x, w, rstd)
    b = o.rmsnorm_bwd(g, x, w, rstd, g_res=gr)
    _close(b["dx_exact"] - a["dx_exact"], numfmt.decode_bf16(gr), 1e-12, "g_res")
    assert np.array_equal(a["dw"], b["dw"])


# ------------------------------------------------------------------- FP8 --

def pin_static_quant(o):
    """Static FP8: v = yv / scale (yv of the forward with the same inputs) and
    the code is the nearest FP8 value of f32(v), saturating; the plain route
    is the fused route with no residual."""
    T, H = 5, 96
    x, u = synth.random_rows(20, T, H, n=2)
    w = synth.random_weight(20, H)
    for kind in (0, 1):
        for scale in (0.04, 1.0, 0.001):
            q = o.rmsnorm_quant(x, w, scale, 1e-6, residual=u, fp8_kind=kind)
            f = o.rmsnorm_fwd(x, w, 1e-6, residual=u)
            assert np.array_equal(q["h_new"], f["h_new"])
            assert np.array_equal(q["rstd"], f["rstd"])
            _close(q["v_exact"], f["y_exact"] / float(np.float32(scale)), 2e-16, "v = y / scale")
            ref = numfmt.nearest_fp8(q["v_exact"].astype(np.float32).astype(np.float64), kind)
            assert np.array_equal(q["q"], ref), (kind, scale)
        p = o.rmsnorm_quant(x, w, 0.5, 1e-6, fp8_kind=kind)
        fp = o.rmsnorm_fwd(x, w, 1e-6)
        _close(p["v_exact"], fp["y_exact"] / 0.5, 2e-16, "plain quant")


def pin_block_quant(o):
    """1x128 block quantisation: normed is the BF16 rounding of the forward's
    y; per row and block the scale is f32(amax/448) stored at [b, t]; the
    block's largest value takes code 448; every code is the nearest E4M3 of
    f32(normed / s); an all-zero row has scale 0 and zero codes; padding
    columns of block_scale are left alone."""
    T, H = 6, 384
    x, u = synth.random_rows(21, T, H, n=2)
    x[5] = u[5] ^ 0x8000                      # x = -u: the row sums to zero
    w = synth.random_weight(21, H)
    r = o.fused_add_rmsnorm_fp8_block_quant(x, u, w, 1e-6, ldT=8)
    f = o.rmsnorm_fwd(x, w, 1e-6, residual=u)
    assert np.array_equal(r["h_new"], f["h_new"])
    assert np.array_equal(r["normed_exact"], f["y_exact"])
    assert np.array_equal(r["normed"], numfmt.nearest_bf16(f["y_exact"]))
    n = numfmt.decode_bf16(r["normed"])
    for t in range(T):
        for b in range(H // 128):
            blk = n[t, b * 128:(b + 1) * 128]
            amax = float(np.max(np.abs(blk)))
            s = np.float32(amax / 448.0)
            assert r["block_scale"][b, t] == s, (t, b)
            codes = r["q"][t, b * 128:(b + 1) * 128]
            if amax == 0:
                assert s == 0 and not codes.any()
                continue
            assert np.any((codes & 0x7F) == 0x7E), (t, b)
            v32 = (blk / np.float64(s)).astype(np.float32).astype(np.float64)
            assert np.array_equal(codes, numfmt.nearest_fp8(v32, 0)), (t, b)
    assert np.isnan(r["block_scale"][:, T:]).all()


def pin_golden_block_quant(o):
    """Hand-derived block: a constant row normalises to 1, the block scale is
    f32(1/448) and every code is 448 (0x7E)."""
    g = json.load(open(GOLDEN))["block_quant"][0]
    Hc = g["H"]
    one = o.fused_add_rmsnorm_fp8_block_quant(
        _bits(np.full((2, Hc), g["x"])), _bits(np.full((2, Hc), g["residual"])),
        _bits(np.full(Hc, g["w"])), g["eps"])
    assert np.all(numfmt.decode_bf16(one["normed"]) == _eval(g["normed"]))
    assert np.all(one["block_scale"][:, :2] == np.float32(_eval(g["scale"])))
    assert np.all(one["q"] == int(g["code"], 16))


def _codes(hexes):
    return [None if h is None else int(h, 16) for h in hexes]


def pin_golden_static_fp8(o):
    """Hand-derived static-scale FP8 cases: v = y / scale and the codes placed
    on the E4M3 / E5M2 grids by hand (divide, not multiply; saturation;
    the residual route)."""
    g = json.load(open(GOLDEN))
    for c in g["static_fp8"]:
        x, w = _bits([c["x"]]), _bits(c["w"])
        res = _bits([c["residual"]]) if "residual" in c else None
        for kind, key in ((0, "e4m3"), (1, "e5m2")):
            if key not in c:
                continue
            r = o.rmsnorm_quant(x, w, c["scale"], c["eps"], residual=res, weight_bias=c["bias"],
                                fp8_kind=kind)
            _close(r["v_exact"][0], [_eval(e) for e in c["v"]], 4e-16, c["name"] + " v")
            assert list(r["q"][0]) == _codes(c[key]), (c["name"], key, list(r["q"][0]))
            if res is not None:
                _close(numfmt.decode_bf16(r["h_new"][0]), [_eval(e) for e in c["h_new"]], 0,
                       c["name"] + " h_new")


def pin_golden_ada(o):
    """Hand-derived AdaRMSNorm row: out = norm * (1 + scale) + shift exactly,
    gate_out the style's last third."""
    g = json.load(open(GOLDEN))
    for c in g["ada"]:
        style = _bits([c["sc"] + c["sh"] + c["gate"]])
        r = o.ada_rms_norm_style(_bits([c["x"]]), _bits(c["w"]), style, c["eps"])
        want = [_eval(e) for e in c["out"]]
        _close(r["out_exact"][0], want, 0, c["name"] + " out")
        _close(numfmt.decode_bf16(r["out"][0]), want, 0, c["name"] + " out (BF16)")
        assert np.array_equal(r["gate_out"][0], _bits(c["gate"])), c["name"]


def pin_golden_gated_ada(o):
    """Hand-derived gated residual + Ada + E4M3 row: the residual update,
    v = Ada output / scale, and the codes placed by hand."""
    g = json.load(open(GOLDEN))
    for c in g["gated_ada"]:
        style = _bits([c["sc"] + c["sh"] + c["gate_chunk"]])
        r = o.gate_residual_ada_norm_fp8(_bits([c["residual"]]), _bits([c["x"]]), _bits([c["gate"]]),
                                         _bits(c["w"]), style, c["scale"], c["eps"])
        _close(numfmt.decode_bf16(r["residual_out"][0]), [_eval(e) for e in c["residual_out"]], 0,
               c["name"] + " residual")
        _close(r["v_exact"][0], [_eval(e) for e in c["v"]], 4e-16, c["name"] + " v")
        assert list(r["q"][0]) == _codes(c["e4m3"]), (c["name"], list(r["q"][0]))
        assert np.array_equal(r["gate_out"][0], _bits(c["gate_chunk"])), c["name"]


def pin_golden_silu(o):
    """Hand-derived SiLU values: SiLU(0) = 0, SiLU(+-ln 3) = (3/4) ln 3 and
    -(1/4) ln 3, SiLU(1) = e/(1+e), and E4M3 codes at scale 1/2."""
    g = json.load(open(GOLDEN))
    for c in g["silu"]:
        w32 = np.array([_eval(e) for e in c["w32"]], np.float32)
        x = _bits([c["x"]])
        r = o.fused_rmsnorm_silu(x, w32, c["eps"])
        _close(r["v_exact"][0], [_eval(e) for e in c["v"]], c["rel"], c["name"] + " v")
        q = o.fused_rmsnorm_silu(x, w32, c["eps"], fp8=True, scale=c["scale"])
        for got, want in zip(q["q"][0], _codes(c["e4m3"])):
            assert want is None or got == want, (c["name"], list(q["q"][0]))


def pin_golden_layernorm(o):
    """Hand-derived two-element LayerNorm row: mean, rstd (population
    variance, eps inside the root), the output with gamma and beta, and its
    FP8 codes (an E5M2 tie rounded to even)."""
    g = json.load(open(GOLDEN))
    for c in g["layernorm"]:
        x = _bits([c["x"]])
        gamma, beta = np.array(c["gamma"], np.float32), np.array(c["beta"], np.float32)
        r = o.layernorm(x, gamma, beta, c["eps"])
        _close(r["mean"][0], _eval(c["mean"]), 0, c["name"] + " mean")
        _close(r["rstd"][0], _eval(c["rstd"]), 1e-15, c["name"] + " rstd")
        want = [_eval(e) for e in c["y"]]
        _close(r["v_exact"][0], want, 1e-15, c["name"] + " y")
        _close(numfmt.decode_bf16(r["y"][0]), want, 0, c["name"] + " y (BF16)")
        for kind, key in ((0, "e4m3"), (1, "e5m2")):
            q = o.layernorm(x, gamma, beta, c["eps"], fp8_kind=kind, scale=c["scale"])
            assert list(q["q"][0]) == _codes(c[key]), (c["name"], key, list(q["q"][0]))


# ------------------------------------------------------------------- Ada --

def pin_ada(o):
    """AdaRMSNorm: zero style scale/shift give the plain RMSNorm output; scale
    1 doubles it; a shift adds to it; gate_out is the style's last third; a
    broadcast style row equals that row repeated; each row uses its own
    style row."""
    T, D = 5, 64
    x = synth.random_rows(22, T, D)[0]
    w = synth.random_weight(22, D)
    st = synth.random_rows(23, T, 3 * D)[0]
    plain = o.rmsnorm_fwd(x, w, 1e-6)
    z = st.copy()
    z[:, :2 * D] = 0
    r = o.ada_rms_norm_style(x, w, z, 1e-6)
    assert np.array_equal(r["out"], plain["y"]) and np.array_equal(r["out_exact"], plain["y_exact"])
    assert np.array_equal(r["gate_out"], st[:, 2 * D:])
    one = z.copy()
    one[:, :D] = 0x3F80                        # style scale = 1.0
    assert np.array_equal(o.ada_rms_norm_style(x, w, one, 1e-6)["out_exact"], 2 * plain["y_exact"])
    sh = z.copy()
    sh[:, D:2 * D] = st[:, D:2 * D]
    _close(o.ada_rms_norm_style(x, w, sh, 1e-6)["out_exact"],
           plain["y_exact"] + numfmt.decode_bf16(st[:, D:2 * D]), 1e-15, "shift")
    b = o.ada_rms_norm_style(x, w, st[:1], 1e-6)
    rep = o.ada_rms_norm_style(x, w, np.repeat(st[:1], T, axis=0), 1e-6)
    for k in b:
        assert np.array_equal(b[k], rep[k]), k
    full = o.ada_rms_norm_style(x, w, st, 1e-6)
    for t in range(T):
        row = o.ada_rms_norm_style(x[t:t + 1], w, st[t:t + 1], 1e-6)
        for k in full:
            assert np.array_equal(full[k][t:t + 1], row[k]), (k, t)


def pin_gated_ada(o):
    """Gated residual + Ada + FP8: the residual update is the BF16 rounding of
    residual + BF16(x * gate) (brute force); a zero gate leaves the residual
    unchanged; v * scale is the Ada output of the updated residual; codes are
    the nearest E4M3 of f32(v), saturating."""
    T, D = 4, 64
    u, x, gt = synth.random_rows(24, T, D, n=3)
    w = synth.random_weight(24, D)
    st = synth.random_rows(25, T, 3 * D)[0]
    for style in (st, st[:1]):
        r = o.gate_residual_ada_norm_fp8(u, x, gt, w, style, 0.04, 1e-6)
        prod = numfmt.nearest_bf16(numfmt.decode_bf16(x) * numfmt.decode_bf16(gt))
        ref = numfmt.nearest_bf16(numfmt.decode_bf16(u) + numfmt.decode_bf16(prod))
        assert np.array_equal(r["residual_out"], ref)
        a = o.ada_rms_norm_style(ref, w, style, 1e-6)
        _close(r["v_exact"] * float(np.float32(0.04)), a["out_exact"], 4e-16, "v * scale")
        assert np.array_equal(r["gate_out"], a["gate_out"])
        want = numfmt.nearest_fp8(r["v_exact"].astype(np.float32).astype(np.float64), 0)
        assert np.array_equal(r["q"], want)
    zero = o.gate_residual_ada_norm_fp8(u, x, np.zeros_like(gt), w, st, 0.04, 1e-6)
    assert np.array_equal(zero["residual_out"], u)


# ------------------------------------------------------------ SiLU, LayerNorm --

def pin_silu(o):
    """RMSNorm + SiLU: v is PyTorch's float64 SiLU of the forward's exact
    value (plain, Gemma and FP32-weight routes); SiLU(v) - SiLU(-v) = v on
    negated rows; a row [a, -a] gives SiLU(+-a*rstd) in closed form; BF16
    outputs are the nearest BF16 and FP8 codes the nearest E4M3 of
    f32(v / scale), saturating."""
    T, H = 6, 160
    x = synth.random_rows(40, T, H)[0]
    for w, bias in ((synth.random_weight(40, H), 0.0), (synth.random_weight(41, H), 1.0),
                    (synth.random_weight(42, H, f32=True), 1.0)):
        r = o.fused_rmsnorm_silu(x, w, 1e-6, weight_bias=bias)
        f = o.rmsnorm_fwd(x, w, 1e-6, weight_bias=bias)
        ref = torch.nn.functional.silu(torch.from_numpy(f["y_exact"])).numpy()
        _close(r["v_exact"], ref, 1e-14, "silu vs torch")
        assert np.array_equal(r["y"], numfmt.nearest_bf16(r["v_exact"]))
        assert np.array_equal(r["rstd"], f["rstd"])
        neg = o.fused_rmsnorm_silu(x ^ np.uint16(0x8000), w, 1e-6, weight_bias=bias)
        _close(r["v_exact"] - neg["v_exact"], f["y_exact"], 1e-12, "silu(v) - silu(-v) = v")
        for scale in (1.0, 0.04):
            qr = o.fused_rmsnorm_silu(x, w, 1e-6, weight_bias=bias, fp8=True, scale=scale)
            _close(qr["v_exact"] * float(np.float32(scale)), r["v_exact"], 4e-16, "v * scale")
            want = numfmt.nearest_fp8(qr["v_exact"].astype(np.float32).astype(np.float64), 0)
            assert np.array_equal(qr["q"], want), scale
    a = 3.0
    row = _bits([[a, -a]])
    r = o.fused_rmsnorm_silu(row, _bits([1.0, 1.0]), 1e-6)
    rs = 1.0 / math.sqrt(a * a + float(np.float32(1e-6)))
    want = [a * rs / (1.0 + math.exp(-a * rs)), -a * rs / (1.0 + math.exp(a * rs))]
    _close(r["v_exact"][0], want, 1e-15, "silu closed form")


def pin_layernorm(o):
    """LayerNorm: v is PyTorch's float64 layer_norm (population variance, eps
    inside the root) with gamma and beta; the mean and rstd are numpy's
    mean and 1/sqrt(var + eps); shifting a row by a constant changes
    nothing; with gamma = 1, beta = 0 a row sums to 0 and its mean square is
    var / (var + eps); a two-element row is +-|a-b|/2 / sqrt(((a-b)/2)^2 +
    eps) in closed form; BF16 outputs are the nearest BF16 and FP8 codes the
    nearest E4M3 / E5M2 of f32(v / scale)."""
    T, H = 5, 192
    x = synth.random_rows(50, T, H)[0]
    gen = torch.Generator().manual_seed(51)
    gamma = (1 + 0.1 * torch.randn(H, generator=gen)).numpy().astype(np.float32)
    beta = (0.1 * torch.randn(H, generator=gen)).numpy().astype(np.float32)
    eps = 1e-5
    e32 = float(np.float32(eps))
    r = o.layernorm(x, gamma, beta, eps)
    xd = numfmt.decode_bf16(x)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(xd), (H,),
                                         torch.from_numpy(gamma.astype(np.float64)),
                                         torch.from_numpy(beta.astype(np.float64)), e32).numpy()
    _close(r["v_exact"], ref, 1e-12, "layernorm vs torch")
    _close(r["mean"], xd.mean(axis=1), 1e-14, "mean")
    _close(r["rstd"], 1.0 / np.sqrt(xd.var(axis=1) + e32), 1e-14, "rstd")
    assert np.array_equal(r["y"], numfmt.nearest_bf16(r["v_exact"]))
    one, zero = np.ones(H, np.float32), np.zeros(H, np.float32)
    p = o.layernorm(x, one, zero, eps)
    var = xd.var(axis=1)
    assert np.all(np.abs(p["v_exact"].sum(axis=1)) <= 1e-12 * H)
    _close((p["v_exact"] ** 2).mean(axis=1), var / (var + e32), 1e-13, "mean square")
    ints = np.arange(-40, 40, dtype=np.float64).reshape(1, 80)
    xi = numfmt.nearest_bf16(ints)
    xs = numfmt.nearest_bf16(ints + 64.0)           # exact: integers below 256
    a1 = o.layernorm(xi, np.ones(80, np.float32), np.zeros(80, np.float32), eps)
    a2 = o.layernorm(xs, np.ones(80, np.float32), np.zeros(80, np.float32), eps)
    _close(a2["v_exact"], a1["v_exact"], 1e-13, "shift invariance")
    a, b = 5.0, 2.0
    two = o.layernorm(_bits([[a, b]]), np.array([2.0, 3.0], np.float32),
                      np.array([0.5, -1.0], np.float32), eps)
    d = abs(a - b) / 2 / math.sqrt(((a - b) / 2) ** 2 + e32)
    _close(two["v_exact"][0], [d * 2.0 + 0.5, -d * 3.0 - 1.0], 1e-15, "two-element row")
    for kind in (0, 1):
        for scale in (0.04, 1.0):
            qr = o.layernorm(x, gamma, beta, eps, fp8_kind=kind, scale=scale)
            _close(qr["v_exact"] * float(np.float32(scale)), r["v_exact"], 4e-16, "v * scale")
            want = numfmt.nearest_fp8(qr["v_exact"].astype(np.float32).astype(np.float64), kind)
            assert np.array_equal(qr["q"], want), (kind, scale)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
