"""Subnormal and near-minimum values through the GPU path.

BF16 has the exponent range of FP32, so its subnormals (magnitudes below
2^-126, multiples of 2^-133) are FP32 subnormals.  These tests feed them to
every operation and compare with the oracle at the usual tolerances:

* residual pairs whose exact sum lies below 2^-126, exact cancellations to
  +-0, sums of two subnormals, and tiny normals plus subnormals (rounding at
  the boundary): h_new / the updated residual must be bit-exact;
* gated products x*gate below 2^-126: the gated residual bit-exact;
* rows of subnormals only (the statistic is eps-dominated, so y is a normal
  number), and rows mixing N(0,1) values with subnormal entries (y, dx, SiLU,
  LayerNorm outputs are themselves subnormal there);
* static FP8 with a scale of 2^-126, so that subnormal normalised values map
  to codes well above zero;
* dw columns whose every term is subnormal (absolute tolerance of one FP32
  subnormal quantum per row).
"""
import numpy as np
import pytest
import torch

import gpu_util as gu
import numfmt
import oracle
import normalization_rmsnorm_fwd_gb300 as crm
from normalization_rmsnorm_fwd_gb300 import synth

pytestmark = pytest.mark.gpu

SUB = (0x0001, 0x0080)        # subnormal magnitude codes
MIN_BINADE = (0x0080, 0x0100)  # [2^-126, 2^-125)
TINY_NORMAL = (0x0080, 0x0800)  # [2^-126, 2^-111): squares underflow FP32


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


def below_min_pairs(seed, shape):
    """x = s*a, u = -s*b with a, b in [2^-126, 2^-125): x + u is a subnormal
    or zero (a multiple of 2^-133, exact in BF16)."""
    a = synth.bf16_codes(seed, shape, *MIN_BINADE)
    b = synth.bf16_codes(seed + 1, shape, *MIN_BINADE, signed=False)
    return a, (b | ((a & 0x8000) ^ 0x8000)).astype(np.uint16)


def mixed_rows(seed, T, H, every=4):
    """N(0,1) rows with every `every`-th column a subnormal."""
    x = synth.random_rows(seed, T, H)[0]
    x[:, ::every] = synth.bf16_codes(seed + 7, (T, (H + every - 1) // every), *SUB)
    return x


def residual_inputs(H=1024):
    parts_x, parts_u = [], []
    a, b = below_min_pairs(1, (16, H))                      # sums below 2^-126
    parts_x.append(a); parts_u.append(b)
    x = synth.random_rows(2, 4, H)[0]                       # exact cancellation to +0
    u = x ^ np.uint16(0x8000)
    x[3], u[3] = 0x8000, 0x8000                             # -0 + -0 = -0
    parts_x.append(x); parts_u.append(u)
    parts_x.append(synth.bf16_codes(3, (8, H), *SUB))       # subnormal + subnormal
    parts_u.append(synth.bf16_codes(4, (8, H), *SUB))
    x, u = synth.random_rows(5, 16, H, n=2)                 # N(0,1) rows with some
    a, b = below_min_pairs(6, (16, H // 4))                 # columns cancelling
    x[:, ::4], u[:, ::4] = a, b
    parts_x.append(x); parts_u.append(u)
    parts_x.append(synth.bf16_codes(7, (20, H), 0x0080, 0x0400))   # tiny normal + subnormal:
    parts_u.append(synth.bf16_codes(8, (20, H), *SUB))             # rounding at the boundary
    return np.concatenate(parts_x), np.concatenate(parts_u)


def plain_inputs(H=1024):
    return np.concatenate([synth.bf16_codes(11, (8, H), *SUB),
                           synth.bf16_codes(12, (8, H), *TINY_NORMAL),
                           mixed_rows(13, 16, H)])


def check_fwd(orc, x, w, y, rstd, eps, residual=None, h_new=None, bias=0.0):
    ref = orc.rmsnorm_fwd(x, w, eps, residual=residual, weight_bias=bias)
    if residual is not None:
        gu.check_exact(h_new, ref["h_new"], "h_new")
    gu.check_rstd(rstd, ref["rstd_exact"])
    gu.check_bf16(y, ref["y_exact"], what="y")


@pytest.mark.parametrize("f32", [False, True])
def test_residual_sums_below_min_normal(orc, f32):
    x, u = residual_inputs()
    H = x.shape[1]
    w = synth.random_weight(20, H, f32=f32)
    bias = 1.0 if f32 else 0.0
    wd = gu.dev_f32(w) if f32 else gu.dev_bf16(w)
    y, rstd, hn = crm.rmsnorm_fwd(gu.dev_bf16(x), wd, 1e-6, residual=gu.dev_bf16(u),
                                  weight_bias=bias)
    torch.cuda.synchronize()
    hb = gu.host_bits(hn)
    exact = numfmt.decode_bf16(x) + numfmt.decode_bf16(u)
    gu.check_exact(hb, numfmt.nearest_bf16(exact), "h_new (brute-force table)")
    assert (hb[16:19] == 0).all() and (hb[19] == 0x8000).all(), "signed zeros of exact cancellation"
    assert ((hb[:16] & 0x7F80) == 0).all() and (hb[:16] & 0x7F).any(), "subnormal sums kept"
    check_fwd(orc, x, w, gu.host_bits(y), rstd.cpu().numpy(), 1e-6, u, hb, bias)


@pytest.mark.parametrize("f32", [False, True])
def test_subnormal_rows_forward(orc, f32):
    x = plain_inputs()
    H = x.shape[1]
    w = synth.random_weight(21, H, f32=f32)
    bias = 1.0 if f32 else 0.0
    wd = gu.dev_f32(w) if f32 else gu.dev_bf16(w)
    y, rstd, _ = crm.rmsnorm_fwd(gu.dev_bf16(x), wd, 1e-6, weight_bias=bias)
    torch.cuda.synchronize()
    yb = gu.host_bits(y)
    check_fwd(orc, x, w, yb, rstd.cpu().numpy(), 1e-6, bias=bias)
    # The mixed rows' subnormal entries give subnormal outputs.
    sub_out = (yb[16:, ::4] & 0x7F80) == 0
    assert sub_out.mean() > 0.75 and (yb[16:, ::4] & 0x7F).any()


def test_static_fp8_of_subnormal_values(orc):
    """Scale 2^-126 (the IEEE-division path): subnormal normalised values
    become codes of order one, normal ones saturate."""
    scale = 2.0 ** -126
    x = plain_inputs()
    T, H = x.shape
    w = synth.random_weight(22, H)
    xd, wd = gu.dev_bf16(x), gu.dev_bf16(w)
    q = torch.empty((T, H), dtype=torch.float8_e4m3fn, device=gu.DEV)
    crm.rmsnorm_quant(q, xd, wd, scale, 1e-6)
    torch.cuda.synchronize()
    ref = orc.rmsnorm_quant(x, w, scale, 1e-6)
    qb = gu.host_u8(q)
    gu.check_fp8(qb, ref["q"], ref["v_exact"], 0, "e4m3 of subnormals")
    assert ((qb[16:, ::4] & 0x7F) > 0x08).mean() > 0.5
    # With the residual route: the sums below 2^-126 quantised at the same scale.
    xr, ur = residual_inputs()
    q = torch.empty(xr.shape, dtype=torch.float8_e4m3fn, device=gu.DEV)
    ud = gu.dev_bf16(ur)
    crm.fused_add_rmsnorm_quant(q, gu.dev_bf16(xr), ud, wd, scale, 1e-6)
    torch.cuda.synchronize()
    ref = orc.rmsnorm_quant(xr, w, scale, 1e-6, residual=ur)
    gu.check_exact(gu.host_bits(ud), ref["h_new"], "residual in place")
    gu.check_fp8(gu.host_u8(q), ref["q"], ref["v_exact"], 0, "e4m3 of residual sums")


def bwd_case(orc, g, x, w, T, H):
    rstd = orc.rmsnorm_fwd(x, w, 1e-6, want_y=False)["rstd"]
    dx, dw = crm.rmsnorm_bwd(gu.dev_bf16(g), gu.dev_bf16(x), gu.dev_bf16(w), gu.dev_f32(rstd))
    torch.cuda.synchronize()
    ref = orc.rmsnorm_bwd(g, x, w, rstd)
    allow = gu.dx_allowance(g, x, orc.weight_eff(w), rstd, ref["m"])
    gu.check_bf16(gu.host_bits(dx), ref["dx_exact"], allowance=allow, what="dx")
    got = dw.cpu().numpy().astype(np.float64)
    # Every term g*x*rstd may be rounded once at the FP32 subnormal quantum.
    bad = ~(np.abs(got - ref["dw"]) <= 1e-5 * ref["dw_abs"] + T * 2.0 ** -149)
    assert not bad.any(), f"dw: {bad.sum()} columns; e.g. got {got[bad][:3]} want {ref['dw'][bad][:3]}"
    return gu.host_bits(dx), got, ref


def test_backward_subnormal_gradient(orc):
    """g subnormal, x ~ N(0,1): dx and every dw term are subnormal."""
    T, H = 64, 2048
    g = synth.bf16_codes(30, (T, H), *SUB)
    x = synth.random_rows(31, T, H)[0]
    w = synth.random_weight(32, H)
    dxb, dw, ref = bwd_case(orc, g, x, w, T, H)
    assert ((dxb & 0x7F80) == 0).mean() > 0.9 and (dxb & 0x7F).any()
    assert np.abs(ref["dw"]).max() < 2.0 ** -120 and (dw != 0).mean() > 0.9


def test_backward_subnormal_input(orc):
    """x subnormal (rstd = 1/sqrt(eps)), g ~ N(0,1); and rows mixing both."""
    T, H = 64, 2048
    w = synth.random_weight(35, H)
    bwd_case(orc, synth.random_rows(33, T, H)[0], synth.bf16_codes(34, (T, H), *SUB), w, T, H)
    bwd_case(orc, mixed_rows(36, T, H, every=3), mixed_rows(37, T, H, every=5), w, T, H)


def test_gated_products_below_min_normal(orc):
    """x ~ 2^-70, gate ~ 2^-60: x*gate lies in [2^-130, 2^-128); the residual
    is subnormal or a tiny normal; one row has gate = 0."""
    T, D = 32, 1024
    x = synth.bf16_codes(40, (T, D), 0x1C80, 0x1D00)       # [2^-70, 2^-69)
    gate = synth.bf16_codes(41, (T, D), 0x2180, 0x2200)    # [2^-60, 2^-59)
    gate[5] = 0
    u = synth.bf16_codes(42, (T, D), 0x0001, 0x0100)
    u[20:] = synth.random_rows(43, T - 20, D)[0]            # normal residual rows
    style = synth.random_rows(44, T, 3 * D)[0]
    w = synth.random_weight(45, D)
    ud = gu.dev_bf16(u)
    res, out, gate_out = crm.gate_residual_ada_norm_fp8(ud, gu.dev_bf16(x), gu.dev_bf16(gate),
                                                        gu.dev_bf16(w), gu.dev_bf16(style),
                                                        0.04, 1e-6)
    torch.cuda.synchronize()
    ref = orc.gate_residual_ada_norm_fp8(u, x, gate, w, style, 0.04, 1e-6)
    rb = gu.host_bits(res)
    gu.check_exact(rb, ref["residual_out"], "gated residual")
    gu.check_exact(rb[5], u[5], "gate = 0 leaves the residual unchanged")
    gu.check_exact(gu.host_bits(gate_out), ref["gate_out"], "gate_out")
    f = orc.rmsnorm_fwd(ref["residual_out"], w, 1e-6)
    sc = numfmt.decode_bf16(style[:, :D])
    sh = numfmt.decode_bf16(style[:, D:2 * D])
    allow = 2.0 ** -20 * (np.abs(f["y_exact"] * (1 + sc)) + np.abs(sh)) / np.float32(0.04)
    gu.check_fp8(gu.host_u8(out), ref["q"], ref["v_exact"], 0, "gated e4m3", allowance=allow)


def test_ada_subnormal_outputs(orc):
    """Mixed rows with zero shift: the style product of subnormal normalised
    values is itself subnormal."""
    T, D = 32, 1024
    x = mixed_rows(50, T, D)
    style = synth.random_rows(51, T, 3 * D)[0]
    style[:, D:2 * D] = 0
    w = synth.random_weight(52, D)
    out, gate_out = crm.ada_rms_norm_style(gu.dev_bf16(x), gu.dev_bf16(w), gu.dev_bf16(style))
    torch.cuda.synchronize()
    ref = orc.ada_rms_norm_style(x, w, style, 1e-6)
    f = orc.rmsnorm_fwd(x, w, 1e-6)
    sc = numfmt.decode_bf16(style[:, :D])
    gu.check_bf16(gu.host_bits(out), ref["out_exact"],
                  allowance=2.0 ** -20 * np.abs(f["y_exact"] * (1 + sc)), what="ada out")
    gu.check_exact(gu.host_bits(gate_out), ref["gate_out"], "gate_out")


def test_silu_and_layernorm_of_subnormals(orc):
    x = plain_inputs(512)
    T, H = x.shape
    w = synth.random_weight(60, H)
    xd = gu.dev_bf16(x)
    y = crm.fused_rmsnorm_silu(xd, gu.dev_bf16(w), 1e-6)
    torch.cuda.synchronize()
    ref = orc.fused_rmsnorm_silu(x, w, 1e-6)
    gu.check_bf16(gu.host_bits(y), ref["v_exact"], what="silu of subnormals")
    gen = torch.Generator().manual_seed(61)
    gamma = (1 + 0.1 * torch.randn(H, generator=gen)).numpy().astype(np.float32)
    beta = np.zeros(H, np.float32)
    yl = crm.layernorm(xd, gu.dev_f32(gamma), gu.dev_f32(beta), 1e-5)
    torch.cuda.synchronize()
    rl = orc.layernorm(x, gamma, beta, 1e-5)
    h = numfmt.decode_bf16(x)
    d = np.abs(h - rl["mean"][:, None]) + np.abs(rl["mean"][:, None])
    allow = 2.0 ** -20 * d * rl["rstd"][:, None] * np.abs(gamma)
    gu.check_bf16(gu.host_bits(yl), rl["v_exact"], allowance=allow, what="layernorm of subnormals")
