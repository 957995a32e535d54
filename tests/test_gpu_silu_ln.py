"""RMSNorm + SiLU and LayerNorm on the GPU against the oracle, element by
element: BF16 outputs within one BF16 ulp of the exact value (plus a
cancellation allowance for LayerNorm's + beta), FP8 codes equal except one
code next to a rounding midpoint, FP32 statistics within a few FP32 ulps."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
from normalization_rmsnorm_fwd_gb300 import synth
import normalization_rmsnorm_fwd_gb300 as crm

pytestmark = pytest.mark.gpu

SILU_H = [2, 64, 128, 160, 256, 320, 512, 640, 1024, 2048, 4096, 8192, 16384]


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


def _silu_gpu(x, w, bias=0.0, fp8=False, scale=None, out=None):
    xd = gu.dev_bf16(x)
    wd = gu.dev_f32(w) if w.dtype == np.float32 else gu.dev_bf16(w)
    if out is None and fp8:
        out = torch.empty(xd.shape, dtype=torch.float8_e4m3fn, device="cuda")
    rstd = torch.empty(x.shape[0], dtype=torch.float32, device="cuda")
    y = crm.fused_rmsnorm_silu(xd, wd, 1e-6, weight_bias=bias, out=out, scale=scale, rstd=rstd)
    torch.cuda.synchronize()
    return y, rstd


def _check_silu(orc, x, w, bias=0.0):
    """Every row: BF16 output, rstd, and E4M3 codes with and without a
    scale."""
    T, H = x.shape
    y, rstd = _silu_gpu(x, w, bias)
    got, r = gu.host_bits(y), rstd.cpu().numpy()
    qs = {}
    for scale in (None, 0.04):
        q, _ = _silu_gpu(x, w, bias, fp8=True, scale=scale)
        qs[scale] = gu.host_u8(q)
        del q

    def check(lo, hi):
        ref = orc.fused_rmsnorm_silu(x[lo:hi], w, 1e-6, weight_bias=bias)
        gu.check_bf16(got[lo:hi], ref["v_exact"], what=f"silu bf16 rows {lo}:{hi}")
        gu.check_rstd(r[lo:hi], ref["rstd"].astype(np.float64), what=f"rstd rows {lo}:{hi}")
        for scale, gq in qs.items():
            refq = orc.fused_rmsnorm_silu(x[lo:hi], w, 1e-6, weight_bias=bias, fp8=True,
                                          scale=1.0 if scale is None else scale)
            gu.check_fp8(gq[lo:hi], refq["q"], refq["v_exact"], 0,
                         what=f"silu e4m3 scale={scale} rows {lo}:{hi}")
    gu.each_block(T, H, check)


@pytest.mark.parametrize("H", SILU_H)
def test_silu_widths(orc, H):
    x = synth.random_rows(H + 1, 67, H)[0]
    _check_silu(orc, x, synth.random_weight(H + 1, H))


@pytest.mark.parametrize("route", ["gemma", "f32"])
def test_silu_weight_routes(orc, route):
    H = 640
    x = synth.random_rows(7, 300, H)[0]
    w = synth.random_weight(7, H, f32=route == "f32")
    _check_silu(orc, x, w, bias=1.0)


@pytest.mark.parametrize("T", [1, 2, 7, 63, 257, 1560])
def test_silu_row_counts(orc, T):
    x = synth.random_rows(T, T, 160)[0]
    _check_silu(orc, x, synth.random_weight(T, 160))


def test_silu_large(orc):
    # The largest point of the B200 sweep grid, T = 399360, H = 1024, every
    # row.
    T, H = 399360, 1024
    gen = torch.Generator().manual_seed(3)
    x = synth.bf16_bits(torch.randn(T, H, generator=gen))
    _check_silu(orc, x, synth.random_weight(3, H))


def test_silu_in_place_and_strided(orc):
    H = 256
    buf = synth.random_rows(9, 40, 2 * H)[0]
    x = buf[:, :H]                        # row stride 2H
    w = synth.random_weight(9, H)
    xd = gu.dev_bf16(buf)[:, :H]
    crm.fused_rmsnorm_silu(xd, gu.dev_bf16(w), 1e-6, out=xd)
    torch.cuda.synchronize()
    ref = orc.fused_rmsnorm_silu(np.ascontiguousarray(x), w, 1e-6)
    gu.check_bf16(gu.host_bits(xd), ref["v_exact"], what="silu in place, strided")


def test_silu_extreme_values(orc):
    # Rows whose normalised values reach +-60 (a few large entries): SiLU of
    # large negative values underflows towards -0, of large positive ones is v.
    H = 128
    gen = torch.Generator().manual_seed(11)
    v = torch.randn(16, H, generator=gen) * 0.01
    v[:, 0] = 60.0
    v[:, 1] = -60.0
    v[:8, 2] = -3.0
    x = synth.bf16_bits(v)
    w = synth.bf16_bits(torch.full((H,), 8.0))
    _check_silu(orc, x, w)


# ---------------------------------------------------------------- LayerNorm --

def _gamma_beta(seed, H):
    gen = torch.Generator().manual_seed(seed)
    gamma = (1 + 0.1 * torch.randn(H, generator=gen)).numpy().astype(np.float32)
    beta = (0.1 * torch.randn(H, generator=gen)).numpy().astype(np.float32)
    return gamma, beta


def _ln_allowance(x, ref, gamma, beta):
    h = x.astype(np.float64)
    d = np.abs(h - ref["mean"][:, None]) + np.abs(ref["mean"][:, None])
    return 2.0 ** -20 * (d * ref["rstd"][:, None] * np.abs(gamma) + np.abs(beta))


def _check_ln(orc, x, gamma, beta, eps=1e-5, kinds=(0, 1)):
    """Every row: BF16 output, mean, rstd, and the FP8 codes of each kind."""
    xd = gu.dev_bf16(x)
    gd, bd = gu.dev_f32(gamma), gu.dev_f32(beta)
    T, H = x.shape
    mean = torch.empty(T, dtype=torch.float32, device="cuda")
    rstd = torch.empty(T, dtype=torch.float32, device="cuda")
    y = crm.layernorm(xd, gd, bd, eps, mean=mean, rstd=rstd)
    torch.cuda.synchronize()
    yb, mb, rb = gu.host_bits(y), mean.cpu().numpy().astype(np.float64), rstd.cpu().numpy()
    del y
    qs = {}
    for kind in kinds:
        dt = torch.float8_e4m3fn if kind == 0 else torch.float8_e5m2
        q = torch.empty(xd.shape, dtype=dt, device="cuda")
        crm.layernorm_quant(q, xd, gd, bd, 0.04, eps)
        torch.cuda.synchronize()
        qs[kind] = gu.host_u8(q)
        del q

    def check(lo, hi):
        xs = x[lo:hi]
        ref = orc.layernorm(xs, gamma, beta, eps)
        xdec = orc.bf16_to_f64(xs)
        allow = _ln_allowance(xdec, ref, gamma, beta)
        gu.check_bf16(yb[lo:hi], ref["v_exact"], allowance=allow, what=f"layernorm rows {lo}:{hi}")
        gu.check_rstd(rb[lo:hi], ref["rstd"], what=f"rstd rows {lo}:{hi}")
        scale_m = np.abs(xdec).mean(axis=1)
        assert np.all(np.abs(mb[lo:hi] - ref["mean"]) <= 2.0 ** -22 * scale_m + 1e-30), "mean"
        for kind, gq in qs.items():
            rq = orc.layernorm(xs, gamma, beta, eps, fp8_kind=kind, scale=0.04)
            gu.check_fp8(gq[lo:hi], rq["q"], rq["v_exact"], kind,
                         what=f"layernorm_quant kind={kind} rows {lo}:{hi}",
                         allowance=allow / float(np.float32(0.04)))
    gu.each_block(T, H, check)


# 6144: the persistent form's gamma/beta table is exactly 48 KB, which with
# the kernel's static shared memory needs the opt-in above the default.
@pytest.mark.parametrize("H", [2, 64, 160, 256, 1000, 2048, 3072, 4096, 5120, 6144, 8192, 8200, 16384])
def test_layernorm_widths(orc, H):
    x = synth.random_rows(H + 2, 45, H)[0]
    g, b = _gamma_beta(H, H)
    _check_ln(orc, x, g, b)


@pytest.mark.parametrize("T", [1, 3, 64, 129, 4097])
def test_layernorm_row_counts(orc, T):
    x = synth.random_rows(T + 5, T, 768)[0]
    g, b = _gamma_beta(T, 768)
    _check_ln(orc, x, g, b)


def test_layernorm_large(orc):
    # The measured LayerNorm workload, T = 16384, H = 4096, every row; the
    # last 1024 rows carry a large common offset (300 + N(0,1)).
    T, H = 16384, 4096
    gen = torch.Generator().manual_seed(8)
    v = torch.randn(T, H, generator=gen)
    v[T - 1024:] += 300.0
    x = synth.bf16_bits(v)
    g, b = _gamma_beta(8, H)
    _check_ln(orc, x, g, b)


def test_layernorm_offset_rows(orc):
    # A large common offset: the mean dominates and the deviations are small
    # (the case a one-pass sum of squares gets wrong).
    H = 1024
    gen = torch.Generator().manual_seed(5)
    v = 300.0 + torch.randn(32, H, generator=gen)
    x = synth.bf16_bits(v)
    g, b = _gamma_beta(5, H)
    _check_ln(orc, x, g, b, eps=1e-6)


def test_layernorm_constant_row(orc):
    # A constant row has zero variance: the output is beta exactly.
    H = 512
    x = synth.bf16_bits(torch.full((4, H), 3.25))
    g, b = _gamma_beta(6, H)
    y = crm.layernorm(gu.dev_bf16(x), gu.dev_f32(g), gu.dev_f32(b), 1e-5)
    torch.cuda.synchronize()
    assert np.array_equal(gu.host_bits(y), orc.bf16_from_f64(b.astype(np.float64)[None, :].repeat(4, 0)))


def test_layernorm_strided_in_place(orc):
    H = 128
    buf = synth.random_rows(12, 64, 3 * H)[0]
    g, b = _gamma_beta(12, H)
    xd = gu.dev_bf16(buf)[:, H:2 * H]
    crm.layernorm(xd, gu.dev_f32(g), gu.dev_f32(b), 1e-5, out=xd)
    torch.cuda.synchronize()
    xs = np.ascontiguousarray(buf[:, H:2 * H])
    ref = orc.layernorm(xs, g, b, 1e-5)
    allow = _ln_allowance(orc.bf16_to_f64(xs), ref, g, b)
    gu.check_bf16(gu.host_bits(xd), ref["v_exact"], allowance=allow, what="layernorm in place")


@pytest.mark.parametrize("H", [4096, 8192])
def test_layernorm_bf16_64_elements_per_thread(orc, H):
    # BF16 LayerNorm at H = 4096 and 8192 runs 64 elements per thread (two or
    # four warps a row, several rows per group, the next row prefetched into
    # L2 only): every row against the oracle, with rows of a large common
    # offset and a constant row; then the same rows at a row stride of 2H with
    # the output in place, bit for bit equal to the contiguous call.
    T = 1500
    gen = torch.Generator().manual_seed(H)
    v = torch.randn(T, H, generator=gen)
    v[::3] += 300.0
    v[7] = 2.5
    x = synth.bf16_bits(v)
    g, b = _gamma_beta(H + 9, H)
    _check_ln(orc, x, g, b, kinds=())
    gd, bd = gu.dev_f32(g), gu.dev_f32(b)
    y = crm.layernorm(gu.dev_bf16(x), gd, bd, 1e-5)
    buf = np.zeros((T, 2 * H), np.uint16)
    buf[:, H:] = x
    xs = gu.dev_bf16(buf)[:, H:]
    crm.layernorm(xs, gd, bd, 1e-5, out=xs)
    torch.cuda.synchronize()
    assert np.array_equal(gu.host_bits(xs), gu.host_bits(y))
