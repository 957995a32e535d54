"""GPU forward (rmsnorm_fwd through the C ABI) against the CPU oracle."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import numfmt
import oracle
import normalization_rmsnorm_fwd_gb300 as crm
from normalization_rmsnorm_fwd_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


def run_fwd(x_bits, w, eps=1e-6, residual_bits=None, bias=0.0):
    x = gu.dev_bf16(x_bits)
    wd = gu.dev_f32(w) if w.dtype == np.float32 else gu.dev_bf16(w)
    r = gu.dev_bf16(residual_bits) if residual_bits is not None else None
    y, rstd, h_new = crm.rmsnorm_fwd(x, wd, eps, residual=r, weight_bias=bias)
    torch.cuda.synchronize()
    return (gu.host_bits(y), rstd.cpu().numpy(),
            gu.host_bits(h_new) if h_new is not None else None)


def compare(orc, x, w, eps=1e-6, residual=None, bias=0.0):
    """Every row of the GPU forward against the oracle (row blocks checked on
    the host's cores)."""
    y, rstd, h_new = run_fwd(x, w, eps, residual, bias)
    T, H = x.shape

    def check(lo, hi):
        r = None if residual is None else residual[lo:hi]
        ref = orc.rmsnorm_fwd(x[lo:hi], w, eps, residual=r, weight_bias=bias)
        gu.check_rstd(rstd[lo:hi], ref["rstd_exact"], what=f"rstd rows {lo}:{hi}")
        gu.check_bf16(y[lo:hi], ref["y_exact"], what=f"y rows {lo}:{hi}")
        if residual is not None:
            gu.check_exact(h_new[lo:hi], ref["h_new"], f"h_new rows {lo}:{hi}")
    gu.each_block(T, H, check)
    return y, rstd, h_new


def test_plain_small_config(orc):
    d = synth.plain_small()
    compare(orc, d["x"], d["w"], d["eps"])


@pytest.mark.parametrize("H", [2, 6, 8, 16, 64, 96, 128, 200, 256, 520, 1000, 1024, 1536, 2048,
                               3072, 4096, 5120, 6144, 8192, 12288, 16384])
@pytest.mark.parametrize("route", ["plain_bf16", "residual_bf16", "plain_f32", "residual_f32"])
def test_widths_and_routes(orc, H, route):
    T = 37
    x, r = synth.random_rows(H, T, H, n=2)
    f32 = route.endswith("f32")
    w = synth.random_weight(H + 1, H, f32=f32)
    compare(orc, x, w, residual=r if route.startswith("residual") else None,
            bias=1.0 if f32 else 0.0)


@pytest.mark.parametrize("T", [1, 2, 7, 63, 64, 65, 127, 128, 129, 255, 257])
def test_row_counts_residual_h4096(orc, T):
    d = synth.residual_large(seed=T, T=T)
    compare(orc, d["x"], d["w"], residual=d["residual"])


def test_residual_large_config(orc):
    """T=16384, H=4096 fused residual route, every row: h_new bit-exact
    (against the oracle and against a brute-force nearest-BF16 table of the
    exact sum), y and rstd within tolerance."""
    d = synth.residual_large()
    y, rstd, h_new = compare(orc, d["x"], d["w"], d["eps"], d["residual"])

    def nearest(lo, hi):
        exact = numfmt.decode_bf16(d["x"][lo:hi]) + numfmt.decode_bf16(d["residual"][lo:hi])
        gu.check_exact(h_new[lo:hi], numfmt.nearest_bf16(exact), f"h_new rows {lo}:{hi} (table)")
    gu.each_block(d["T"], d["H"], nearest)


@pytest.mark.parametrize("T", [1, 7, 128, 1024, 1025, 4096, 16384])
def test_zero_centred_weight_config(orc, T):
    """H=5120, FP32 zero-centred weight (effective 1 + w), x ~ 4 N(0,1),
    every row."""
    d = synth.zero_centred(T)
    compare(orc, d["x"], d["w"], d["eps"], bias=1.0)


def test_strided_heads_config(orc):
    """[2048, 32, 256] buffer viewed as [2048, 32, 128]: 65536 rows of stride
    256 read in place; the outputs match the contiguous copy bitwise."""
    d = synth.strided_heads()
    buf = gu.dev_bf16(d["buf"])
    view = buf[..., :d["H"]]
    w = gu.dev_f32(d["w"])
    y, rstd, _ = crm.rmsnorm_fwd(view, w, d["eps"], weight_bias=1.0)
    yc, rstdc, _ = crm.rmsnorm_fwd(view.contiguous(), w, d["eps"], weight_bias=1.0)
    # A strided output: the other half of a second buffer.
    obuf = torch.zeros_like(buf)
    crm.rmsnorm_fwd(view, w, d["eps"], weight_bias=1.0, y=obuf[..., d["H"]:])
    torch.cuda.synchronize()
    assert rstd.shape == (d["T"], d["heads"])
    gu.check_exact(gu.host_bits(y), gu.host_bits(yc), "strided vs contiguous y")
    gu.check_exact(gu.host_bits(obuf[..., d["H"]:]), gu.host_bits(y), "strided output")
    assert not obuf[..., :d["H"]].any()
    assert torch.equal(rstd, rstdc)
    x2 = d["buf"].reshape(-1, d["W"])[:, :d["H"]]        # row stride 256, every row checked
    yb = gu.host_bits(y).reshape(-1, d["H"])
    rb = rstd.cpu().numpy().reshape(-1)

    def check(lo, hi):
        ref = orc.rmsnorm_fwd(x2[lo:hi], d["w"], d["eps"], weight_bias=1.0)
        gu.check_bf16(yb[lo:hi], ref["y_exact"], what=f"y rows {lo}:{hi}")
        gu.check_rstd(rb[lo:hi], ref["rstd_exact"], what=f"rstd rows {lo}:{hi}")
    gu.each_block(x2.shape[0], d["H"], check)


def test_in_place_fused_add(orc):
    """fused_add_rmsnorm: input <- y and residual <- h_new in place."""
    x_bits, r_bits = synth.random_rows(11, 100, 2048, n=2)
    w = synth.random_weight(11, 2048)
    x, r = gu.dev_bf16(x_bits), gu.dev_bf16(r_bits)
    crm.rmsnorm_fwd(x, gu.dev_bf16(w), 1e-6, residual=r, y=x, h_new=r, want_rstd=False)
    torch.cuda.synchronize()
    ref = orc.rmsnorm_fwd(x_bits, w, 1e-6, residual=r_bits)
    gu.check_exact(gu.host_bits(r), ref["h_new"], "residual in place")
    gu.check_bf16(gu.host_bits(x), ref["y_exact"], what="input in place")


def test_gemma_equals_fp32_weight_route():
    """Gemma (BF16 w, bias 1) and the FP32 route fed the same weight values
    with bias 1 give identical bits on the GPU."""
    x = synth.random_rows(12, 64, 3072)[0]
    w = synth.random_weight(12, 3072)
    a = run_fwd(x, w, bias=1.0)
    b = run_fwd(x, numfmt.decode_bf16(w).astype(np.float32), bias=1.0)
    gu.check_exact(a[0], b[0], "y")
    assert np.array_equal(a[1], b[1])


@pytest.mark.parametrize("scale", [1e-3, 1e3])
def test_input_scales_and_zero_rows(orc, scale):
    x = synth.random_rows(13, 40, 1024, scale=scale)[0]
    x[3] = 0
    x[17] = 0x8000          # -0.0 everywhere
    w = synth.random_weight(13, 1024)
    y, rstd, _ = compare(orc, x, w)
    assert not numfmt.decode_bf16(y[3]).any() and not numfmt.decode_bf16(y[17]).any()


def test_unaligned_and_narrow_paths(orc):
    """4-byte-aligned views (an odd column offset of 2 elements) and widths
    that are not multiples of 8 take the 4-byte path."""
    buf = synth.random_rows(14, 50, 1040)[0]
    w = synth.random_weight(14, 1024)
    x = gu.dev_bf16(buf)[:, 2:1026]
    assert x.data_ptr() % 16 != 0
    y, rstd, _ = crm.rmsnorm_fwd(x, gu.dev_bf16(w), 1e-6)
    torch.cuda.synchronize()
    ref = orc.rmsnorm_fwd(np.ascontiguousarray(buf[:, 2:1026]), w, 1e-6)
    gu.check_bf16(gu.host_bits(y), ref["y_exact"])
    gu.check_rstd(rstd.cpu().numpy(), ref["rstd_exact"])
    for H in (250, 1002, 4094):
        xb = synth.random_rows(H, 9, H)[0]
        wb = synth.random_weight(H, H)
        compare(orc, xb, wb)


def test_rows_do_not_depend_on_T():
    """A row's y and rstd are the same bits whatever the token count."""
    x, r = synth.random_rows(15, 1025, 4096, n=2)
    w = synth.random_weight(15, 4096)
    big = run_fwd(x, w, residual_bits=r)
    for T in (1, 7, 640):
        small = run_fwd(x[:T], w, residual_bits=r[:T])
        gu.check_exact(small[0], big[0][:T], f"y at T={T}")
        assert np.array_equal(small[1], big[1][:T])


def test_outputs_stay_inside_their_rows():
    """Canary: an output written into the middle of a larger buffer leaves
    the surrounding elements (row padding and guard rows) untouched."""
    T, H, ld = 33, 1000, 1016
    x = synth.random_rows(16, T, H)[0]
    w = synth.random_weight(16, H)
    guard = torch.full((T + 2, ld), -7.0, dtype=torch.bfloat16, device=gu.DEV)
    out = guard[1:T + 1, :H]
    crm.rmsnorm_fwd(gu.dev_bf16(x), gu.dev_bf16(w), 1e-6, y=out)
    torch.cuda.synchronize()
    g = guard.float().cpu()
    assert (g[0] == -7).all() and (g[T + 1] == -7).all() and (g[1:T + 1, H:] == -7).all()


def test_zero_rows_launch_nothing():
    x = torch.empty((0, 4096), dtype=torch.bfloat16, device=gu.DEV)
    w = torch.ones(4096, dtype=torch.bfloat16, device=gu.DEV)
    y, rstd, _ = crm.rmsnorm_fwd(x, w)
    assert y.shape == (0, 4096) and rstd.shape == (0,)


@pytest.mark.parametrize("H", [1024, 4096, 8192, 16384])
@pytest.mark.parametrize("form", ["y", "e4m3"])
def test_persistent_forms_every_row(orc, H, form):
    """The persistent plain forms (BF16 y and static FP8), whose row groups
    of one to sixteen warps walk many rows per CTA with shared per-warp
    reduction slots: at T=16384 every row matches the oracle and is bitwise
    equal to the same row normalised alone (one launch per row, T=1)."""
    T = 16384
    x = synth.random_rows(H + 40, T, H)[0]
    w = synth.random_weight(H + 41, H)
    xd, wd = gu.dev_bf16(x), gu.dev_bf16(w)
    rstd, rstd1 = torch.empty(T, device=gu.DEV), torch.empty(T, device=gu.DEV)
    if form == "y":
        out, out1 = torch.empty_like(xd), torch.empty_like(xd)
        crm.rmsnorm_fwd(xd, wd, 1e-6, y=out, rstd=rstd)
        for t in range(T):
            crm.rmsnorm_fwd(xd[t:t + 1], wd, 1e-6, y=out1[t:t + 1], rstd=rstd1[t:t + 1])
    else:
        sc = torch.tensor([0.04], device=gu.DEV)
        out = torch.empty((T, H), dtype=torch.float8_e4m3fn, device=gu.DEV)
        out1 = torch.empty_like(out)
        crm.rmsnorm_quant(out, xd, wd, sc, 1e-6, rstd=rstd)
        for t in range(T):
            crm.rmsnorm_quant(out1[t:t + 1], xd[t:t + 1], wd, sc, 1e-6, rstd=rstd1[t:t + 1])
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.uint8), out1.view(torch.uint8)), "differs from one row per launch"
    assert torch.equal(rstd.view(torch.int32), rstd1.view(torch.int32)), "rstd differs from one row per launch"
    o = gu.host_bits(out) if form == "y" else gu.host_u8(out)
    r = rstd.cpu().numpy()

    def check(lo, hi):
        ref = orc.rmsnorm_fwd(x[lo:hi], w, 1e-6, want_y=form == "y")
        gu.check_rstd(r[lo:hi], ref["rstd_exact"], what=f"rstd rows {lo}:{hi}")
        if form == "y":
            gu.check_bf16(o[lo:hi], ref["y_exact"], what=f"y rows {lo}:{hi}")
        else:
            q = orc.rmsnorm_quant(x[lo:hi], w, 0.04, 1e-6, fp8_kind=0)
            gu.check_fp8(o[lo:hi], q["q"], q["v_exact"], 0, what=f"e4m3 rows {lo}:{hi}")
    gu.each_block(T, H, check)
