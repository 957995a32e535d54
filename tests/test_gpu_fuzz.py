"""Seeded random shapes against the oracle: forward, backward and the static
FP8 epilogue on widths, row counts, row strides, weight routes, input scales
and eps drawn at random (every row checked), so that combinations no other
test names -- a ragged width on the 4-byte path with a padded stride and a
g_residual, a row count just above the column form's limit, a large or tiny
input scale -- still meet the same tolerances."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import numfmt
import oracle
import normalization_rmsnorm_fwd_gb300 as crm

pytestmark = pytest.mark.gpu
N_CASES = 96


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


def _case(seed):
    rng = np.random.default_rng(1000 + seed)
    if rng.random() < 0.5:
        H = int(8 * np.round(2 ** rng.uniform(0, 11)))          # multiples of 8: 16-byte path
    else:
        H = int(2 * np.round(2 ** rng.uniform(0, 13)))          # even: often the 4-byte path
    H = max(2, min(H, 16384))
    T = int(np.round(2 ** rng.uniform(0, 12.2)))                 # 1 .. ~4700 rows
    if seed % 8 == 0:
        T = int(rng.choice([2048, 2049, 2050]))                  # either side of the column form's limit
    pad = int(rng.choice([0, 2, 8, 64]))
    if H % 8 == 0 and pad == 2:
        pad = 8
    route = str(rng.choice(["plain", "residual", "gemma", "f32"]))
    gres = bool(rng.random() < 0.4)
    scale = float(10.0 ** rng.uniform(-2, 2))
    eps = float(rng.choice([1e-6, 1e-5, 0.1]))
    kind = int(rng.integers(0, 2))
    return dict(H=H, T=T, pad=pad, route=route, gres=gres, scale=scale, eps=eps, kind=kind, rng=rng)


def _rows(rng, T, H, scale, shift=0.0):
    """BF16 bits of shift + scale * N(0, 1), rounded to nearest even."""
    v = (shift + scale * rng.standard_normal((T, H))).astype(np.float64)
    return numfmt.nearest_bf16(v)


def _device_rows(bits, pad):
    """Device BF16 rows of `bits` in a buffer of row stride H + pad."""
    T, H = bits.shape
    buf = torch.full((T, H + pad), 77.0, dtype=torch.bfloat16, device=gu.DEV)
    buf[:, :H] = gu.dev_bf16(bits)
    return buf[:, :H]


@pytest.mark.parametrize("seed", range(N_CASES))
def test_random_shapes(orc, seed):
    c = _case(seed)
    rng, H, T, pad = c["rng"], c["H"], c["T"], c["pad"]
    x = _rows(rng, T, H, c["scale"])
    r = _rows(rng, T, H, c["scale"]) if c["route"] == "residual" else None
    g = _rows(rng, T, H, 1.0)
    gr = _rows(rng, T, H, 1.0) if c["gres"] else None
    f32 = c["route"] == "f32"
    bias = 1.0 if c["route"] in ("gemma", "f32") else 0.0
    if f32:
        w = (0.02 * rng.standard_normal(H)).astype(np.float32)     # zero-centred: 1 + w
    elif c["route"] == "gemma":
        w = _rows(rng, 1, H, 0.1)[0]                               # Gemma: w + 1
    else:
        w = _rows(rng, 1, H, 0.1, shift=1.0)[0]
    wd = gu.dev_f32(w) if f32 else gu.dev_bf16(w)
    eps = c["eps"]

    # Forward.
    xd = _device_rows(x, pad)
    rd = _device_rows(r, pad) if r is not None else None
    y, rstd, h_new = crm.rmsnorm_fwd(xd, wd, eps, residual=rd, weight_bias=bias)
    # Backward on the forward's normalised input.
    hb = gu.host_bits(h_new) if h_new is not None else x
    gd = _device_rows(g, pad)
    grd = _device_rows(gr, pad) if gr is not None else None
    hd = _device_rows(hb, pad)
    dx, dw = crm.rmsnorm_bwd(gd, hd, wd, rstd, bias, g_residual=grd)
    # Static FP8 on the same inputs.
    dt = torch.float8_e4m3fn if c["kind"] == 0 else torch.float8_e5m2
    q = torch.empty((T, H), dtype=dt, device=gu.DEV)
    rq = _device_rows(r, pad) if r is not None else None
    crm.fused_add_rmsnorm_quant(q, xd, rq, wd, 0.04, eps, bias)
    torch.cuda.synchronize()
    yb, rs, dxb, dwh, qb = (gu.host_bits(y), rstd.cpu().numpy(), gu.host_bits(dx),
                            dw.cpu().numpy(), gu.host_u8(q))
    w_eff = orc.weight_eff(w, bias)
    what = f"case {seed} (T={T}, H={H}, pad={pad}, {c['route']}, gres={c['gres']}, eps={eps})"

    def check(lo, hi):
        rr = None if r is None else r[lo:hi]
        f = orc.rmsnorm_fwd(x[lo:hi], w, eps, residual=rr, weight_bias=bias)
        gu.check_rstd(rs[lo:hi], f["rstd_exact"], what=f"{what}: rstd rows {lo}:{hi}")
        gu.check_bf16(yb[lo:hi], f["y_exact"], what=f"{what}: y rows {lo}:{hi}")
        if r is not None:
            gu.check_exact(hb[lo:hi], f["h_new"], f"{what}: h_new rows {lo}:{hi}")
        b = orc.rmsnorm_bwd(g[lo:hi], hb[lo:hi], w, rs[lo:hi], weight_bias=bias,
                            g_res=None if gr is None else gr[lo:hi])
        allow = gu.dx_allowance(g[lo:hi], hb[lo:hi], w_eff, rs[lo:hi], b["m"])
        gu.check_bf16(dxb[lo:hi], b["dx_exact"], allowance=allow, what=f"{what}: dx rows {lo}:{hi}")
        fq = orc.rmsnorm_quant(x[lo:hi], w, 0.04, eps, residual=rr, weight_bias=bias,
                               fp8_kind=c["kind"])
        gu.check_fp8(qb[lo:hi], fq["q"], fq["v_exact"], c["kind"], what=f"{what}: fp8 rows {lo}:{hi}")
        return b["dw"], b["dw_abs"]
    parts = gu.each_block(T, H, check)
    gu.check_dw(dwh, sum(p[0] for p in parts), sum(p[1] for p in parts), what=f"{what}: dw")


# The other operations on random shapes, through the checks of their own test
# files: 1x128 block quantisation, AdaRMSNorm (per-row or broadcast style),
# the gated FP8 path, RMSNorm + SiLU and LayerNorm.
from test_gpu_ada import compare_ada, compare_gated            # noqa: E402
from test_gpu_quant import compare_block                       # noqa: E402
from test_gpu_silu_ln import _check_ln, _check_silu            # noqa: E402

N_OTHER = 40


@pytest.mark.parametrize("seed", range(N_OTHER))
def test_random_shapes_other_ops(orc, seed):
    rng = np.random.default_rng(5000 + seed)
    op = seed % 5
    T = int(np.round(2 ** rng.uniform(0, 11.5)))
    scale = float(10.0 ** rng.uniform(-1.5, 1.5))
    if op == 0:
        H = 128 * int(rng.integers(1, 65))
        x, r = _rows(rng, T, H, scale), _rows(rng, T, H, scale)
        compare_block(orc, x, r, _rows(rng, 1, H, 0.1, shift=1.0)[0])
        return
    D = int(2 * np.round(2 ** rng.uniform(0, 12)))
    D = max(2, min(D, 8192))
    if op in (1, 2):
        x = _rows(rng, T, D, scale)
        style = _rows(rng, 1 if rng.random() < 0.5 else T, 3 * D, 0.5)
        w = _rows(rng, 1, D, 0.1, shift=1.0)[0]
        if op == 1:
            compare_ada(orc, x, w, style)
        else:
            compare_gated(orc, _rows(rng, T, D, scale), x, _rows(rng, T, D, 1.0), w, style)
    elif op == 3:
        x = _rows(rng, T, D, scale)
        if rng.random() < 0.5:
            compare_w, bias = (0.02 * rng.standard_normal(D)).astype(np.float32), 1.0
        else:
            compare_w, bias = _rows(rng, 1, D, 0.1, shift=1.0)[0], 0.0
        _check_silu(orc, x, compare_w, bias)
    else:
        shift = float(rng.choice([0.0, 0.0, 50.0]))
        x = _rows(rng, T, D, scale, shift=shift)
        gamma = (1 + 0.1 * rng.standard_normal(D)).astype(np.float32)
        beta = (0.1 * rng.standard_normal(D)).astype(np.float32)
        _check_ln(orc, x, gamma, beta)
