"""GPU FP8 epilogues against the CPU oracle: static-scale (fused add or plain,
E4M3FN and E5M2) and 1x128 block quantisation."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import numfmt
import oracle
import normalization_rmsnorm_fwd_gb300 as crm
from normalization_rmsnorm_fwd_gb300 import synth

pytestmark = pytest.mark.gpu
FP8 = {0: torch.float8_e4m3fn, 1: torch.float8_e5m2}


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


def run_static(x, w, scale, kind, residual=None, bias=0.0):
    T, H = x.shape
    out = torch.empty((T, H), dtype=FP8[kind], device=gu.DEV)
    r = gu.dev_bf16(residual) if residual is not None else None
    wd = gu.dev_f32(w) if w.dtype == np.float32 else gu.dev_bf16(w)
    rstd = torch.empty(T, device=gu.DEV)
    crm.fused_add_rmsnorm_quant(out, gu.dev_bf16(x), r, wd, scale, 1e-6, bias, rstd=rstd)
    torch.cuda.synchronize()
    return gu.host_u8(out), (gu.host_bits(r) if r is not None else None), rstd.cpu().numpy()


def compare_static(orc, x, w, scale, kind, residual=None, bias=0.0):
    """Every row: codes, the in-place residual and rstd against the oracle."""
    q, h_new, rstd = run_static(x, w, scale, kind, residual, bias)
    T, H = x.shape

    def check(lo, hi):
        r = None if residual is None else residual[lo:hi]
        ref = orc.rmsnorm_quant(x[lo:hi], w, scale, 1e-6, residual=r, weight_bias=bias,
                                fp8_kind=kind)
        gu.check_fp8(q[lo:hi], ref["q"], ref["v_exact"], kind, what=f"fp8 rows {lo}:{hi}")
        if residual is not None:
            gu.check_exact(h_new[lo:hi], ref["h_new"], f"residual in place, rows {lo}:{hi}")
        f = orc.rmsnorm_fwd(x[lo:hi], w, 1e-6, residual=r, weight_bias=bias, want_y=False)
        gu.check_rstd(rstd[lo:hi], f["rstd_exact"], what=f"rstd rows {lo}:{hi}")
    gu.each_block(T, H, check)


@pytest.mark.parametrize("kind", [0, 1])
@pytest.mark.parametrize("H", [8, 128, 1000, 4096, 8192])
@pytest.mark.parametrize("residual", [False, True])
def test_static_small(orc, kind, H, residual):
    x, r = synth.random_rows(H + kind, 45, H, n=2)
    w = synth.random_weight(H, H)
    compare_static(orc, x, w, 0.04, kind, r if residual else None)


def test_static_fp32_weight_and_saturation(orc):
    x, r = synth.random_rows(31, 33, 2048, n=2)
    w = synth.random_weight(31, 2048, f32=True)
    compare_static(orc, x, w, 0.004, 0, r, bias=1.0)     # many values beyond 448: saturate


def test_static_fp8_config(orc):
    """T = H = 8192, scale 0.04, E4M3FN: fused add, residual updated in place;
    every row."""
    d = synth.fp8()
    compare_static(orc, d["x"], d["w"], d["scale"], 0, d["residual"])


def run_block(x, r, w, ldT=None):
    T, H = x.shape
    ldT = ldT or (T + 3) // 4 * 4
    out = torch.empty((T, H), dtype=torch.float8_e4m3fn, device=gu.DEV)
    bs = torch.full((H // 128, ldT), float("nan"), device=gu.DEV)
    normed = torch.empty((T, H), dtype=torch.bfloat16, device=gu.DEV)
    rd = gu.dev_bf16(r)
    crm.fused_add_rmsnorm_fp8_block_quant(out, bs, normed, gu.dev_bf16(x), rd, gu.dev_bf16(w))
    torch.cuda.synchronize()
    return gu.host_u8(out), bs.cpu().numpy(), gu.host_bits(normed), gu.host_bits(rd)


def compare_block(orc, x, r, w):
    """Every row: residual, normed_out, block scales and codes."""
    q, bs, normed, h_new = run_block(x, r, w)
    T, H = x.shape
    assert np.isnan(bs[:, T:]).all(), "padding columns of block_scale were written"
    nb = H // 128

    def check(lo, hi):
        n = hi - lo
        ref = orc.fused_add_rmsnorm_fp8_block_quant(x[lo:hi], r[lo:hi], w, 1e-6)
        gu.check_exact(h_new[lo:hi], ref["h_new"], f"residual in place, rows {lo}:{hi}")
        gu.check_bf16(normed[lo:hi], ref["normed_exact"], what=f"normed_out rows {lo}:{hi}")
        same_block = (normed[lo:hi] == ref["normed"]).reshape(n, nb, 128).all(axis=2)   # [t, b]
        s_ref = ref["block_scale"][:, :n].T                                             # [t, b]
        s_gpu = bs[:, lo:hi].T
        assert np.array_equal(s_gpu[same_block], s_ref[same_block]), f"block scale rows {lo}:{hi}"
        assert np.all(np.abs(s_gpu - s_ref) <= 2.0 ** -7 * s_ref), "block scale (differing normed)"
        qb = q[lo:hi].reshape(n, nb, 128)
        rb = ref["q"].reshape(n, nb, 128)
        assert np.array_equal(qb[same_block], rb[same_block]), f"block codes rows {lo}:{hi}"
        d = qb[~same_block].astype(np.int32) - rb[~same_block].astype(np.int32)
        assert np.all(np.abs(d) <= 1), "block codes in blocks whose normed values differ by an ulp"
        return int((~same_block).sum())
    return sum(gu.each_block(T, H, check))


@pytest.mark.parametrize("H", [128, 256, 384, 1024, 4096, 8192, 16384])
@pytest.mark.parametrize("T", [1, 5, 66])
def test_block_small(orc, H, T):
    x, r = synth.random_rows(H + T, T, H, n=2)
    w = synth.random_weight(H, H)
    x[0, :128] = r[0, :128] ^ 0x8000          # a block that sums to zero
    compare_block(orc, x, r, w)


def test_block_fp8_config(orc):
    d = synth.fp8()
    compare_block(orc, d["x"], d["residual"], d["w"])
