"""GPU backward (rmsnorm_bwd through the C ABI) against the CPU oracle, and
dw determinism.  The backward's inputs (g, the normalised x, the FP32 rstd)
come from the seeded generator and the oracle's forward, never from the GPU."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
import normalization_rmsnorm_fwd_gb300 as crm
from normalization_rmsnorm_fwd_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


def run_bwd(g, x, w, rstd, bias=0.0, g_res=None, workspace=None):
    wd = gu.dev_f32(w) if w.dtype == np.float32 else gu.dev_bf16(w)
    dx, dw = crm.rmsnorm_bwd(gu.dev_bf16(g), gu.dev_bf16(x), wd, gu.dev_f32(rstd), bias,
                             g_residual=gu.dev_bf16(g_res) if g_res is not None else None,
                             workspace=workspace)
    torch.cuda.synchronize()
    return gu.host_bits(dx), dw.cpu().numpy()


def compare(orc, g, x, w, eps=1e-6, bias=0.0, g_res=None, rows=None):
    rstd = orc.rmsnorm_fwd(x, w, eps, weight_bias=bias, want_y=False)["rstd"]
    dx, dw = run_bwd(g, x, w, rstd, bias, g_res)
    full = orc.rmsnorm_bwd(g, x, w, rstd, weight_bias=bias, g_res=g_res, want_dx=rows is None)
    gu.check_dw(dw, full["dw"], full["dw_abs"])
    if rows is None:
        ref, sel = full, slice(None)
    else:
        sel = rows
        ref = orc.rmsnorm_bwd(g[rows], x[rows], w, rstd[rows], weight_bias=bias,
                              g_res=None if g_res is None else g_res[rows])
    w_eff = orc.weight_eff(w, bias)
    allow = gu.dx_allowance(g[sel], x[sel], w_eff, rstd[sel], ref["m"])
    gu.check_bf16(dx[sel], ref["dx_exact"], allowance=allow, what="dx")
    return dx, dw


def test_plain_small_config(orc):
    d = synth.plain_small()
    compare(orc, d["g"], d["x"], d["w"], d["eps"])


# 8192 with g_residual, 9002 with g_residual (4-byte path) and 12288 run the
# backward with two rows in flight (three ring stages fit, four do not).
@pytest.mark.parametrize("H", [2, 8, 64, 128, 200, 256, 520, 1024, 2048, 3072, 4096, 5120,
                               6144, 8192, 9002, 12288, 16384])
@pytest.mark.parametrize("route", ["bf16", "f32", "bf16_gres"])
def test_widths_and_routes(orc, H, route):
    T = 300
    g, x, gr = synth.random_rows(H + 3, T, H, n=3)
    f32 = route == "f32"
    w = synth.random_weight(H + 4, H, f32=f32)
    compare(orc, g, x, w, bias=1.0 if f32 else 0.0, g_res=gr if route.endswith("gres") else None)


@pytest.mark.parametrize("T", [1, 2, 7, 63, 64, 65, 127, 128, 129, 255, 257, 16172, 16231])
def test_row_counts(orc, T):
    g, x = synth.random_rows(T, T, 512, n=2)
    w = synth.random_weight(T, 512)
    compare(orc, g, x, w, rows=None if T < 1000 else gu.sample_rows(T))


def test_residual_large_config(orc):
    """T=16384, H=4096 on the residual route: the backward of h_new with the
    gradient g; dw over all rows, dx on a spread of rows."""
    d = synth.residual_large()
    h_new = orc.rmsnorm_fwd(d["x"], d["w"], d["eps"], residual=d["residual"], want_y=False)["h_new"]
    compare(orc, d["g"], h_new, d["w"], d["eps"], rows=gu.sample_rows(d["T"]))


@pytest.mark.parametrize("T", [1024, 4096])
def test_zero_centred_weight_config(orc, T):
    d = synth.zero_centred(T)
    compare(orc, d["g"], d["x"], d["w"], d["eps"], bias=1.0, rows=gu.sample_rows(T, 256))


def test_strided_heads_config(orc):
    d = synth.strided_heads()
    H = d["H"]
    x = gu.dev_bf16(d["buf"])[..., :H]
    g = gu.dev_bf16(d["gbuf"])[..., H:]
    x2 = np.ascontiguousarray(d["buf"].reshape(-1, d["W"])[:, :H])
    g2 = np.ascontiguousarray(d["gbuf"].reshape(-1, d["W"])[:, H:])
    rstd = orc.rmsnorm_fwd(x2, d["w"], d["eps"], weight_bias=1.0, want_y=False)["rstd"]
    w = gu.dev_f32(d["w"])
    dx, dw = crm.rmsnorm_bwd(g, x, w, gu.dev_f32(rstd).view(d["T"], d["heads"]), 1.0)
    dxc, dwc = crm.rmsnorm_bwd(g.contiguous(), x.contiguous(), w,
                               gu.dev_f32(rstd).view(d["T"], d["heads"]), 1.0)
    torch.cuda.synchronize()
    gu.check_exact(gu.host_bits(dx), gu.host_bits(dxc), "strided vs contiguous dx")
    assert torch.equal(dw, dwc)
    ref = orc.rmsnorm_bwd(g2, x2, d["w"], rstd, weight_bias=1.0, want_dx=False)
    gu.check_dw(dw.cpu().numpy(), ref["dw"], ref["dw_abs"])


def test_dw_is_bitwise_reproducible():
    """Three runs, and a run on a second stream with a reused workspace, give
    identical dw and dx bits."""
    g, x = synth.random_rows(21, 16384, 4096, n=2)
    w = synth.random_weight(21, 4096)
    rstd = np.abs(synth.Draw(21).f32((16384,), 0.1, 1.0))
    ws = crm.rmsnorm_bwd_workspace(16384, 4096, gu.DEV)
    runs = [run_bwd(g, x, w, rstd, workspace=ws) for _ in range(3)]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        runs.append(run_bwd(g, x, w, rstd, workspace=ws))
    for dx, dw in runs[1:]:
        assert np.array_equal(dw.view(np.uint32), runs[0][1].view(np.uint32))
        assert np.array_equal(dx, runs[0][0])


def test_workspace_does_not_depend_on_rows():
    a = crm.rmsnorm_bwd_workspace_bytes(1, 4096, gu.DEV)
    b = crm.rmsnorm_bwd_workspace_bytes(1 << 20, 4096, gu.DEV)
    assert a == b and a % 256 == 0 and a >= 4096 * 4


def test_short_workspace_is_rejected():
    g, x = synth.random_rows(22, 64, 256, n=2)
    w = synth.random_weight(22, 256)
    need = crm.rmsnorm_bwd_workspace_bytes(64, 256, gu.DEV)
    ws = torch.empty(need - 256, dtype=torch.uint8, device=gu.DEV)
    with pytest.raises(crm.CrmsnError, match="WORKSPACE"):
        crm.rmsnorm_bwd(gu.dev_bf16(g), gu.dev_bf16(x), gu.dev_bf16(w),
                        torch.ones(64, device=gu.DEV), workspace=ws)
    big = torch.empty(need + 512, dtype=torch.uint8, device=gu.DEV)
    with pytest.raises(crm.CrmsnError, match="WORKSPACE"):
        crm.rmsnorm_bwd(gu.dev_bf16(g), gu.dev_bf16(x), gu.dev_bf16(w),
                        torch.ones(64, device=gu.DEV), workspace=big[16:])


def test_zero_rows_give_zero_dw():
    x = torch.empty((0, 1024), dtype=torch.bfloat16, device=gu.DEV)
    dw = torch.full((1024,), 5.0, device=gu.DEV)
    crm.rmsnorm_bwd(x, x, torch.ones(1024, dtype=torch.bfloat16, device=gu.DEV),
                    torch.empty(0, device=gu.DEV), dw=dw)
    torch.cuda.synchronize()
    assert not dw.any()


def test_dx_in_place_over_g(orc):
    g, x = synth.random_rows(23, 50, 768, n=2)
    w = synth.random_weight(23, 768)
    rstd = orc.rmsnorm_fwd(x, w, 1e-6, want_y=False)["rstd"]
    gd = gu.dev_bf16(g)
    crm.rmsnorm_bwd(gd, gu.dev_bf16(x), gu.dev_bf16(w), gu.dev_f32(rstd), dx=gd)
    torch.cuda.synchronize()
    ref = orc.rmsnorm_bwd(g, x, w, rstd)
    allow = gu.dx_allowance(g, x, orc.weight_eff(w), rstd, ref["m"])
    gu.check_bf16(gu.host_bits(gd), ref["dx_exact"], allowance=allow, what="dx in place")


@pytest.mark.parametrize("H", [1024, 4096])
@pytest.mark.parametrize("T", [305, 608, 913, 1500, 2431])
def test_pipelined_chunk_lengths(orc, H, T):
    # Multi-warp rows run the software-pipelined loop (row i+1's sum formed
    # while row i's dx is written); these row counts give chunks of one to
    # eight rows, so the prologue, the steady state and the tail (rows past
    # the chunk) all occur, with one and two row groups per CTA (H = 4096 and
    # H = 1024).
    g, x = synth.random_rows(T + H, T, H, n=2)
    w = synth.random_weight(T + 7, H)
    compare(orc, g, x, w, rows=None if T < 1000 else gu.sample_rows(T))

