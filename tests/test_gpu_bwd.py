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


def oracle_rstd(orc, x, w, eps, bias=0.0):
    """The oracle forward's FP32 rstd of every row (row blocks in parallel)."""
    T, H = x.shape
    parts = gu.each_block(T, H, lambda lo, hi: orc.rmsnorm_fwd(x[lo:hi], w, eps, weight_bias=bias,
                                                               want_y=False)["rstd"])
    return np.concatenate(parts) if parts else np.empty(0, np.float32)


def check_every_row(orc, g, x, w, rstd, dx, dw, bias=0.0, g_res=None):
    """dx of every row against the oracle, and dw against the oracle's sum
    over all rows (formed block by block in double precision)."""
    T, H = x.shape
    w_eff = orc.weight_eff(w, bias)

    def check(lo, hi):
        gr = None if g_res is None else g_res[lo:hi]
        ref = orc.rmsnorm_bwd(g[lo:hi], x[lo:hi], w, rstd[lo:hi], weight_bias=bias, g_res=gr)
        allow = gu.dx_allowance(g[lo:hi], x[lo:hi], w_eff, rstd[lo:hi], ref["m"])
        gu.check_bf16(dx[lo:hi], ref["dx_exact"], allowance=allow, what=f"dx rows {lo}:{hi}")
        return ref["dw"], ref["dw_abs"]
    parts = gu.each_block(T, H, check)
    gu.check_dw(dw, sum(p[0] for p in parts), sum(p[1] for p in parts))


def compare(orc, g, x, w, eps=1e-6, bias=0.0, g_res=None):
    rstd = oracle_rstd(orc, x, w, eps, bias)
    dx, dw = run_bwd(g, x, w, rstd, bias, g_res)
    check_every_row(orc, g, x, w, rstd, dx, dw, bias, g_res)
    return dx, dw


def test_plain_small_config(orc):
    d = synth.plain_small()
    compare(orc, d["g"], d["x"], d["w"], d["eps"])


# 8192 with g_residual, 9002 with g_residual (4-byte path) and 12288 run the
# backward with two rows in flight (three ring stages fit, four do not);
# 16384 holds the BF16 weight as BF16 in shared memory (two rows in flight,
# one with g_residual; the FP32 weight: one, or with g_residual no ring).
# 300 rows take dw from the column CTAs, 2500 rows from the chunks' partial
# rows and the reduction kernel.
@pytest.mark.parametrize("H", [2, 8, 64, 128, 200, 256, 520, 1024, 2048, 3072, 4096, 5120,
                               6144, 8192, 9002, 12288, 16384])
@pytest.mark.parametrize("route", ["bf16", "f32", "bf16_gres"])
@pytest.mark.parametrize("T", [300, 2500])
def test_widths_and_routes(orc, H, route, T):
    g, x, gr = synth.random_rows(H + 3, T, H, n=3)
    f32 = route == "f32"
    w = synth.random_weight(H + 4, H, f32=f32)
    compare(orc, g, x, w, bias=1.0 if f32 else 0.0, g_res=gr if route.endswith("gres") else None)


@pytest.mark.parametrize("T", [1, 2, 7, 63, 64, 65, 127, 128, 129, 255, 257, 16172, 16231])
def test_row_counts(orc, T):
    g, x = synth.random_rows(T, T, 512, n=2)
    w = synth.random_weight(T, 512)
    compare(orc, g, x, w)


def test_residual_large_config(orc):
    """T=16384, H=4096 on the residual route: the backward of h_new with the
    gradient g; dx on every row, dw over all rows."""
    d = synth.residual_large()
    T, H = d["T"], d["H"]
    h_new = np.concatenate(gu.each_block(T, H, lambda lo, hi: orc.rmsnorm_fwd(
        d["x"][lo:hi], d["w"], d["eps"], residual=d["residual"][lo:hi], want_y=False)["h_new"]))
    compare(orc, d["g"], h_new, d["w"], d["eps"])


@pytest.mark.parametrize("T", [1, 7, 128, 1024, 1025, 4096, 16384])
def test_zero_centred_weight_config(orc, T):
    """H=5120, FP32 zero-centred weight, every row of every token count."""
    d = synth.zero_centred(T)
    compare(orc, d["g"], d["x"], d["w"], d["eps"], bias=1.0)


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
    check_every_row(orc, g2, x2, d["w"], rstd, gu.host_bits(dx).reshape(-1, H),
                    dw.cpu().numpy(), bias=1.0)


@pytest.mark.parametrize("T", [1000, 16384])
def test_dw_is_bitwise_reproducible(T):
    """Three runs, and a run on a second stream with a reused workspace, give
    identical dw and dx bits (1000 rows: the column form; 16384: the chunk
    table)."""
    g, x = synth.random_rows(21, T, 4096, n=2)
    w = synth.random_weight(21, 4096)
    rstd = np.abs(synth.Draw(21).f32((T,), 0.1, 1.0))
    ws = crm.rmsnorm_bwd_workspace(T, 4096, gu.DEV)
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
@pytest.mark.parametrize("T", [305, 608, 913, 1500, 2048, 2049, 2431])
def test_pipelined_chunk_lengths(orc, H, T):
    # Multi-warp rows run the software-pipelined loop (row i+1's sum formed
    # while row i's dx is written); these row counts give chunks of one to
    # eight rows, so the prologue, the steady state and the tail (rows past
    # the chunk) all occur, with one and two row groups per CTA (H = 4096 and
    # H = 1024).  Up to 2048 rows dw comes from the column CTAs of the same
    # launch, above it from the chunks' partial rows.
    g, x = synth.random_rows(T + H, T, H, n=2)
    w = synth.random_weight(T + 7, H)
    compare(orc, g, x, w)



@pytest.mark.parametrize("H,gres", [(16384, False), (11264, True)])
@pytest.mark.parametrize("bias", [0.0, -0.0, 1.0])
@pytest.mark.parametrize("T", [300, 2500])
def test_bf16_weight_held_as_bf16_matches_fp32_weight(orc, H, gres, bias, T):
    # At these widths a BF16 weight is held as BF16 in shared memory (which
    # leaves room for a deeper ring than the FP32 weight does); the same
    # weight values given as FP32 take the FP32 table and a shallower ring.
    # Both run the same pipelined arithmetic, so dx and dw agree bit for bit;
    # a few weights are -0 (with a bias of +0 the FP32 table holds +0 there,
    # with a bias of -0 it keeps -0).
    g, x, gr = synth.random_rows(H + T + 5, T, H, n=3)
    w = synth.random_weight(H + 6, H)
    w[::997] = 0x8000
    w32 = (w.astype(np.uint32) << 16).view(np.float32)       # the same values, exactly
    rstd = np.abs(synth.Draw(H + 7).f32((T,), 0.1, 1.0))
    g_res = gr if gres else None
    dx_b, dw_b = run_bwd(g, x, w, rstd, bias, g_res)
    dx_f, dw_f = run_bwd(g, x, w32, rstd, bias, g_res)
    assert np.array_equal(dx_b, dx_f)
    assert np.array_equal(dw_b.view(np.uint32), dw_f.view(np.uint32))
    if T == 300:
        check_every_row(orc, g, x, w, rstd, dx_b, dw_b, bias, g_res)
