"""Row strides, T-independence of the persistent forward, output canaries for
the backward, and capture of the forward + backward in a CUDA graph."""
import numpy as np
import pytest
import torch

import gpu_util as gu
import oracle
from normalization_rmsnorm_fwd_gb300 import synth
import normalization_rmsnorm_fwd_gb300 as crm

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return oracle.Oracle()


def _strided(bits, pad):
    """A device view of `bits` [T, H] whose rows sit in a buffer of row stride
    H + pad (the pad filled with garbage)."""
    T, H = bits.shape
    buf = torch.full((T, H + pad), 123.0, dtype=torch.bfloat16, device=gu.DEV)
    buf[:, :H] = gu.dev_bf16(bits)
    return buf[:, :H]


@pytest.mark.parametrize("pad", [0, 64, "2H"])
@pytest.mark.parametrize("H", [512, 4096])
def test_stride_pads_forward_and_backward(orc, pad, H):
    # The guide's layout matrix: row stride H, H + 64 and 3H (pad 2H) for
    # x, residual, g and the outputs.
    p = 2 * H if pad == "2H" else pad
    T = 200
    xb, ub, gb = synth.random_rows(H + p, T, H, n=3)
    wb = synth.random_weight(H + p, H)
    x, u, g = _strided(xb, p), _strided(ub, p), _strided(gb, p)
    w = gu.dev_bf16(wb)
    y = _strided(np.zeros_like(xb), p)
    yp, rp, _ = crm.rmsnorm_fwd(x, w, 1e-6, y=y)               # plain (persistent form)
    y2, r2, hn = crm.rmsnorm_fwd(x, w, 1e-6, residual=u)       # residual route
    dx = _strided(np.zeros_like(xb), p)
    crm.rmsnorm_bwd(g, x, w, rp, dx=dx)
    torch.cuda.synchronize()
    f = orc.rmsnorm_fwd(xb, wb, 1e-6)
    gu.check_bf16(gu.host_bits(yp), f["y_exact"], what=f"y pad {pad}")
    fr = orc.rmsnorm_fwd(xb, wb, 1e-6, residual=ub)
    assert np.array_equal(gu.host_bits(hn), fr["h_new"])
    gu.check_bf16(gu.host_bits(y2), fr["y_exact"], what=f"y residual pad {pad}")
    ref = orc.rmsnorm_bwd(gb, xb, wb, rp.cpu().numpy())
    allow = gu.dx_allowance(gb, xb, orc.weight_eff(wb), rp.cpu().numpy(), ref["m"])
    gu.check_bf16(gu.host_bits(dx), ref["dx_exact"], allowance=allow, what=f"dx pad {pad}")


def test_persistent_forward_rows_do_not_depend_on_T():
    # The plain forward runs on a grid capped at the resident CTAs; a row's
    # outputs must not depend on how many rows the call has (or on the grid).
    H = 4096
    x = synth.random_rows(30, 20000, H)[0]
    w = gu.dev_bf16(synth.random_weight(30, H))
    xd = gu.dev_bf16(x)
    big_y, big_r, _ = crm.rmsnorm_fwd(xd, w, 1e-6)
    torch.cuda.synchronize()
    for T in (1, 5, 152, 1000, 12345):
        y, r, _ = crm.rmsnorm_fwd(xd[:T], w, 1e-6)
        torch.cuda.synchronize()
        assert torch.equal(y, big_y[:T]) and torch.equal(r, big_r[:T]), T


@pytest.mark.parametrize("H,route", [(4096, "bf16"), (5120, "f32"), (1024, "bf16_gres"), (128, "bf16")])
def test_backward_dx_rows_do_not_depend_on_T(H, route):
    # A row's dx must not depend on how many rows the call has: neither on
    # the chunk table nor on the form (up to 2048 rows strip CTAs reduce dw
    # beside the chunks; above, the chunks write partial rows).  dw differs
    # only by the rows added, and matches the sum of the parts closely.
    T = 3000
    g, x, gr = synth.random_rows(31 + H, T, H, n=3)
    f32 = route == "f32"
    w = synth.random_weight(32, H, f32=f32)
    wd = gu.dev_f32(w) if f32 else gu.dev_bf16(w)
    gd, xd = gu.dev_bf16(g), gu.dev_bf16(x)
    grd = gu.dev_bf16(gr) if route == "bf16_gres" else None
    rstd = gu.dev_f32(np.abs(synth.Draw(33).f32((T,), 0.1, 1.0)))
    bias = 1.0 if f32 else 0.0
    big_dx, _ = crm.rmsnorm_bwd(gd, xd, wd, rstd, bias, g_residual=grd)
    torch.cuda.synchronize()
    for T2 in (1, 7, 2048, 2049, 2999):
        dx, _ = crm.rmsnorm_bwd(gd[:T2], xd[:T2], wd, rstd[:T2], bias,
                                g_residual=None if grd is None else grd[:T2])
        torch.cuda.synchronize()
        assert torch.equal(dx.view(torch.int16), big_dx[:T2].view(torch.int16)), T2
    _, dw_a = crm.rmsnorm_bwd(gd[:2048], xd[:2048], wd, rstd[:2048], bias,
                              g_residual=None if grd is None else grd[:2048])
    _, dw_b = crm.rmsnorm_bwd(gd[2048:], xd[2048:], wd, rstd[2048:], bias,
                              g_residual=None if grd is None else grd[2048:])
    _, dw_all = crm.rmsnorm_bwd(gd, xd, wd, rstd, bias, g_residual=grd)
    torch.cuda.synchronize()
    a, b, c = (t.double().cpu().numpy() for t in (dw_a, dw_b, dw_all))
    assert np.linalg.norm(a + b - c) <= 1e-6 * np.linalg.norm(c)


def test_backward_outputs_stay_inside_their_rows():
    T, H, ld = 70, 1000, 1040
    g, x = synth.random_rows(31, T, H, n=2)
    w = gu.dev_bf16(synth.random_weight(31, H))
    rstd = torch.rand(T, device=gu.DEV) + 0.5
    guard = torch.full((T + 2, ld), -7.0, dtype=torch.bfloat16, device=gu.DEV)
    dx = guard[1:T + 1, :H]
    dw_guard = torch.full((H + 64,), -7.0, device=gu.DEV)
    crm.rmsnorm_bwd(gu.dev_bf16(g), gu.dev_bf16(x), w, rstd, dx=dx, dw=dw_guard[32:32 + H])
    torch.cuda.synchronize()
    gd = guard.float().cpu()
    assert (gd[0] == -7).all() and (gd[T + 1] == -7).all() and (gd[1:T + 1, H:] == -7).all()
    dwg = dw_guard.cpu()
    assert (dwg[:32] == -7).all() and (dwg[32 + H:] == -7).all()


@pytest.mark.parametrize("T", [1024, 2500])
def test_cuda_graph_replay_matches_eager(T):
    # The residual forward and the backward (one launch in the column form at
    # 1024 rows; the chunks and the reduce at 2500, launched with programmatic
    # dependent launch) captured once in a CUDA graph and replayed on new
    # inputs copied into the captured buffers: every replay equals an eager
    # run bit for bit, and the workspace needs no reset between replays.
    H = 2048
    w = gu.dev_bf16(synth.random_weight(40, H))
    ws = crm.rmsnorm_bwd_workspace(T, H, gu.DEV)
    xs = torch.empty((T, H), dtype=torch.bfloat16, device=gu.DEV)
    us = torch.empty_like(xs)
    gs = torch.empty_like(xs)
    y, hn, dx = torch.empty_like(xs), torch.empty_like(xs), torch.empty_like(xs)
    rstd = torch.empty(T, device=gu.DEV)
    dw = torch.empty(H, device=gu.DEV)

    def step():
        crm.rmsnorm_fwd(xs, w, 1e-6, residual=us, y=y, rstd=rstd, h_new=hn)
        crm.rmsnorm_bwd(gs, hn, w, rstd, workspace=ws, dx=dx, dw=dw)

    def load(seed):
        xb, ub, gb = synth.random_rows(seed, T, H, n=3)
        xs.copy_(gu.dev_bf16(xb)); us.copy_(gu.dev_bf16(ub)); gs.copy_(gu.dev_bf16(gb))

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        load(41)
        step()                       # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in (42, 43, 44):
        load(seed)
        graph.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (y, hn, dx, dw, rstd)]
        load(seed)
        step()
        torch.cuda.synchronize()
        want = [y, hn, dx, dw, rstd]
        for a, b, name in zip(got, want, ("y", "h_new", "dx", "dw", "rstd")):
            assert torch.equal(a, b), (seed, name)


def test_back_to_back_dependent_calls_match_serialised_calls():
    # Every grid is launched with programmatic dependent launch, so the next
    # grid may be scheduled while the previous one still runs; each call here
    # reads what the call before it wrote (forward -> backward -> forward on
    # the backward's dx ...), so a missing dependency wait would read stale
    # rows.  The chain enqueued back to back equals the same chain with a
    # device synchronisation after every call, bit for bit.
    T, H = 3000, 2048
    xb, gb = synth.random_rows(50, T, H, n=2)
    w = gu.dev_bf16(synth.random_weight(50, H))
    ws = crm.rmsnorm_bwd_workspace(T, H, gu.DEV)

    def chain(sync):
        x = gu.dev_bf16(xb)
        g = gu.dev_bf16(gb)
        outs = []
        for _ in range(6):
            y, rstd, _ = crm.rmsnorm_fwd(x, w, 1e-6)
            if sync:
                torch.cuda.synchronize()
            dx, dw = crm.rmsnorm_bwd(g, y, w, rstd, workspace=ws)
            if sync:
                torch.cuda.synchronize()
            q = torch.empty((T, H), dtype=torch.float8_e4m3fn, device=gu.DEV)
            crm.rmsnorm_quant(q, dx, w, 0.5)
            if sync:
                torch.cuda.synchronize()
            outs += [y, rstd, dx, dw, q.view(torch.uint8)]
            x, g = dx, y
        torch.cuda.synchronize()
        return outs

    for a, b in zip(chain(False), chain(True)):
        assert torch.equal(a, b)
