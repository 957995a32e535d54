"""The debug build's bounds guard (-DCRMSN_DEBUG).

In that build every global load and store of every kernel is checked against
the byte ranges of the call's tensors and every dynamic shared-memory access
against the launch's size; a violation is skipped and recorded, and
crmsn_debug_status() reads the record back.  Each case below runs one entry
point on small and ragged shapes (one and several tiles, strided rows, the
persistent forms, both backward forms, g_residual, the 4-byte path) in the
normal and in the debug library: the debug run must record nothing and give
the same bits.  A last case checks that the guard does report: it narrows the
guard's view of the output (an environment switch read by the debug build
only; the buffer itself is untouched) and expects the stores there to be
reported and skipped.
"""
import ctypes

import pytest
import torch

from normalization_rmsnorm_fwd_gb300 import _abi, build
import normalization_rmsnorm_fwd_gb300 as crm

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module")
def dbg():
    return _abi.load(build.build(debug=True))


def _word(lib) -> int:
    w = ctypes.c_uint64(0)
    st = lib.crmsn_debug_status(ctypes.byref(w))
    assert st == 0, _abi.STATUS.get(st, st)
    return w.value


def _describe(w: int) -> str:
    kinds = {1: "load", 2: "store", 3: "async copy", 4: "shared memory"}
    return (f"{kinds.get((w >> 56) & 0x7f, '?')} by CTA {(w >> 32) & 0xffffff}, "
            f"thread {(w >> 22) & 0x3ff}, address ...{w & 0x3fffff:06x}")


def _same(a: torch.Tensor, b: torch.Tensor) -> bool:
    if a.dtype in (torch.float8_e4m3fn, torch.float8_e5m2):
        return torch.equal(a.view(torch.uint8), b.view(torch.uint8))
    if a.element_size() == 2:
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    return torch.equal(a.view(torch.int32), b.view(torch.int32))


def run_both(dbg, monkeypatch, case):
    """case() builds its seeded inputs, runs one entry point and returns its
    outputs; run it on the normal and on the debug library."""
    ref = case()
    torch.cuda.synchronize()
    with monkeypatch.context() as m:
        m.setattr(_abi, "_lib", dbg)
        _word(dbg)                        # start from a clear record
        got = case()
        w = _word(dbg)
    assert w == 0, "bounds guard: " + _describe(w)
    for i, (a, b) in enumerate(zip(ref, got)):
        assert _same(a, b), f"output {i} differs between the normal and the debug build"


def _rows(gen, T, H, ld=None, scale=1.0):
    ld = ld or H
    buf = (scale * torch.randn(T, ld, generator=gen)).bfloat16().to(DEV)
    return buf[:, :H]


def _gen(seed):
    return torch.Generator().manual_seed(seed)


@pytest.mark.parametrize("T,H,ld", [(37, 2, 2), (37, 200, 200), (5, 4096, 4104), (300, 4096, 4096),
                                    (1000, 4096, 4096), (9, 5120, 5120), (3, 16384, 16384),
                                    (65, 1022, 1022)])
@pytest.mark.parametrize("route", ["plain", "residual", "f32"])
def test_forward(dbg, monkeypatch, T, H, ld, route):
    def case():
        g = _gen(T + H)
        x = _rows(g, T, H, ld)
        r = _rows(g, T, H, ld) if route == "residual" else None
        w = (1 + 0.1 * torch.randn(H, generator=g))
        w = w.to(DEV) if route == "f32" else w.bfloat16().to(DEV)
        if r is not None:
            r = r.clone()
        out = crm.rmsnorm_fwd(x, w, 1e-6, residual=r, weight_bias=1.0 if route == "f32" else 0.0)
        return [t for t in out if t is not None]
    run_both(dbg, monkeypatch, case)


@pytest.mark.parametrize("T,H", [(37, 256), (1000, 4096), (7, 8192)])
@pytest.mark.parametrize("residual", [False, True])
@pytest.mark.parametrize("kind", [torch.float8_e4m3fn, torch.float8_e5m2])
def test_static_fp8(dbg, monkeypatch, T, H, residual, kind):
    def case():
        g = _gen(3 * T + H)
        x = _rows(g, T, H)
        r = _rows(g, T, H).clone() if residual else None
        w = (1 + 0.1 * torch.randn(H, generator=g)).bfloat16().to(DEV)
        scale = torch.tensor([0.04], device=DEV)
        out = torch.empty(T, H, dtype=kind, device=DEV)
        rstd = torch.empty(T, device=DEV)
        if residual:
            crm.fused_add_rmsnorm_quant(out, x, r, w, scale, rstd=rstd)
            return [out, r, rstd]
        crm.rmsnorm_quant(out, x, w, scale, rstd=rstd)
        return [out, rstd]
    run_both(dbg, monkeypatch, case)


@pytest.mark.parametrize("T,H", [(37, 1024), (130, 4096)])
def test_block_fp8(dbg, monkeypatch, T, H):
    def case():
        g = _gen(5 * T + H)
        x = _rows(g, T, H)
        r = _rows(g, T, H).clone()
        w = (1 + 0.1 * torch.randn(H, generator=g)).bfloat16().to(DEV)
        ldT = (T + 3) // 4 * 4
        out = torch.empty(T, H, dtype=torch.float8_e4m3fn, device=DEV)
        bs = torch.zeros(H // 128, ldT, device=DEV)
        normed = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
        crm.fused_add_rmsnorm_fp8_block_quant(out, bs, normed, x, r, w)
        return [out, bs, normed, r]
    run_both(dbg, monkeypatch, case)


@pytest.mark.parametrize("T,D", [(37, 384), (40, 3072)])
@pytest.mark.parametrize("style_rows", ["per_row", "broadcast"])
@pytest.mark.parametrize("gated", [False, True])
def test_ada(dbg, monkeypatch, T, D, style_rows, gated):
    def case():
        g = _gen(7 * T + D)
        x = _rows(g, T, D)
        w = torch.ones(D, dtype=torch.bfloat16, device=DEV)
        S = T if style_rows == "per_row" else 1
        style = (0.1 * torch.randn(S, 3 * D, generator=g)).bfloat16().to(DEV)
        if not gated:
            out, gate_out = crm.ada_rms_norm_style(x, w, style)
            return [out, gate_out]
        gate = _rows(g, T, D)
        r = _rows(g, T, D).clone()
        scale = torch.tensor([0.05], device=DEV)
        r, out, gate_out = crm.gate_residual_ada_norm_fp8(r, x, gate, w, style, scale)
        return [out, gate_out, r]
    run_both(dbg, monkeypatch, case)


@pytest.mark.parametrize("T,H", [(100, 128), (37, 1024), (300, 2048)])
@pytest.mark.parametrize("fmt", ["bf16", "e4m3", "e4m3_scaled"])
def test_silu(dbg, monkeypatch, T, H, fmt):
    def case():
        g = _gen(11 * T + H)
        x = _rows(g, T, H)
        w = (1 + 0.1 * torch.randn(H, generator=g)).bfloat16().to(DEV)
        if fmt == "bf16":
            out = crm.fused_rmsnorm_silu(x, w)
        else:
            out = torch.empty(T, H, dtype=torch.float8_e4m3fn, device=DEV)
            scale = torch.tensor([0.5], device=DEV) if fmt == "e4m3_scaled" else None
            out = crm.fused_rmsnorm_silu(x, w, out=out, scale=scale)
        return [out if not isinstance(out, tuple) else out[0]]
    run_both(dbg, monkeypatch, case)


@pytest.mark.parametrize("T,H", [(100, 4096), (37, 16384), (33, 258)])
@pytest.mark.parametrize("fp8", [False, True])
def test_layernorm(dbg, monkeypatch, T, H, fp8):
    def case():
        g = _gen(13 * T + H)
        x = _rows(g, T, H, scale=3.0)
        gamma = (1 + 0.1 * torch.randn(H, generator=g)).to(DEV)
        beta = (0.1 * torch.randn(H, generator=g)).to(DEV)
        mean, rstd = torch.empty(T, device=DEV), torch.empty(T, device=DEV)
        if fp8:
            out = torch.empty(T, H, dtype=torch.float8_e4m3fn, device=DEV)
            crm.layernorm_quant(out, x, gamma, beta, torch.tensor([0.25], device=DEV), mean=mean, rstd=rstd)
        else:
            out = crm.layernorm(x, gamma, beta, mean=mean, rstd=rstd)
            out = out[0] if isinstance(out, tuple) else out
        return [out, mean, rstd]
    run_both(dbg, monkeypatch, case)


@pytest.mark.parametrize("T,H", [(1, 4096), (37, 128), (37, 1022), (300, 4096), (300, 5120),
                                 (2500, 4096), (2500, 128), (2049, 1024), (40, 16384), (2100, 11264)])
@pytest.mark.parametrize("route", ["bf16", "f32", "bf16_gres"])
def test_backward(dbg, monkeypatch, T, H, route):
    # Up to 2048 rows the column form (strip CTAs beside the chunks), above
    # it the chunk table, its partial rows and the reduction kernel; at
    # H = 16384 (and 11264 with g_residual) a BF16 weight is held as BF16.
    def case():
        g = _gen(17 * T + H)
        gr = _rows(g, T, H)
        x = _rows(g, T, H)
        gres = _rows(g, T, H) if route == "bf16_gres" else None
        w = 1 + 0.1 * torch.randn(H, generator=g)
        w = w.to(DEV) if route == "f32" else w.bfloat16().to(DEV)
        rstd = (0.5 + torch.rand(T, generator=g)).to(DEV)
        dx, dw = crm.rmsnorm_bwd(gr, x, w, rstd, 1.0 if route == "f32" else 0.0, g_residual=gres)
        dx2, dw2 = crm.rmsnorm_bwd_noalloc(gr, x, w, rstd, 1.0 if route == "f32" else 0.0, g_residual=gres)
        return [dx, dw, dx2, dw2]
    run_both(dbg, monkeypatch, case)


def test_guard_reports_and_skips(dbg, monkeypatch):
    """With the guard's view of y narrowed by 64 bytes, the stores of the
    last 32 elements are reported (kind 2, a store) and skipped: those keep
    their earlier contents and every other element equals the normal
    build's."""
    T, H = 64, 1024
    g = _gen(99)
    x = _rows(g, T, H)
    w = (1 + 0.1 * torch.randn(H, generator=g)).bfloat16().to(DEV)
    ref = crm.rmsnorm_fwd(x, w, 1e-6, want_rstd=False)[0]
    y = torch.full((T, H), 7.0, dtype=torch.bfloat16, device=DEV)
    with monkeypatch.context() as m:
        m.setattr(_abi, "_lib", dbg)
        m.setenv("CRMSN_DEBUG_TRIM_OUTPUT", "64")
        _word(dbg)
        crm.rmsnorm_fwd(x, w, 1e-6, y=y, want_rstd=False)
        w_ = _word(dbg)
    assert w_ >> 63 == 1, "the guard recorded nothing"
    assert (w_ >> 56) & 0x7f == 2, _describe(w_)
    flat, rflat = y.view(-1), ref.reshape(-1)
    assert torch.equal(flat[-32:], torch.full((32,), 7.0, dtype=torch.bfloat16, device=DEV))
    assert _same(flat[:-32], rflat[:-32])
    assert _word(dbg) == 0, "the record was not cleared"


def test_normal_build_has_no_guard():
    w = ctypes.c_uint64(5)
    st = _abi.load().crmsn_debug_status(ctypes.byref(w))
    assert _abi.STATUS[st] == "CRMSN_ERR_NOT_DEBUG_BUILD" and w.value == 0
