"""GPU AdaRMSNorm epilogues against the CPU oracle (per-row and broadcast
style; the gated residual + static FP8 path)."""
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


def ada_allowance(orc, x, w, style, eps):
    """2^-20 * (|yv * (1 + sc)| + |sh|) for the FP32 evaluation of the shift."""
    T, D = x.shape
    f = orc.rmsnorm_fwd(x, w, eps)
    st = np.broadcast_to(style, (T, 3 * D))
    sc = numfmt.decode_bf16(st[:, :D])
    sh = numfmt.decode_bf16(st[:, D:2 * D])
    return 2.0 ** -20 * (np.abs(f["y_exact"] * (1 + sc)) + np.abs(sh))


def compare_ada(orc, x, w, style, eps=1e-6):
    out, gate_out = crm.ada_rms_norm_style(gu.dev_bf16(x), gu.dev_bf16(w), gu.dev_bf16(style), eps)
    torch.cuda.synchronize()
    ref = orc.ada_rms_norm_style(x, w, style, eps)
    gu.check_bf16(gu.host_bits(out), ref["out_exact"], allowance=ada_allowance(orc, x, w, style, eps),
                  what="ada out")
    gu.check_exact(gu.host_bits(gate_out), ref["gate_out"], "gate_out")


def compare_gated(orc, u, x, gate, w, style, scale=0.04, eps=1e-6):
    ud = gu.dev_bf16(u)
    res, out, gate_out = crm.gate_residual_ada_norm_fp8(ud, gu.dev_bf16(x), gu.dev_bf16(gate),
                                                        gu.dev_bf16(w), gu.dev_bf16(style),
                                                        scale, eps)
    torch.cuda.synchronize()
    r_gpu, q_gpu, g_gpu = gu.host_bits(res), gu.host_u8(out), gu.host_bits(gate_out)
    ref = orc.gate_residual_ada_norm_fp8(u, x, gate, w, style, scale, eps)
    gu.check_exact(r_gpu, ref["residual_out"], "residual")
    gu.check_exact(g_gpu, ref["gate_out"], "gate_out")
    allow = ada_allowance(orc, ref["residual_out"], w, style, eps) / np.float32(scale)
    gu.check_fp8(q_gpu, ref["q"], ref["v_exact"], 0, "ada fp8", allowance=allow)


@pytest.mark.parametrize("D", [2, 6, 64, 250, 1024, 3072, 3070, 5120])
@pytest.mark.parametrize("broadcast", [False, True])
def test_ada_small(orc, D, broadcast):
    T = 29
    x = synth.random_rows(D, T, D)[0]
    style = synth.random_rows(D + 1, 1 if broadcast else T, 3 * D)[0]
    w = synth.random_weight(D, D)
    compare_ada(orc, x, w, style)


@pytest.mark.parametrize("D", [2, 64, 250, 3072, 3070])
@pytest.mark.parametrize("broadcast", [False, True])
def test_gated_small(orc, D, broadcast):
    T = 29
    u, x, g = synth.random_rows(D + 2, T, D, n=3)
    style = synth.random_rows(D + 3, 1 if broadcast else T, 3 * D)[0]
    w = synth.random_weight(D, D)
    compare_gated(orc, u, x, g, w, style)


@pytest.mark.parametrize("broadcast", [False, True])
def test_ada_config(orc, broadcast):
    """rows = 2520, dim = 3072, w = 1, style (rows, 3*dim) or (1, 3*dim)."""
    d = synth.ada()
    style = d["style1"] if broadcast else d["style"]
    compare_ada(orc, d["x"], d["w"], style, d["eps"])


@pytest.mark.parametrize("broadcast", [False, True])
def test_gated_config(orc, broadcast):
    d = synth.ada()
    style = d["style1"] if broadcast else d["style"]
    compare_gated(orc, d["residual"], d["x"], d["gate"], d["w"], style, d["scale"], d["eps"])


def test_broadcast_equals_repeated_style():
    d = synth.ada(T=64, D=1024)
    x, w = gu.dev_bf16(d["x"]), gu.dev_bf16(d["w"])
    a = crm.ada_rms_norm_style(x, w, gu.dev_bf16(d["style1"]))
    b = crm.ada_rms_norm_style(x, w, gu.dev_bf16(np.repeat(d["style1"], 64, axis=0)))
    torch.cuda.synchronize()
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1].view(torch.int16), b[1].view(torch.int16))
