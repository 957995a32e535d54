"""The C ABI without a GPU: the library loads, exports every function that
include/crmsnorm.h declares, and rejects invalid arguments on the host before
any CUDA call (fake device addresses are never dereferenced)."""
import os
import re
import subprocess

import pytest

from normalization_rmsnorm_fwd_gb300 import _abi
from normalization_rmsnorm_fwd_gb300 import build as nbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]

OK, NULL, SHAPE, UNSUP, ALIGN, DTYPE, WS, ALIAS, CUDA, TIMEOUT, ARG, SCRATCH = range(12)
A = 1 << 40            # a fake, 256-byte aligned device address (never dereferenced)
MB = 1 << 20


@pytest.fixture(scope="module")
def L():
    nbuild.build()
    return _abi.load()


def declared_functions():
    names = []
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(\w+)\s*\([^;]*\)\s*;", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(L):
    names = declared_functions()
    assert "rmsnorm_fwd" in names and "crmsn_status_str" in names and len(names) >= 9
    out = subprocess.run(["nm", "-D", "--defined-only", _abi.library_path()],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r" T (\w+)$", out, flags=re.M))
    for n in names:
        assert n in exported, f"{n} declared in include/ but not exported"
        assert n in _abi.SIGNATURES, f"{n} missing from the Python binding"
        getattr(L, n)


def test_status_strings(L):
    for s in range(12):
        assert L.crmsn_status_str(s)
    assert L.crmsn_status_str(99) == b"unknown status"


def fwd(L, **kw):
    a = dict(x=A, ldx=256, residual=None, ldr=0, w=A + 64 * MB, w_dtype=0, bias=0.0, eps=1e-6,
             T=4, H=256, y=A + 128 * MB, ldy=256, rstd=None, h_new=None, ldh=0, stream=None)
    a.update(kw)
    return L.rmsnorm_fwd(a["x"], a["ldx"], a["residual"], a["ldr"], a["w"], a["w_dtype"],
                         a["bias"], a["eps"], a["T"], a["H"], a["y"], a["ldy"], a["rstd"],
                         a["h_new"], a["ldh"], a["stream"])


def test_fwd_validation(L):
    assert fwd(L, T=-1) == SHAPE
    assert fwd(L, H=0) == SHAPE
    assert fwd(L, H=255) == UNSUP
    assert fwd(L, H=16386, ldx=16386, ldy=16386) == UNSUP
    assert fwd(L, w_dtype=7) == DTYPE
    assert fwd(L, x=None) == NULL
    assert fwd(L, y=None) == NULL
    assert fwd(L, residual=A + 256 * MB, ldr=256) == NULL          # residual without h_new
    assert fwd(L, eps=float("nan")) == ARG
    assert fwd(L, eps=-1.0) == ARG
    assert fwd(L, ldx=100) == SHAPE
    assert fwd(L, T=0) == OK                                        # no launch, no CUDA call
    assert fwd(L, T=0, x=None, y=None) == OK                        # empty tensors: NULL data
    assert fwd(L, x=A + 1) == ALIGN                                 # not even 4-byte aligned
    assert fwd(L, ldx=257) == ALIGN                                 # odd row stride


def test_fwd_alias_rules(L):
    # y overlapping the residual input, or the weight: rejected.
    assert fwd(L, residual=A + 256 * MB, ldr=256, h_new=A + 512 * MB, ldh=256,
               y=A + 256 * MB + 64) == ALIAS
    assert fwd(L, y=A + 64 * MB) == ALIAS
    # y == x with the same stride (in place) passes validation: without a GPU
    # the launch itself is what fails.
    assert fwd(L, y=A, ldy=256) == CUDA
    # h_new == residual in place passes; h_new == x does not.
    assert fwd(L, residual=A + 256 * MB, ldr=256, h_new=A + 256 * MB, ldh=256) == CUDA
    assert fwd(L, residual=A + 256 * MB, ldr=256, h_new=A, ldh=256) == ALIAS
    # Interleaved column slices of one buffer (row period 512) are disjoint.
    assert fwd(L, ldx=512, y=A + 512, ldy=512) == CUDA
    assert fwd(L, ldx=512, y=A + 256, ldy=512) == ALIAS
    # rstd inside x.
    assert fwd(L, rstd=A + 16) == ALIAS


def test_fwd_unaligned_fallback_passes_validation(L):
    # 4-byte aligned but not 16-byte aligned: the 4-byte path is chosen.
    assert fwd(L, x=A + 4, y=A + 128 * MB + 4) == CUDA
    assert fwd(L, H=250, ldx=250, ldy=250) == CUDA


def test_other_entry_points_validation(L):
    # fused_add_rmsnorm_quant
    q = lambda **kw: L.fused_add_rmsnorm_quant(
        kw.get("out", A), kw.get("ldo", 256), kw.get("kind", 0), kw.get("x", A + 64 * MB), 256,
        kw.get("res", A + 128 * MB), 256, A + 192 * MB, kw.get("wd", 0), 0.0,
        kw.get("scale", A + 200 * MB), 1e-6, 4, kw.get("H", 256), None, None)
    assert q(kind=3) == DTYPE
    assert q(scale=None) == NULL
    assert q(H=255) == UNSUP
    assert q(res=A + 64 * MB) == ALIAS
    assert q() == CUDA
    # block quant: H must be a multiple of 128; ldT >= T
    b = lambda **kw: L.fused_add_rmsnorm_fp8_block_quant(
        A, A + 64 * MB, kw.get("ldT", 4), A + 128 * MB, A + 192 * MB, kw.get("H", 256),
        A + 256 * MB, kw.get("H", 256), A + 320 * MB, 1e-6, 4, kw.get("H", 256), None)
    assert b(H=200) == UNSUP
    assert b(ldT=3) == SHAPE
    assert b() == CUDA
    # ada: odd D, bad style_rows
    ada = lambda **kw: L.ada_rms_norm_style(A, A + 64 * MB, A + 128 * MB, kw.get("sr", 4), 1e-6,
                                            4, kw.get("D", 256), A + 192 * MB, A + 256 * MB,
                                            None)
    assert ada(D=255) == SHAPE
    assert ada(sr=3) == SHAPE
    assert ada() == CUDA
    assert ada(sr=1) == CUDA
    gated = L.gate_residual_ada_norm_fp8(A, A + 64 * MB, None, A + 128 * MB, A + 192 * MB, 4,
                                         A + 256 * MB, 1e-6, 4, 256, A + 320 * MB, A + 384 * MB,
                                         None)
    assert gated == NULL
    # backward: required pointers
    bw = L.rmsnorm_bwd(A, 256, A + 64 * MB, 256, A + 128 * MB, 0, 0.0, None, None, 0, 4, 256,
                       A + 192 * MB, 256, A + 256 * MB, A + 320 * MB, 1 << 20, None)
    assert bw == NULL


def test_supports(L):
    assert L.rmsnorm_supports(4096, 0, 0) == OK
    assert L.rmsnorm_supports(5120, 1, 1) == OK
    assert L.rmsnorm_supports(4097, 0, 0) == UNSUP
    assert L.rmsnorm_supports(4096, 2, 0) == DTYPE
    assert L.rmsnorm_supports(8192, 0, 3) == OK
    assert L.rmsnorm_supports(200, 0, 3) == UNSUP
    assert L.rmsnorm_supports(8192, 1, 3) == DTYPE
    assert L.rmsnorm_supports(3072, 0, 5) == OK
    assert L.rmsnorm_supports(3071, 0, 4) == SHAPE
    assert L.rmsnorm_supports(3072, 0, 9) == ARG


def test_silu_and_layernorm_validation(L):
    silu = lambda **kw: L.fused_rmsnorm_silu(
        kw.get("out", A), 256, kw.get("fmt", 0), kw.get("x", A + 64 * MB), 256, A + 128 * MB,
        kw.get("wd", 0), 0.0, kw.get("scale", None), 1e-6, 4, kw.get("H", 256), None, None)
    assert silu(fmt=2) == DTYPE
    assert silu(wd=3) == DTYPE
    assert silu(H=255) == UNSUP
    assert silu(out=A + 64 * MB + 2) == ALIAS        # partial overlap with x
    assert silu(out=A + 64 * MB) == CUDA             # in place over x is allowed
    assert silu(fmt=1, out=A + 64 * MB) == ALIAS     # an FP8 out cannot replace x
    assert silu(fmt=1) == CUDA                       # no scale: the plain cast
    assert silu(x=None) == NULL
    ln = lambda **kw: L.layernorm(
        kw.get("y", A), 256, kw.get("x", A + 64 * MB), 256, kw.get("g", A + 128 * MB),
        kw.get("b", A + 129 * MB), kw.get("eps", 1e-5), 4, kw.get("H", 256), None, None, None)
    assert ln(b=None) == NULL
    assert ln(eps=-1.0) == ARG
    assert ln(H=0) == SHAPE
    assert ln(g=A + 128 * MB + 4) == ALIGN           # 4-byte aligned: the 8-element path
    assert ln(g=A + 128 * MB + 2) == ALIGN
    assert ln(y=A + 64 * MB) == CUDA
    assert ln() == CUDA
    lq = lambda **kw: L.layernorm_quant(
        A, 256, kw.get("kind", 0), A + 64 * MB, 256, A + 128 * MB, A + 129 * MB,
        kw.get("scale", A + 130 * MB), 1e-5, 4, 256, None, None, None)
    assert lq(kind=2) == DTYPE
    assert lq(scale=None) == NULL
    assert lq(kind=1) == CUDA
    assert L.rmsnorm_supports(1024, 0, 6) == OK
    assert L.rmsnorm_supports(1024, 1, 7) == OK
    assert L.rmsnorm_supports(1024, 0, 7) == DTYPE
