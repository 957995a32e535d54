"""Plain FP64 CPU oracle for the RMSNorm hot path -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package.  It wraps ``rmsnorm_oracle.c`` (a
single-threaded C library evaluated in double precision, written from the
pages' definitions) through ctypes and shares nothing with the CUDA library.

BF16 tensors are passed as numpy ``uint16`` bit patterns, FP8 as ``uint8``
codes, FP32 as ``float32``.  Every wrapper allocates its own outputs and
returns them in a dict.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rmsnorm_oracle.c")
_HDR = os.path.join(_HERE, "rmsnorm_oracle.h")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liborc_rmsnorm.so")
# -ffp-contract=off: no fused multiply-add contraction, so x86_64 and aarch64
# builds round identically.  No fast-math of any kind.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-Wall", "-Wextra"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/_build`` and return the path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(_SRC),
                                                   os.path.getmtime(_HDR))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def compile_variant(src_text: str, out_path: str) -> str:
    """Compile an edited copy of the oracle source (used by the mutation test)."""
    src = out_path + ".c"
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", *CFLAGS, "-I", _HERE, "-o", out_path, src, "-lm"],
                   check=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


_P = ctypes.c_void_p
_I = ctypes.c_int64
_F = ctypes.c_float
_D = ctypes.c_double
_INT = ctypes.c_int

_SIGS = {
    "orc_bf16_to_f64": (_D, [ctypes.c_uint16]),
    "orc_bf16_from_f64": (ctypes.c_uint16, [_D]),
    "orc_e4m3_to_f64": (_D, [ctypes.c_uint8]),
    "orc_e4m3_from_f32": (ctypes.c_uint8, [_F]),
    "orc_e5m2_to_f64": (_D, [ctypes.c_uint8]),
    "orc_e5m2_from_f32": (ctypes.c_uint8, [_F]),
    "orc_bf16_to_f64_n": (None, [_I, _P, _P]),
    "orc_bf16_from_f64_n": (None, [_I, _P, _P]),
    "orc_fp8_to_f64_n": (None, [_I, _INT, _P, _P]),
    "orc_fp8_from_f32_n": (None, [_I, _INT, _P, _P]),
    "orc_row_fwd_f64": (_D, [_I, _P, _P, _D, _P]),
    "orc_row_bwd_f64": (_D, [_I, _P, _P, _P, _D, _P, _P, _P]),
    "orc_weight_eff": (None, [_I, _P, _INT, _F, _P]),
    "orc_rmsnorm_fwd": (None, [_I, _I, _P, _I, _P, _I, _P, _INT, _F, _F,
                               _P, _P, _P, _P, _P]),
    "orc_rmsnorm_bwd": (None, [_I, _I, _P, _I, _P, _I, _P, _INT, _F, _P,
                               _P, _I, _P, _P, _P, _P, _P]),
    "orc_rmsnorm_quant": (None, [_I, _I, _P, _I, _P, _I, _P, _INT, _F, _F,
                                 _F, _INT, _P, _P, _P, _P]),
    "orc_fused_add_rmsnorm_fp8_block_quant": (None, [_I, _I, _P, _I, _P, _I,
                                                     _P, _F, _P, _P, _P, _P,
                                                     _I, _P]),
    "orc_ada_rms_norm_style": (None, [_I, _I, _P, _P, _P, _I, _F, _P, _P, _P]),
    "orc_gate_residual_ada_norm_fp8": (None, [_I, _I, _P, _P, _P, _P, _P, _I,
                                              _F, _F, _P, _P, _P, _P]),
    "orc_fused_rmsnorm_silu": (None, [_I, _I, _P, _I, _P, _INT, _F, _F, _INT, _F,
                                      _P, _P, _P, _P]),
    "orc_layernorm": (None, [_I, _I, _P, _I, _P, _P, _F, _INT, _INT, _F, _P, _P,
                             _P, _P, _P]),
}


def load_path(path: str) -> ctypes.CDLL:
    lib_ = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib_, name)
        fn.restype = res
        fn.argtypes = args
    return lib_


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            _lib = load_path(build())
        return _lib


# --------------------------------------------------------------------------
# numpy wrappers
# --------------------------------------------------------------------------

def _ptr(a):
    return None if a is None else a.ctypes.data


def _rows(a: np.ndarray, dtype) -> tuple[np.ndarray, int]:
    """Return (array, row stride in elements) for a 2-D row-strided view."""
    assert a.dtype == dtype, (a.dtype, dtype)
    assert a.ndim == 2
    item = a.itemsize
    if a.shape[1] > 1:
        assert a.strides[1] == item, "feature dimension must be contiguous"
    if a.shape[0] <= 1:
        return a, a.shape[1]
    assert a.strides[0] % item == 0
    return a, a.strides[0] // item


def _weight(w: np.ndarray):
    if w.dtype == np.float32:
        return np.ascontiguousarray(w), 1
    assert w.dtype == np.uint16
    return np.ascontiguousarray(w), 0


class Oracle:
    """Thin numpy front end over one loaded oracle library (the default build
    or a variant compiled from an edited source)."""

    def __init__(self, cdll: ctypes.CDLL | None = None):
        self.L = cdll if cdll is not None else lib()

    # -- formats -------------------------------------------------------------
    def bf16_from_f64(self, v) -> np.ndarray:
        v = np.ascontiguousarray(v, np.float64)
        out = np.empty(v.shape, np.uint16)
        self.L.orc_bf16_from_f64_n(v.size, _ptr(v), _ptr(out))
        return out

    def bf16_to_f64(self, b) -> np.ndarray:
        b = np.ascontiguousarray(b, np.uint16)
        out = np.empty(b.shape, np.float64)
        self.L.orc_bf16_to_f64_n(b.size, _ptr(b), _ptr(out))
        return out

    def fp8_from_f32(self, v, fp8_kind=0) -> np.ndarray:
        v = np.ascontiguousarray(v, np.float32)
        out = np.empty(v.shape, np.uint8)
        self.L.orc_fp8_from_f32_n(v.size, int(fp8_kind), _ptr(v), _ptr(out))
        return out

    def fp8_to_f64(self, c, fp8_kind=0) -> np.ndarray:
        c = np.ascontiguousarray(c, np.uint8)
        out = np.empty(c.shape, np.float64)
        self.L.orc_fp8_to_f64_n(c.size, int(fp8_kind), _ptr(c), _ptr(out))
        return out

    # -- row math in double -------------------------------------------------
    def row_fwd_f64(self, h, w_eff, eps):
        h = np.ascontiguousarray(h, np.float64)
        w_eff = np.ascontiguousarray(w_eff, np.float64)
        yv = np.empty_like(h)
        r = self.L.orc_row_fwd_f64(h.size, _ptr(h), _ptr(w_eff), float(eps), _ptr(yv))
        return yv, r

    def row_bwd_f64(self, g, h, w_eff, rstd, g_res=None):
        g = np.ascontiguousarray(g, np.float64)
        h = np.ascontiguousarray(h, np.float64)
        w_eff = np.ascontiguousarray(w_eff, np.float64)
        gr = None if g_res is None else np.ascontiguousarray(g_res, np.float64)
        dxv = np.empty_like(h)
        dwr = np.empty_like(h)
        m = self.L.orc_row_bwd_f64(h.size, _ptr(g), _ptr(h), _ptr(w_eff), float(rstd),
                                   _ptr(gr), _ptr(dxv), _ptr(dwr))
        return dxv, dwr, m

    def weight_eff(self, w, weight_bias=0.0):
        w, is32 = _weight(w)
        out = np.empty(w.size, np.float64)
        self.L.orc_weight_eff(w.size, _ptr(w), is32, float(weight_bias), _ptr(out))
        return out

    # -- operations -------------------------------------------------------------
    def rmsnorm_fwd(self, x, w, eps, residual=None, weight_bias=0.0, want_y=True):
        x, ldx = _rows(x, np.uint16)
        T, H = x.shape
        w, is32 = _weight(w)
        ldr = 0
        if residual is not None:
            residual, ldr = _rows(residual, np.uint16)
        y_exact = np.empty((T, H), np.float64) if want_y else None
        y = np.empty((T, H), np.uint16) if want_y else None
        rstd_exact = np.empty(T, np.float64)
        rstd32 = np.empty(T, np.float32)
        h_new = np.empty((T, H), np.uint16) if residual is not None else None
        self.L.orc_rmsnorm_fwd(T, H, _ptr(x), ldx, _ptr(residual), ldr, _ptr(w), is32,
                               float(weight_bias), float(eps), _ptr(y_exact), _ptr(y),
                               _ptr(rstd_exact), _ptr(rstd32), _ptr(h_new))
        return dict(y_exact=y_exact, y=y, rstd_exact=rstd_exact, rstd=rstd32, h_new=h_new)

    def rmsnorm_bwd(self, g, x, w, rstd, weight_bias=0.0, g_res=None, want_dx=True):
        g, ldg = _rows(g, np.uint16)
        x, ldx = _rows(x, np.uint16)
        T, H = x.shape
        w, is32 = _weight(w)
        rstd = np.ascontiguousarray(rstd, np.float32)
        ldgr = 0
        if g_res is not None:
            g_res, ldgr = _rows(g_res, np.uint16)
        dx_exact = np.empty((T, H), np.float64) if want_dx else None
        dx = np.empty((T, H), np.uint16) if want_dx else None
        m = np.empty(T, np.float64)
        dw = np.empty(H, np.float64)
        dw_abs = np.empty(H, np.float64)
        self.L.orc_rmsnorm_bwd(T, H, _ptr(g), ldg, _ptr(x), ldx, _ptr(w), is32,
                               float(weight_bias), _ptr(rstd), _ptr(g_res), ldgr,
                               _ptr(dx_exact), _ptr(dx), _ptr(m), _ptr(dw), _ptr(dw_abs))
        return dict(dx_exact=dx_exact, dx=dx, m=m, dw=dw, dw_abs=dw_abs)

    def rmsnorm_quant(self, x, w, scale, eps, residual=None, weight_bias=0.0, fp8_kind=0):
        x, ldx = _rows(x, np.uint16)
        T, H = x.shape
        w, is32 = _weight(w)
        ldr = 0
        if residual is not None:
            residual, ldr = _rows(residual, np.uint16)
        h_new = np.empty((T, H), np.uint16) if residual is not None else None
        v_exact = np.empty((T, H), np.float64)
        q = np.empty((T, H), np.uint8)
        rstd32 = np.empty(T, np.float32)
        self.L.orc_rmsnorm_quant(T, H, _ptr(x), ldx, _ptr(residual), ldr, _ptr(w), is32,
                                 float(weight_bias), float(scale), float(eps), int(fp8_kind),
                                 _ptr(h_new), _ptr(v_exact), _ptr(q), _ptr(rstd32))
        return dict(h_new=h_new, v_exact=v_exact, q=q, rstd=rstd32)

    def fused_add_rmsnorm_fp8_block_quant(self, x, residual, w, eps, ldT=None):
        x, ldx = _rows(x, np.uint16)
        residual, ldr = _rows(residual, np.uint16)
        T, H = x.shape
        assert H % 128 == 0
        w = np.ascontiguousarray(w, np.uint16)
        if ldT is None:
            ldT = (T + 3) // 4 * 4
        h_new = np.empty((T, H), np.uint16)
        normed_exact = np.empty((T, H), np.float64)
        normed = np.empty((T, H), np.uint16)
        block_scale = np.full((H // 128, ldT), np.nan, np.float32)
        q = np.empty((T, H), np.uint8)
        self.L.orc_fused_add_rmsnorm_fp8_block_quant(
            T, H, _ptr(x), ldx, _ptr(residual), ldr, _ptr(w), float(eps), _ptr(h_new),
            _ptr(normed_exact), _ptr(normed), _ptr(block_scale), ldT, _ptr(q))
        return dict(h_new=h_new, normed_exact=normed_exact, normed=normed,
                    block_scale=block_scale, q=q)

    def ada_rms_norm_style(self, x, w, style, eps):
        x = np.ascontiguousarray(x, np.uint16)
        style = np.ascontiguousarray(style, np.uint16)
        T, D = x.shape
        assert style.shape[1] == 3 * D and style.shape[0] in (1, T)
        w = np.ascontiguousarray(w, np.uint16)
        out_exact = np.empty((T, D), np.float64)
        out = np.empty((T, D), np.uint16)
        gate_out = np.empty((T, D), np.uint16)
        self.L.orc_ada_rms_norm_style(T, D, _ptr(x), _ptr(w), _ptr(style), style.shape[0],
                                      float(eps), _ptr(out_exact), _ptr(out), _ptr(gate_out))
        return dict(out_exact=out_exact, out=out, gate_out=gate_out)

    def gate_residual_ada_norm_fp8(self, residual, x, gate, w, style, scale, eps):
        residual = np.ascontiguousarray(residual, np.uint16)
        x = np.ascontiguousarray(x, np.uint16)
        gate = np.ascontiguousarray(gate, np.uint16)
        style = np.ascontiguousarray(style, np.uint16)
        T, D = x.shape
        assert style.shape[1] == 3 * D and style.shape[0] in (1, T)
        w = np.ascontiguousarray(w, np.uint16)
        residual_out = np.empty((T, D), np.uint16)
        v_exact = np.empty((T, D), np.float64)
        q = np.empty((T, D), np.uint8)
        gate_out = np.empty((T, D), np.uint16)
        self.L.orc_gate_residual_ada_norm_fp8(
            T, D, _ptr(residual), _ptr(x), _ptr(gate), _ptr(w), _ptr(style), style.shape[0],
            float(scale), float(eps), _ptr(residual_out), _ptr(v_exact), _ptr(q), _ptr(gate_out))
        return dict(residual_out=residual_out, v_exact=v_exact, q=q, gate_out=gate_out)


    def fused_rmsnorm_silu(self, x, w, eps, weight_bias=0.0, fp8=False, scale=1.0):
        x, ldx = _rows(x, np.uint16)
        T, H = x.shape
        w, is32 = _weight(w)
        v_exact = np.empty((T, H), np.float64)
        y = None if fp8 else np.empty((T, H), np.uint16)
        q = np.empty((T, H), np.uint8) if fp8 else None
        rstd32 = np.empty(T, np.float32)
        self.L.orc_fused_rmsnorm_silu(T, H, _ptr(x), ldx, _ptr(w), is32, float(weight_bias),
                                      float(eps), int(bool(fp8)), float(scale), _ptr(v_exact),
                                      _ptr(y), _ptr(q), _ptr(rstd32))
        return dict(v_exact=v_exact, y=y, q=q, rstd=rstd32)

    def layernorm(self, x, gamma, beta, eps, fp8_kind=None, scale=1.0):
        x, ldx = _rows(x, np.uint16)
        T, H = x.shape
        gamma = np.ascontiguousarray(gamma, np.float32)
        beta = np.ascontiguousarray(beta, np.float32)
        fp8 = fp8_kind is not None
        v_exact = np.empty((T, H), np.float64)
        y = None if fp8 else np.empty((T, H), np.uint16)
        q = np.empty((T, H), np.uint8) if fp8 else None
        mean = np.empty(T, np.float64)
        rstd = np.empty(T, np.float64)
        self.L.orc_layernorm(T, H, _ptr(x), ldx, _ptr(gamma), _ptr(beta), float(eps), int(fp8),
                             int(fp8_kind or 0), float(scale), _ptr(v_exact), _ptr(y), _ptr(q),
                             _ptr(mean), _ptr(rstd))
        return dict(v_exact=v_exact, y=y, q=q, mean=mean, rstd=rstd)

_default: Oracle | None = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle()
    return _default
