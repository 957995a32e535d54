"""ctypes view of ``libcrmsnorm.so`` (the C ABI of ``include/crmsnorm.h``).

The library is built in-tree by ``build.py``; loading fails loudly when it is
missing -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading


_P = ctypes.c_void_p
_I = ctypes.c_int64
_F = ctypes.c_float
_INT = ctypes.c_int
_ST = ctypes.c_int

# name -> (restype, argtypes); mirrors include/crmsnorm.h
SIGNATURES = {
    "rmsnorm_fwd": (_ST, [_P, _I, _P, _I, _P, _INT, _F, _F, _I, _I, _P, _I, _P, _P, _I, _P]),
    "rmsnorm_bwd": (_ST, [_P, _I, _P, _I, _P, _INT, _F, _P, _P, _I, _I, _I, _P, _I, _P, _P,
                          ctypes.c_size_t, _P]),
    "rmsnorm_bwd_workspace_bytes": (ctypes.c_size_t, [_I, _I, _INT, _INT]),
    "rmsnorm_bwd_noalloc": (_ST, [_P, _I, _P, _I, _P, _INT, _F, _P, _P, _I, _I, _I, _P, _I, _P, _P]),
    "fused_add_rmsnorm_quant": (_ST, [_P, _I, _INT, _P, _I, _P, _I, _P, _INT, _F, _P, _F, _I, _I,
                                      _P, _P]),
    "fused_add_rmsnorm_fp8_block_quant": (_ST, [_P, _P, _I, _P, _P, _I, _P, _I, _P, _F, _I, _I,
                                                _P]),
    "ada_rms_norm_style": (_ST, [_P, _P, _P, _I, _F, _I, _I, _P, _P, _P]),
    "gate_residual_ada_norm_fp8": (_ST, [_P, _P, _P, _P, _P, _I, _P, _F, _I, _I, _P, _P, _P]),
    "rmsnorm_supports": (_ST, [_I, _INT, _INT]),
    "crmsn_status_str": (ctypes.c_char_p, [_ST]),
    "fused_rmsnorm_silu": (_ST, [_P, _I, _INT, _P, _I, _P, _INT, _F, _P, _F, _I, _I, _P, _P]),
    "layernorm": (_ST, [_P, _I, _P, _I, _P, _P, _F, _I, _I, _P, _P, _P]),
    "layernorm_quant": (_ST, [_P, _I, _INT, _P, _I, _P, _P, _P, _F, _I, _I, _P, _P, _P]),
    "crmsn_debug_status": (_ST, [ctypes.POINTER(ctypes.c_uint64)]),
}

STATUS = {
    0: "CRMSN_OK", 1: "CRMSN_ERR_NULL", 2: "CRMSN_ERR_SHAPE", 3: "CRMSN_ERR_UNSUPPORTED_H",
    4: "CRMSN_ERR_ALIGNMENT", 5: "CRMSN_ERR_DTYPE", 6: "CRMSN_ERR_WORKSPACE",
    7: "CRMSN_ERR_ALIAS", 8: "CRMSN_ERR_CUDA", 9: "CRMSN_ERR_DEVICE_TIMEOUT", 10: "CRMSN_ERR_ARG",
    11: "CRMSN_ERR_SCRATCH_LIMIT", 12: "CRMSN_ERR_NOT_DEBUG_BUILD",
}
OK = 0
BF16, F32 = 0, 1
E4M3, E5M2 = 0, 1
OP_FWD, OP_BWD, OP_QUANT, OP_BLOCK_QUANT, OP_ADA_STYLE, OP_GATED_ADA_FP8, OP_SILU, OP_LAYERNORM = range(8)
OUT_BF16, OUT_E4M3 = 0, 1
MAX_H = 16384

_lock = threading.Lock()
_lib = None


class CrmsnError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn}: {STATUS.get(status, status)} ({text})")
        self.status = status


_LIB = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libcrmsnorm.so")


def library_path() -> str:
    return _LIB


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (once) and return the CUDA library; raise if it was never built."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    with _lock:
        if _lib is None or path is not None:
            p = path or _LIB
            if not os.path.exists(p):
                raise RuntimeError(
                    f"libcrmsnorm.so not found at {p}: build it with "
                    "`python -m normalization_rmsnorm_fwd_gb300.build` (needs nvcc)")
            lib = ctypes.CDLL(p)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            if path is not None:
                return lib
            _lib = lib
        return _lib


def check(fn: str, status: int) -> None:
    if status != OK:
        raise CrmsnError(fn, status, load().crmsn_status_str(status).decode())
