"""GB300-native (sm_103a) RMSNorm forward / backward library.

The computation lives in ``libcrmsnorm.so`` (hand-written CUDA behind the C
ABI of ``include/crmsnorm.h``); this package builds it (``build``) and binds
it (``binding``).  Importing the package does not load the library; the first
call does, and raises when the library has not been built.
"""
from .binding import (  # noqa: F401
    CrmsnError,
    ada_rms_norm_style,
    as_rows,
    fused_add_rmsnorm_fp8_block_quant,
    fused_add_rmsnorm_quant,
    fused_rmsnorm_silu,
    gate_residual_ada_norm_fp8,
    layernorm,
    layernorm_quant,
    rmsnorm_bwd,
    rmsnorm_bwd_noalloc,
    rmsnorm_bwd_workspace,
    rmsnorm_bwd_workspace_bytes,
    rmsnorm_fwd,
    rmsnorm_quant,
    rmsnorm_supports,
)
from .autograd import RMSNormFunction, rmsnorm  # noqa: F401,E402
