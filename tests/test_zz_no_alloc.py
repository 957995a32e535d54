"""rmsnorm_bwd_noalloc: the backward for callers that cannot allocate.

Engines and plugin hosts that plan every device buffer in advance, and C
callers with no device allocator, cannot pass rmsnorm_bwd a workspace; this
entry point uses the library's built-in scratch instead.  The test calls it
through the C ABI twice in a row (different shapes) and requires dx and dw
to be bit-identical to rmsnorm_bwd with a caller-owned workspace on the same
inputs: both run the same kernels with the same chunk table.  Before each
call the scratch is filled with NaN partial rows by a wider call whose
gradient is NaN, so a partial row read before it was written would show.
The first problem is also checked against the oracle on every row.  A
width whose workspace exceeds the built-in scratch must be refused without
a launch (no width does on a 152-SM GB300).  This file
sorts last so that a run stopping at its first failure has already run
every other test.
"""
import numpy as np
import pytest
import torch

import gpu_util as gu
from normalization_rmsnorm_fwd_gb300 import _abi, synth

pytestmark = pytest.mark.gpu


def _dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _bits(t):
    return t.contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def _poison_scratch(L, stream):
    """A no-allocation call whose partial rows are all NaN, on a problem that
    uses more of the scratch than the problems below."""
    T, H = 4096, 5120
    g = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
    x = torch.ones((T, H), dtype=torch.bfloat16, device="cuda")
    w = torch.ones(H, dtype=torch.bfloat16, device="cuda")
    rstd = torch.ones(T, device="cuda")
    dx = torch.empty_like(x)
    dw = torch.empty(H, device="cuda")
    st = L.rmsnorm_bwd_noalloc(g.data_ptr(), H, x.data_ptr(), H, w.data_ptr(), 0, 0.0,
                               rstd.data_ptr(), None, 0, T, H, dx.data_ptr(), H, dw.data_ptr(),
                               stream)
    assert st == 0, _abi.STATUS[st]
    torch.cuda.synchronize()
    assert torch.isnan(dw).all(), "the poisoning call left finite partials"


def test_noalloc_backward_matches_rmsnorm_bwd(orc):
    L = _abi.load()
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream().cuda_stream
    # The first problem runs the chunked form (partial rows in the scratch),
    # the second the column form (no scratch).
    for seed, (T, H, gres) in enumerate([(3000, 4096, False), (333, 5120, True)]):
        g_b, x_b, r_b = synth.random_rows(100 + seed, T, H, n=3)
        w_b = synth.random_weight(100 + seed, H)
        g, x, w = _dev_bf16(g_b), _dev_bf16(x_b), _dev_bf16(w_b)
        gr = _dev_bf16(r_b) if gres else None
        rstd_h = np.abs(synth.Draw(seed).f32((T,), 0.1, 1.0))
        rstd = torch.from_numpy(rstd_h).cuda()
        # Existing entry point with a caller-owned workspace.
        nbytes = L.rmsnorm_bwd_workspace_bytes(T, H, 0, int(gres))
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        dx_ref = torch.empty_like(x)
        dw_ref = torch.empty(H, device="cuda")
        st = L.rmsnorm_bwd(g.data_ptr(), H, x.data_ptr(), H, w.data_ptr(), 0, 0.0, rstd.data_ptr(),
                           gr.data_ptr() if gres else None, H, T, H, dx_ref.data_ptr(), H,
                           dw_ref.data_ptr(), ws.data_ptr(), nbytes, stream)
        assert st == 0, _abi.STATUS[st]
        # The no-allocation entry point on the same inputs, its scratch full
        # of NaN partial rows from the call before.
        _poison_scratch(L, stream)
        dx = torch.full_like(x, float("nan"))
        dw = torch.full((H,), float("nan"), device="cuda")
        st = L.rmsnorm_bwd_noalloc(g.data_ptr(), H, x.data_ptr(), H, w.data_ptr(), 0, 0.0,
                                   rstd.data_ptr(), gr.data_ptr() if gres else None, H, T, H,
                                   dx.data_ptr(), H, dw.data_ptr(), stream)
        assert st == 0, _abi.STATUS[st]
        torch.cuda.synchronize()
        assert torch.equal(dx.view(torch.int16), dx_ref.view(torch.int16)), "dx differs from rmsnorm_bwd"
        assert torch.equal(dw.view(torch.int32), dw_ref.view(torch.int32)), "dw differs from rmsnorm_bwd"
        if seed == 0:
            ref = orc.rmsnorm_bwd(g_b, x_b, w_b, rstd_h)
            allow = gu.dx_allowance(g_b, x_b, orc.weight_eff(w_b), rstd_h, ref["m"])
            gu.check_bf16(_bits(dx), ref["dx_exact"], allowance=allow, what="dx vs oracle")
            gu.check_dw(dw.cpu().numpy(), ref["dw"], ref["dw_abs"], what="dw vs oracle")


def test_noalloc_scratch_limit_is_the_workspace_size():
    """Every width either runs (its workspace fits the 16 MiB scratch) or is
    refused with CRMSN_ERR_SCRATCH_LIMIT and no launch, exactly as
    rmsnorm_bwd_workspace_bytes says (on a 152-SM GB300 every width fits;
    GPUs with many more SMs need larger workspaces)."""
    L = _abi.load()
    torch.cuda.set_device(0)
    st = torch.cuda.current_stream().cuda_stream
    T = 4
    for H in (128, 4096, 8192, 9728, 12288, 16384):
        need = L.rmsnorm_bwd_workspace_bytes(T, H, 0, 0)
        t = torch.ones((T, H), dtype=torch.bfloat16, device="cuda")
        w = torch.ones(H, dtype=torch.bfloat16, device="cuda")
        rstd = torch.ones(T, device="cuda")
        dw = torch.full((H,), float("nan"), device="cuda")
        dx = torch.empty_like(t)
        s = L.rmsnorm_bwd_noalloc(t.data_ptr(), H, t.data_ptr(), H, w.data_ptr(), 0, 0.0,
                                  rstd.data_ptr(), None, 0, T, H, dx.data_ptr(), H, dw.data_ptr(), st)
        torch.cuda.synchronize()
        if need > 16 << 20:
            assert _abi.STATUS[s] == "CRMSN_ERR_SCRATCH_LIMIT", (H, need)
            assert torch.isnan(dw).all(), "a refused call launched"
        else:
            assert s == 0, (H, _abi.STATUS[s])
            assert torch.equal(dw, torch.full_like(dw, float(T))), H   # g = x = rstd = 1
