"""Host logic of the autograd wrapper, without a GPU: which layouts are
passed to the kernels in place and which are copied once, and that CPU
tensors are refused loudly (there is no CPU path)."""
import pytest
import torch

from normalization_rmsnorm_fwd_gb300 import autograd as ag
import normalization_rmsnorm_fwd_gb300 as crm


def test_readable_layouts():
    base = torch.zeros(8, 64, dtype=torch.bfloat16)
    assert ag._readable(base) is base                              # contiguous rows
    assert ag._readable(base.view(2, 4, 64)) is not None
    strided = torch.zeros(8, 128, dtype=torch.bfloat16)[:, :64]    # row stride 128
    assert ag._readable(strided) is strided
    expanded = torch.ones(1, 64, dtype=torch.bfloat16).expand(8, 64)   # row stride 0
    out = ag._readable(expanded)
    assert out is not expanded and out.is_contiguous()
    transposed = torch.zeros(64, 8, dtype=torch.bfloat16).t()       # features strided
    assert ag._readable(transposed).is_contiguous()
    odd = torch.zeros(8 * 64 + 1, dtype=torch.bfloat16)[1:].view(8, 64)   # 2-byte offset
    assert ag._readable(odd) is not odd


def test_cpu_tensors_are_refused():
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    w = torch.ones(64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        crm.rmsnorm(x, w)
