"""Host logic of the Python binding, without a GPU: how a tensor's layout
becomes (rows, H, row stride), and which layouts are refused."""
import pytest
import torch

from normalization_rmsnorm_fwd_gb300 import binding as B


def rows(t):
    return B.as_rows(t, "x")


def test_two_dimensional_rows():
    t = torch.zeros(7, 64)
    assert rows(t) == (7, 64, 64)
    assert rows(torch.zeros(7, 128)[:, :64]) == (7, 64, 128)        # row stride 128
    assert rows(torch.zeros(1, 64)) == (1, 64, 64)
    # One row: its stride is not meaningful and is reported as at least H.
    assert rows(torch.zeros(4, 256)[:1, :64]) == (1, 64, 256)
    assert rows(torch.zeros(1, 64).expand(1, 64)) == (1, 64, 64)


def test_leading_dimensions_collapse():
    assert rows(torch.zeros(2, 3, 5, 64)) == (30, 64, 64)
    # [T, heads, H] slice of a [T, heads, W] buffer: T*heads rows of stride W.
    buf = torch.zeros(6, 4, 256)
    assert rows(buf[:, :, :128]) == (24, 128, 256)
    # Size-1 leading dimensions impose nothing on their strides.
    assert rows(torch.zeros(5, 64)[None]) == (5, 64, 64)


def test_one_dimensional_row():
    assert rows(torch.zeros(64)) == (1, 64, 64)
    assert rows(torch.zeros(1)) == (1, 1, 1)


def test_refused_layouts():
    with pytest.raises(ValueError):
        rows(torch.zeros(64, 8).t())                                # features strided
    # Every second row of each block keeps one row stride (128): accepted.
    assert rows(torch.zeros(4, 6, 64)[:, ::2]) == (12, 64, 128)
    with pytest.raises(ValueError):
        rows(torch.zeros(4, 6, 64)[:, :3])                          # a gap after every 3 rows
    with pytest.raises(ValueError):
        rows(torch.zeros(6, 4, 64).transpose(0, 1))                 # leading dims out of order
    with pytest.raises(ValueError):
        rows(torch.zeros(()))                                       # no feature dimension


def test_operations_refuse_cpu_tensors():
    x = torch.zeros(4, 64, dtype=torch.bfloat16)
    w = torch.ones(64, dtype=torch.bfloat16)
    with pytest.raises(TypeError):
        B.rmsnorm_fwd(x, w)
    with pytest.raises(TypeError):
        B.rmsnorm_bwd(x, x, w, torch.ones(4))
    with pytest.raises(TypeError):
        B.layernorm(x, w.float(), w.float())
