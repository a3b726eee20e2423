"""The guard-region helper used by the GPU out-of-bounds tests, checked on
the CPU: writes inside the tensor leave the guards intact, a write one byte
past either end is seen, and the tensor keeps the alignment the library
requires."""

import pytest
import torch

from tests.guard import LEAD, Guarded


@pytest.mark.parametrize("dtype", [torch.uint8, torch.bfloat16, torch.float32, torch.int32])
def test_guards_see_writes_past_either_end(dtype):
    g = Guarded((7, 24), dtype, "cpu")
    assert g.t.shape == (7, 24) and g.t.dtype == dtype
    assert g.t.data_ptr() % 16 == 0 and g.t.is_contiguous()
    g.t.fill_(3)
    assert g.intact() and g.first_overwrite() is None
    g.raw[LEAD + g.nbytes] = 0
    assert not g.intact() and g.first_overwrite() == g.nbytes
    g2 = Guarded((7, 24), dtype, "cpu")
    g2.raw[LEAD - 1] = 0
    assert not g2.intact() and g2.first_overwrite() == -1


def test_empty_and_filled_tensors():
    g = Guarded((0, 128), torch.bfloat16, "cpu")
    assert g.t.numel() == 0 and g.intact()
    src = torch.arange(12, dtype=torch.float32).view(3, 4)
    g = Guarded((3, 4), torch.float32, "cpu", fill=src)
    assert torch.equal(g.t, src) and g.intact()
