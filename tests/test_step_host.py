"""Host-side logic of the step driver that needs no GPU."""

import numpy as np
import torch

from context_paged_attention_gb300.step import pack_tensors


def test_pack_tensors_views_alignment_and_contents():
    rng = np.random.default_rng(0)
    ts = [
        torch.tensor(rng.standard_normal((3, 5, 7)), dtype=torch.bfloat16),
        torch.tensor(rng.integers(-9, 9, size=13), dtype=torch.int32),
        torch.empty((0,), dtype=torch.int32),
        torch.tensor(rng.standard_normal((2, 3)), dtype=torch.float32),
        torch.tensor(rng.integers(0, 5, size=1), dtype=torch.int32),
    ]
    buf, views = pack_tensors(ts, "cpu")
    assert buf.dtype == torch.uint8 and buf.dim() == 1
    base = buf.data_ptr()
    prev_end = 0
    for t, v in zip(ts, views):
        assert v.dtype == t.dtype and v.shape == t.shape and v.is_contiguous()
        assert torch.equal(v, t)
        if v.numel() == 0:
            continue  # an empty view has no storage address to check
        off = v.data_ptr() - base
        assert off % 256 == 0 and off >= prev_end  # aligned, in order, no overlap
        prev_end = off + v.numel() * v.element_size()
        assert prev_end <= buf.numel()
    # the views alias the buffer: writing the buffer changes them (one copy feeds them all)
    snapshot = buf.clone()
    buf.zero_()
    assert all(int(v.float().abs().sum()) == 0 for v in views if v.numel())
    buf.copy_(snapshot)
    assert all(torch.equal(v, t) for t, v in zip(ts, views))


def test_pack_tensors_empty_list():
    buf, views = pack_tensors([], "cpu")
    assert views == [] and buf.numel() >= 1
