"""The guard-band allocator the GPU tests route every library output
through (tests/conftest.py), checked on the CPU: it returns a view of the
requested shape inside a larger buffer, poisons it, and reports any byte
written before or after it."""
import torch

from conftest import GuardedAllocator


def test_writes_inside_the_output_pass():
    g = GuardedAllocator()
    x = g((3, 5, 7), torch.bfloat16, "cpu")
    assert x.shape == (3, 5, 7) and x.is_contiguous()
    assert torch.all(x.view(torch.uint8) == GuardedAllocator.SENTINEL)  # poisoned
    x.fill_(1.5)
    assert g.check() == []


def test_a_write_past_either_end_is_reported():
    for where in ("before", "after"):
        g = GuardedAllocator()
        x = g((10, 3), torch.float32, "cpu")
        raw, nbytes = g.bufs[0]
        off = GuardedAllocator.GUARD - 1 if where == "before" else GuardedAllocator.GUARD + nbytes + 100
        raw[off] = 0
        x.zero_()
        bad = g.check()
        assert len(bad) == 1 and where in bad[0]


def test_the_padding_after_an_odd_size_is_guarded():
    g = GuardedAllocator()
    x = g((7,), torch.bfloat16, "cpu")  # 14 bytes; the rest of its 256 belongs to the tail guard
    raw, nbytes = g.bufs[0]
    raw[GuardedAllocator.GUARD + nbytes] = 0
    assert len(g.check()) == 1
