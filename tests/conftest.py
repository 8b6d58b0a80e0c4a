import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    try:
        import torch

        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this environment")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


class GuardedAllocator:
    """Output buffers with guard bands: each allocation is one byte buffer of
    guard | output (rounded up to 256 bytes) | guard, every byte set to a
    sentinel first.  After the test every guard byte must still hold it, so a
    kernel that writes past either end of an output (a tail tile, a
    transposed store, a TMA store, a partial-sum slot) fails the test even
    when the output itself compares equal.  The sentinel also poisons the
    output: an element the library never writes shows up in the parity
    comparison."""

    SENTINEL = 0xA5
    GUARD = 1 << 19  # 512 KB before and after every output

    def __init__(self):
        self.bufs = []

    def __call__(self, shape, dtype, device):
        import torch

        n = 1
        for d in shape:
            n *= int(d)
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        padded = (nbytes + 255) // 256 * 256
        raw = torch.full((2 * self.GUARD + padded,), self.SENTINEL, dtype=torch.uint8, device=device)
        self.bufs.append((raw, nbytes))
        return raw[self.GUARD:self.GUARD + nbytes].view(dtype).view(shape)

    def check(self):
        import torch

        if torch.cuda.is_available():
            torch.cuda.synchronize()
        bad = []
        for raw, nbytes in self.bufs:
            head, tail = raw[:self.GUARD], raw[self.GUARD + nbytes:]
            for name, g in (("before", head), ("after", tail)):
                hit = torch.nonzero(g != self.SENTINEL)
                if hit.numel():
                    bad.append(f"{int(hit.numel())} guard bytes {name} an output of {nbytes} bytes were written "
                               f"(first at offset {int(hit[0])})")
        self.bufs.clear()
        return bad


@pytest.fixture(autouse=True)
def _guard_outputs(request):
    """Every GPU test allocates the library's outputs through GuardedAllocator
    and checks the guards when it ends."""
    if "gpu" not in request.node.keywords:
        yield
        return
    import torch

    if not torch.cuda.is_available():
        yield
        return
    import prefix_tree_block_gb300 as pt

    guard = GuardedAllocator()
    pt.set_output_allocator(guard)
    try:
        yield
    finally:
        pt.set_output_allocator(None)
    bad = guard.check()
    assert not bad, "; ".join(bad)
