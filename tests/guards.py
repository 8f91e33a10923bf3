"""Canary guard bands around device output buffers: a stand-in for a device memory checker.

Every output a guarded test passes to libfq is carved out of a larger device allocation. GUARD bytes
before and GUARD bytes after it hold a fixed byte pattern, and `check()` confirms after the call that
none of them changed. That catches a stray store past a ragged last stage, a row written past the end
of the tensor, a wrong token stride or a workspace overrun. It does not catch a store that lands
further away than the band. The output itself starts 256-byte aligned, as a fresh torch allocation
does, so the call takes the same kernels it takes on an ordinary tensor.
"""
from __future__ import annotations

import torch

GUARD = 256       # bytes on each side (a multiple of 256: keeps the output's own alignment)
PATTERN = 0xA5


class Guarded:
    """A device tensor of `shape` and `dtype` with guard bands on both sides."""

    def __init__(self, shape, dtype, device="cuda", fill=None):
        shape = tuple(int(s) for s in shape)
        numel = 1
        for s in shape:
            numel *= s
        self.nbytes = numel * torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((2 * GUARD + self.nbytes,), PATTERN, dtype=torch.uint8, device=device)
        self.t = self.buf[GUARD:GUARD + self.nbytes].view(dtype).view(shape)
        if fill is not None and numel:
            self.t.fill_(fill)

    def check(self, what: str = "output"):
        """Assert that the bytes before and after the tensor still hold the pattern."""
        torch.cuda.synchronize()
        b = self.buf.cpu()
        head = (b[:GUARD] != PATTERN).nonzero().flatten()
        tail = (b[GUARD + self.nbytes:] != PATTERN).nonzero().flatten()
        assert head.numel() == 0, (
            f"{what}: {head.numel()} guard bytes before the tensor were written (nearest at offset "
            f"{int(head.max()) - GUARD})")
        assert tail.numel() == 0, (
            f"{what}: {tail.numel()} guard bytes after the tensor were written (first at +{int(tail.min())} "
            f"past its end)")


def check_all(**outs: Guarded):
    for name, g in outs.items():
        if g is not None:
            g.check(name)
