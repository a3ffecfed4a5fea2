"""Canary guards for the outputs of GPU calls (a stand-in for a device memory checker, which this
test suite cannot rely on): an output tensor is carved out of a larger buffer whose leading and
trailing guard regions hold a known bit pattern -- NaN for floating-point outputs, a sentinel for
integer ones.  A kernel that writes past either end of its output lands in a guard, and
``check`` compares the guards with the pattern bit for bit after the call."""
from __future__ import annotations

import math

import torch

GUARD_ELEMS = 4096          # per side; a multiple of 8 elements keeps every view 16-byte aligned
INT_SENTINEL = -0x2B2B2B2B

_BITS = {torch.bfloat16: torch.int16, torch.float16: torch.int16, torch.float32: torch.int32,
         torch.int32: torch.int32}


class Guarded:
    """``t`` is a contiguous tensor of ``shape`` between two guard regions of one allocation."""

    def __init__(self, shape, dtype, device, guard: int = GUARD_ELEMS):
        n = math.prod(shape)
        fill = INT_SENTINEL if dtype == torch.int32 else float("nan")
        self.buf = torch.full((n + 2 * guard,), fill, dtype=dtype, device=device)
        self.guard, self.n = guard, n
        self.t = self.buf[guard:guard + n].view(shape)
        self.pattern = self.buf[:1].clone()

    def check(self, what: str = "output") -> None:
        bits = _BITS[self.buf.dtype]
        want = self.pattern.view(bits)
        for name, region in (("leading", self.buf[:self.guard]), ("trailing", self.buf[self.guard + self.n:])):
            bad = (region.view(bits) != want).nonzero()
            assert bad.numel() == 0, (f"{what}: {bad.numel()} {name} guard elements overwritten "
                                      f"(first at offset {int(bad[0])})")


def guarded(shape, dtype, device):
    return Guarded(tuple(shape), dtype, device)


def check_all(guards, what: str = "output") -> None:
    for i, g in enumerate(guards):
        g.check(f"{what}[{i}]")
