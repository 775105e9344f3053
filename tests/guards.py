"""Poisoned, guarded output buffers for the GPU parity tests.

Every output a test hands to the library is the middle of a larger buffer: 256 canary bytes
(0xA5) on each side catch writes past either end, and the output itself starts poisoned, so
an element the kernel never writes fails the comparison with the oracle instead of passing
on memory a previous call left behind.  Poison: NaN for floating-point outputs, 0x7F (the
E4M3 NaN code, never produced by a saturating conversion) for code bytes, 0xFF (the E8M0 NaN
code; scales are clamped to 0..254) for scale bytes.  Buffers the library accumulates into
(dprob) start at zero instead.
"""
from __future__ import annotations

import math

import torch

PAD_BYTES = 256
CANARY = 0xA5


class Guarded:
    def __init__(self, shape, dtype, fill, device="cuda"):
        shape = tuple(int(s) for s in shape)
        es = torch.empty((), dtype=dtype).element_size()
        n = math.prod(shape)
        self.pad = PAD_BYTES // es
        self.buf = torch.empty(n + 2 * self.pad, dtype=dtype, device=device)
        self.buf.view(torch.uint8).fill_(CANARY)
        self.view = self.buf[self.pad:self.pad + n].view(shape)
        self.view.fill_(fill)

    def intact(self) -> bool:
        raw = self.buf.view(torch.uint8)
        pb = self.pad * self.buf.element_size()
        return bool(torch.all(raw[:pb] == CANARY)) and bool(torch.all(raw[-pb:] == CANARY))


class Outputs:
    """A set of guarded outputs; ``check()`` asserts every canary is intact."""

    def __init__(self):
        self._all = {}

    def float(self, name, shape, dtype):
        g = Guarded(shape, dtype, float("nan"))
        self._all[name] = g
        return g.view

    def codes(self, name, shape):
        g = Guarded(shape, torch.uint8, 0x7F)
        self._all[name] = g
        return g.view

    def scales(self, name, shape):
        g = Guarded(shape if isinstance(shape, tuple) else (shape,), torch.uint8, 0xFF)
        self._all[name] = g
        return g.view

    def zeros(self, name, shape, dtype=torch.float32):
        g = Guarded(shape, dtype, 0)
        self._all[name] = g
        return g.view

    def check(self):
        bad = [k for k, g in self._all.items() if not g.intact()]
        assert not bad, f"writes outside the output buffers: {bad}"
