"""Guard bytes around device outputs: a stand-in for a memory checker.

Every output a parity test hands to the library (Y, acc_out, Xq_out, sa_out,
P) and every workspace lives inside a larger allocation whose first and last
GUARD bytes hold a fixed pattern.  After the call the test asserts that the
pattern is intact, so a kernel that writes past the end (or before the start)
of an output is caught even when the values it was meant to write are right.
"""
from __future__ import annotations

import numpy as np
import torch

GUARD = 4096        # bytes on each side; keeps every view 4096-byte aligned
PATTERN = 0xA5      # guard byte
WS_FILL = 0x00      # workspaces start zeroed, as the C header requires


class Guarded:
    """A contiguous tensor of `shape`/`dtype` with guard bytes on both sides."""

    def __init__(self, shape, dtype, device="cuda", fill=None):
        self.shape = tuple(int(s) for s in shape)
        self.dtype = dtype
        esize = torch.empty((), dtype=dtype).element_size()
        self.nbytes = int(np.prod(self.shape, dtype=np.int64)) * esize
        self.buf = torch.full((self.nbytes + 2 * GUARD,), PATTERN, dtype=torch.uint8, device=device)
        inner = self.buf[GUARD:GUARD + self.nbytes]
        if fill is not None:
            inner.fill_(fill)
        self.t = inner.view(dtype).view(self.shape) if self.nbytes else \
            torch.empty(self.shape, dtype=dtype, device=device)

    def intact(self) -> bool:
        head = self.buf[:GUARD]
        tail = self.buf[GUARD + self.nbytes:]
        return bool(torch.all(head == PATTERN).item()) and bool(torch.all(tail == PATTERN).item())

    def check(self, what="output"):
        torch.cuda.synchronize()
        assert self.intact(), "guard bytes around %s %s were overwritten" % (what, self.shape)


def out(shape, dtype):
    """A guarded output tensor (its contents are left as the guard pattern,
    so a kernel that skips an element is caught by the value comparison)."""
    return Guarded(shape, dtype)


def workspace(nbytes: int):
    """A guarded, zero-filled workspace of `nbytes` (None when 0)."""
    if nbytes == 0:
        return None
    return Guarded((nbytes,), torch.uint8, fill=WS_FILL)


def check_all(*gs):
    torch.cuda.synchronize()
    for i, g in enumerate(gs):
        if g is not None:
            assert g.intact(), "guard bytes around argument %d %s were overwritten" % (i, g.shape)


def t(g):
    """The tensor of a Guarded (None passes through)."""
    return None if g is None else g.t
