"""Canary guard regions around the device outputs of the GPU parity tests.

No memory checker runs on the GPU pool, so the parity tests look for
out-of-bounds writes themselves: every output buffer is cut from a larger
allocation whose PAD bytes before and after it hold a known byte pattern,
and after each call the pattern must still be there. An overrun past the end
of an output (or a write before its start) lands in a guard region instead
of in a neighbouring allocation, and the check names the buffer.
"""
import math

import torch

PAD = 4096
PATTERN = 0x5A


class Guarded:
    """A device tensor of `shape` and `dtype` with guard regions on both sides."""

    def __init__(self, shape, dtype, device="cuda", fill=None, name="buffer"):
        shape = tuple(shape) if isinstance(shape, (tuple, list)) else (shape,)
        esize = torch.empty((), dtype=dtype).element_size()
        self.nbytes = math.prod(shape) * esize
        body = (self.nbytes + 255) // 256 * 256
        self.raw = torch.full((PAD + body + PAD,), PATTERN, dtype=torch.uint8, device=device)
        self.tensor = self.raw[PAD:PAD + self.nbytes].view(dtype).view(shape)
        if fill is not None:
            self.tensor.fill_(fill)
        self.name = name

    def check(self):
        head = self.raw[:PAD]
        tail = self.raw[PAD + self.nbytes:]
        bad_head = int((head != PATTERN).sum().item())
        bad_tail = int((tail != PATTERN).sum().item())
        assert bad_head == 0 and bad_tail == 0, (
            f"{self.name}: {bad_head} guard bytes before and {bad_tail} after it were written")


def guarded(shape, dtype, fill=None, name="buffer"):
    g = Guarded(shape, dtype, fill=fill, name=name)
    return g.tensor, g


def guard_attrs(obj, names, fill_from_original=True):
    """Replaces each named tensor attribute of obj (a buffer set of the binding)
    with a guarded tensor of the same shape and dtype (and contents), and
    returns the guards."""
    guards = []
    for n in names:
        t = getattr(obj, n)
        g = Guarded(t.shape, t.dtype, device=t.device, name=n)
        if fill_from_original:
            g.tensor.copy_(t)
        setattr(obj, n, g.tensor)
        guards.append(g)
    return guards


def check_all(guards):
    torch.cuda.synchronize()
    for g in guards:
        g.check()
