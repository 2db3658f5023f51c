"""Helpers for the GPU tests: guarded output buffers and error metrics."""
import numpy as np
import torch

CANARY = 4096  # elements of poison before and after every output


class Guarded:
    """An output tensor carved from the middle of a poisoned buffer (NaN for
    floating point, ``poison`` for integers); the regions before and after it
    must still hold the poison afterwards. For integer outputs, where every
    value is legal, completeness is checked by writing twice into buffers with
    different poisons (see ``run_twice``)."""

    def __init__(self, shape, dtype, device="cuda", poison=0x5A5A, lead=0):
        """``lead`` extra poisoned elements before the output move its base
        address off the buffer's (256-byte aligned) allocation."""
        n = int(np.prod(shape))
        self.is_float = dtype.is_floating_point
        fill = float("nan") if self.is_float else poison
        self.poison = fill
        self.buf = torch.full((CANARY + lead + n + CANARY,), fill, dtype=dtype, device=device)
        self.n = n
        self.start = CANARY + lead
        self.out = self.buf[self.start:self.start + n].view(*shape)

    def check(self):
        torch.cuda.synchronize()
        head = self.buf[:self.start]
        tail = self.buf[self.start + self.n:]
        if self.is_float:
            assert torch.isnan(head).all() and torch.isnan(tail).all(), "write outside the output tensor"
            assert not torch.isnan(self.out).any(), "part of the output was not written"
        else:
            assert (head == self.poison).all() and (tail == self.poison).all(), "write outside the output tensor"
        return self.out


def run_twice(shape, dtype, launch):
    """Integer outputs: ``launch(out)`` into two guarded buffers poisoned with
    different values; equal results mean every element was written."""
    a = Guarded(shape, dtype, poison=0x5A5A)
    launch(a.out)
    b = Guarded(shape, dtype, poison=-0x3C3D)
    launch(b.out)
    ra, rb = a.check(), b.check()
    assert torch.equal(ra, rb), "part of the output was not written (or the result is not deterministic)"
    return ra


def errors(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    diff = np.abs(got - want)
    rel_l2 = float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))
    return float(diff.max()), float(diff.mean()), rel_l2
