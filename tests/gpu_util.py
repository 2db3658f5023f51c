"""Helpers for the GPU tests: guarded output buffers and error metrics."""
import numpy as np
import torch

CANARY = 4096  # elements of poison before and after every output


class Guarded:
    """An output tensor carved from the middle of a NaN-filled buffer; the
    regions before and after it must still hold the poison afterwards."""

    def __init__(self, shape, dtype, device="cuda"):
        n = int(np.prod(shape))
        self.buf = torch.full((CANARY + n + CANARY,), float("nan"), dtype=dtype, device=device)
        self.n = n
        self.out = self.buf[CANARY:CANARY + n].view(*shape)
        self._poison = self.buf[:CANARY].clone()

    def check(self):
        torch.cuda.synchronize()
        head = self.buf[:CANARY]
        tail = self.buf[CANARY + self.n:]
        assert torch.isnan(head).all() and torch.isnan(tail).all(), "write outside the output tensor"
        assert not torch.isnan(self.out).any(), "part of the output was not written"
        return self.out


def errors(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    diff = np.abs(got - want)
    rel_l2 = float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))
    return float(diff.max()), float(diff.mean()), rel_l2
