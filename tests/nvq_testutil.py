"""Shared helpers of the GPU parity tests (no quantisation arithmetic)."""
import numpy as np
import torch

GUARD = 4096
CANARY = 0xA5


def u16(t):
    """bf16 / int16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def u8(t):
    return t.contiguous().cpu().numpy().astype(np.uint8)


def f32(t):
    return t.contiguous().cpu().numpy().astype(np.float32)


def bf16_from_u16(a, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


class Guarded:
    """A device tensor with canary-filled guard bands on both sides; stands in
    for a memory checker on writes past either end."""

    def __init__(self, shape, dtype, device="cuda"):
        n = int(np.prod(shape)) if len(shape) else 1
        self.nbytes = n * torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((self.nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8, device=device)
        self.t = self.buf[GUARD:GUARD + self.nbytes].view(dtype).view(shape)

    def intact(self):
        b = self.buf.cpu().numpy()
        return bool((b[:GUARD] == CANARY).all() and (b[GUARD + self.nbytes:] == CANARY).all())


def first_mismatch(a, b):
    a = np.asarray(a).ravel()
    b = np.asarray(b).ravel()
    if a.shape != b.shape:
        return "shape %s vs %s" % (a.shape, b.shape)
    bad = np.nonzero(a != b)[0]
    if bad.size == 0:
        return None
    i = bad[0]
    return "%d mismatches, first at %d: %r vs %r" % (bad.size, i, a[i], b[i])


def assert_same(a, b, what=""):
    m = first_mismatch(a, b)
    assert m is None, "%s: %s" % (what, m)
