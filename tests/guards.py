"""Canary regions around device buffers (the GPU tests' bounds check).

guarded(shape, dtype) returns a contiguous device tensor of that shape whose
storage sits between two 4 KiB guard regions filled with a byte pattern, and
a function that asserts the guards still hold it. A kernel that writes past
either end of an output or workspace changes a guard. The tensor itself
starts 4 KiB into the allocation, so its alignment (16 bytes for TMA and
more) is the allocation's.
"""
import torch

GUARD = 4096
PATTERN = 0xA5


class Guarded:
    def __init__(self, shape, dtype=torch.float32, device="cuda", fill=None):
        n = 1
        for x in shape:
            n *= int(x)
        esize = torch.empty((), dtype=dtype).element_size()
        nbytes = n * esize
        body = (nbytes + 255) // 256 * 256
        self.raw = torch.full((GUARD + body + GUARD,), PATTERN, dtype=torch.uint8, device=device)
        self.nbytes = nbytes
        self.body = body
        inner = self.raw[GUARD:GUARD + nbytes]
        self.tensor = inner.view(dtype).view(*shape) if n > 0 else torch.empty(shape, dtype=dtype,
                                                                                device=device)
        if fill is not None and n > 0:
            self.tensor.fill_(fill)

    def check(self, name):
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.body:]
        pad = self.raw[GUARD + self.nbytes:GUARD + self.body]
        for part, where in ((head, "before"), (tail, "after"), (pad, "in the padding after")):
            bad = (part != PATTERN).nonzero()
            assert bad.numel() == 0, f"{name}: guard bytes {where} the buffer were overwritten " \
                                     f"(first at offset {int(bad[0])})"


def guarded(shape, dtype=torch.float32, device="cuda", fill=None):
    g = Guarded(shape, dtype, device, fill)
    return g.tensor, g
