"""Output buffers wrapped in guard bands, for the GPU parity tests.

Every output tensor a parity test hands to the library is a view into a
larger device buffer: BAND bytes of a sentinel pattern before it and at least
BAND bytes after it (the space between the end of the view and the next
256-byte boundary belongs to the trailing band).  After the call the bands
must still hold the sentinel, so a kernel that stores outside its output
(a 16-byte store past the end of a row, a stray scatter of a partial tile,
an id or weight written for a slot past k) fails the test even where the
stray bytes would land in memory nobody reads.
"""

import torch

BAND = 4096        # bytes on each side (a multiple of 256: the view stays 256-byte aligned)
SENTINEL = 0xA5    # every byte of a band


class Guarded:
    """One output tensor of `shape` and `dtype` inside sentinel bands."""

    def __init__(self, shape, dtype, device="cuda", fill=None):
        shape = tuple(int(s) for s in shape)
        elem = torch.empty((), dtype=dtype).element_size()
        n = 1
        for s in shape:
            n *= s
        self.nbytes = n * elem
        body = (self.nbytes + 255) // 256 * 256
        self.buf = torch.full((BAND + body + BAND,), SENTINEL, dtype=torch.uint8, device=device)
        self.t = self.buf[BAND:BAND + self.nbytes].view(dtype).view(shape)
        if fill is not None:
            self.t.fill_(fill)

    def check(self, name="output"):
        head = self.buf[:BAND]
        tail = self.buf[BAND + self.nbytes:]
        bad_h = int((head != SENTINEL).sum().item())
        bad_t = int((tail != SENTINEL).sum().item())
        assert bad_h == 0 and bad_t == 0, (
            f"{name}: {bad_h} bytes before and {bad_t} bytes after the buffer were overwritten")


def guarded(shape, dtype, fill=None):
    return Guarded(shape, dtype, fill=fill)


def check_all(**named):
    """Check the bands of every Guarded given by keyword (None is skipped)."""
    for name, g in named.items():
        if g is not None:
            g.check(name)
