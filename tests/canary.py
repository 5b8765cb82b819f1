"""Guard bands around device buffers that a kernel writes (a stand-in for a memory
checker): each buffer is a view into a larger allocation whose bytes before and
after it hold 0xFF (a NaN in bf16 and in fp32).  After a call, check() asserts
that no band byte changed, i.e. that no kernel wrote outside the buffer it was
given.  Views start 4096 bytes into the allocation, so they keep its alignment."""
import torch

BAND = 4096


class Guarded:
    """A `shape`/`dtype` CUDA tensor `t` inside a 0xFF-filled allocation."""

    def __init__(self, shape, dtype, device="cuda", band: int = BAND, fill=None):
        n = 1
        for s in shape:
            n *= int(s)
        self.nbytes = n * torch.empty(0, dtype=dtype).element_size()
        self.band = band
        self.raw = torch.full((band + self.nbytes + band,), 0xFF, dtype=torch.uint8, device=device)
        self.t = self.raw[band:band + self.nbytes].view(dtype).view(*shape)
        if fill is not None:
            self.t.fill_(fill)

    @classmethod
    def like(cls, t, fill=None):
        return cls(tuple(t.shape), t.dtype, t.device, fill=fill)

    @classmethod
    def copy_of(cls, t):
        g = cls(tuple(t.shape), t.dtype, t.device)
        g.t.copy_(t)
        return g

    def check(self, what="buffer"):
        torch.cuda.synchronize()
        lo = self.raw[:self.band]
        hi = self.raw[self.band + self.nbytes:]
        bad_lo = int((lo != 0xFF).sum())
        bad_hi = int((hi != 0xFF).sum())
        assert bad_lo == 0 and bad_hi == 0, "%s: %d bytes written before it, %d after it" % (what, bad_lo, bad_hi)


def check_all(**guards):
    for name, g in guards.items():
        if g is not None:
            g.check(name)
