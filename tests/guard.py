"""Guard regions around output buffers: a tensor is carved out of a larger
allocation whose bytes before and after it hold a canary pattern, so that a
kernel writing past either end of its output (or of its workspace) is seen
on the host afterwards.  This stands in for a memory checker on a pool where
none can be run."""

import torch

CANARY = 0xA5
LEAD = 256          # guard bytes before the tensor (keeps 256-byte alignment)
TAIL = 64 * 1024    # guard bytes after it


class Guarded:
    """A tensor of `shape` and `dtype` on `device` with canary-filled guard
    regions on both sides; `.t` is the tensor, `.intact()` checks the guards."""

    def __init__(self, shape, dtype, device, fill=None):
        esize = torch.empty((), dtype=dtype).element_size()
        numel = 1
        for s in shape:
            numel *= int(s)
        self.nbytes = numel * esize
        self.raw = torch.full((LEAD + self.nbytes + TAIL,), CANARY, dtype=torch.uint8, device=device)
        self.t = self.raw[LEAD:LEAD + self.nbytes].view(dtype).view(tuple(shape))
        if fill is not None:
            self.t.copy_(fill)

    def intact(self):
        lead = self.raw[:LEAD]
        tail = self.raw[LEAD + self.nbytes:]
        return bool((lead == CANARY).all()) and bool((tail == CANARY).all())

    def first_overwrite(self):
        """Byte offset (relative to the tensor's start) of the first guard
        byte that changed, or None."""
        bad = torch.nonzero(self.raw != CANARY).flatten().cpu().tolist()
        for i in bad:
            if i < LEAD or i >= LEAD + self.nbytes:
                return i - LEAD
        return None
