"""Guard bytes around every buffer a test hands to the library.

compute-sanitizer cannot be used here, so out-of-bounds writes are caught
the old way: an Arena is one allocation from which each buffer is cut with a
stretch of seeded random bytes before and after it.  A kernel or copy that
writes past either end of its buffer changes guard bytes, and Arena.check()
reports every changed byte with the buffers on either side of it.  Each
buffer starts at an odd multiple of its required alignment (32 bytes for
fp32 state, 16 for 16-bit vectors, 256 for staging), the least-aligned
placement the ABI accepts, so that no extra alignment hides an overrun."""

import bisect

import torch

GUARD = 64 * 1024       # wider than any tile or vector a kernel moves at once


def _align_of(dtype: torch.dtype) -> int:
    if dtype == torch.uint8:
        return 256
    return 32 if torch.empty(0, dtype=dtype).element_size() == 4 else 16


class Arena:
    def __init__(self, nbytes: int, device, seed: int = 0, guard: int = GUARD):
        self.device = torch.device(device)
        self.guard = guard
        self.nbytes = int(nbytes) + 2 * guard
        gen = torch.Generator().manual_seed(seed)
        pattern = torch.randint(0, 256, (self.nbytes,), dtype=torch.uint8, generator=gen)
        if self.device.type == "cpu":
            self.buf = torch.empty(self.nbytes, dtype=torch.uint8)
            if torch.cuda.is_available():       # page-locked, as host buffers of the library should be
                self.buf = self.buf.pin_memory()
            self.pattern = pattern
        else:
            self.buf = torch.empty(self.nbytes, dtype=torch.uint8, device=self.device)
            self.pattern = pattern.to(self.device)
        self.buf.copy_(self.pattern)
        self.pos = guard
        self.regions = []          # (lo, hi, name), in address order

    def zeros(self, numel: int, dtype: torch.dtype, name: str = "") -> torch.Tensor:
        """A zero-filled buffer of ``numel`` values, guarded on both sides."""
        size = int(numel) * torch.empty(0, dtype=dtype).element_size()
        align = _align_of(dtype)
        base = self.buf.data_ptr()
        lo = self.pos + (-(base + self.pos)) % align
        if (base + lo) % (2 * align) == 0:
            lo += align
        hi = lo + size
        if hi + self.guard > self.nbytes:
            raise MemoryError(f"arena of {self.nbytes} bytes is full")
        self.pos = hi + self.guard
        self.regions.append((lo, hi, name or f"buffer {len(self.regions)} ({numel} x {dtype})"))
        out = self.buf[lo:hi].view(dtype)
        out.zero_()
        return out

    def __call__(self, numel, dtype):
        return self.zeros(numel, dtype)

    def changed_outside(self):
        """(offset, name of the buffer before it, name of the buffer after it)
        for each guard byte that no longer holds the pattern (waits for the
        device first)."""
        if self.device.type == "cuda":
            torch.cuda.synchronize(self.device)
        diff = self.buf != self.pattern
        for lo, hi, _ in self.regions:
            diff[lo:hi] = False
        where = diff.nonzero().flatten().cpu().tolist()
        starts = [lo for lo, _, _ in self.regions]
        out = []
        for off in where:
            k = bisect.bisect_right(starts, off)
            before = self.regions[k - 1][2] if k > 0 else "(arena start)"
            after = self.regions[k][2] if k < len(self.regions) else "(arena end)"
            out.append((off, before, after))
        return out

    def check(self):
        bad = self.changed_outside()
        assert not bad, f"{len(bad)} guard bytes written, first at {bad[:4]}"
