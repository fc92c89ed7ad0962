"""The guard-byte checker itself, on host memory (no GPU): placement at the
least alignment the ABI accepts, and a write one byte past a buffer, or one
byte before it, reported with its neighbours."""

import torch

from tests.canary import Arena


def test_buffers_sit_at_odd_multiples_of_their_alignment():
    a = Arena(1 << 20, "cpu", seed=3)
    for numel, dtype, align in [(5, torch.float32, 32), (7, torch.bfloat16, 16), (3, torch.uint8, 256),
                                (0, torch.float16, 16), (9, torch.int64, 16)]:
        t = a.zeros(numel, dtype)
        assert t.numel() == numel and t.dtype == dtype
        if numel:   # torch gives an empty view address 0 (NULL, which the ABI accepts for empty buffers)
            assert t.data_ptr() % align == 0 and t.data_ptr() % (2 * align) == align
        assert bool((t == 0).all())
    a.check()


def test_writes_inside_buffers_pass_and_past_them_are_reported():
    a = Arena(1 << 20, "cpu", seed=4)
    x = a.zeros(100, torch.float32, "x")
    y = a.zeros(64, torch.bfloat16, "y")
    x.fill_(1.5)
    y.fill_(-2.0)
    a.check()
    # one byte after x's end, one byte before y's start
    lo_x, hi_x, _ = a.regions[0]
    lo_y, _, _ = a.regions[1]
    a.buf[hi_x] ^= 0xFF
    a.buf[lo_y - 1] ^= 0x01
    bad = a.changed_outside()
    assert [(off, before, after) for off, before, after in bad] == [(hi_x, "x", "y"), (lo_y - 1, "x", "y")]
    a.buf[hi_x] ^= 0xFF
    a.buf[lo_y - 1] ^= 0x01
    a.check()
    # before the first buffer and after the last
    a.buf[lo_x - 1] ^= 0x10
    assert a.changed_outside() == [(lo_x - 1, "(arena start)", "x")]
