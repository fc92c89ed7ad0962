"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""

import os

import numpy as np
import pytest

from oracle import zero_oracle as z
from tests import oracle_pins as pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(check):
    check(z)


def test_golden_file_covers_every_page_figure_kind():
    rows = pins.load_accounting_pins()
    kinds = {r["qty"] for r in rows}
    assert kinds == {"resident", "bytes_pp", "lab_peak_pp", "comm_elems_collective",
                     "comm_bytes_step", "paper_volume"}
    assert {r["scheme"] for r in rows if r["qty"] == "resident"} == {0, 1, 2, 3}


def test_layout_padding_and_offsets():
    L = z.Layout(4, [13, 24, 3])
    assert L.S == [4, 6, 1] and L.off == [0, 16, 40] and L.off16 == [0, 4, 10]
    assert L.n == 40 and L.n_pad == 44 and L.S_total == 11
    assert list(L.real_index()[:14]) == list(range(13)) + [16]
    assert z.shard_size(0, 3) == 0 and z.shard_size(1, 3) == 1 and z.shard_size(9, 3) == 3
    with pytest.raises(ValueError):
        z.shard_size(5, 0)


def test_step_counter_starts_at_one():
    with pytest.raises(ValueError):
        z.bias_corrections(0.9, 0.999, 0)
    bc1, bc2 = z.bias_corrections(0.9, 0.999, 1)
    assert bc1 == pytest.approx(0.1) and bc2 == pytest.approx(0.001)


def test_ulp_distance():
    a = np.array([0x3C00, 0x3C01, 0x8001, 0x0000], np.uint16)
    b = np.array([0x3C00, 0x3C00, 0x0001, 0x8000], np.uint16)
    assert list(z.ulp_distance16(a, b)) == [0, 1, 2, 0]


@pytest.mark.skipif(os.environ.get("ZERO_EXHAUSTIVE_ROUNDING") != "1",
                    reason="all 2^32 fp32 patterns take ~10 minutes; set ZERO_EXHAUSTIVE_ROUNDING=1")
def test_rounding_exhaustive():
    import torch
    chunk = 1 << 24
    for k in range(1 << 8):
        u = np.arange(k * chunk, (k + 1) * chunk, dtype=np.uint64).astype(np.uint32)
        x = u.view(np.float32)
        x = x[~np.isnan(x)]
        t = torch.from_numpy(x)
        assert np.array_equal(z.cast16(x, "bf16"), t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
        assert np.array_equal(z.bits16(z.cast16(x, "fp16"), "fp16"),
                              t.to(torch.float16).view(torch.int16).numpy().view(np.uint16))
