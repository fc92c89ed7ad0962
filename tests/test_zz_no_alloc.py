"""The ZeRO-3 step that allocates nothing (zero_step_z3_static), against the
ZeRO-3 step of a context (zero_step), through the C ABI on the GPU.

zero_step_z3_static is for callers that cannot allocate device memory and so
cannot hand zero_step the two unit buffers ZeRO-3 gathers into: it gathers
into a fixed array that belongs to the library.  Here the caller owns only
its state (master, m, v, the ranks' 16-bit shard stores, the gradients);
two calls in a row must leave that state where two zero_step calls leave
it, within the parity tolerances, and the hook must see every gathered unit
in the library's array.  This file is collected last and needs nothing
from the tests before it.
"""

import numpy as np
import pytest
import torch

import workloads as wk
import zero_sharded_mixed_step_gb300 as zs
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu

W = 8
UNITS = [1_000_003, 4_194_304, 17, 0, 262_147]


class _DeviceWords:
    """A raw device pointer as a tensor-compatible object (no copy)."""

    def __init__(self, ptr: int, count: int):
        self.__cuda_array_interface__ = {"shape": (count,), "typestr": "<i2", "data": (ptr, False),
                                         "version": 3, "strides": None}


def _caller_state(ref: zs.ZeroStep):
    """master / m / v and shard stores the way a caller would hold them,
    equal to the reference context's initial state."""
    master, m, v = ref.master.clone(), torch.zeros_like(ref.m), torch.zeros_like(ref.v)
    shards = []
    for r in range(W):
        parts = [master[o + r * s:o + (r + 1) * s] for o, s in zip(ref.off, ref.shard)]
        shards.append(torch.cat(parts).to(torch.bfloat16))
    return master, m, v, shards


def test_static_scratch_step_matches_zero_step():
    from zero_sharded_mixed_step_gb300 import build
    build.build()
    wl = wk.scaled(wk.LAYER_UNITS, unit_sizes=UNITS, steps=2, name="static_scratch")
    ref = zs.ZeroStep(zs.ZERO_SCHEME_Z3, W, UNITS, "bf16", theta0=wk.draw_theta0(wl, "cuda"))
    master, m, v, shards = _caller_state(ref)
    torch.cuda.synchronize()
    for r in range(W):
        assert torch.equal(shards[r], ref.shard16[r])
    src = wk.GradSource(wl, "bf16", "cuda")
    hp = (wl.lr, wl.beta1, wl.beta2, wl.eps)
    seen = []

    def hook(_user, phase, unit, buf, stream):
        n = ref.shard[unit] * W
        s = torch.cuda.ExternalStream(stream) if stream else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            got = torch.as_tensor(_DeviceWords(buf, n), device="cuda").clone() if n else None
        seen.append((phase, unit, buf, got))

    for t in (1, 2):                                  # two calls in a row
        grads = []
        for d in src.step(t):
            g = torch.zeros(ref.n_pad, dtype=torch.bfloat16, device="cuda")
            ref.place_(g, d)
            grads.append(g)
        torch.cuda.synchronize()
        flat_before = torch.cat([torch.cat([shards[r][o16:o16 + s] for r in range(W)])
                                 for s, o16 in zip(ref.shard, ref.off16)]).view(torch.int16)
        seen.clear()
        ref.step(grads, *hp, t)
        zs.zero_step_z3_static(W, UNITS, zs.ZERO_BF16, zs.ZERO_BF16, master, m, v, shards, grads, *hp, t,
                               hook=hook)
        torch.cuda.synchronize()

        # the state equals zero_step's, within the parity tolerances (and in fact bit for bit)
        for mine, theirs, what in ((master, ref.master, "master"), (m, ref.m, "m"), (v, ref.v, "v")):
            gh.assert_f32_close(mine.cpu().numpy(), theirs.cpu().numpy(), f"t={t} {what}")
            assert torch.equal(mine, theirs), f"t={t} {what}"
        for r in range(W):
            gh.assert_16bit_band(gh.bits_of(shards[r]), _rank_master(ref, r), "bf16", f"t={t} shard store {r}")
            assert torch.equal(shards[r], ref.shard16[r]), f"t={t} shard store {r}"

        # every unit gathered twice, in the ZeRO-3 order, into the library's one array
        U = len(UNITS)
        assert [(p, u) for p, u, _, _ in seen] == [(0, u) for u in range(U)] + [(1, u) for u in reversed(range(U))]
        assert len({b for _, u, b, _ in seen if ref.shard[u]}) == 1
        for _phase, u, _buf, got in seen:
            if got is None:
                continue
            lo = ref.off[u]
            assert torch.equal(got, flat_before[lo:lo + ref.shard[u] * W]), f"t={t} gathered unit {u}"
    assert zs.zero_stat(ref.ctx, zs.ZERO_STAT_T) == 2
    ref.close()


def _rank_master(ref: zs.ZeroStep, r: int) -> np.ndarray:
    """Rank r's slice of every unit of the reference master, in shard-store order."""
    parts = [ref.master[o + r * s:o + (r + 1) * s] for o, s in zip(ref.off, ref.shard)]
    return torch.cat(parts).cpu().numpy()


def test_static_scratch_rejects_units_beyond_its_size():
    from zero_sharded_mixed_step_gb300 import build
    build.build()
    big = [8_388_609]                                  # one value past the array, with W = 1
    x = torch.zeros(8_388_616, dtype=torch.float32, device="cuda")
    s16 = torch.zeros(8_388_616, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(zs.ZeroError) as e:
        zs.zero_step_z3_static(1, big, zs.ZERO_BF16, zs.ZERO_BF16, x, x, x, [s16], [s16], 1e-3, 0.9, 0.95, 1e-8, 1)
    assert e.value.code == zs.ZERO_E_ARG
    assert "static gather buffer" in zs.zero_last_error()
    torch.cuda.synchronize()
    assert bool((x == 0).all()) and bool((s16 == 0).all())   # nothing ran
