"""Seeded random configurations against the oracle at every position (GPU
needed): scheme, rank count (1 to 64), vector or unit sizes (empty, tiny,
ragged and several tiles long), gradient and working-copy formats, and the
fused-pass variant are drawn per case, then three steps run and every
element of master, m, v and the 16-bit copy is compared, with the padding
still zero and the traffic counter equal to its closed form (ZeRO-3: to
three ring collectives per unit)."""

import numpy as np
import pytest
import torch

import workloads as wk
import zero_sharded_mixed_step_gb300 as zs
from oracle import zero_oracle as z
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu

RANKS = [1, 2, 3, 4, 5, 7, 8, 12, 16, 31, 64]
VARIANTS = [zs.ZERO_VARIANT_AUTO, zs.ZERO_VARIANT_VECTOR, zs.ZERO_VARIANT_BULK]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from zero_sharded_mixed_step_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _size(rng) -> int:
    kind = rng.random()
    if kind < 0.15:
        return int(rng.integers(0, 3))
    if kind < 0.4:
        return int(rng.integers(3, 200))
    return int(rng.integers(1_000, 300_000))


def draw(seed: int):
    rng = np.random.default_rng(9000 + seed)
    scheme = int(rng.integers(0, 4))
    W = int(rng.choice(RANKS))
    if scheme == zs.ZERO_SCHEME_Z3:
        units = [_size(rng) for _ in range(int(rng.integers(1, 6)))]
        if sum(units) == 0:
            units[0] = 1
    else:
        units = [max(1, _size(rng))]
    gdt, wdt = (str(rng.choice(["fp16", "bf16"])) for _ in range(2))
    variant = int(rng.choice(VARIANTS))
    return scheme, W, units, gdt, wdt, variant


@pytest.mark.parametrize("seed", range(32))
def test_random_configuration_against_the_oracle(seed):
    scheme, W, units, gdt, wdt, variant = draw(seed)
    base = wk.LAYER_UNITS if scheme == zs.ZERO_SCHEME_Z3 else wk.GPT2_SMALL
    wl = wk.scaled(base, W=W, steps=3, unit_sizes=units, name=f"random{seed}")
    run = gh.Run(wl, scheme, gdt, units=units, work_dtype=wdt, variant=variant)
    what = f"seed {seed}: scheme {scheme}, W {W}, units {units}, {gdt}->{wdt}, variant {variant}"
    for _ in range(wl.steps):
        run.step()
        run.compare(what)
    assert run.padding_is_zero(), what
    comm = zs.zero_comm_bytes_per_rank(run.zs.ctx)
    if scheme == zs.ZERO_SCHEME_Z3:
        _, shard, _ = zs.zero_layout(W, units)
        assert comm == wl.steps * sum(3 * (W - 1) * s * 2 for s in shard), what
    else:
        assert comm == wl.steps * z.comm_bytes_closed_form(scheme, sum(units), W), what
    run.close()


def draw_one_size(seed: int):
    """ZeRO-3 with every unit of one size: the forward gathers in one launch
    when the padded shard is a multiple of 16 values (32 bytes), else a launch
    per pair; the step from a CUDA graph (backward on two chains) or not."""
    rng = np.random.default_rng(7000 + seed)
    W = int(rng.choice(RANKS))
    aligned, graph = seed % 2 == 0, seed % 4 < 2          # each combination on 4 seeds
    U = int(rng.integers(1, 8))
    S = int(rng.integers(1, max(2, 3_000_000 // (16 * W * U))))   # at most ~3M parameters in all
    S = S * 16 if aligned else (S * 16 + int(rng.integers(1, 16)))
    units = [S * W - int(rng.integers(0, W))] * U
    dt = str(rng.choice(["fp16", "bf16"]))
    return W, units, dt, graph


@pytest.mark.parametrize("seed", range(16))
def test_random_one_size_units_against_the_oracle_and_plain_launches(seed):
    W, units, dt, graph = draw_one_size(seed)
    what = f"seed {seed}: W {W}, units {units}, {dt}, graph {graph}"
    wl = wk.scaled(wk.LAYER_UNITS, W=W, steps=3, unit_sizes=units, name=f"one_size{seed}")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        run = gh.Run(wl, zs.ZERO_SCHEME_Z3, dt, units=units, gather_stream=False)
        plain = zs.ZeroStep(zs.ZERO_SCHEME_Z3, W, units, dt, theta0=wk.draw_theta0(wl, "cuda"), stream=s)
        run.zs.set_graph(graph)
        for _ in range(wl.steps):
            run.step()
            plain.step(run.zs.grads, wl.lr, wl.beta1, wl.beta2, wl.eps, run.t)
            run.compare(what)
        torch.cuda.synchronize()
        for x, y in ((run.zs.master, plain.master), (run.zs.m, plain.m), (run.zs.v, plain.v)):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32)), what
        for a, b in zip(run.zs.shard16, plain.shard16):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16)), what
        # the unit buffers end the same in both contexts (the last units gathered)
        for b in range(2):
            assert torch.equal(run.zs.unit_bufs[b].view(torch.int16), plain.unit_bufs[b].view(torch.int16)), what
        _, shard, _ = zs.zero_layout(W, units)
        assert zs.zero_comm_bytes_per_rank(run.zs.ctx) == wl.steps * sum(3 * (W - 1) * x * 2 for x in shard), what
        assert run.zs.stat(zs.ZERO_STAT_PEAK_LIVE_ELEMS) == 2 * shard[0] * W, what
        assert run.padding_is_zero(), what
        plain.close()
        run.close()
