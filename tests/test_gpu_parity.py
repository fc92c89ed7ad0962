"""CUDA path against the CPU oracle on the same seeded inputs (GPU needed).

Element by element at sizes the oracle finishes in seconds (several tiles
and ragged tails), and on sampled positions at the full sizes of the five
workloads, in the launch configuration the benchmark times."""

import numpy as np
import pytest
import torch

import workloads as wk
import zero_sharded_mixed_step_gb300 as zs
from oracle import zero_oracle as z
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu

SCHEMES = [zs.ZERO_SCHEME_DP, zs.ZERO_SCHEME_Z1, zs.ZERO_SCHEME_Z2, zs.ZERO_SCHEME_Z3]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from zero_sharded_mixed_step_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def test_tiny_lab_case_all_schemes():
    """Psi = 8 on 4 ranks, 5 steps, all four schemes: each equals its oracle
    scheme at every step, all four are bit-identical, and the traffic the
    context counted equals the oracle's event count."""
    wl = wk.TINY
    finals = []
    for scheme in SCHEMES:
        run = gh.Run(wl, scheme, "fp16")
        units = run.units
        orc = z.make_scheme(scheme, wl.W, wk.draw_theta0(wl, "cuda").cpu().numpy(), "fp16",
                            units if scheme == zs.ZERO_SCHEME_Z3 else None)
        for _ in range(wl.steps):
            run.step()
            grads_np = [wk.to_numpy16(g) for g in run.zs.grads]
            orc.step(grads_np, wl.lr, wl.beta1, wl.beta2, wl.eps)
            run.compare()
            th, m, v, p16 = run.gpu_state()
            gh.assert_f32_close(th, orc.full_master()[:8], "scheme oracle master")
            gh.assert_16bit_band(p16, orc.full_master()[:8], "fp16", "scheme oracle 16-bit")
        assert zs.zero_comm_bytes_per_rank(run.zs.ctx) == orc.comm_bytes()
        assert zs.zero_comm_bytes_per_rank(run.zs.ctx) == wl.steps * z.comm_bytes_closed_form(scheme, 8, 4)
        finals.append([x.copy() for x in run.gpu_state()])
        run.close()
    for other in finals[1:]:
        for a, b in zip(finals[0], other):
            assert np.array_equal(a.view(np.uint32) if a.dtype == np.float32 else a,
                                  b.view(np.uint32) if b.dtype == np.float32 else b)


@pytest.mark.parametrize("scheme", [zs.ZERO_SCHEME_Z1, zs.ZERO_SCHEME_Z2])
def test_flat_2p20_full_compare(scheme):
    """Psi = 2^20 on 8 ranks with 1% exact-zero gradients, 10 steps, every
    element against the oracle."""
    wl = wk.FLAT_1M
    run = gh.Run(wl, scheme, "fp16")
    for _ in range(wl.steps):
        run.step()
    run.compare()
    assert zs.zero_comm_bytes_per_rank(run.zs.ctx) == wl.steps * z.comm_bytes_closed_form(scheme, wl.n, wl.W)
    run.close()


RAGGED = [
    # (n, W, scheme, grad dtype, work dtype, units)
    (3_000_007, 8, zs.ZERO_SCHEME_Z2, "bf16", "bf16", None),
    (3_000_007, 3, zs.ZERO_SCHEME_Z1, "fp16", "fp16", None),
    (1_000_001, 5, zs.ZERO_SCHEME_DP, "bf16", "fp16", None),
    (777_777, 16, zs.ZERO_SCHEME_Z1, "fp16", "bf16", None),
    (400_003, 64, zs.ZERO_SCHEME_Z2, "bf16", "bf16", None),
    (300_001, 12, zs.ZERO_SCHEME_Z1, "fp16", "fp16", None),
    (5, 4, zs.ZERO_SCHEME_Z1, "fp16", "fp16", None),
    (1, 1, zs.ZERO_SCHEME_DP, "bf16", "bf16", None),
    (None, 5, zs.ZERO_SCHEME_Z3, "bf16", "bf16", [1_000_003, 17, 0, 250_000, 7]),
    (None, 8, zs.ZERO_SCHEME_Z3, "fp16", "fp16", [262_144, 262_147, 100_000]),
    (None, 2, zs.ZERO_SCHEME_Z3, "bf16", "fp16", [9, 1, 33]),
]


VARIANTS = {"auto": zs.ZERO_VARIANT_AUTO, "vector": zs.ZERO_VARIANT_VECTOR, "bulk": zs.ZERO_VARIANT_BULK}


@pytest.mark.parametrize("variant", sorted(VARIANTS))
@pytest.mark.parametrize("case", RAGGED, ids=lambda c: f"n{c[0]}_W{c[1]}_s{c[2]}_{c[3]}_{c[4]}")
def test_ragged_full_compare(case, variant):
    """Sizes that leave ragged tails, W that is not a power of two (the mean
    divides), W = 64 (any-W path), mixed gradient / working-copy formats,
    ZeRO-3 units with padding and an empty unit: every element for 4 steps,
    padding exactly zero, under each fused-kernel variant."""
    n, W, scheme, gdt, wdt, units = case
    if units is not None:
        n = sum(units)
    wl = wk.scaled(wk.GPT2_SMALL, n=n, W=W, steps=4, unit_sizes=units, name=f"ragged_{n}_{W}",
                   outlier_frac=1e-3)
    run = gh.Run(wl, scheme, gdt, units=units, work_dtype=wdt, variant=VARIANTS[variant])
    for _ in range(wl.steps):
        run.step()
        run.compare()
    assert run.padding_is_zero()
    run.close()


@pytest.mark.parametrize("case", [(124_439_808, 8, zs.ZERO_SCHEME_Z2, "bf16", None),
                                  (50_331_651, 16, zs.ZERO_SCHEME_Z1, "fp16", None),
                                  (None, 8, zs.ZERO_SCHEME_Z3, "bf16", [50_331_648, 6_291_459, 4096]),
                                  (3_000_005, 4, zs.ZERO_SCHEME_DP, "bf16", None)],
                         ids=["gpt2small_w8", "w16_ragged", "zero3_w8", "w4"])
def test_bulk_and_vector_kernels_bit_identical(case):
    """The bulk-staged and the register kernel leave the same bits in every
    element, full-size GPT-2-small included, and report which one ran."""
    n, W, scheme, dtype, units = case
    if units is not None:
        n = sum(units)
    wl = wk.scaled(wk.GPT2_SMALL, n=n, W=W, steps=2, unit_sizes=units, name="variants")
    states = []
    for variant in (zs.ZERO_VARIANT_VECTOR, zs.ZERO_VARIANT_BULK):
        run = gh.Run(wl, scheme, dtype, units=units, sample=np.arange(min(n, 4096)), variant=variant)
        for _ in range(wl.steps):
            run.step()
        torch.cuda.synchronize()
        assert run.zs.stat(zs.ZERO_STAT_LAST_VARIANT) == variant
        states.append([x.clone() for x in (run.zs.master, run.zs.m, run.zs.v, run.zs.working_copy())])
        run.compare()
        run.close()
    for a, b in zip(*states):
        assert torch.equal(a.view(torch.int16) if a.element_size() == 2 else a.view(torch.int32),
                           b.view(torch.int16) if b.element_size() == 2 else b.view(torch.int32))


def test_schemes_bit_identical_on_gpu():
    """Data parallel, ZeRO-1, ZeRO-2 and ZeRO-3 (one unit, and ten ragged
    units) leave bit-identical master, m, v and 16-bit copies."""
    n, W = 1_000_003, 8
    wl = wk.scaled(wk.GPT2_SMALL, n=n, W=W, steps=3, name="invariance")
    cases = [(s, None) for s in SCHEMES] + [(zs.ZERO_SCHEME_Z3, [100_000] * 9 + [100_003])]
    results = []
    for scheme, units in cases:
        run = gh.Run(wl, scheme, "bf16", units=units, sample=np.arange(n))
        for _ in range(wl.steps):
            run.step()
        th, m, v, p16 = run.gpu_state()
        results.append((th.view(np.uint32), m.view(np.uint32), v.view(np.uint32), p16))
        run.close()
    for other in results[1:]:
        for a, b in zip(results[0], other):
            assert np.array_equal(a, b)


def test_zero3_overlap_equals_serial():
    """The ZeRO-3 step with a unit hook (gathers on their own stream, each
    overlapping the work on the unit before) and without one (everything in
    order on one stream, each backward gather done by the unit's update
    pass) give bit-identical results."""
    units = [65_536 * 3 + 5] * 6
    wl = wk.scaled(wk.LAYER_UNITS, unit_sizes=units, steps=3, name="overlap")
    out = []
    for with_hook in (True, False):
        run = gh.Run(wl, zs.ZERO_SCHEME_Z3, "bf16", units=units, sample=np.arange(wl.n), gather_stream=True)
        sums = []
        if with_hook:
            def hook(_user, phase, unit, buf, stream):
                s = torch.cuda.ExternalStream(stream) if stream else torch.cuda.current_stream()
                with torch.cuda.stream(s):
                    b = next(x for x in run.zs.unit_bufs if x.data_ptr() == buf)
                    sums.append(b.float().abs().sum())       # some work that reads the gathered unit
            run.zs.set_unit_hook(hook)
        for _ in range(wl.steps):
            run.step()
        run.compare()
        if with_hook:
            torch.cuda.synchronize()
            assert len(sums) == 2 * len(units) * wl.steps and all(bool(torch.isfinite(x)) for x in sums)
        out.append([x.copy() for x in run.gpu_state()])
        run.close()
    for a, b in zip(*out):
        assert np.array_equal(a.view(np.uint16), b.view(np.uint16))
