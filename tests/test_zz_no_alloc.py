"""The ZeRO-3 step that allocates nothing (zero_step_z3_static), against the
ZeRO-3 step of a context (zero_step), through the C ABI on the GPU.

zero_step_z3_static is for callers that cannot allocate device memory and so
cannot hand zero_step the two unit buffers ZeRO-3 gathers into: it gathers
into a fixed array that belongs to the library.  Here the caller owns only
its state (master, m, v, the ranks' 16-bit shard stores, the gradients);
two calls in a row must leave that state where two zero_step calls leave
it, within the parity tolerances, and the hook must see every gathered unit
in the library's array; the same must hold across a cudaDeviceReset.  This
file is collected last and needs nothing from the tests before it.
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


@pytest.mark.parametrize("with_hook", [True, False], ids=["hook", "no_hook"])
def test_static_scratch_step_matches_zero_step(with_hook):
    """With a hook every gather is a copy of its own; without one each
    backward gather is done by the unit's update pass, as in zero_step."""
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
                               hook=hook if with_hook else None)
        torch.cuda.synchronize()

        # the state equals zero_step's, within the parity tolerances (and in fact bit for bit)
        for mine, theirs, what in ((master, ref.master, "master"), (m, ref.m, "m"), (v, ref.v, "v")):
            gh.assert_f32_close(mine.cpu().numpy(), theirs.cpu().numpy(), f"t={t} {what}")
            assert torch.equal(mine, theirs), f"t={t} {what}"
        for r in range(W):
            gh.assert_16bit_band(gh.bits_of(shards[r]), _rank_master(ref, r), "bf16", f"t={t} shard store {r}")
            assert torch.equal(shards[r], ref.shard16[r]), f"t={t} shard store {r}"

        if not with_hook:
            continue
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
    x = torch.zeros(8_388_616, dtype=torch.float32, device="cuda")
    s16 = torch.zeros(8_388_616, dtype=torch.bfloat16, device="cuda")
    # one value past the array (W = 1); one that only padding takes past it
    # (W = 3); sizes whose padding would overflow int64 if computed first
    for W, big in ((1, [8_388_609]), (3, [8_388_607]), (1, [2**63 - 1]), (5, [2**63 - 2]), (2, [17, 2**62])):
        with pytest.raises(zs.ZeroError) as e:
            zs.zero_step_z3_static(W, big, zs.ZERO_BF16, zs.ZERO_BF16, x, x, x, [s16] * W, [s16] * W,
                                   1e-3, 0.9, 0.95, 1e-8, 1)
        assert e.value.code == zs.ZERO_E_ARG, (W, big)
        assert "static gather buffer" in zs.zero_last_error()
    torch.cuda.synchronize()
    assert bool((x == 0).all()) and bool((s16 == 0).all())   # nothing ran


def test_static_scratch_step_survives_a_device_reset(tmp_path):
    """A plain C client (tests/c_static_reset.c) runs the step without
    allocations beside zero_step, resets the device with cudaDeviceReset
    (freeing everything and unloading the library's device code, the
    gather array with it), allocates again and runs both once more: the
    same bits both times.  The array's address is looked up on each call,
    so the call after the reset uses the reloaded array, not a stale
    address.  Runs in its own process, so it neither needs nor disturbs
    the state of this one."""
    import os
    import subprocess
    from zero_sharded_mixed_step_gb300 import build
    lib = build.build()
    # the client and the library must share one CUDA runtime for the reset to reach the library
    deps = subprocess.run(["ldd", lib], capture_output=True, text=True).stdout
    assert "libcudart.so" in deps, deps
    here = os.path.dirname(os.path.abspath(__file__))
    root = os.path.dirname(here)
    cuda = build.cuda_home()
    libdir = os.path.dirname(lib)
    exe = str(tmp_path / "c_static_reset")
    res = subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(root, "include"), "-I",
                          os.path.join(cuda, "include"), os.path.join(here, "c_static_reset.c"), "-o", exe,
                          "-L", libdir, "-lzero_gb300", "-L", build.cudart_dir(), "-lcudart",
                          f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{build.cudart_dir()}"],
                         capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "before and after cudaDeviceReset" in run.stdout


@pytest.mark.parametrize("seed", range(8))
def test_static_scratch_random_configurations(seed):
    """Seeded random rank counts (1 to 64), units (empty, ragged, up to the
    array's limit once padded), 16-bit formats, with and without a hook: two
    calls in a row equal to zero_step's state bit for bit."""
    rng = np.random.default_rng(3000 + seed)
    Wr = int(rng.choice([1, 2, 3, 5, 8, 16, 31, 64]))
    limit = 8_388_608 // Wr * Wr                       # the largest padded unit the array holds
    units = [int(rng.choice([0, 1, 17, int(rng.integers(2, 200_000)), limit - int(rng.integers(0, Wr))]))
             for _ in range(int(rng.integers(1, 5)))]
    if sum(units) == 0:
        units[0] = 5
    gdt, wdt = (str(rng.choice(["fp16", "bf16"])) for _ in range(2))
    with_hook = bool(rng.random() < 0.5)
    what = f"seed {seed}: W {Wr}, units {units}, {gdt}->{wdt}, hook {with_hook}"
    wl = wk.scaled(wk.LAYER_UNITS, W=Wr, unit_sizes=units, steps=2, name=f"static_random{seed}")
    ref = zs.ZeroStep(zs.ZERO_SCHEME_Z3, Wr, units, gdt, wdt, theta0=wk.draw_theta0(wl, "cuda"))
    master, m, v = ref.master.clone(), torch.zeros_like(ref.m), torch.zeros_like(ref.v)
    shards = [s.clone() for s in ref.shard16]
    calls = []
    src = wk.GradSource(wl, gdt, "cuda")
    hp = (wl.lr, wl.beta1, wl.beta2, wl.eps)
    G = {"fp16": zs.ZERO_FP16, "bf16": zs.ZERO_BF16}
    for t in (1, 2):
        grads = ref.new_grad_buffers()
        for g, d in zip(grads, src.step(t)):
            ref.place_(g, d)
        torch.cuda.synchronize()
        ref.step(grads, *hp, t)
        zs.zero_step_z3_static(Wr, units, G[gdt], G[wdt], master, m, v, shards, grads, *hp, t,
                               hook=(lambda _u, ph, un, _b, _s: calls.append((ph, un))) if with_hook else None)
        torch.cuda.synchronize()
        for mine, theirs, name in ((master, ref.master, "master"), (m, ref.m, "m"), (v, ref.v, "v")):
            assert torch.equal(mine.view(torch.int32), theirs.view(torch.int32)), (what, t, name)
        for r in range(Wr):
            assert torch.equal(shards[r].view(torch.int16), ref.shard16[r].view(torch.int16)), (what, t, r)
    U = len(units)
    if with_hook:
        order = [(0, u) for u in range(U)] + [(1, u) for u in reversed(range(U))]
        assert calls == order * 2, what
    ref.close()
