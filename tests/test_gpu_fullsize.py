"""The three large workloads at their full sizes, in the launch configuration
the benchmark times, against the oracle on sampled positions (the update is
elementwise, so the oracle computes each sampled position on its own), plus
properties checked over every element."""

import numpy as np
import pytest
import torch

import workloads as wk
import zero_sharded_mixed_step_gb300 as zs
from oracle import zero_oracle as z
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu

TORCH16 = {"fp16": torch.float16, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from zero_sharded_mixed_step_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def first_step_property(run, theta0: torch.Tensor):
    """After step 1 every parameter moved by -lr g / (|g| + eps): by lr sign(g)
    up to lr eps / (|g| + eps), and not at all where g = 0 (checked on every
    element).  g is the rank mean as the kernel forms it: fp32 additions in
    rank order, then the division by W (exact for W a power of two)."""
    wl = run.wl
    acc = run.zs.grads[0].float()
    for g in run.zs.grads[1:]:
        acc = acc + g.float()
    gbar = (acc / wl.W).double()
    del acc
    d = run.zs.master.double() - theta0.double()
    ulp = torch.abs(torch.nextafter(run.zs.master, torch.full_like(run.zs.master, float("inf"))) - run.zs.master)
    bound = wl.lr * wl.eps / (gbar.abs() + wl.eps) + 2 * ulp.double() + 1e-5 * wl.lr
    assert bool(((d + wl.lr * torch.sign(gbar)).abs() <= bound).all())
    assert bool((d[gbar == 0] == 0).all())
    del gbar, d, ulp, bound


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_gpt2_small_zero2(dtype):
    wl = wk.GPT2_SMALL
    sample = gh.sample_real_indices(wl.n, wl.W, [wl.n], k=16384)
    run = gh.Run(wl, zs.ZERO_SCHEME_Z2, dtype, sample=sample)
    theta0 = run.zs.master.clone()
    run.step()
    torch.cuda.synchronize()
    first_step_property(run, theta0)
    del theta0
    run.compare("after step 1")
    for _ in range(wl.steps - 1):
        run.step()
    run.compare()
    # the 16-bit copy is the round-to-nearest-even of the master, everywhere
    assert torch.equal(run.zs.p16, run.zs.master.to(TORCH16[dtype]))
    assert zs.zero_comm_bytes_per_rank(run.zs.ctx) == wl.steps * z.comm_bytes_closed_form(2, wl.n, wl.W)
    assert run.zs.stat(zs.ZERO_STAT_LAUNCHES) == 1 + wl.steps
    run.close()


def test_gpt2_xl_zero1():
    wl = wk.GPT2_XL
    sample = gh.sample_real_indices(wl.n, wl.W, [wl.n], k=16384)
    run = gh.Run(wl, zs.ZERO_SCHEME_Z1, "fp16", sample=sample)
    for _ in range(wl.steps):
        run.step()
    run.compare()
    assert torch.equal(run.zs.p16, run.zs.master.to(torch.float16))
    assert zs.zero_comm_bytes_per_rank(run.zs.ctx) == wl.steps * z.comm_bytes_closed_form(1, wl.n, wl.W)
    run.close()


def test_zero3_layer_units():
    """24 units of 50,331,648 on 8 ranks: sampled parity, the gathered units
    hold the 16-bit cast of the master as it was before the step (forward in
    unit order, backward in reverse), traffic 3 (N-1)/N 2 Psi per step, at
    most two unit buffers live, 3 launches per unit per step."""
    wl = wk.LAYER_UNITS
    U, S_u = len(wl.units()), wl.units()[0] // wl.W
    sample = gh.sample_real_indices(wl.n, wl.W, wl.units(), k=16384)
    run = gh.Run(wl, zs.ZERO_SCHEME_Z3, "bf16", sample=sample)
    unit_of = sample // wl.units()[0]
    seen = []
    bufs = {b.data_ptr(): b for b in run.zs.unit_bufs}

    def hook(_user, phase, unit, buf, stream):
        local = torch.from_numpy(sample[unit_of == unit] - unit * wl.units()[0]).cuda()
        s = torch.cuda.ExternalStream(stream) if stream else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            seen.append((phase, unit, bufs[buf][local].clone()))

    run.zs.set_unit_hook(hook)
    launches0 = run.zs.stat(zs.ZERO_STAT_LAUNCHES)
    for t in range(1, wl.steps + 1):
        torch.cuda.synchronize()
        before_gpu = gh.bits_of(run.zs.working_copy()[run.sample_flat])
        before_orc = run.oracle.master.copy()
        seen.clear()
        run.step()
        torch.cuda.synchronize()
        assert [(p, u) for p, u, _ in seen] == [(0, u) for u in range(U)] + [(1, u) for u in reversed(range(U))]
        for phase, u, vals in seen:
            sel = unit_of == u
            got = gh.bits_of(vals)
            assert np.array_equal(got, before_gpu[sel]), f"gathered unit {u} phase {phase} t={t}"
            gh.assert_16bit_band(got, before_orc[sel], "bf16", f"gathered unit {u} phase {phase} t={t}")
    run.compare()
    assert zs.zero_comm_bytes_per_rank(run.zs.ctx) == wl.steps * 6_341_787_648
    assert run.zs.stat(zs.ZERO_STAT_LAUNCHES) - launches0 == wl.steps * 3 * U
    assert run.zs.stat(zs.ZERO_STAT_PEAK_LIVE_ELEMS) == 2 * S_u * wl.W
    assert run.zs.stat(zs.ZERO_STAT_LIVE_ELEMS) == 0
    run.close()


def test_schemes_bit_identical_at_gpt2_small_size():
    """Scheme invariance at full size: DP, ZeRO-1, ZeRO-2 and ZeRO-3 (the whole
    vector as one unit, and as 12 layer-sized units) on the same 124,439,808
    gradients leave the same master, m, v and 16-bit copy, bit for bit."""
    wl = wk.scaled(wk.GPT2_SMALL, steps=2)
    theta0 = wk.draw_theta0(wl, "cuda")
    twelve = [wl.n // 12] * 11 + [wl.n - 11 * (wl.n // 12)]
    cases = [(zs.ZERO_SCHEME_DP, [wl.n]), (zs.ZERO_SCHEME_Z1, [wl.n]), (zs.ZERO_SCHEME_Z2, [wl.n]),
             (zs.ZERO_SCHEME_Z3, [wl.n]), (zs.ZERO_SCHEME_Z3, twelve)]
    steps = [zs.ZeroStep(s, wl.W, u, "bf16", theta0=theta0) for s, u in cases]
    src = wk.GradSource(wl, "bf16", "cuda")
    for t in range(1, wl.steps + 1):
        draws = src.step(t)
        for st in steps:
            g = st.new_grad_buffers()
            for b, d in zip(g, draws):
                st.place_(b, d)
            st.step(g, wl.lr, wl.beta1, wl.beta2, wl.eps, t)
            del g
        del draws
    torch.cuda.synchronize()
    ref = steps[0]
    ref_idx = ref.real_index()
    for st in steps[1:]:
        idx = st.real_index()
        for a, b in ((ref.master, st.master), (ref.m, st.m), (ref.v, st.v)):
            assert torch.equal(a[ref_idx].view(torch.int32), b[idx].view(torch.int32))
        assert torch.equal(ref.working_copy()[ref_idx].view(torch.int16), st.working_copy()[idx].view(torch.int16))
    for st in steps:
        st.close()
