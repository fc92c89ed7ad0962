"""The ZeRO-3 two-stream schedule under perturbed timing (GPU needed).

With a unit hook, each gather runs on its own stream and waits only for the
event that released the buffer it reuses.  If that wait were missing or
misplaced, the next gather would overwrite a unit while the caller's work
on it still reads it.  Here the caller's work on every gathered unit first
sleeps for a random, bounded number of GPU cycles, which widens any such
window to tens of microseconds, then snapshots the unit.  Every snapshot
must equal the working copy from before the step (no unit is updated before
its backward gather), released buffers are poisoned with NaN so that a
late read cannot pass by luck, and the final state must equal that of the
one-stream schedule bit for bit."""

import numpy as np
import pytest
import torch

import workloads as wk
import zero_sharded_mixed_step_gb300 as zs

pytestmark = pytest.mark.gpu

UNITS = [65_536 * 3 + 5, 1_000_003, 17, 262_144, 65_536 * 3 + 5, 9]
STEPS = 3


@pytest.fixture(scope="module", autouse=True)
def _built():
    from zero_sharded_mixed_step_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _flat_before(st):
    """The working copy in flat order, as the gathers must deliver it."""
    return st.working_copy().clone()


@pytest.mark.parametrize("seed", [0, 1])
def test_two_stream_schedule_under_random_delays(seed):
    wl = wk.scaled(wk.LAYER_UNITS, unit_sizes=UNITS, W=8, steps=STEPS, name="races")
    theta0 = wk.draw_theta0(wl, "cuda")
    s_up, s_g = torch.cuda.Stream(), torch.cuda.Stream()
    st = zs.ZeroStep(zs.ZERO_SCHEME_Z3, wl.W, UNITS, "bf16", theta0=theta0, stream=s_up, gather_stream=s_g,
                     with_grad_buffers=True)
    ref = zs.ZeroStep(zs.ZERO_SCHEME_Z3, wl.W, UNITS, "bf16", theta0=theta0, with_grad_buffers=True)
    st.set_debug(zs.ZERO_DEBUG_POISON_RELEASED)
    rng = np.random.default_rng(seed)
    bufs = {b.data_ptr(): b for b in st.unit_bufs}
    seen = []

    def hook(_user, phase, unit, buf, stream):
        s = torch.cuda.ExternalStream(stream)
        n = st.shard[unit] * wl.W
        with torch.cuda.stream(s):
            torch.cuda._sleep(int(rng.integers(0, 200_000)))    # bounded: at most ~0.1 ms at 2 GHz
            seen.append((phase, unit, bufs[buf][:n].clone()))

    st.set_unit_hook(hook)
    src = wk.GradSource(wl, "bf16", "cuda")
    for t in range(1, STEPS + 1):
        torch.cuda.synchronize()
        for r, d in enumerate(src.step(t)):
            st.place_(st.grads[r], d)
            ref.grads[r].copy_(st.grads[r])
        before = _flat_before(st)
        torch.cuda.synchronize()
        seen.clear()
        st.step(st.grads, wl.lr, wl.beta1, wl.beta2, wl.eps, t)
        ref.step(ref.grads, wl.lr, wl.beta1, wl.beta2, wl.eps, t)
        torch.cuda.synchronize()
        U = len(UNITS)
        assert [(p, u) for p, u, _ in seen] == [(0, u) for u in range(U)] + [(1, u) for u in reversed(range(U))]
        for phase, u, got in seen:
            o = st.off[u]
            want = before[o:o + got.numel()]
            assert torch.equal(got.view(torch.int16), want.view(torch.int16)), f"t={t} phase {phase} unit {u}"
    st.sync()
    for a, b, what in ((st.master, ref.master, "master"), (st.m, ref.m, "m"), (st.v, ref.v, "v")):
        assert torch.equal(a, b), what
    assert torch.equal(st.working_copy(), ref.working_copy())
    st.close()
    ref.close()
