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


@pytest.mark.parametrize("scheme,units,W,chunk", [(zs.ZERO_SCHEME_Z2, [1_000_003], 8, 100_000),
                                                  (zs.ZERO_SCHEME_Z3, [262_147, 5, 500_000, 17], 5, 0)])
def test_host_fed_ring_under_random_delays(scheme, units, W, chunk):
    """zero_step_host's three streams, each held back by a random bounded
    sleep before every step, with three steps enqueued back to back and no
    host synchronisation between them: the two-slot staging ring, the
    read-back of each step and the next step's update of the same values
    must keep their order.  Each step's read-back must equal the working
    copy the device step had after that step; the final state must equal it
    bit for bit."""
    n = sum(units)
    wl = wk.scaled(wk.GPT2_SMALL, unit_sizes=units if scheme == zs.ZERO_SCHEME_Z3 else None, n=n, W=W, steps=3,
                   name="host_races")
    theta0 = wk.draw_theta0(wl, "cuda")
    s_up, sh, sd = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    a = zs.ZeroStep(scheme, W, units, "bf16", theta0=theta0)
    b = zs.ZeroStep(scheme, W, units, "bf16", theta0=theta0, stream=s_up)
    need = zs.zero_host_staging_bytes(scheme, W, units, chunk)
    staging = torch.empty(need, dtype=torch.uint8, device="cuda")
    out_elems = b.n_pad if scheme != zs.ZERO_SCHEME_Z3 else W * b.sizes["shard_store"]
    hp = (wl.lr, wl.beta1, wl.beta2, wl.eps)
    src = wk.GradSource(wl, "bf16", "cuda")

    def result(st):
        return (st.p16 if scheme != zs.ZERO_SCHEME_Z3 else torch.cat(list(st.shard16))).cpu()

    host_grads, host_out, want = [], [], []
    for t in range(1, wl.steps + 1):
        dev = []
        for d in src.step(t):
            g = torch.zeros(a.n_pad, dtype=a.grad_torch_dtype, device="cuda")
            a.place_(g, d)
            dev.append(g)
        a.step(dev, *hp, t)
        torch.cuda.synchronize()
        host_grads.append([g.cpu().pin_memory() for g in dev])
        host_out.append(torch.zeros(out_elems, dtype=b.work_torch_dtype).pin_memory())
        want.append(result(a))
    torch.cuda.synchronize()
    rng = np.random.default_rng(len(units))
    for t in range(1, wl.steps + 1):
        for s in (s_up, sh, sd):
            with torch.cuda.stream(s):
                torch.cuda._sleep(int(rng.integers(0, 400_000)))   # bounded: at most ~0.2 ms at 2 GHz
        zs.zero_step_host(b.ctx, scheme, W, n, host_grads[t - 1], host_out[t - 1], staging, need, chunk, *hp, t,
                          sh, sd)
    b.sync(timeout_ms=60_000)
    torch.cuda.synchronize()
    for t in range(1, wl.steps + 1):
        assert torch.equal(host_out[t - 1].view(torch.int16), want[t - 1].view(torch.int16)), f"read-back of step {t}"
    for x, y, what in ((a.master, b.master, "master"), (a.m, b.m, "m"), (a.v, b.v, "v")):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32)), what
    a.close()
    b.close()
