"""Behaviour of the C ABI on the GPU: checkpoint and resume, ZeRO-3 driven by
the caller, the bounded wait, launch counts, rank fault injection."""

import numpy as np
import pytest
import torch

import workloads as wk
import zero_sharded_mixed_step_gb300 as zs
from oracle import zero_oracle as z
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from zero_sharded_mixed_step_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _grads(wl, dtype, steps, zstep):
    src = wk.GradSource(wl, dtype, "cuda")
    out = []
    for t in range(1, steps + 1):
        per = []
        for d in src.step(t):
            buf = torch.zeros(zstep.n_pad, dtype=zstep.grad_torch_dtype, device="cuda")
            zstep.place_(buf, d)
            per.append(buf)
        out.append(per)
    return out


def _state(zstep):
    torch.cuda.synchronize()
    return [x.clone() for x in (zstep.master, zstep.m, zstep.v, zstep.working_copy())]


@pytest.mark.parametrize("scheme,units", [(zs.ZERO_SCHEME_Z1, [300_007]), (zs.ZERO_SCHEME_Z3, [100_000, 200_007])])
def test_checkpoint_resume_is_bitwise(scheme, units):
    """10 steps in one go equal 5 steps, a round trip of master / m / v / t
    through host memory into a fresh context, and 5 more steps."""
    wl = wk.scaled(wk.GPT2_SMALL, unit_sizes=units, W=4, steps=10, name="ckpt")
    theta0 = wk.draw_theta0(wl, "cuda")
    a = zs.ZeroStep(scheme, 4, units, "bf16", theta0=theta0)
    grads = _grads(wl, "bf16", 10, a)
    for t in range(1, 11):
        a.step(grads[t - 1], wl.lr, wl.beta1, wl.beta2, wl.eps, t)
    want = _state(a)
    b = zs.ZeroStep(scheme, 4, units, "bf16", theta0=theta0)
    for t in range(1, 6):
        b.step(grads[t - 1], wl.lr, wl.beta1, wl.beta2, wl.eps, t)
    host = [np.empty(b.n_pad, np.float32) for _ in range(3)]
    t_saved = zs.zero_get_state(b.ctx, *[h.ctypes.data for h in host])
    assert t_saved == 5
    c = zs.ZeroStep(scheme, 4, units, "bf16")
    zs.zero_set_state(c.ctx, *[h.ctypes.data for h in host], t_saved)
    with pytest.raises(zs.ZeroError) as e:
        c.step(grads[5], wl.lr, wl.beta1, wl.beta2, wl.eps, 5)
    assert e.value.code == zs.ZERO_E_STATE
    for t in range(6, 11):
        c.step(grads[t - 1], wl.lr, wl.beta1, wl.beta2, wl.eps, t)
    got = _state(c)
    for x, y in zip(want, got):
        assert torch.equal(x.view(torch.int16) if x.element_size() == 2 else x.view(torch.int32),
                           y.view(torch.int16) if y.element_size() == 2 else y.view(torch.int32))
    for s in (a, b, c):
        s.close()


def test_zero3_driven_by_caller_equals_step():
    """gather / release / update driven unit by unit through the ABI gives the
    same bits, the same traffic and the same counters as zero_step."""
    units = [70_001, 0, 65_536, 9]
    wl = wk.scaled(wk.LAYER_UNITS, unit_sizes=units, steps=3, name="manual")
    theta0 = wk.draw_theta0(wl, "cuda")
    a = zs.ZeroStep(zs.ZERO_SCHEME_Z3, wl.W, units, "bf16", theta0=theta0)
    b = zs.ZeroStep(zs.ZERO_SCHEME_Z3, wl.W, units, "bf16", theta0=theta0)
    grads = _grads(wl, "bf16", wl.steps, a)
    buf = torch.zeros(a.sizes["unit_buf"], dtype=torch.bfloat16, device="cuda")
    hp = (wl.lr, wl.beta1, wl.beta2, wl.eps)
    for t in range(1, wl.steps + 1):
        a.step(grads[t - 1], *hp, t)
        for u in range(len(units)):
            zs.zero_gather_unit(b.ctx, u, buf)
            with pytest.raises(zs.ZeroError) as e:
                zs.zero_gather_unit(b.ctx, u, buf)
            assert e.value.code == zs.ZERO_E_STATE
            zs.zero_release_unit(b.ctx, u)
        for u in reversed(range(len(units))):
            zs.zero_gather_unit(b.ctx, u, buf)
            torch.cuda.synchronize()
            o, s = b.off[u], b.shard[u]
            assert torch.equal(buf[: s * wl.W], b.working_copy()[o:o + s * wl.W])
            zs.zero_update_unit(b.ctx, u, grads[t - 1], *hp, t)
            zs.zero_release_unit(b.ctx, u)
    for x, y in zip(_state(a), _state(b)):
        assert torch.equal(x, y)
    assert zs.zero_comm_bytes_per_rank(a.ctx) == zs.zero_comm_bytes_per_rank(b.ctx)
    L = z.Layout(wl.W, units)
    assert zs.zero_comm_bytes_per_rank(a.ctx) == wl.steps * 3 * sum(z.ring_bytes_per_rank(wl.W, s) for s in L.S)
    for k in (zs.ZERO_STAT_GATHERS, zs.ZERO_STAT_SCATTERS, zs.ZERO_STAT_T):
        assert a.stat(k) == b.stat(k)
    assert b.stat(zs.ZERO_STAT_LIVE_ELEMS) == 0
    a.close()
    b.close()


def test_sync_deadline_and_recovery():
    """zero_sync gives up at its deadline while the stream is still busy (a
    bounded GPU sleep ahead of the step), leaves the work running, and a
    later wait succeeds: the context stays usable."""
    wl = wk.scaled(wk.GPT2_SMALL, n=1 << 16, W=4, steps=2, name="sync")
    s = zs.ZeroStep(zs.ZERO_SCHEME_Z1, 4, [wl.n], "fp16", theta0=wk.draw_theta0(wl, "cuda"))
    grads = _grads(wl, "fp16", 2, s)
    torch.cuda.synchronize()
    torch.cuda._sleep(400_000_000)       # a few hundred ms of spinning on the context's stream
    s.step(grads[0], wl.lr, wl.beta1, wl.beta2, wl.eps, 1)
    with pytest.raises(zs.ZeroError) as e:
        s.sync(timeout_ms=1)
    assert e.value.code == zs.ZERO_E_TIMEOUT
    s.sync(timeout_ms=60_000)
    s.step(grads[1], wl.lr, wl.beta1, wl.beta2, wl.eps, 2)
    s.sync()
    assert s.stat(zs.ZERO_STAT_DEVICE_ERRORS) == 0
    s.close()


def test_rank_fault_injection_launches_nothing():
    wl = wk.scaled(wk.LAYER_UNITS, unit_sizes=[4096, 4096], steps=2, name="fault")
    s = zs.ZeroStep(zs.ZERO_SCHEME_Z3, wl.W, [4096, 4096], "bf16", theta0=wk.draw_theta0(wl, "cuda"))
    grads = _grads(wl, "bf16", 1, s)
    n0 = s.stat(zs.ZERO_STAT_LAUNCHES)
    zs.zero_mark_rank(s.ctx, 3, False)
    with pytest.raises(zs.ZeroError) as e:
        s.step(grads[0], wl.lr, wl.beta1, wl.beta2, wl.eps, 1)
    assert e.value.code == zs.ZERO_E_RANK
    assert s.stat(zs.ZERO_STAT_LAUNCHES) == n0 and s.stat(zs.ZERO_STAT_COMM_BYTES) == 0
    zs.zero_mark_rank(s.ctx, 3, True)
    s.step(grads[0], wl.lr, wl.beta1, wl.beta2, wl.eps, 1)
    s.sync()
    # no hook: one launch gathers both units for the forward pass, and one pass per
    # unit gathers and updates it for the backward pass
    assert s.stat(zs.ZERO_STAT_LAUNCHES) == n0 + 1 + 2
    s.close()


def test_zero3_backward_gather_fused_into_update():
    """Without a unit hook the backward gather of each unit is done by the
    unit's update pass: after the step the two unit buffers hold the last two
    units gathered (units 1 and 0, in backward order) as they were before the
    update, bit for bit, and the traffic counts three collectives per unit."""
    units = [100_003, 65_536, 70_001]
    wl = wk.scaled(wk.LAYER_UNITS, unit_sizes=units, steps=2, name="fused_gather")
    s = zs.ZeroStep(zs.ZERO_SCHEME_Z3, wl.W, units, "bf16", theta0=wk.draw_theta0(wl, "cuda"))
    grads = _grads(wl, "bf16", 2, s)
    for t in (1, 2):
        torch.cuda.synchronize()
        before = s.working_copy().clone()
        s.step(grads[t - 1], wl.lr, wl.beta1, wl.beta2, wl.eps, t)
        torch.cuda.synchronize()
        U = len(units)
        for u, seq in ((1, 2 * U - 2), (0, 2 * U - 1)):
            buf = s.unit_bufs[seq & 1]
            o, sh = s.off[u], s.shard[u]
            assert torch.equal(buf[: sh * wl.W].view(torch.int16), before[o:o + sh * wl.W].view(torch.int16)), (t, u)
        assert not torch.equal(before, s.working_copy())
    L = z.Layout(wl.W, units)
    assert zs.zero_comm_bytes_per_rank(s.ctx) == 2 * 3 * sum(z.ring_bytes_per_rank(wl.W, x) for x in L.S)
    # a cast per unit, then per step the forward gathers two units per launch (the
    # units have different sizes) and one pass per unit gathers and updates it
    U = len(units)
    assert s.stat(zs.ZERO_STAT_LAUNCHES) == U + 2 * ((U + 1) // 2 + U)
    s.close()


def test_tiny_and_empty_vectors():
    """n = 0 (nothing to do), n below one vector group, a single rank."""
    for n, W in ((0, 4), (3, 4), (7, 1), (9, 8)):
        wl = wk.scaled(wk.TINY, n=n, W=W, steps=2, name=f"edge{n}")
        if n == 0:
            s = zs.ZeroStep(zs.ZERO_SCHEME_Z1, W, [0], "fp16")
            s.step(s.new_grad_buffers(), 1e-3, 0.9, 0.999, 1e-8, 1)
            s.sync()
            s.close()
            continue
        run = gh.Run(wl, zs.ZERO_SCHEME_Z1, "fp16")
        for _ in range(2):
            run.step()
            run.compare()
        assert run.padding_is_zero()
        run.close()


def test_bounded_device_wait_reports_and_recovers():
    """A bulk-staged launch whose tile never loads (injected on purpose) gives
    up after its bounded wait instead of hanging: zero_sync reports
    ZERO_E_STATE, the device error count rises, and the context keeps
    working for the next steps."""
    n, W = 8 * 2048 * 200, 8
    wl = wk.scaled(wk.GPT2_SMALL, n=n, W=W, steps=3, name="stall")
    s = zs.ZeroStep(zs.ZERO_SCHEME_Z2, W, [n], "bf16", theta0=wk.draw_theta0(wl, "cuda"))
    s.set_variant(zs.ZERO_VARIANT_BULK)
    grads = _grads(wl, "bf16", 3, s)
    s.step(grads[0], wl.lr, wl.beta1, wl.beta2, wl.eps, 1)
    s.sync(timeout_ms=60_000)
    assert s.stat(zs.ZERO_STAT_DEVICE_ERRORS) == 0 and s.stat(zs.ZERO_STAT_LAST_VARIANT) == zs.ZERO_VARIANT_BULK
    zs.zero_inject_stall(s.ctx, 1)
    s.step(grads[1], wl.lr, wl.beta1, wl.beta2, wl.eps, 2)
    with pytest.raises(zs.ZeroError) as e:
        s.sync(timeout_ms=60_000)
    assert e.value.code == zs.ZERO_E_STATE and "bounded device waits" in str(e.value)
    assert s.stat(zs.ZERO_STAT_DEVICE_ERRORS) == 1
    s.step(grads[2], wl.lr, wl.beta1, wl.beta2, wl.eps, 3)     # still usable, and no new error
    s.sync(timeout_ms=60_000)
    assert s.stat(zs.ZERO_STAT_DEVICE_ERRORS) == 1
    s.close()


def test_poison_released_units():
    """With ZERO_DEBUG_POISON_RELEASED a released unit buffer holds NaN
    (0x7FFF), both through the caller-driven API and inside zero_step, while
    everything read before the release, and the step's results, are unchanged."""
    units = [4096 * 3 + 5, 70_001]
    W = 8
    wl = wk.scaled(wk.LAYER_UNITS, unit_sizes=units, steps=2, name="poison")
    theta0 = wk.draw_theta0(wl, "cuda")
    plain = zs.ZeroStep(zs.ZERO_SCHEME_Z3, W, units, "bf16", theta0=theta0)
    s = zs.ZeroStep(zs.ZERO_SCHEME_Z3, W, units, "bf16", theta0=theta0)
    s.set_debug(zs.ZERO_DEBUG_POISON_RELEASED)
    grads = _grads(wl, "bf16", 2, s)
    hp = (wl.lr, wl.beta1, wl.beta2, wl.eps)
    # caller-driven: gather, check, release, check the poison
    buf = torch.zeros(s.sizes["unit_buf"], dtype=torch.bfloat16, device="cuda")
    n0 = s.shard[0] * W
    zs.zero_gather_unit(s.ctx, 0, buf)
    torch.cuda.synchronize()
    assert torch.equal(buf[:n0], s.working_copy()[:n0])
    zs.zero_release_unit(s.ctx, 0)
    torch.cuda.synchronize()
    assert bool((buf[:n0].view(torch.int16) == 0x7FFF).all())
    # inside zero_step: what the hook reads comes before the release
    seen = []

    def hook(_user, phase, unit, ptr, stream):
        st = torch.cuda.ExternalStream(stream) if stream else torch.cuda.current_stream()
        with torch.cuda.stream(st):
            b = next(x for x in s.unit_bufs if x.data_ptr() == ptr)
            seen.append((unit, b[: s.shard[unit] * W].clone()))

    s.set_unit_hook(hook)
    before = s.working_copy().clone()
    s.step(grads[0], *hp, 1)
    plain.set_unit_hook(lambda *a: None)
    plain.step(grads[0], *hp, 1)
    torch.cuda.synchronize()
    for unit, vals in seen:
        o = s.off[unit]
        assert torch.equal(vals, before[o:o + vals.numel()])
    for b in s.unit_bufs:
        assert bool((b.view(torch.int16) == 0x7FFF).all())
    for x, y in ((plain.master, s.master), (plain.m, s.m), (plain.v, s.v)):
        assert torch.equal(x, y)
    assert torch.equal(plain.working_copy(), s.working_copy())
    with pytest.raises(zs.ZeroError):
        zs.zero_set_debug(s.ctx, 8)
    plain.close()
    s.close()
