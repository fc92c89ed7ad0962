"""ZeRO-3 steps replayed from a CUDA graph (zero_set_graph) against ordinary
launches: the same bits, the same counters, and the fallbacks (a hook,
timing brackets, a variant change) (GPU needed)."""

import pytest
import torch

import workloads as wk
import zero_sharded_mixed_step_gb300 as zs
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu

STATS = (zs.ZERO_STAT_COMM_BYTES, zs.ZERO_STAT_LAUNCHES, zs.ZERO_STAT_GATHERS, zs.ZERO_STAT_SCATTERS,
         zs.ZERO_STAT_PEAK_LIVE_ELEMS, zs.ZERO_STAT_LIVE_ELEMS, zs.ZERO_STAT_T, zs.ZERO_STAT_DEVICE_ERRORS)


# Graph capture needs a created stream (not the legacy default stream); every
# test runs all its work, torch's included, on this one.
STREAM = None


def _stream():
    global STREAM
    if STREAM is None:
        STREAM = torch.cuda.Stream()
    return STREAM


def _pair(units, W, dtype="bf16"):
    wl = wk.scaled(wk.LAYER_UNITS, unit_sizes=units, W=W, steps=6, name="graph")
    theta0 = wk.draw_theta0(wl, "cuda")
    made = []
    for graph in (False, True):
        st = zs.ZeroStep(zs.ZERO_SCHEME_Z3, W, units, dtype, theta0=theta0, stream=_stream())
        if graph:
            st.set_graph(True)
        made.append(st)
    return wl, made


def _draw(wl, st, src, t):
    bufs = st.new_grad_buffers()
    for b, d in zip(bufs, src.step(t)):
        st.place_(b, d)
    return bufs


def _same(a, b, what):
    for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
        assert torch.equal(x.view(torch.int32), y.view(torch.int32)), what
    assert torch.equal(a.working_copy().view(torch.int16), b.working_copy().view(torch.int16)), what
    for k in STATS:
        assert a.stat(k) == b.stat(k), (what, k)


def test_graph_steps_equal_launched_steps():
    """Six steps, a new set of gradient buffers every step (the graph must pick
    up the new pointers and each step's coefficients), bit for bit."""
    with torch.cuda.stream(_stream()):
        _graph_steps_equal_launched_steps()


def _graph_steps_equal_launched_steps():
    units = [50_331_648 // 8, 1_000_003, 17, 0, 4096]
    wl, (plain, graph) = _pair(units, 8)
    src = wk.GradSource(wl, "bf16", "cuda")
    for t in range(1, wl.steps + 1):
        grads = _draw(wl, plain, src, t)
        plain.step(grads, wl.lr, wl.beta1, wl.beta2, wl.eps, t)
        graph.step(grads, wl.lr, wl.beta1, wl.beta2, wl.eps, t)
        torch.cuda.synchronize()
        _same(plain, graph, f"t={t}")
    plain.close()
    graph.close()


@pytest.mark.parametrize("units", [[262_144, 262_147, 100_000], [262_144, 262_144, 262_144]],
                         ids=["ragged", "one_size"])
def test_graph_steps_fall_back_and_recapture(units):
    """A hook, timing brackets and a variant change run the ordinary launches
    (or capture anew); every step still matches the plain context.  Units of
    one size take the one-launch forward gathers, ragged ones a launch per
    pair, in the graph and outside it."""
    with torch.cuda.stream(_stream()):
        _graph_steps_fall_back_and_recapture(units)


def _graph_steps_fall_back_and_recapture(units):
    wl, (plain, graph) = _pair(units, 8, "fp16")
    src = wk.GradSource(wl, "fp16", "cuda")
    hp = (wl.lr, wl.beta1, wl.beta2, wl.eps)
    calls = []
    for t in range(1, 7):
        grads = _draw(wl, plain, src, t)
        if t == 2:
            graph.set_unit_hook(lambda user, phase, unit, buf, stream: calls.append((phase, unit)))
            plain.set_unit_hook(lambda user, phase, unit, buf, stream: None)
        if t == 3:
            graph.set_unit_hook(None)
            plain.set_unit_hook(None)
            zs.zero_enable_timing(graph.ctx, True)
        if t == 4:
            zs.zero_enable_timing(graph.ctx, False)
            graph.set_variant(zs.ZERO_VARIANT_VECTOR)
            plain.set_variant(zs.ZERO_VARIANT_VECTOR)
        plain.step(grads, *hp, t)
        graph.step(grads, *hp, t)
        torch.cuda.synchronize()
        _same(plain, graph, f"t={t}")
    assert len(calls) == 2 * len(units)          # the hooked step ran unit by unit
    ms, n = zs.zero_read_timing(graph.ctx, zs.ZERO_KERNEL_FUSED)
    assert n == len(units)                        # the timed step ran as ordinary launches
    ms, n = zs.zero_read_timing(graph.ctx, zs.ZERO_KERNEL_GATHER)
    assert n == (1 if len(set(units)) == 1 else (len(units) + 1) // 2)   # its forward gathers
    graph.set_graph(False)
    plain.close()
    graph.close()


def test_graph_steps_against_the_oracle():
    units = [1_000_003, 17, 250_000, 7]
    W = 5
    wl = wk.scaled(wk.LAYER_UNITS, unit_sizes=units, W=W, steps=4, name="graph_oracle")
    with torch.cuda.stream(_stream()):
        run = gh.Run(wl, zs.ZERO_SCHEME_Z3, "bf16", units=units, gather_stream=False)
        run.zs.set_graph(True)
        for _ in range(wl.steps):
            run.step()
            run.compare()
        assert run.padding_is_zero()
        run.close()


def test_full_zero3_workload_as_the_benchmark_runs_it():
    """The 24 x 50,331,648 workload on 8 ranks without a hook and with graph
    replay, the launch configuration the benchmark times: sampled parity with
    the oracle, bit-identical to ordinary launches on the same gradients,
    traffic 6,341,787,648 B and U + 1 launches per step (every unit has the
    same size, so the forward gathers go in one launch), two unit buffers at
    most."""
    wl = wk.scaled(wk.LAYER_UNITS, steps=3)
    U, S_u = len(wl.units()), wl.units()[0] // wl.W
    sample = gh.sample_real_indices(wl.n, wl.W, wl.units(), k=16384)
    with torch.cuda.stream(_stream()):
        run = gh.Run(wl, zs.ZERO_SCHEME_Z3, "bf16", sample=sample, gather_stream=False)
        run.zs.set_graph(True)
        plain = zs.ZeroStep(zs.ZERO_SCHEME_Z3, wl.W, wl.units(), "bf16",
                            theta0=wk.draw_theta0(wl, "cuda"), stream=_stream())
        launches0 = run.zs.stat(zs.ZERO_STAT_LAUNCHES)
        for _ in range(wl.steps):
            run.step()
            plain.step(run.zs.grads, wl.lr, wl.beta1, wl.beta2, wl.eps, run.t)
        torch.cuda.synchronize()
        run.compare()
        for x, y in ((run.zs.master, plain.master), (run.zs.m, plain.m), (run.zs.v, plain.v)):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32))
        for a, b in zip(run.zs.shard16, plain.shard16):
            assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        assert zs.zero_comm_bytes_per_rank(run.zs.ctx) == wl.steps * 6_341_787_648
        assert run.zs.stat(zs.ZERO_STAT_LAUNCHES) - launches0 == wl.steps * (U + 1)
        assert run.zs.stat(zs.ZERO_STAT_PEAK_LIVE_ELEMS) == 2 * S_u * wl.W
        assert run.zs.stat(zs.ZERO_STAT_LIVE_ELEMS) == 0
        plain.close()
        run.close()
