"""Every entry point writes only inside the buffers it is given (GPU needed).

Each device and host buffer is cut from an Arena with 64 KB of seeded random
bytes before and after it, at the least alignment the ABI accepts; after the
steps every guard byte must still hold its pattern.  Sizes are ragged (n not
a multiple of W or of any tile, units of 0, 5 and 17 values, n = 1) so that
every tail path runs.  Each case also steps a context whose buffers come
from ordinary allocations and requires the same state bit for bit, so the
placement changes nothing."""

import numpy as np
import pytest
import torch

import zero_sharded_mixed_step_gb300 as zs
from tests.canary import GUARD, Arena

pytestmark = pytest.mark.gpu

HP = (1e-3, 0.9, 0.95, 1e-8)
SLACK = GUARD + 1024            # room per buffer for its guard and its alignment


@pytest.fixture(scope="module", autouse=True)
def _built():
    from zero_sharded_mixed_step_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def theta0_of(n, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn(n, generator=g, device="cuda") * 0.02


def fill_grads(grads, real_index, t):
    """Rank r's gradient at step t: N(0, 1e-3) at the real positions, zero in the padding."""
    for r, g in enumerate(grads):
        gen = torch.Generator(device="cuda").manual_seed(1000 * t + r)
        g.zero_()
        if real_index.numel():
            g[real_index] = (torch.randn(real_index.numel(), generator=gen, device="cuda") * 1e-3).to(g.dtype)


def z_bytes(scheme, W, units):
    """Device bytes of a context's buffers and its W gradient vectors, with slack."""
    s = zs.zero_buffer_sizes(scheme, W, units)
    payload = 12 * s["n_pad"] + 2 * s["p16"] + 2 * W * s["n_pad"]
    buffers = 3 + 1 + W
    if scheme == zs.ZERO_SCHEME_Z3:
        payload += 2 * W * s["shard_store"] + 4 * s["unit_buf"]
        buffers += W + 2
    return payload, buffers


def assert_same_state(a, b):
    for x, y, what in ((a.master, b.master, "master"), (a.m, b.m, "m"), (a.v, b.v, "v")):
        assert torch.equal(x, y), what
    assert torch.equal(a.working_copy(), b.working_copy()), "working copy"


FLAT = [(3, 1), (8, 4097), (16, 1_000_003), (5, 262_147), (8, 2_000_001)]


@pytest.mark.parametrize("scheme", [zs.ZERO_SCHEME_DP, zs.ZERO_SCHEME_Z1, zs.ZERO_SCHEME_Z2])
@pytest.mark.parametrize("W,n", FLAT)
def test_flat_step_writes_only_its_buffers(scheme, W, n):
    for variant in (zs.ZERO_VARIANT_VECTOR, zs.ZERO_VARIANT_BULK):
        payload, buffers = z_bytes(scheme, W, [n])
        arena = Arena(payload + buffers * SLACK, "cuda", seed=n + W + variant)
        theta0 = theta0_of(n, seed=n)
        st = zs.ZeroStep(scheme, W, [n], "bf16", theta0=theta0, alloc=arena)
        ref = zs.ZeroStep(scheme, W, [n], "bf16", theta0=theta0)
        st.set_variant(variant)
        ref.set_variant(variant)
        grads = st.new_grad_buffers()
        for t in (1, 2, 3):
            fill_grads(grads, st.real_index(), t)
            st.step(grads, *HP, t)
            ref.step(grads, *HP, t)
        arena.check()
        assert_same_state(st, ref)
        st.close()
        ref.close()


UNITS = [17, 0, 4096, 1_000_003, 5, 262_144]


@pytest.mark.parametrize("W", [5, 8])
@pytest.mark.parametrize("mode", ["fused", "hook", "graph", "poison"])
def test_zero3_step_writes_only_its_buffers(W, mode):
    payload, buffers = z_bytes(zs.ZERO_SCHEME_Z3, W, UNITS)
    arena = Arena(payload + buffers * SLACK, "cuda", seed=W)
    theta0 = theta0_of(sum(UNITS), seed=W)
    s_up, s_g = torch.cuda.Stream(), torch.cuda.Stream()
    st = zs.ZeroStep(zs.ZERO_SCHEME_Z3, W, UNITS, "bf16", theta0=theta0, alloc=arena, stream=s_up,
                     gather_stream=s_g if mode == "hook" else None)
    ref = zs.ZeroStep(zs.ZERO_SCHEME_Z3, W, UNITS, "bf16", theta0=theta0)
    if mode == "hook":
        st.set_unit_hook(lambda user, phase, unit, buf, stream: None)
    elif mode == "graph":
        st.set_graph(True)
    elif mode == "poison":
        st.set_debug(zs.ZERO_DEBUG_POISON_RELEASED)
    grads = st.new_grad_buffers()
    for t in (1, 2, 3):
        torch.cuda.synchronize()
        fill_grads(grads, st.real_index(), t)
        torch.cuda.synchronize()
        st.step(grads, *HP, t)
        ref.step(grads, *HP, t)
    torch.cuda.synchronize()
    arena.check()
    assert_same_state(st, ref)
    st.close()
    ref.close()


def test_zero3_caller_driven_units_write_only_their_buffers():
    """zero_gather_unit into the caller's buffers, zero_update_unit in reverse order."""
    W = 8
    payload, buffers = z_bytes(zs.ZERO_SCHEME_Z3, W, UNITS)
    s = zs.zero_buffer_sizes(zs.ZERO_SCHEME_Z3, W, UNITS)
    arena = Arena(payload + 2 * s["unit_buf"] * len(UNITS) + (buffers + len(UNITS)) * SLACK, "cuda", seed=11)
    theta0 = theta0_of(sum(UNITS), seed=11)
    st = zs.ZeroStep(zs.ZERO_SCHEME_Z3, W, UNITS, "bf16", theta0=theta0, alloc=arena)
    ref = zs.ZeroStep(zs.ZERO_SCHEME_Z3, W, UNITS, "bf16", theta0=theta0)
    dsts = [arena.zeros(max(1, st.shard[u] * W), torch.bfloat16, f"gather of unit {u}") for u in range(len(UNITS))]
    grads = st.new_grad_buffers()
    for t in (1, 2):
        fill_grads(grads, st.real_index(), t)
        for u in range(len(UNITS)):
            zs.zero_gather_unit(st.ctx, u, dsts[u])
            zs.zero_release_unit(st.ctx, u)
        for u in reversed(range(len(UNITS))):
            zs.zero_gather_unit(st.ctx, u, dsts[u])
            zs.zero_update_unit(st.ctx, u, grads, *HP, t)
            zs.zero_release_unit(st.ctx, u)
        ref.step(grads, *HP, t)
    st.sync()
    arena.check()
    assert_same_state(st, ref)
    st.close()
    ref.close()


def test_bucketed_step_writes_only_its_buffers():
    W, n = 8, 1_000_003
    payload, buffers = z_bytes(zs.ZERO_SCHEME_Z2, W, [n])
    n_pad = zs.zero_buffer_sizes(zs.ZERO_SCHEME_Z2, W, [n])["n_pad"]
    rng = np.random.default_rng(5)
    cuts = sorted(set([0, n_pad] + [int(c) * 8 for c in rng.integers(1, n_pad // 8, 9)]))
    spans = list(zip(cuts[:-1], cuts[1:]))
    rng.shuffle(spans)
    arena = Arena(payload + 2 * W * n_pad + (buffers + W * len(spans)) * SLACK, "cuda", seed=5)
    theta0 = theta0_of(n, seed=5)
    st = zs.ZeroStep(zs.ZERO_SCHEME_Z2, W, [n], "fp16", theta0=theta0, alloc=arena)
    ref = zs.ZeroStep(zs.ZERO_SCHEME_Z2, W, [n], "fp16", theta0=theta0)
    grads = ref.new_grad_buffers()
    buckets = {span: [arena.zeros(span[1] - span[0], torch.float16) for _ in range(W)] for span in spans}
    for t in (1, 2):
        fill_grads(grads, ref.real_index(), t)
        for lo, hi in spans:
            for r in range(W):
                buckets[(lo, hi)][r].copy_(grads[r][lo:hi])
            zs.zero_step_bucket(st.ctx, lo, hi - lo, buckets[(lo, hi)], *HP, t)
        ref.step(grads, *HP, t)
    st.sync()
    arena.check()
    assert_same_state(st, ref)
    st.close()
    ref.close()


@pytest.mark.parametrize("scheme,units,chunk", [(zs.ZERO_SCHEME_Z2, [1_000_003], 65_536),
                                                (zs.ZERO_SCHEME_Z1, [4097], 0),
                                                (zs.ZERO_SCHEME_Z3, UNITS, 0)])
def test_host_fed_step_writes_only_its_buffers(scheme, units, chunk):
    W = 8
    payload, buffers = z_bytes(scheme, W, units)
    need = zs.zero_host_staging_bytes(scheme, W, units, chunk)
    dev = Arena(payload + need + (buffers + 1) * SLACK, "cuda", seed=21)
    s = zs.zero_buffer_sizes(scheme, W, units)
    out_elems = s["n_pad"] if scheme != zs.ZERO_SCHEME_Z3 else W * s["shard_store"]
    host = Arena(2 * W * s["n_pad"] + 2 * out_elems + (W + 1) * SLACK, "cpu", seed=22)
    theta0 = theta0_of(sum(units), seed=21)
    st = zs.ZeroStep(scheme, W, units, "bf16", theta0=theta0, alloc=dev)
    ref = zs.ZeroStep(scheme, W, units, "bf16", theta0=theta0)
    staging = dev.zeros(need, torch.uint8, "staging")
    host_grads = [host.zeros(s["n_pad"], torch.bfloat16, f"host grads {r}") for r in range(W)]
    host_out = host.zeros(out_elems, torch.bfloat16, "host out")
    grads = ref.new_grad_buffers()
    for t in (1, 2):
        fill_grads(grads, ref.real_index(), t)
        torch.cuda.synchronize()
        for h, g in zip(host_grads, grads):
            h.copy_(g)
        zs.zero_step_host(st.ctx, scheme, W, sum(units), host_grads, host_out, staging, need, chunk, *HP, t)
        ref.step(grads, *HP, t)
        st.sync()
    torch.cuda.synchronize()
    dev.check()
    host.check()
    assert_same_state(st, ref)
    want = ref.p16 if scheme != zs.ZERO_SCHEME_Z3 else torch.cat(ref.shard16)
    assert torch.equal(host_out, want.cpu())
    st.close()
    ref.close()


@pytest.mark.parametrize("W,n", [(3, 4097), (8, 1_000_003)])
def test_dp_replicas_write_only_their_buffers(W, n):
    n_pad = zs.zero_buffer_sizes(zs.ZERO_SCHEME_DP, W, [n])["n_pad"]
    arena = Arena(W * n_pad * (14 + 2) + 8 + (5 * W + 1) * SLACK, "cuda", seed=W)
    theta0 = theta0_of(n, seed=W)
    rep = zs.DpReplicas(W, n, "bf16", theta0=theta0, alloc=arena)
    ref = zs.ZeroStep(zs.ZERO_SCHEME_DP, W, [n], "bf16", theta0=theta0)
    grads = rep.new_grad_buffers()
    for t in (1, 2, 3):
        fill_grads(grads, ref.real_index(), t)
        rep.step(grads, *HP, t)
        ref.step(grads, *HP, t)
    assert rep.mismatches() == 0
    arena.check()
    for r in range(W):
        assert torch.equal(rep.master[r], ref.master) and torch.equal(rep.p16[r], ref.p16)
    ref.close()


def test_offload_writes_only_its_buffers():
    W, n, chunk = 8, 1_000_003, 262_144
    n_pad = zs.zero_buffer_sizes(zs.ZERO_SCHEME_Z2, W, [n])["n_pad"]
    staging = zs.zero_offload_staging_bytes(chunk)
    dev = Arena(2 * n_pad + staging + 2 * W * n_pad + (W + 2) * SLACK, "cuda", seed=31)
    host = Arena(18 * n_pad + 5 * SLACK, "cpu", seed=32)
    theta0 = theta0_of(n, seed=31)
    off = zs.ZeroOffload(W, n, "bf16", theta0=theta0, chunk_elems=chunk, threads=4, alloc=dev, host_alloc=host)
    ref = zs.ZeroStep(zs.ZERO_SCHEME_Z2, W, [n], "bf16", theta0=theta0)
    grads = off.new_grad_buffers()
    for t in (1, 2):
        fill_grads(grads, ref.real_index(), t)
        torch.cuda.synchronize()
        off.step(grads, *HP, t)
        ref.step(grads, *HP, t)
    torch.cuda.synchronize()
    dev.check()
    host.check()
    assert torch.equal(off.master, ref.master.cpu()) and torch.equal(off.p16, ref.p16)
    off.close()
    ref.close()


def test_static_zero3_step_writes_only_the_callers_buffers():
    W, units = 8, [17, 4096, 1_000_003, 0, 5]
    s = zs.zero_buffer_sizes(zs.ZERO_SCHEME_Z3, W, units)
    arena = Arena(12 * s["n_pad"] + 2 * W * s["shard_store"] + 2 * W * s["n_pad"] + (2 * W + 3) * SLACK, "cuda",
                  seed=41)
    theta0 = theta0_of(sum(units), seed=41)
    ref = zs.ZeroStep(zs.ZERO_SCHEME_Z3, W, units, "bf16", theta0=theta0)
    torch.cuda.synchronize()
    master, m, v = (arena.zeros(s["n_pad"], torch.float32, name) for name in ("master", "m", "v"))
    master.copy_(ref.master)
    shards = [arena.zeros(s["shard_store"], torch.bfloat16, f"shard store {r}") for r in range(W)]
    for r in range(W):
        shards[r].copy_(ref.shard16[r])
    grads = [arena.zeros(s["n_pad"], torch.bfloat16, f"grads {r}") for r in range(W)]
    for t in (1, 2):
        fill_grads(grads, ref.real_index(), t)
        zs.zero_step_z3_static(W, units, zs.ZERO_BF16, zs.ZERO_BF16, master, m, v, shards, grads, *HP, t)
        ref.step(grads, *HP, t)
    torch.cuda.synchronize()
    arena.check()
    assert torch.equal(master, ref.master) and torch.equal(m, ref.m) and torch.equal(v, ref.v)
    for r in range(W):
        assert torch.equal(shards[r], ref.shard16[r])
    ref.close()
