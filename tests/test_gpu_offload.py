"""ZeRO-2 with the optimizer offloaded to the host (zero_offload_*):
bitwise against the device step zero_step on the same gradients, and
against the oracle."""

import pytest
import torch

import workloads as wk
import zero_sharded_mixed_step_gb300 as zs
from oracle import zero_oracle as z
from tests.gpu_harness import assert_16bit_band, assert_f32_parity, bits_of, sample_real_indices

pytestmark = pytest.mark.gpu

CASES = [
    # n, W, grad dtype, working dtype, chunk_elems (0: default; others rounded up to 8)
    (1001, 3, wk.FP16, wk.FP16, 64),
    (3_000_005, 8, wk.BF16, wk.BF16, 1 << 20),
    (2_000_000, 16, wk.FP16, wk.BF16, 0),
    (7, 1, wk.BF16, wk.FP16, 8),
    (250_001, 5, wk.BF16, wk.BF16, 100),
    (20_000, 64, wk.FP16, wk.FP16, 1000),   # the most ranks a context takes
]


def _equal(a, b):
    return torch.equal(a.view(torch.int32) if a.dtype == torch.float32 else a.view(torch.int16),
                       b.view(torch.int32) if b.dtype == torch.float32 else b.view(torch.int16))


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"n{c[0]}_W{c[1]}_{c[2]}_{c[3]}_chunk{c[4]}")
def test_offloaded_step_equals_device_step(case):
    n, W, gdt, wdt, chunk = case
    wl = wk.scaled(wk.GPT2_SMALL, n=n, W=W, steps=3, name="offload")
    theta0 = wk.draw_theta0(wl, "cuda")
    dev = zs.ZeroStep(zs.ZERO_SCHEME_Z2, W, [n], gdt, wdt, theta0=theta0)
    off = zs.ZeroOffload(W, n, gdt, wdt, theta0=theta0.cpu(), chunk_elems=chunk, threads=4)
    src = wk.GradSource(wl, gdt, "cuda")
    grads = dev.new_grad_buffers()
    hp = (wl.lr, wl.beta1, wl.beta2, wl.eps)
    for t in range(1, wl.steps + 1):
        for g, d in zip(grads, src.step(t)):
            g[:n].copy_(d)
        dev.step(grads, *hp, t)
        off.step(grads, *hp, t)
        torch.cuda.synchronize()
        for mine, theirs in ((off.master, dev.master), (off.m, dev.m), (off.v, dev.v)):
            assert _equal(mine, theirs.cpu()), t
        assert _equal(off.p16, dev.p16), t
        assert bool((off.master[n:] == 0).all())
    st = off.stats()
    assert st["t"] == wl.steps
    assert st["d2h_bytes"] == 4 * off.n_pad * wl.steps
    assert st["h2d_bytes"] == 2 * off.n_pad * wl.steps
    with pytest.raises(zs.ZeroError) as e:
        off.step(grads, *hp, wl.steps + 2)
    assert e.value.code == zs.ZERO_E_STATE
    off.close()
    dev.close()


def test_tiny_offloaded_step_against_the_oracle():
    wl = wk.TINY
    theta0 = wk.draw_theta0(wl, "cuda")
    off = zs.ZeroOffload(wl.W, wl.n, wk.FP16, theta0=theta0.cpu(), threads=2)
    orc = z.make_scheme(z.ZERO2, wl.W, theta0.cpu().numpy(), wk.FP16)
    src = wk.GradSource(wl, wk.FP16, "cuda")
    grads = off.new_grad_buffers()
    for t in range(1, wl.steps + 1):
        for g, d in zip(grads, src.step(t)):
            g[:wl.n].copy_(d)
        off.step(grads, wl.lr, wl.beta1, wl.beta2, wl.eps, t)
        orc.step([z.place(wk.to_numpy16(g[:wl.n]), orc.layout) for g in grads], wl.lr, wl.beta1, wl.beta2,
                 wl.eps)
        torch.cuda.synchronize()
        assert_f32_parity(off.master.numpy(), orc.full_master(), f"t={t} master")
        assert_f32_parity(off.m.numpy(), orc.full_m(), f"t={t} m")
        assert_f32_parity(off.v.numpy(), orc.full_v(), f"t={t} v")
        assert_16bit_band(bits_of(off.p16), orc.full_master(), wk.FP16, f"t={t} working copy")
    off.close()


def test_gpt2_small_sized_offloaded_step():
    """124,439,808 parameters on 8 ranks, bf16, two steps: bitwise equal to
    ZeRO-2 on the device, and a sample against the oracle."""
    wl = wk.scaled(wk.GPT2_SMALL, steps=2)
    theta0 = wk.draw_theta0(wl, "cuda")
    dev = zs.ZeroStep(zs.ZERO_SCHEME_Z2, wl.W, [wl.n], wk.BF16, theta0=theta0)
    off = zs.ZeroOffload(wl.W, wl.n, wk.BF16, theta0=theta0.cpu())
    idx = sample_real_indices(wl.n, wl.W, [wl.n], k=4096)
    orc = z.SingleReplica(theta0.cpu().numpy()[idx], wk.BF16)
    del theta0
    src = wk.GradSource(wl, wk.BF16, "cuda")
    grads = dev.new_grad_buffers()
    tidx = torch.from_numpy(idx).cuda()
    for t in range(1, wl.steps + 1):
        for g, d in zip(grads, src.step(t)):
            g[:wl.n].copy_(d)
        dev.step(grads, wl.lr, wl.beta1, wl.beta2, wl.eps, t)
        off.step(grads, wl.lr, wl.beta1, wl.beta2, wl.eps, t)
        orc.step([wk.to_numpy16(g[tidx]) for g in grads], wl.lr, wl.beta1, wl.beta2, wl.eps)
        torch.cuda.synchronize()
        assert _equal(off.master, dev.master.cpu())
        assert _equal(off.p16, dev.p16)
        assert_f32_parity(off.master.numpy()[idx], orc.master, f"t={t} master sample")
    off.close()
    dev.close()


def test_offloaded_step_resumes_from_a_checkpoint():
    """Save master, m, v and t after 3 steps, restore them into a new context,
    set its step counter, and the next step equals the uninterrupted run."""
    n, W = 300_001, 4
    wl = wk.scaled(wk.GPT2_SMALL, n=n, W=W, steps=4, name="offload_resume")
    theta0 = wk.draw_theta0(wl, "cuda")
    a = zs.ZeroOffload(W, n, wk.BF16, theta0=theta0.cpu(), threads=3)
    src = wk.GradSource(wl, wk.BF16, "cuda")
    steps = []
    for t in range(1, 5):
        g = a.new_grad_buffers()
        for b, d in zip(g, src.step(t)):
            b[:n].copy_(d)
        steps.append(g)
    hp = (wl.lr, wl.beta1, wl.beta2, wl.eps)
    for t in range(1, 4):
        a.step(steps[t - 1], *hp, t)
    saved = [x.clone() for x in (a.master, a.m, a.v)]
    a.step(steps[3], *hp, 4)
    torch.cuda.synchronize()
    b = zs.ZeroOffload(W, n, wk.BF16, threads=2)
    for dst, src_ in zip((b.master, b.m, b.v), saved):
        dst.copy_(src_)
    with pytest.raises(zs.ZeroError) as e:
        b.step(steps[3], *hp, 4)              # a fresh context expects step 1
    assert e.value.code == zs.ZERO_E_STATE
    b.set_step(3)
    b.step(steps[3], *hp, 4)
    torch.cuda.synchronize()
    for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
        assert _equal(x, y)
    assert _equal(a.p16, b.p16)
    with pytest.raises(zs.ZeroError):
        b.set_step(-1)
    a.close()
    b.close()


def _random_case(seed):
    import numpy as np
    rng = np.random.default_rng(8000 + seed)
    W = int(rng.choice([1, 2, 3, 5, 8, 16, 31, 64]))
    n = int(rng.integers(1, 1_200_000 if W <= 16 else 200_000))
    gdt, wdt = (str(rng.choice([wk.FP16, wk.BF16])) for _ in range(2))
    chunk = int(rng.choice([0, 8, 4096, int(rng.integers(8, 500_000))]))
    if chunk and n // chunk > 2000:                  # keep the number of chunks per step modest
        chunk = 0
    return n, W, gdt, wdt, chunk, int(rng.integers(1, 9))


@pytest.mark.parametrize("seed", range(10))
def test_random_offloaded_configurations(seed):
    """Seeded random rank counts (1 to 64), sizes, 16-bit formats, chunk
    lengths and host thread counts: the offloaded step bit for bit equal to
    the device step, three steps each."""
    n, W, gdt, wdt, chunk, threads = _random_case(seed)
    what = f"seed {seed}: n {n}, W {W}, {gdt}->{wdt}, chunk {chunk}, threads {threads}"
    wl = wk.scaled(wk.GPT2_SMALL, n=n, W=W, steps=3, name=f"offload_random{seed}")
    theta0 = wk.draw_theta0(wl, "cuda")
    dev = zs.ZeroStep(zs.ZERO_SCHEME_Z2, W, [n], gdt, wdt, theta0=theta0)
    off = zs.ZeroOffload(W, n, gdt, wdt, theta0=theta0.cpu(), chunk_elems=chunk, threads=threads)
    src = wk.GradSource(wl, gdt, "cuda")
    grads = dev.new_grad_buffers()
    hp = (wl.lr, wl.beta1, wl.beta2, wl.eps)
    for t in range(1, wl.steps + 1):
        for g, d in zip(grads, src.step(t)):
            g[:n].copy_(d)
        dev.step(grads, *hp, t)
        off.step(grads, *hp, t)
        torch.cuda.synchronize()
        for mine, theirs in ((off.master, dev.master), (off.m, dev.m), (off.v, dev.v)):
            assert _equal(mine, theirs.cpu()), (what, t)
        assert _equal(off.p16, dev.p16), (what, t)
    off.close()
    dev.close()
