"""zero_step_bucket: a DP/Z1/Z2 step applied bucket by bucket, from bucket
buffers that hold only each range's gradients, against zero_step and the
oracle (GPU needed)."""

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


def buckets_of(n_pad, rng, min_len=8, max_len=300_000):
    """Random bucket boundaries at multiples of 8, the last one ragged, in shuffled order."""
    cuts, pos = [0], 0
    while pos < n_pad:
        pos = min(n_pad, pos + int(rng.integers(min_len // 8, max_len // 8 + 1)) * 8)
        cuts.append(pos)
    spans = list(zip(cuts[:-1], cuts[1:]))
    rng.shuffle(spans)
    return spans


@pytest.mark.parametrize("scheme,n,W,dtype", [(zs.ZERO_SCHEME_Z2, 2_000_003, 8, "bf16"),
                                              (zs.ZERO_SCHEME_Z1, 1_000_001, 5, "fp16"),
                                              (zs.ZERO_SCHEME_DP, 777_777, 16, "bf16")])
def test_bucketed_step_equals_full_step(scheme, n, W, dtype):
    wl = wk.scaled(wk.GPT2_SMALL, n=n, W=W, steps=3, name="bucketed")
    theta0 = wk.draw_theta0(wl, "cuda")
    a = zs.ZeroStep(scheme, W, [n], dtype, theta0=theta0)
    b = zs.ZeroStep(scheme, W, [n], dtype, theta0=theta0)
    oracle = z.SingleReplica(theta0.cpu().numpy(), dtype)
    src = wk.GradSource(wl, dtype, "cuda")
    rng = np.random.default_rng(5)
    hp = (wl.lr, wl.beta1, wl.beta2, wl.eps)
    for t in range(1, wl.steps + 1):
        full = []
        for d in src.step(t):
            g = torch.zeros(a.n_pad, dtype=a.grad_torch_dtype, device="cuda")
            a.place_(g, d)
            full.append(g)
        a.step(full, *hp, t)
        for lo, hi in buckets_of(b.n_pad, rng):
            bucket = [g[lo:hi].clone() for g in full]      # only this range's gradients exist
            zs.zero_step_bucket(b.ctx, lo, hi - lo, bucket, *hp, t)
        oracle.step([wk.to_numpy16(g[:n]) for g in full], *hp)
        torch.cuda.synchronize()
        for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32)), t
        assert torch.equal(a.p16.view(torch.int16), b.p16.view(torch.int16)), t
        gh.assert_f32_parity(b.master[:n].cpu().numpy(), oracle.master, f"bucketed t={t}")
        gh.assert_16bit_band(gh.bits_of(b.p16[:n]), oracle.master, dtype, f"bucketed t={t}")
    assert zs.zero_comm_bytes_per_rank(b.ctx) == zs.zero_comm_bytes_per_rank(a.ctx)
    assert b.stat(zs.ZERO_STAT_SCATTERS) == a.stat(zs.ZERO_STAT_SCATTERS) == wl.steps
    a.close()
    b.close()


def test_bucketed_step_coverage_rules():
    n, W = 4096, 4
    wl = wk.scaled(wk.GPT2_SMALL, n=n, W=W, steps=2, name="coverage")
    s = zs.ZeroStep(zs.ZERO_SCHEME_Z2, W, [n], "bf16", theta0=wk.draw_theta0(wl, "cuda"))
    g = [torch.zeros(n, dtype=torch.bfloat16, device="cuda") for _ in range(W)]
    hp = (wl.lr, wl.beta1, wl.beta2, wl.eps)

    def code(fn, *args):
        with pytest.raises(zs.ZeroError) as e:
            fn(*args)
        return e.value.code

    zs.zero_step_bucket(s.ctx, 0, 1024, [x[:1024] for x in g], *hp, 1)
    # overlapping what step 1 already covered
    assert code(zs.zero_step_bucket, s.ctx, 1016, 16, [x[1016:1032] for x in g], *hp, 1) == zs.ZERO_E_STATE
    # a new step, or a whole step, while step 1 is incomplete
    assert code(zs.zero_step_bucket, s.ctx, 1024, 8, [x[1024:1032] for x in g], *hp, 2) == zs.ZERO_E_STATE
    assert code(s.step, g, *hp, 2) == zs.ZERO_E_STATE
    assert zs.zero_comm_bytes_per_rank(s.ctx) == 0
    zs.zero_step_bucket(s.ctx, 1024, n - 1024, [x[1024:] for x in g], *hp, 1)
    assert zs.zero_comm_bytes_per_rank(s.ctx) == z.comm_bytes_closed_form(2, n, W)
    # step 1 complete: step 2 may start either way
    s.step(g, *hp, 2)
    s.sync()
    assert s.stat(zs.ZERO_STAT_T) == 2
    s.close()


@pytest.mark.parametrize("seed", range(12))
def test_random_bucketed_configurations(seed):
    """Seeded random configurations of the bucketed step: scheme (DP, ZeRO-1,
    ZeRO-2), W from 1 to 64, both 16-bit formats, a ragged n, buckets from 8
    values to the whole vector in shuffled order, a variant of the fused
    pass, and each bucket's gradients in a buffer of its own at any 16-byte
    aligned address.  Bit for bit against zero_step, every position against
    the oracle, three steps."""
    rng = np.random.default_rng(4000 + seed)
    scheme = int(rng.integers(0, 3))
    W = int(rng.choice([1, 2, 3, 5, 8, 16, 31, 64]))
    max_len = int(rng.choice([64, 4096, 100_000, 1 << 40]))         # 2^40: one bucket for the whole vector
    n = int(rng.integers(1, 600_000 if max_len > 64 else 30_000))    # tiny buckets only on short vectors
    gdt, wdt = (str(rng.choice(["fp16", "bf16"])) for _ in range(2))
    variant = int(rng.choice([zs.ZERO_VARIANT_AUTO, zs.ZERO_VARIANT_VECTOR, zs.ZERO_VARIANT_BULK]))
    what = f"seed {seed}: scheme {scheme}, W {W}, n {n}, {gdt}->{wdt}, variant {variant}"
    wl = wk.scaled(wk.GPT2_SMALL, n=n, W=W, steps=3, name=f"bucket_random{seed}")
    theta0 = wk.draw_theta0(wl, "cuda")
    a = zs.ZeroStep(scheme, W, [n], gdt, wdt, theta0=theta0)
    b = zs.ZeroStep(scheme, W, [n], gdt, wdt, theta0=theta0)
    a.set_variant(variant)
    b.set_variant(variant)
    oracle = z.SingleReplica(theta0.cpu().numpy(), wdt, grad_dtype=gdt)
    src = wk.GradSource(wl, gdt, "cuda")
    hp = (wl.lr, wl.beta1, wl.beta2, wl.eps)
    for t in range(1, wl.steps + 1):
        full = []
        for d in src.step(t):
            g = torch.zeros(a.n_pad, dtype=a.grad_torch_dtype, device="cuda")
            a.place_(g, d)
            full.append(g)
        a.step(full, *hp, t)
        for lo, hi in buckets_of(b.n_pad, rng, max_len=min(max_len, b.n_pad + 8)):
            # each bucket in a buffer of its own, at an odd multiple of 16 bytes
            bucket = []
            for g in full:
                room = torch.empty(hi - lo + 8, dtype=g.dtype, device="cuda")
                view = room[8:] if room.data_ptr() % 32 == 0 else room[:hi - lo]
                view.copy_(g[lo:hi])
                bucket.append(view)
            zs.zero_step_bucket(b.ctx, lo, hi - lo, bucket, *hp, t)
        oracle.step([wk.to_numpy16(g[:n]) for g in full], *hp)
        torch.cuda.synchronize()
        for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32)), (what, t)
        assert torch.equal(a.p16.view(torch.int16), b.p16.view(torch.int16)), (what, t)
        gh.assert_f32_parity(b.master[:n].cpu().numpy(), oracle.master, f"{what} t={t} master")
        gh.assert_f32_parity(b.m[:n].cpu().numpy(), oracle.m, f"{what} t={t} m")
        gh.assert_f32_parity(b.v[:n].cpu().numpy(), oracle.v, f"{what} t={t} v")
        gh.assert_16bit_band(gh.bits_of(b.p16[:n]), oracle.master, wdt, f"{what} t={t}")
    assert zs.zero_comm_bytes_per_rank(b.ctx) == zs.zero_comm_bytes_per_rank(a.ctx), what
    a.close()
    b.close()
