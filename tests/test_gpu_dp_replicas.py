"""Data parallelism with W literal replicas (zero_step_dp_replicas and
zero_dp_replicas_mismatches) against the oracle's DP class, which keeps its
W replicas literally too, and bitwise against the one-copy DP step."""

import numpy as np
import pytest
import torch

import zero_sharded_mixed_step_gb300 as zs
import workloads as wk
from oracle import zero_oracle as z
from tests.gpu_harness import assert_16bit_band, assert_f32_parity, bits_of, sample_real_indices

pytestmark = pytest.mark.gpu


def _replicas(wl, dtype, work_dtype=None):
    dev = torch.device("cuda")
    theta0 = wk.draw_theta0(wl, dev)
    rep = zs.DpReplicas(wl.W, wl.n, dtype, work_dtype or dtype, theta0=theta0, device=dev)
    return rep, theta0


def _fill(bufs, draws, n):
    for b, d in zip(bufs, draws):
        b[:n].copy_(d)


def _check_replica(rep, r, master, m, v, dtype, tag, idx=None):
    sel = (lambda x: x) if idx is None else (lambda x: x[idx])
    assert_f32_parity(sel(rep.master[r]).cpu().numpy(), master, f"{tag} replica {r} master")
    assert_f32_parity(sel(rep.m[r]).cpu().numpy(), m, f"{tag} replica {r} m")
    assert_f32_parity(sel(rep.v[r]).cpu().numpy(), v, f"{tag} replica {r} v")
    p16 = bits_of(sel(rep.p16[r]))
    assert_16bit_band(p16, master, dtype, f"{tag} replica {r} 16-bit copy")
    own = bits_of(sel(rep.master[r]).to(rep.work_torch_dtype))
    assert np.array_equal(p16, own), f"{tag}: replica {r}'s 16-bit copy is not the RNE of its master"


def test_tiny_replicas_follow_the_oracle_replicas():
    """Psi = 8 on 4 ranks, 5 steps: every GPU replica against the matching
    replica of the oracle's DP class (which asserts its own replicas equal)."""
    wl = wk.TINY
    rep, theta0 = _replicas(wl, wk.FP16)
    orc = z.DataParallel(wl.W, theta0.cpu().numpy(), wk.FP16)
    src = wk.GradSource(wl, wk.FP16, "cuda")
    grads = rep.new_grad_buffers()
    for t in range(1, wl.steps + 1):
        _fill(grads, src.step(t), wl.n)
        rep.step(grads, wl.lr, wl.beta1, wl.beta2, wl.eps, t)
        orc.step([wk.to_numpy16(g) for g in grads], wl.lr, wl.beta1, wl.beta2, wl.eps)
        torch.cuda.synchronize()
        for r in range(wl.W):
            _check_replica(rep, r, orc.master[r], orc.m[r], orc.v[r], wk.FP16, f"tiny t={t}")
        assert rep.mismatches() == 0


RAGGED = [
    # (n, W, grad dtype, working dtype): a rank count with no compiled
    # specialisation, power-of-two counts, one rank, mixed formats, ragged tails
    (1001, 3, wk.FP16, wk.FP16),
    (20_011, 8, wk.BF16, wk.BF16),
    (65_537, 16, wk.FP16, wk.BF16),
    (7, 1, wk.BF16, wk.FP16),
    (333_333, 5, wk.BF16, wk.BF16),
    (10_001, 64, wk.FP16, wk.FP16),         # the most ranks a context takes
]


@pytest.mark.parametrize("n,W,gdt,wdt", RAGGED)
def test_ragged_replicas_match_the_oracle_and_the_one_copy_step(n, W, gdt, wdt):
    wl = wk.scaled(wk.FLAT_1M, n=n, W=W, steps=3, outlier_frac=1e-3, outlier_scale=50.0)
    rep, theta0 = _replicas(wl, gdt, wdt)
    one = zs.ZeroStep(zs.ZERO_SCHEME_DP, W, [n], gdt, wdt, theta0=theta0, device="cuda")
    orc = z.SingleReplica(theta0.cpu().numpy(), wdt, grad_dtype=gdt)
    src = wk.GradSource(wl, gdt, "cuda")
    grads = rep.new_grad_buffers()
    for t in range(1, wl.steps + 1):
        _fill(grads, src.step(t), n)
        rep.step(grads, wl.lr, wl.beta1, wl.beta2, wl.eps, t)
        one.step(grads, wl.lr, wl.beta1, wl.beta2, wl.eps, t)
        orc.step([wk.to_numpy16(g[:n]) for g in grads], wl.lr, wl.beta1, wl.beta2, wl.eps)
        torch.cuda.synchronize()
        for r in range(W):
            for mine, theirs in ((rep.master[r], one.master), (rep.m[r], one.m), (rep.v[r], one.v)):
                assert torch.equal(mine.view(torch.int32), theirs.view(torch.int32)), f"t={t} replica {r}"
            assert torch.equal(rep.p16[r].view(torch.int16), one.p16.view(torch.int16)), f"t={t} replica {r}"
        _check_replica(rep, W - 1, orc.master, orc.m, orc.v, wdt, f"n={n} W={W} t={t}", idx=slice(0, n))
        for r in range(W):
            tail = slice(n, rep.n_pad)
            assert all(bool((x[r][tail] == 0).all()) for x in (rep.master, rep.m, rep.v, rep.p16))
        assert rep.mismatches() == 0
    one.close()


def test_mismatch_counter_counts_replica_element_pairs():
    """Plant differences in the data (no fault involved): each (replica,
    element) pair counts once, whichever of its four values differ."""
    wl = wk.scaled(wk.FLAT_1M, n=4096 + 3, W=4, steps=1)
    rep, _ = _replicas(wl, wk.BF16)
    grads = rep.new_grad_buffers()
    _fill(grads, wk.GradSource(wl, wk.BF16, "cuda").step(1), wl.n)
    rep.step(grads, wl.lr, wl.beta1, wl.beta2, wl.eps, 1)
    assert rep.mismatches() == 0
    rep.master[1].view(torch.int32)[5] ^= 1
    rep.v[1].view(torch.int32)[5] ^= 1          # same pair as above
    rep.p16[2].view(torch.int16)[7] ^= 1
    rep.m[3].view(torch.int32)[4098] ^= 1       # in the ragged tail
    rep.master[3].view(torch.int32)[0] ^= 1
    assert rep.mismatches() == 4
    # replica 0 is the reference: a change there differs from all W - 1 others
    rep.master[0].view(torch.int32)[100] ^= 1
    assert rep.mismatches() == 4 + wl.W - 1


def test_gpt2_small_sized_replicas():
    """124,439,808 parameters on 8 ranks, bf16, two steps: every replica
    bitwise equal to the ZeRO-2 step on the same inputs, and a sample of
    positions (every rank boundary included) against the oracle."""
    wl = wk.scaled(wk.GPT2_SMALL, steps=2)
    rep, theta0 = _replicas(wl, wk.BF16)
    z2 = zs.ZeroStep(zs.ZERO_SCHEME_Z2, wl.W, [wl.n], wk.BF16, theta0=theta0, device="cuda")
    idx = sample_real_indices(wl.n, wl.W, [wl.n], k=4096)
    orc = z.SingleReplica(theta0.cpu().numpy()[idx], wk.BF16)
    del theta0
    src = wk.GradSource(wl, wk.BF16, "cuda")
    grads = rep.new_grad_buffers()
    tidx = torch.from_numpy(idx).cuda()
    for t in range(1, wl.steps + 1):
        _fill(grads, src.step(t), wl.n)
        rep.step(grads, wl.lr, wl.beta1, wl.beta2, wl.eps, t)
        z2.step(grads, wl.lr, wl.beta1, wl.beta2, wl.eps, t)
        orc.step([wk.to_numpy16(g[tidx]) for g in grads], wl.lr, wl.beta1, wl.beta2, wl.eps)
        torch.cuda.synchronize()
        assert rep.mismatches() == 0
        assert torch.equal(rep.master[0].view(torch.int32), z2.master.view(torch.int32))
        assert torch.equal(rep.p16[0].view(torch.int16), z2.p16.view(torch.int16))
        _check_replica(rep, wl.W - 1, orc.master, orc.m, orc.v, wk.BF16, f"gpt2-small t={t}", idx=tidx)
    z2.close()


def test_replicas_beyond_device_memory_are_refused_before_allocating():
    """GPT-2-1.5B on 16 ranks: 16 replicas of 14 bytes per parameter are
    349 GB, more than the device holds; the owner says so instead of
    allocating part of it."""
    before = torch.cuda.memory_allocated()
    with pytest.raises(MemoryError, match="replicas"):
        zs.DpReplicas(16, wk.GPT2_XL.n, wk.FP16, device="cuda")
    assert torch.cuda.memory_allocated() == before


def test_mismatch_counter_with_replicas_off_the_vector_grain():
    """zero_dp_replicas_mismatches accepts buffers aligned only to their
    element size; replicas one element off a 32-byte boundary take the
    element-at-a-time path and count the same pairs as aligned ones."""
    W, n = 3, 10_001
    n_pad = -(-n // W) * W                 # the compare reads n_pad values of every vector
    base = [torch.zeros(n_pad + 1, dtype=torch.float32, device="cuda") for _ in range(3 * W)]
    b16 = [torch.zeros(n_pad + 1, dtype=torch.int16, device="cuda") for _ in range(W)]
    th, m, v = (base[k * W:(k + 1) * W] for k in range(3))
    vals = torch.linspace(-1, 1, n_pad + 1, device="cuda")
    for x in th + m + v:
        x.copy_(vals)
    for x in b16:
        x.copy_(torch.arange(n_pad + 1, device="cuda", dtype=torch.int16))
    views = [[x[1:] for x in grp] for grp in (th, m, v)] + [[x[1:] for x in b16]]   # 4 and 2 bytes off
    count = torch.zeros(1, dtype=torch.int64, device="cuda")

    def mismatches():
        zs.zero_dp_replicas_mismatches(W, n, *views, count)
        torch.cuda.synchronize()
        return int(count.item())

    assert mismatches() == 0
    th[1][1 + 17] += 1.0                  # element 17 of replica 1
    v[2][1 + 17] += 1.0                   # element 17 of replica 2
    b16[2][1 + n_pad - 1] += 1            # the last (padding) element of replica 2
    m[1][1 + 17] += 1.0                   # the same pair as the first
    assert mismatches() == 3
    th[0][1 + 5000] += 1.0                # replica 0 is the reference
    assert mismatches() == 3 + W - 1
