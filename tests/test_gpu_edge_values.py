"""Degenerate values through every step entry point (GPU needed): masters
beyond the fp16 range (the working copy becomes +-inf, reading 5), gradients
at the fp16 maximum, and all-zero gradients (nothing may move).  The device
step, DP with literal replicas and the offloaded step must agree bit for bit
and stay within the tolerance of the oracle.  Then the hyper-parameters at
their edges, through the ZeRO-2 and ZeRO-3 kernels."""

import numpy as np
import pytest
import torch

import workloads as wk
import zero_sharded_mixed_step_gb300 as zs
from oracle import zero_oracle as z
from tests.gpu_harness import assert_16bit_band, assert_f32_parity, bits_of

pytestmark = pytest.mark.gpu

W = 4
HP = (1e-2, 0.9, 0.999, 1e-8)


def _theta0():
    edge = np.array([65503.0, 65519.99, 65520.0, 65536.0, 70000.0, -70000.0, 1e6, -65504.0, 65504.0, 0.0,
                     6e-8, -6e-8, 1e-30], np.float32)
    rng = np.random.default_rng(5)
    return np.concatenate([edge, (rng.standard_normal(1000) * 0.02).astype(np.float32)])


def _grads(theta0, kind, t):
    n = theta0.size
    rng = np.random.default_rng(100 + t)
    if kind == "zero":
        g = np.zeros((W, n), np.float32)
    elif kind == "fp16max":
        g = np.where(rng.random((W, n)) < 0.5, -65504.0, 65504.0).astype(np.float32)
    else:
        g = (rng.standard_normal((W, n)) * 1e-3).astype(np.float32)
        g[:, :13] = -1.0        # push the edge masters upwards
    return [torch.from_numpy(x).to(torch.float16) for x in g]


@pytest.mark.parametrize("kind", ["normal", "fp16max", "zero"])
def test_edge_values_agree_everywhere(kind):
    theta0 = _theta0()
    n = theta0.size
    dev = zs.ZeroStep(zs.ZERO_SCHEME_Z2, W, [n], "fp16", "fp16", theta0=torch.from_numpy(theta0), device="cuda")
    rep = zs.DpReplicas(W, n, "fp16", "fp16", theta0=torch.from_numpy(theta0).cuda(), device="cuda")
    off = zs.ZeroOffload(W, n, "fp16", "fp16", theta0=torch.from_numpy(theta0), threads=2, chunk_elems=256)
    orc = z.SingleReplica(theta0.copy(), "fp16")
    grads = dev.new_grad_buffers()
    for t in range(1, 4):
        draws = _grads(theta0, kind, t)
        for g, d in zip(grads, draws):
            g[:n].copy_(d)
        dev.step(grads, *HP, t)
        rep.step(grads, *HP, t)
        off.step(grads, *HP, t)
        orc.step([d.numpy() for d in draws], *HP)
        torch.cuda.synchronize()
        th = dev.master[:n].cpu().numpy()
        assert_f32_parity(th, orc.master, f"{kind} t={t} master")
        p16 = bits_of(dev.p16[:n])
        assert_16bit_band(p16, orc.master, "fp16", f"{kind} t={t} working copy")
        assert np.array_equal(p16, bits_of(dev.master[:n].to(torch.float16)))
        for r in range(W):
            assert torch.equal(rep.master[r].view(torch.int32), dev.master.view(torch.int32))
            assert torch.equal(rep.p16[r].view(torch.int16), dev.p16.view(torch.int16))
        assert torch.equal(off.master.view(torch.int32), dev.master.cpu().view(torch.int32))
        assert torch.equal(off.p16.view(torch.int16), dev.p16.view(torch.int16))
    final = dev.master[:n].cpu().numpy()
    wc = bits_of(dev.p16[:n])
    # beyond the fp16 range the working copy is infinite, with the master's sign
    big = np.abs(final) >= 65520.0
    assert big.sum() >= 4
    assert np.all(wc[big & (final > 0)] == 0x7C00) and np.all(wc[big & (final < 0)] == 0xFC00)
    if kind == "zero":
        assert np.array_equal(final.view(np.uint32), theta0.view(np.uint32))
        assert bool((dev.m == 0).all()) and bool((dev.v == 0).all())
    assert rep.mismatches() == 0
    off.close()
    dev.close()


@pytest.mark.parametrize("hp,t0", [((1e-3, 0.0, 0.0, 1e-8), 0),
                                   ((0.0, 0.9, 0.95, 1e-8), 0),
                                   ((1e-3, 0.9, 0.95, 1.0), 0),
                                   ((1e-3, 0.9, 0.95, 1e-30), 0),
                                   ((1e-3, 0.9, 0.999, 1e-8), 999_999)])
@pytest.mark.parametrize("scheme", [zs.ZERO_SCHEME_Z2, zs.ZERO_SCHEME_Z3])
def test_hyperparameter_edges_on_the_gpu(scheme, hp, t0):
    """No momentum (beta = 0), lr = 0, eps above and far below every |g|, and
    a step counter so large that beta^t underflows: the kernels against the
    oracle and bit for bit against the host update, which repeats their
    arithmetic.  The state is restored at step t0 through zero_set_state."""
    n, Wr = 20_011, 8
    rng = np.random.default_rng(int(1e6 * hp[0]) + t0)
    theta0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    units = [n] if scheme != zs.ZERO_SCHEME_Z3 else [7_001, 13_010]
    st = zs.ZeroStep(scheme, Wr, units, "bf16", theta0=torch.from_numpy(theta0), device="cuda",
                     stream=torch.cuda.Stream())
    idx = st.real_index()
    if t0:
        zs.zero_set_state(st.ctx, st.master.clone(), st.m.clone(), st.v.clone(), t0)
    orc = z.SingleReplica(theta0.copy(), "bf16")
    orc.t = t0
    host = [torch.from_numpy(theta0.copy()), torch.zeros(n), torch.zeros(n)]
    host16 = torch.zeros(n, dtype=torch.int16)
    grads = st.new_grad_buffers()
    for t in range(t0 + 1, t0 + 4):
        per_rank = (rng.standard_normal((Wr, n)) * 1e-3).astype(np.float32)
        per_rank[:, rng.random(n) < 0.01] = 0.0
        draws = [torch.from_numpy(x).to(torch.bfloat16) for x in per_rank]
        torch.cuda.synchronize()
        for g, d in zip(grads, draws):
            g.zero_()
            g[idx] = d.cuda()
        torch.cuda.synchronize()
        st.step(grads, *hp, t)
        # the rank mean as the kernel forms it: fp32 additions in rank order, then / W (exact for W = 8)
        acc = draws[0].float()
        for d in draws[1:]:
            acc = acc + d.float()
        mean = acc / Wr
        zs.zero_adam_host(n, mean, *host, host16, zs.ZERO_BF16, *hp, t, Wr, 2)
        orc.step([wk.to_numpy16(d) for d in draws], *hp)
    st.sync()
    got = [st.master[idx].cpu(), st.m[idx].cpu(), st.v[idx].cpu()]
    for a, b, what in zip(got, host, ("master", "m", "v")):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32)), what
    assert_f32_parity(got[0].numpy(), orc.master, "master")
    assert_f32_parity(got[1].numpy(), orc.m, "m")
    assert_f32_parity(got[2].numpy(), orc.v, "v")
    assert torch.equal(st.working_copy()[idx].cpu().view(torch.int16), host16)
    if hp[0] == 0.0:
        assert np.array_equal(got[0].numpy().view(np.uint32), theta0.view(np.uint32))
    st.close()
