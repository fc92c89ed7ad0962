"""The offloaded step's host half (zero_adam_host), on the CPU: against the
oracle, the first-step closed form, thread-count invariance, and the
argument checks of the offload entry points (no GPU needed)."""

import numpy as np
import pytest
import torch

import zero_sharded_mixed_step_gb300 as zs
from oracle import zero_oracle as z

from tests.gpu_harness import assert_f32_parity


def _run(g_steps, theta0, dtype, threads, hp=(1e-3, 0.9, 0.95, 1e-8)):
    n = theta0.size
    th = torch.from_numpy(theta0.copy())
    m, v = torch.zeros(n), torch.zeros(n)
    out = torch.zeros(n, dtype=torch.int16)
    for t, g in enumerate(g_steps, start=1):
        zs.zero_adam_host(n, torch.from_numpy(g), th, m, v, out, zs._DT[dtype], *hp, t, 8, threads)
    return th.numpy(), m.numpy(), v.numpy(), out.numpy().view(np.uint16)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_host_adam_matches_the_oracle(zlib, dtype):
    rng = np.random.default_rng(7)
    n = 70_001                                  # ragged against the 65,536-element pieces
    theta0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g_steps = []
    for _ in range(4):
        g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        g[rng.random(n) < 0.01] = 0.0
        g_steps.append(g)
    th, m, v, out = _run(g_steps, theta0, dtype, threads=3)
    o = z.SingleReplica(theta0.copy(), dtype)
    for t, g in enumerate(g_steps, start=1):
        z.adam_update(o.master, o.m, o.v, g.astype(np.float64), 1e-3, 0.9, 0.95, 1e-8, t)
    assert_f32_parity(th, o.master, "master")
    assert_f32_parity(m, o.m, "m")
    assert_f32_parity(v, o.v, "v")
    # the 16-bit copy is exactly the round-to-nearest-even of the host master
    assert np.array_equal(out, z.bits16(z.cast16(th, dtype), dtype))


def test_host_adam_first_step_closed_form(zlib):
    """t = 1: m_hat = g and v_hat = g^2, so theta moves by -lr g / (|g| + eps);
    where g = 0 it does not move."""
    rng = np.random.default_rng(3)
    n = 10_000
    theta0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    g[::97] = 0.0
    lr, eps = 1e-3, 1e-8
    th, _, _, _ = _run([g], theta0, "bf16", threads=2, hp=(lr, 0.9, 0.999, eps))
    d = th.astype(np.float64) - theta0.astype(np.float64)
    gd = g.astype(np.float64)
    ulp = np.abs(np.spacing(th.astype(np.float32))).astype(np.float64)
    bound = lr * eps / (np.abs(gd) + eps) + 2 * ulp + 1e-5 * lr
    assert (np.abs(d + lr * np.sign(gd)) <= bound).all()
    assert (d[gd == 0] == 0).all()


def test_host_adam_is_the_same_on_any_thread_count(zlib):
    rng = np.random.default_rng(11)
    n = 300_007
    theta0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    g_steps = [(rng.standard_normal(n) * 1e-3).astype(np.float32) for _ in range(2)]
    ref = _run(g_steps, theta0, "fp16", threads=1)
    for threads in (2, 5, 16):
        got = _run(g_steps, theta0, "fp16", threads=threads)
        for a, b in zip(ref, got):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8)), threads


def _err(fn, *args):
    with pytest.raises(zs.ZeroError) as e:
        fn(*args)
    return e.value.code


@pytest.mark.parametrize("hp,t0", [((1e-3, 0.0, 0.0, 1e-8), 0),        # no momentum: m = g, v = g^2
                                   ((0.0, 0.9, 0.95, 1e-8), 0),        # lr 0: theta stays, m and v move
                                   ((1e-3, 0.9, 0.95, 1.0), 0),        # eps above every |g|
                                   ((1e-3, 0.9, 0.95, 1e-30), 0),      # eps far below every |g|
                                   ((1e-3, 0.9, 0.999, 1e-8), 999_999)])   # beta^t underflows: no bias correction
def test_host_adam_hyperparameter_edges_match_the_oracle(zlib, hp, t0):
    """The update at the edges of its hyper-parameters, with about 1% zero
    gradients, against the oracle; the same fp32 arithmetic as the kernels."""
    rng = np.random.default_rng(int(1e6 * hp[0]) + t0)
    n = 20_011
    theta0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    th, m, v = torch.from_numpy(theta0.copy()), torch.zeros(n), torch.zeros(n)
    out = torch.zeros(n, dtype=torch.int16)
    o = z.SingleReplica(theta0.copy(), "bf16")
    for t in range(t0 + 1, t0 + 4):
        g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        g[rng.random(n) < 0.01] = 0.0
        zs.zero_adam_host(n, torch.from_numpy(g), th, m, v, out, zs.ZERO_BF16, *hp, t, 8, 2)
        z.adam_update(o.master, o.m, o.v, g.astype(np.float64), *hp, t)
    assert_f32_parity(th.numpy(), o.master, "master")
    assert_f32_parity(m.numpy(), o.m, "m")
    assert_f32_parity(v.numpy(), o.v, "v")
    if hp[0] == 0.0:
        assert np.array_equal(th.numpy().view(np.uint32), theta0.view(np.uint32))


def test_host_adam_refuses_what_fp32_cannot_carry(zlib):
    """eps that rounds to 0 in fp32, or beyond its range, and a step size
    lr / (1 - beta1^t) beyond it, are refused before any arithmetic."""
    x = torch.zeros(8)
    o = torch.zeros(8, dtype=torch.int16)
    assert _err(zs.zero_adam_host, 8, x, x, x, x, o, 0, 1e-3, 0.9, 0.95, 1e-50, 1) == zs.ZERO_E_ARG
    assert "eps" in zs.zero_last_error()
    assert _err(zs.zero_adam_host, 8, x, x, x, x, o, 0, 1e-3, 0.9, 0.95, 1e39, 1) == zs.ZERO_E_ARG
    assert _err(zs.zero_adam_host, 8, x, x, x, x, o, 0, 1e38, 0.9, 0.95, 1e-8, 1) == zs.ZERO_E_ARG  # 1e38 / 0.1
    assert "overflows" in zs.zero_last_error()
    zs.zero_adam_host(8, x, x, x, x, o, 0, 1e38, 0.9, 0.95, 1e-8, 100)   # 1 - 0.9^100 is about 1: fits
    zs.zero_adam_host(8, x, x, x, x, o, 0, 1e-3, 0.9, 0.95, 1e-44, 1)    # a subnormal fp32 eps is still > 0


def test_host_adam_checks(zlib):
    x = torch.zeros(8)
    o = torch.zeros(8, dtype=torch.int16)
    assert _err(zs.zero_adam_host, -1, x, x, x, x, o, 0, 1e-3, 0.9, 0.95, 1e-8, 1) == zs.ZERO_E_ARG
    assert _err(zs.zero_adam_host, 8, x, x, x, x, o, 2, 1e-3, 0.9, 0.95, 1e-8, 1) == zs.ZERO_E_ARG
    assert _err(zs.zero_adam_host, 8, x, x, x, x, o, 0, 1e-3, 0.9, 0.95, 1e-8, 0) == zs.ZERO_E_STATE
    assert _err(zs.zero_adam_host, 8, None, x, x, x, o, 0, 1e-3, 0.9, 0.95, 1e-8, 1) == zs.ZERO_E_ARG
    zs.zero_adam_host(0, None, None, None, None, None, 0, 1e-3, 0.9, 0.95, 1e-8, 1)


A = 0x7F0000000000


def fake(k):
    return A + k * (1 << 30)


def test_offload_init_checks_before_any_cuda_call(zlib):
    need = zs.zero_offload_staging_bytes(1000)
    assert need == 2 * 1000 * 4
    assert zs.zero_offload_staging_bytes(0) == 2 * (4 << 20) * 4
    assert zs.zero_offload_staging_bytes(13) == 2 * 16 * 4
    h = [fake(k) for k in range(5)]
    ok = (h[0], h[1], h[2], h[3], h[4], fake(10), fake(11), need, 1000)
    init = zs.zero_offload_init
    assert _err(init, 0, 100, 0, 0, *ok) == zs.ZERO_E_ARG
    assert _err(init, 4, -1, 0, 0, *ok) == zs.ZERO_E_ARG
    assert _err(init, 4, 100, 3, 0, *ok) == zs.ZERO_E_ARG
    assert _err(init, 4, 100, 0, 0, None, *ok[1:]) == zs.ZERO_E_ARG
    assert _err(init, 4, 100, 0, 0, *ok[:5], fake(10) + 2, *ok[6:]) == zs.ZERO_E_ALIGN
    assert _err(init, 4, 100, 0, 0, *ok[:6], fake(11) + 16, *ok[7:]) == zs.ZERO_E_ALIGN
    assert _err(init, 4, 100, 0, 0, *ok[:7], need - 1, 1000) == zs.ZERO_E_ARG
    assert _err(init, 4, 100, 0, 0, h[0] + 1, *ok[1:]) == zs.ZERO_E_ALIGN


def test_offload_init_refuses_overlapping_host_buffers(zlib):
    need = zs.zero_offload_staging_bytes(1000)
    h = [fake(k) for k in range(5)]
    # m inside master
    assert _err(zs.zero_offload_init, 4, 100, 0, 0, h[0], h[0] + 64, h[2], h[3], h[4], fake(10), fake(11), need,
                1000) == zs.ZERO_E_ARG
    assert "overlap" in zs.zero_last_error()
