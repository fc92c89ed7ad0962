"""The synthetic inputs against their stated recipe (no GPU): the normal
draws' standard deviations, the fraction of exact zeros, the fraction and
scale of the outliers, and the seed rules (which generator feeds which rank
at which step, and that the draws come in step order)."""

import math

import pytest
import torch

import workloads as wk

N = 1 << 20


def _frac_ok(got, p, n, sigmas=5.0):
    """got within `sigmas` binomial standard deviations of p."""
    return abs(got - p) <= sigmas * math.sqrt(p * (1 - p) / n)


def test_theta0_is_normal_with_the_stated_sigma():
    wl = wk.scaled(wk.GPT2_SMALL, n=N)
    x = wk.draw_theta0(wl).double()
    assert abs(x.mean().item()) < 5 * wl.theta_sigma / math.sqrt(N)
    assert abs(x.std().item() / wl.theta_sigma - 1) < 0.01
    assert torch.equal(wk.draw_theta0(wl), wk.draw_theta0(wl))      # seeded


def test_exact_zeros_at_the_stated_fraction():
    wl = wk.scaled(wk.FLAT_1M, n=N, W=2)
    g = wk.GradSource(wl, "fp16").step(1)[0].float()
    assert wl.zero_frac == 0.01
    assert _frac_ok((g == 0).double().mean().item(), wl.zero_frac, N)
    nz = g[g != 0].double()
    assert abs(nz.std().item() / wl.grad_sigma - 1) < 0.01


def test_outliers_at_the_stated_fraction_and_scale():
    wl = wk.scaled(wk.GPT2_SMALL, n=N, W=2)
    assert (wl.outlier_frac, wl.outlier_scale) == (1e-3, 50.0)
    g = wk.GradSource(wl, "bf16").step(1)[0].double()
    # an outlier is a N(0, sigma) draw times 50: beyond 10 sigma unless the draw was under 0.2 sigma
    big = (g.abs() > 10 * wl.grad_sigma).double().mean().item()
    p_big = wl.outlier_frac * math.erfc(0.2 / math.sqrt(2))
    assert _frac_ok(big, p_big, N)
    # without the outliers the rest is N(0, sigma) (none beyond 10 sigma in 2^20 draws)
    assert abs(g[g.abs() <= 10 * wl.grad_sigma].std().item() / wl.grad_sigma - 1) < 0.01
    assert g.abs().max().item() <= 50 * 6 * wl.grad_sigma


def test_step_rank_seed_rule():
    """Rank r's draw at step t comes from a generator seeded 1000 t + r."""
    wl = wk.scaled(wk.GPT2_SMALL, n=4096, W=3)
    src = wk.GradSource(wl, "bf16")
    src.step(1)
    got = src.step(2)
    for r in range(wl.W):
        g = torch.Generator().manual_seed(1000 * 2 + r)
        x = torch.randn(wl.n, generator=g).mul_(wl.grad_sigma)
        mask = torch.rand(wl.n, generator=g) < wl.outlier_frac
        want = torch.where(mask, x * wl.outlier_scale, x).to(torch.bfloat16)
        assert torch.equal(got[r], want), r


def test_per_rank_and_one_stream_seed_rules():
    xl = wk.scaled(wk.GPT2_XL, n=4096, W=4)
    assert xl.seed_rule == "per_rank_stream"
    a, b = wk.GradSource(xl, "fp16"), wk.GradSource(xl, "fp16")
    a1, a2 = a.step(1), a.step(2)
    assert all(torch.equal(x, y) for x, y in zip(a1, b.step(1)))      # rank r's stream is seeded r
    assert not torch.equal(a1[0], a2[0])                               # and advances across steps
    assert not torch.equal(a1[0], a1[1])
    tiny = wk.TINY
    assert tiny.seed_rule == "one_stream"
    s = wk.GradSource(tiny, "fp16")
    t1 = s.step(1)
    assert not torch.equal(t1[0], t1[1])                               # one stream, ranks in order


def test_draws_come_in_step_order():
    src = wk.GradSource(wk.scaled(wk.GPT2_SMALL, n=64, W=2), "bf16")
    with pytest.raises(ValueError):
        src.step(2)
    src.step(1)
    with pytest.raises(ValueError):
        src.step(1)


def test_workload_sizes_are_the_benchmarks():
    assert wk.GPT2_SMALL.n == 124_439_808 and wk.GPT2_SMALL.W == 8
    assert wk.GPT2_XL.n == 1_557_611_200 and wk.GPT2_XL.W == 16
    assert wk.LAYER_UNITS.units() == [50_331_648] * 24 and wk.LAYER_UNITS.W == 8
    assert wk.TINY.n == 8 and wk.TINY.W == 4
