"""Seeded synthetic workloads for the ZeRO step: sizes, hyper-parameters and
random draws.

This module holds no arithmetic of the method.  It describes the seven
workloads (sizes, rank counts, schemes, Adam hyper-parameters, step counts,
value distributions and seeds) and draws their random inputs with
``torch.Generator``: the initial fp32 master and each rank's 16-bit
gradients.  Both the CUDA path and the CPU oracle consume exactly the same
draws, so the bits produced here are the single source of every input.
Nothing here pads, shards or lays out a vector: callers place the drawn
length-n vectors into their own layout.

Distributions (the sigma of every normal is its standard deviation):

* a fraction ``zero_frac`` of gradient entries is set exactly to 0, chosen
  per entry by an independent uniform draw;
* a fraction ``outlier_frac`` is multiplied by ``outlier_scale``, sign kept.

Seeding rules:

* ``"one_stream"``: one generator seeded ``grad_seed`` draws every step's
  gradients, rank 0 first, in step order;
* ``"step_rank"``: a fresh generator per (step t, rank r), seed ``1000 t + r``;
* ``"per_rank_stream"``: one generator per rank, seed ``r``, advanced from
  step to step.

The initial master always comes from its own generator seeded
``theta_seed``.
"""

from __future__ import annotations

from dataclasses import dataclass

import torch

DP, ZERO1, ZERO2, ZERO3 = 0, 1, 2, 3
FP16, BF16 = "fp16", "bf16"
TORCH_DTYPE = {FP16: torch.float16, BF16: torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    n: int
    W: int
    schemes: tuple
    dtypes: tuple
    lr: float
    beta1: float
    beta2: float
    eps: float
    steps: int
    theta_sigma: float
    grad_sigma: float
    seed_rule: str
    zero_frac: float = 0.0
    outlier_frac: float = 0.0
    outlier_scale: float = 1.0
    theta_seed: int = 0
    grad_seed: int = 1
    unit_sizes: tuple | None = None
    description: str = ""
    # data parallelism with its W replicas kept literally (scheme DP only)
    dp_replicas: bool = False
    # ZeRO-2 with the optimizer state and update on the host CPU
    offload: bool = False

    def units(self):
        return list(self.unit_sizes) if self.unit_sizes else [self.n]


TINY = Workload(
    name="tiny_lab_psi8_w4", n=8, W=4, schemes=(DP, ZERO1, ZERO2, ZERO3), dtypes=(FP16,),
    lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8, steps=5,
    theta_sigma=1.0, grad_sigma=0.1, seed_rule="one_stream", theta_seed=0, grad_seed=1,
    unit_sizes=(8,),
    description="Psi=8 on 4 ranks (shard 2), all four schemes, 5 steps",
)

FLAT_1M = Workload(
    name="flat_2p20_w8", n=1 << 20, W=8, schemes=(ZERO1, ZERO2), dtypes=(FP16,),
    lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, steps=10,
    theta_sigma=0.02, grad_sigma=1e-3, seed_rule="step_rank", zero_frac=0.01,
    description="Psi=2^20 on 8 ranks, ZeRO-1 and ZeRO-2, 1% exact zeros, 10 steps",
)

GPT2_SMALL = Workload(
    name="gpt2_small_124m_w8_zero2", n=124_439_808, W=8, schemes=(ZERO2,), dtypes=(BF16, FP16),
    lr=6e-4, beta1=0.9, beta2=0.95, eps=1e-8, steps=20,
    theta_sigma=0.02, grad_sigma=1e-3, seed_rule="step_rank",
    outlier_frac=1e-3, outlier_scale=50.0,
    description="GPT-2-small sized flat vector, 8 ranks, ZeRO-2, 0.1% outliers at 50x",
)

GPT2_XL = Workload(
    name="gpt2_1p5b_w16_zero1", n=1_557_611_200, W=16, schemes=(ZERO1,), dtypes=(FP16,),
    lr=1.5e-4, beta1=0.9, beta2=0.95, eps=1e-8, steps=5,
    theta_sigma=0.02, grad_sigma=5e-4, seed_rule="per_rank_stream",
    description="GPT-2-1.5B sized flat vector, 16 ranks, ZeRO-1",
)

LAYER_UNITS = Workload(
    name="zero3_24x50m_w8", n=24 * 50_331_648, W=8, schemes=(ZERO3,), dtypes=(BF16,),
    lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, steps=5,
    theta_sigma=0.02, grad_sigma=1e-3, seed_rule="step_rank",
    unit_sizes=(50_331_648,) * 24,
    description="ZeRO-3, 24 transformer-layer units of 50,331,648 parameters, 8 ranks",
)

GPT2_SMALL_DP_REPLICAS = Workload(
    name="gpt2_small_124m_w8_dp_replicas", n=124_439_808, W=8, schemes=(DP,), dtypes=(BF16, FP16),
    lr=6e-4, beta1=0.9, beta2=0.95, eps=1e-8, steps=20,
    theta_sigma=0.02, grad_sigma=1e-3, seed_rule="step_rank",
    outlier_frac=1e-3, outlier_scale=50.0, dp_replicas=True,
    description="the GPT-2-small vector under plain data parallelism, its 8 replicas kept literally",
)

GPT2_SMALL_OFFLOAD = Workload(
    name="gpt2_small_124m_w8_zero2_offload", n=124_439_808, W=8, schemes=(ZERO2,), dtypes=(BF16, FP16),
    lr=6e-4, beta1=0.9, beta2=0.95, eps=1e-8, steps=20,
    theta_sigma=0.02, grad_sigma=1e-3, seed_rule="step_rank",
    outlier_frac=1e-3, outlier_scale=50.0, offload=True,
    description="the GPT-2-small vector under ZeRO-2 with the optimizer state and update on the host",
)

WORKLOADS = {w.name: w for w in (TINY, FLAT_1M, GPT2_SMALL, GPT2_XL, LAYER_UNITS, GPT2_SMALL_DP_REPLICAS,
                                 GPT2_SMALL_OFFLOAD)}


def scaled(wl: Workload, n: int | None = None, W: int | None = None, steps: int | None = None,
           unit_sizes=None, name: str | None = None, **kw) -> Workload:
    """A copy of ``wl`` with other sizes (same distributions and seeds)."""
    fields = dict(wl.__dict__)
    if n is not None:
        fields["n"] = n
    if W is not None:
        fields["W"] = W
    if steps is not None:
        fields["steps"] = steps
    if unit_sizes is not None:
        fields["unit_sizes"] = tuple(unit_sizes)
        fields["n"] = int(sum(unit_sizes))
    elif n is not None and wl.unit_sizes is not None:
        fields["unit_sizes"] = None
    fields["name"] = name or f"{wl.name}_scaled"
    fields.update(kw)
    return Workload(**fields)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def draw_theta0(wl: Workload, device="cpu") -> torch.Tensor:
    """Initial fp32 master of n entries, N(0, theta_sigma)."""
    g = _gen(wl.theta_seed, device)
    x = torch.randn(wl.n, generator=g, device=device, dtype=torch.float32)
    return x.mul_(wl.theta_sigma)


def _draw_grad(wl: Workload, g: torch.Generator, dtype: str, device, out=None) -> torch.Tensor:
    x = torch.randn(wl.n, generator=g, device=device, dtype=torch.float32).mul_(wl.grad_sigma)
    if wl.zero_frac > 0:
        mask = torch.rand(wl.n, generator=g, device=device) < wl.zero_frac
        x.masked_fill_(mask, 0.0)
        del mask
    if wl.outlier_frac > 0:
        mask = torch.rand(wl.n, generator=g, device=device) < wl.outlier_frac
        x = torch.where(mask, x * wl.outlier_scale, x)
        del mask
    if out is None:
        return x.to(TORCH_DTYPE[dtype])
    out.copy_(x)
    return out


class GradSource:
    """Each rank's 16-bit gradients, step by step.

    ``step(t)`` must be called with t = 1, 2, ... in order; it returns W
    tensors of n entries (or fills ``out``, a list of W tensors whose first
    n entries receive the draw).
    """

    def __init__(self, wl: Workload, dtype: str, device="cpu"):
        self.wl, self.dtype, self.device = wl, dtype, device
        self.t = 0
        if wl.seed_rule == "one_stream":
            self._one = _gen(wl.grad_seed, device)
        elif wl.seed_rule == "per_rank_stream":
            self._per_rank = [_gen(r, device) for r in range(wl.W)]
        elif wl.seed_rule != "step_rank":
            raise ValueError(wl.seed_rule)

    def _generator(self, t: int, r: int) -> torch.Generator:
        rule = self.wl.seed_rule
        if rule == "one_stream":
            return self._one
        if rule == "per_rank_stream":
            return self._per_rank[r]
        return _gen(1000 * t + r, self.device)

    def step(self, t: int, out=None):
        if t != self.t + 1:
            raise ValueError(f"gradients are drawn in step order: expected t={self.t + 1}, got {t}")
        self.t = t
        res = []
        for r in range(self.wl.W):
            g = self._generator(t, r)
            dst = None if out is None else out[r][: self.wl.n]
            res.append(_draw_grad(self.wl, g, self.dtype, self.device, dst))
        return res if out is None else out


def to_numpy16(x: torch.Tensor):
    """A 16-bit torch tensor as NumPy: float16 for fp16, raw uint16 bits for bf16."""
    import numpy as np
    x = x.detach().cpu().contiguous()
    if x.dtype == torch.float16:
        return x.numpy()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16)
    raise TypeError(x.dtype)
