"""zero_step_host: the step fed from host memory through the staging ring,
against zero_step on the same gradients (GPU needed)."""

import numpy as np
import pytest
import torch

import workloads as wk
import zero_sharded_mixed_step_gb300 as zs

pytestmark = pytest.mark.gpu

CASES = [
    # scheme, n or units, W, dtype, chunk_elems, pinned, read back
    (zs.ZERO_SCHEME_Z2, 3_000_005, 8, "bf16", 1_000_000, True, True),
    (zs.ZERO_SCHEME_Z1, 1_000_003, 3, "fp16", 100_001, True, True),
    (zs.ZERO_SCHEME_DP, 2_500_000, 16, "bf16", 0, False, True),
    (zs.ZERO_SCHEME_Z1, 777_777, 8, "bf16", 65_536, True, False),
    (zs.ZERO_SCHEME_Z3, [1_000_003, 17, 0, 250_000, 7], 5, "bf16", 0, True, True),
    (zs.ZERO_SCHEME_Z3, [262_144, 262_144, 262_144], 8, "fp16", 0, False, True),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from zero_sharded_mixed_step_gb300 import build
    build.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"s{c[0]}_W{c[2]}_{c[3]}_chunk{c[4]}_pin{int(c[5])}_out{int(c[6])}")
def test_host_step_equals_device_step(case):
    scheme, size, W, dtype, chunk, pinned, read_back = case
    units = size if isinstance(size, list) else [size]
    n = sum(units)
    wl = wk.scaled(wk.GPT2_SMALL, unit_sizes=units if scheme == zs.ZERO_SCHEME_Z3 else None, n=n, W=W, steps=3,
                   name="host_step")
    theta0 = wk.draw_theta0(wl, "cuda")
    a = zs.ZeroStep(scheme, W, units, dtype, theta0=theta0)
    b = zs.ZeroStep(scheme, W, units, dtype, theta0=theta0)
    need = zs.zero_host_staging_bytes(scheme, W, units, chunk)
    staging = torch.empty(need, dtype=torch.uint8, device="cuda")
    out_elems = b.n_pad if scheme != zs.ZERO_SCHEME_Z3 else W * b.sizes["shard_store"]
    host_out = torch.zeros(out_elems, dtype=b.work_torch_dtype, pin_memory=True) if read_back else None
    sh, sd = torch.cuda.Stream(), torch.cuda.Stream()
    src = wk.GradSource(wl, dtype, "cuda")
    hp = (wl.lr, wl.beta1, wl.beta2, wl.eps)
    for t in range(1, wl.steps + 1):
        dev_grads = []
        for d in src.step(t):
            g = torch.zeros(a.n_pad, dtype=a.grad_torch_dtype, device="cuda")
            a.place_(g, d)
            dev_grads.append(g)
        host = [g.cpu().pin_memory() if pinned else g.cpu() for g in dev_grads]
        torch.cuda.synchronize()
        a.step(dev_grads, *hp, t)
        zs.zero_step_host(b.ctx, scheme, W, n, host, host_out, staging, need, chunk, *hp, t, sh, sd)
        b.sync(timeout_ms=60_000)
        for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32)), t
        assert torch.equal(a.working_copy().view(torch.int16), b.working_copy().view(torch.int16)), t
        if read_back:
            if scheme != zs.ZERO_SCHEME_Z3:
                want = b.p16.cpu()
            else:
                want = torch.cat([x.cpu() for x in b.shard16])
            assert torch.equal(host_out.view(torch.int16), want.view(torch.int16)), t
    for k in (zs.ZERO_STAT_COMM_BYTES, zs.ZERO_STAT_GATHERS, zs.ZERO_STAT_SCATTERS, zs.ZERO_STAT_T):
        assert a.stat(k) == b.stat(k), k
    assert b.stat(zs.ZERO_STAT_LIVE_ELEMS) == 0
    a.close()
    b.close()
