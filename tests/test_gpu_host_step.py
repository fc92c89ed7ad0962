"""zero_step_host: the step fed from host memory through the staging ring,
against zero_step on the same gradients (GPU needed)."""

import os

import pytest
import torch

import workloads as wk
import zero_sharded_mixed_step_gb300 as zs

pytestmark = pytest.mark.gpu

CASES = [
    # scheme, n or units, W, dtype, chunk_elems, host memory, read back;
    # host memory: "pin" torch pinned, "page" pageable, "huge" zero_host_alloc
    (zs.ZERO_SCHEME_Z2, 3_000_005, 8, "bf16", 1_000_000, "pin", True),
    (zs.ZERO_SCHEME_Z1, 1_000_003, 3, "fp16", 100_001, "pin", True),
    (zs.ZERO_SCHEME_DP, 2_500_000, 16, "bf16", 0, "page", True),
    (zs.ZERO_SCHEME_Z1, 777_777, 8, "bf16", 65_536, "pin", False),
    (zs.ZERO_SCHEME_Z3, [1_000_003, 17, 0, 250_000, 7], 5, "bf16", 0, "pin", True),
    (zs.ZERO_SCHEME_Z3, [262_144, 262_144, 262_144], 8, "fp16", 0, "page", True),
    (zs.ZERO_SCHEME_Z2, 2_000_003, 8, "bf16", 500_000, "huge", True),
    (zs.ZERO_SCHEME_Z3, [500_000, 3, 700_001], 8, "bf16", 0, "huge", True),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from zero_sharded_mixed_step_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _host_copy(g, mem, keep):
    if mem == "pin":
        return g.cpu().pin_memory()
    if mem == "page":
        return g.cpu()
    buf = zs.HostBuffer(g.numel(), g.dtype)
    keep.append(buf)
    buf.tensor.copy_(g)
    return buf.tensor


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"s{c[0]}_W{c[2]}_{c[3]}_chunk{c[4]}_{c[5]}_out{int(c[6])}")
def test_host_step_equals_device_step(case):
    scheme, size, W, dtype, chunk, mem, read_back = case
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
    keep = []
    if not read_back:
        host_out = None
    elif mem == "huge":
        keep.append(zs.HostBuffer(out_elems, b.work_torch_dtype))
        host_out = keep[-1].tensor
    else:
        host_out = torch.zeros(out_elems, dtype=b.work_torch_dtype, pin_memory=True)
    sh, sd = torch.cuda.Stream(), torch.cuda.Stream()
    src = wk.GradSource(wl, dtype, "cuda")
    hp = (wl.lr, wl.beta1, wl.beta2, wl.eps)
    for t in range(1, wl.steps + 1):
        dev_grads = []
        for d in src.step(t):
            g = torch.zeros(a.n_pad, dtype=a.grad_torch_dtype, device="cuda")
            a.place_(g, d)
            dev_grads.append(g)
        host = [_host_copy(g, mem, keep) for g in dev_grads]
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
    torch.cuda.synchronize()
    for buf in keep:
        buf.close()


def test_host_alloc_is_page_locked_aligned_and_zeroed():
    """zero_host_alloc: a block of a huge page or more starts on a huge-page
    boundary (a small one on a page boundary), reads as
    zeros, counts as page-locked for CUDA copies, and is returned by
    zero_host_free (twice is an error: the address is no longer known)."""
    try:
        huge = int(open("/sys/kernel/mm/transparent_hugepage/hpage_pmd_size").read())
    except OSError:
        huge = 2 << 20
    page = os.sysconf("SC_PAGE_SIZE")
    small = zs.HostBuffer(1000, torch.float32)
    assert small.ptr % page == 0 and small.tensor.is_pinned()
    small.close()
    buf = zs.HostBuffer(huge // 2 + 5, torch.float16)      # just over one huge page of bytes
    assert buf.ptr % huge == 0
    assert buf.tensor.is_pinned()
    assert int(buf.tensor.view(torch.int16).abs().max()) == 0
    d = torch.arange(buf.tensor.numel(), device="cuda").to(torch.float16)
    buf.tensor.copy_(d, non_blocking=True)
    torch.cuda.synchronize()
    assert torch.equal(buf.tensor, d.cpu())
    ptr = buf.ptr
    buf.close()
    with pytest.raises(zs.ZeroError) as e:
        zs.zero_host_free(ptr)
    assert e.value.code == zs.ZERO_E_ARG


def test_host_step_with_the_benchmark_units():
    """The benchmark's ZeRO-3 units (50,331,648 parameters on 8 ranks; the first
    three of its 24, to keep the test's host memory small) fed from host
    memory the way the benchmark's end-to-end leg feeds them (one huge-page
    block for the W gradient vectors and the read-back): two steps,
    bit-identical to the device step, the read-back equal to the device's
    shard stores."""
    wl = wk.scaled(wk.LAYER_UNITS, unit_sizes=wk.LAYER_UNITS.unit_sizes[:3], steps=2)
    units, W = wl.units(), wl.W
    theta0 = wk.draw_theta0(wl, "cuda")
    a = zs.ZeroStep(zs.ZERO_SCHEME_Z3, W, units, "bf16", theta0=theta0, with_grad_buffers=True)
    b = zs.ZeroStep(zs.ZERO_SCHEME_Z3, W, units, "bf16", theta0=theta0)
    del theta0
    n_pad, out_elems = a.n_pad, W * a.sizes["shard_store"]
    block = zs.HostBuffer(W * n_pad + out_elems, torch.int16)
    host = [block.tensor[r * n_pad:(r + 1) * n_pad].view(torch.bfloat16) for r in range(W)]
    host_out = block.tensor[W * n_pad:].view(torch.bfloat16)
    need = zs.zero_host_staging_bytes(zs.ZERO_SCHEME_Z3, W, units, 0)
    staging = torch.empty(need, dtype=torch.uint8, device="cuda")
    sh, sd = torch.cuda.Stream(), torch.cuda.Stream()
    src = wk.GradSource(wl, "bf16", "cuda")
    hp = (wl.lr, wl.beta1, wl.beta2, wl.eps)
    for t in range(1, wl.steps + 1):
        for g, d in zip(a.grads, src.step(t)):
            a.place_(g, d)
        for h, g in zip(host, a.grads):
            h.copy_(g)
        torch.cuda.synchronize()
        a.step(a.grads, *hp, t)
        zs.zero_step_host(b.ctx, zs.ZERO_SCHEME_Z3, W, wl.n, host, host_out, staging, need, 0, *hp, t, sh, sd)
        b.sync(timeout_ms=120_000)
        for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32)), t
        want = torch.cat([x.cpu() for x in b.shard16])
        assert torch.equal(host_out.view(torch.int16), want.view(torch.int16)), t
        for x, y in zip(a.shard16, b.shard16):
            assert torch.equal(x.view(torch.int16), y.view(torch.int16)), t
    assert a.stat(zs.ZERO_STAT_COMM_BYTES) == b.stat(zs.ZERO_STAT_COMM_BYTES)
    del host, host_out
    block.close()
    a.close()
    b.close()


def test_host_step_with_the_headline_chunking():
    """The GPT-2-1.5B workload's ranks and format (W = 16, fp16, ZeRO-1) on a
    vector long enough that the default chunk is above 2^24 elements
    (25 x 2^24 + 12,345 parameters: chunks of 17,825,792), fed from one
    huge-page block the way the benchmark's end-to-end leg feeds it: two
    steps, bit-identical to the device step, the read-back equal to the
    device's working copy."""
    n = 25 * (1 << 24) + 12_345
    wl = wk.scaled(wk.GPT2_XL, n=n, steps=2, name="headline_chunking")
    W = wl.W
    theta0 = wk.draw_theta0(wl, "cuda")
    a = zs.ZeroStep(zs.ZERO_SCHEME_Z1, W, [n], "fp16", theta0=theta0, with_grad_buffers=True)
    b = zs.ZeroStep(zs.ZERO_SCHEME_Z1, W, [n], "fp16", theta0=theta0)
    del theta0
    n_pad = a.n_pad
    chunk = -(-(-(-n_pad // 24)) // (1 << 20)) * (1 << 20)        # n_pad / 24, up to a multiple of 2^20
    assert chunk > 1 << 24
    need = zs.zero_host_staging_bytes(zs.ZERO_SCHEME_Z1, W, [n], 0)
    assert need == 2 * W * (((chunk + 8) * 2 + 255) // 256 * 256)
    staging = torch.empty(need, dtype=torch.uint8, device="cuda")
    block = zs.HostBuffer(W * n_pad + n_pad, torch.int16)
    host = [block.tensor[r * n_pad:(r + 1) * n_pad].view(torch.float16) for r in range(W)]
    host_out = block.tensor[W * n_pad:].view(torch.float16)
    sh, sd = torch.cuda.Stream(), torch.cuda.Stream()
    src = wk.GradSource(wl, "fp16", "cuda")
    hp = (wl.lr, wl.beta1, wl.beta2, wl.eps)
    for t in range(1, wl.steps + 1):
        for g, d in zip(a.grads, src.step(t)):
            a.place_(g, d)
            del d
        for h, g in zip(host, a.grads):
            h.copy_(g)
        torch.cuda.synchronize()
        a.step(a.grads, *hp, t)
        zs.zero_step_host(b.ctx, zs.ZERO_SCHEME_Z1, W, n, host, host_out, staging, need, 0, *hp, t, sh, sd)
        b.sync(timeout_ms=120_000)
        for x, y in ((a.master, b.master), (a.m, b.m), (a.v, b.v)):
            assert torch.equal(x.view(torch.int32), y.view(torch.int32)), t
        assert torch.equal(a.p16.view(torch.int16), b.p16.view(torch.int16)), t
        assert torch.equal(host_out.view(torch.int16), b.p16.cpu().view(torch.int16)), t
    assert a.stat(zs.ZERO_STAT_COMM_BYTES) == b.stat(zs.ZERO_STAT_COMM_BYTES)
    del host, host_out
    block.close()
    a.close()
    b.close()


def _random_case(seed):
    """A seeded random case of test_host_step_equals_device_step's form."""
    import numpy as np
    rng = np.random.default_rng(6000 + seed)
    scheme = int(rng.integers(0, 4))
    W = int(rng.choice([1, 2, 3, 5, 8, 16, 24]))
    if scheme == zs.ZERO_SCHEME_Z3:
        size = [int(rng.choice([0, 1, 7, 4096, int(rng.integers(10, 400_000))])) for _ in range(int(rng.integers(1, 6)))]
        if sum(size) == 0:
            size[0] = 1
    else:
        size = int(rng.integers(1, 1_500_000))
    chunk = int(rng.choice([0, 1000, 65_536, int(rng.integers(8, 300_000))]))
    mem = str(rng.choice(["pin", "page", "huge"]))
    return (scheme, size, W, str(rng.choice(["fp16", "bf16"])), chunk, mem, bool(rng.random() < 0.8))


@pytest.mark.parametrize("seed", range(12))
def test_random_host_fed_configurations(seed):
    """Seeded random schemes, rank counts, sizes (ZeRO-3: ragged and empty
    units), chunk lengths, kinds of host memory and read-back: the host-fed
    step bit for bit equal to the device step, three steps each."""
    test_host_step_equals_device_step(_random_case(seed))
