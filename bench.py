#!/usr/bin/env python3
"""Throughput of the ZeRO step on GB300: parameters updated per second and
achieved HBM bandwidth, through the library's C ABI.

A step is one pass of the whole hot path over one batch of synthetic
gradients: the mean reduce-scatter of W ranks' 16-bit gradients, Adam with
bias correction on the fp32 master / m / v, the recast and gather of the
16-bit working copy and, for ZeRO-3, the per-unit gather / release /
re-gather schedule.  The default workload is the largest that fits one GPU:
a GPT-2-1.5B-sized flat vector (1,557,611,200 parameters, 16 simulated
ranks, fp16, ZeRO-1).  The same process then times the other configurations
on the device and reports them under ``also``: the ZeRO-3 layer-unit
schedule (24 units of 50,331,648 parameters, 8 ranks, bf16), the only one
that passes through every stage, and the GPT-2-small-sized vector (ZeRO-2,
8 ranks) with bf16 and with fp16 gradients, with bf16 applied bucket by
bucket (zero_step_bucket, 8 buckets of 2^24), as data parallelism with its 8
replicas kept literally, and as ZeRO-2 with the optimizer on the host.  ``--workload`` selects another
headline; ``--no-also`` leaves the others out.

Prints one JSON line.  ``value`` is whole-job parameters per second with the
inputs resident in HBM; ``e2e`` is the same metric with the gradients copied
in from page-locked host memory and the 16-bit working copy read back every step;
``roofline`` is for the fused reduce-scatter + Adam + recast kernel, timed
per launch with CUDA events on its own stream inside the timed region;
``cpu_baseline`` is the CPU oracle timed on a bounded sample on this host.

``--impl reference`` times the CPU oracle instead (on the host cores, a
bounded sample per step) and prints the same line with ``"impl": "reference"``.

Several GPUs (``--gpus N`` under torchrun) run N independent replicas of the
single-GPU step: the method's ranks are simulated inside one GPU, so there is
no data-path collective; a barrier and a max over ranks bracket the timing.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "params updated/sec per ZeRO step and achieved HBM GB/s vs GB300 peak (1 GPU)"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 126 * 1024 * 1024


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="gpt2_1p5b_w16_zero1",
                   choices=["zero3_24x50m_w8", "gpt2_small_124m_w8_zero2", "gpt2_1p5b_w16_zero1",
                            "gpt2_small_124m_w8_dp_replicas", "gpt2_small_124m_w8_zero2_offload"])
    p.add_argument("--dtype", choices=["bf16", "fp16"], default=None)
    p.add_argument("--params", type=int, default=None,
                   help="flat workloads only: a smaller copy with this many parameters (same W, dtype, "
                        "distributions and kernel), for profiling")
    p.add_argument("--units", type=int, default=None,
                   help="ZeRO-3 only: keep the first N units (a smaller copy of the workload with the same "
                        "per-unit launches, for profiling)")
    p.add_argument("--variant", choices=["auto", "vector", "bulk"], default="auto",
                   help="the fused kernel the headline workload runs (zero_set_variant; for profiling)")
    p.add_argument("--hook", action="store_true",
                   help="ZeRO-3 headline: register an empty unit hook, so the step runs its prefetch schedule "
                        "(a gather launch per unit on the gather stream; for profiling)")
    p.add_argument("--no-also", action="store_true",
                   help="time only the headline workload (not the other configurations under 'also')")
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="CPU oracle sample budget")
    p.add_argument("--reference-seconds", type=float, default=150.0,
                   help="--impl reference: oracle seconds for the whole run (split over warmup + steps)")
    return p.parse_args(argv)


# ---- workload arithmetic ----------------------------------------------------------

def workload(name, units=None, params=None):
    import workloads as wk
    wl = wk.WORKLOADS[name]
    if units is not None and wl.unit_sizes is not None and units < len(wl.unit_sizes):
        wl = wk.scaled(wl, unit_sizes=wl.unit_sizes[:units], name=f"{wl.name}_first{units}units")
    if params is not None and wl.unit_sizes is None and params < wl.n:
        wl = wk.scaled(wl, n=params, name=f"{wl.name}_{params}params")
    return wl


def scheme_of(wl):
    return wl.schemes[0]


def layout_sizes(wl):
    """(n_pad, unit elements per fused launch, units) of the flat layout."""
    W = wl.W
    units = wl.units() if scheme_of(wl) == 3 else [wl.n]
    padded = [-(-u // W) * W for u in units]
    return sum(padded), padded, units


def gather_kernel(wl):
    """The kernel of a ZeRO-3 step's forward gathers without a hook: all units
    in one launch (gather_units) when they share one padded shard size whose
    bytes are a multiple of 32, else two units per launch (copy_segments)."""
    W = wl.W
    shards = {-(-u // W) for u in wl.units()}
    return "gather_units" if len(shards) == 1 and (2 * shards.pop()) % 32 == 0 else "copy_segments"


def bytes_per_element(wl):
    """Bytes the fused pass moves per element: the W 16-bit gradients read
    once, then 12 read + 14 written per copy of the state (W copies when the
    DP replicas are kept literally)."""
    return 2 * wl.W + 26 * (wl.W if wl.dp_replicas else 1)


def algorithmic_bytes(wl):
    """Bytes a step must move: the fused pass (bytes_per_element per
    element); each ZeRO-3 gather reads and writes 2 bytes per element, twice
    per step."""
    n_pad, _, _ = layout_sizes(wl)
    fused = bytes_per_element(wl) * n_pad
    gathers = 8 * n_pad if scheme_of(wl) == 3 else 0
    return fused, gathers


# ---- environment facts -------------------------------------------------------------

def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(profile: str, kernel_sources):
    """Per-launch DRAM bytes from the committed ncu summary ``profiles/<profile>.md``,
    or None when there is none or the kernel's sources (the files named, in
    order) changed since it was taken."""
    path = os.path.join(ROOT, "profiles", f"{profile}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m1 = re.search(r"traffic_bytes_per_launch\s*=\s*(\d+)", text)
    m2 = re.search(r"kernel_source_sha256\s*=\s*([0-9a-f]{64})", text)
    if not (m1 and m2):
        return None
    if kernel_source_sha256(kernel_sources) != m2.group(1):
        return None
    return int(m1.group(1))


def kernel_source_sha256(kernel_sources) -> str:
    h = hashlib.sha256()
    for name in kernel_sources:
        h.update(open(os.path.join(ROOT, "zero_sharded_mixed_step_gb300", "csrc", name), "rb").read())
    return h.hexdigest()


FUSED_SOURCES = ("fused_step.cu", "step_math.cuh")
COPY_SOURCES = ("copy_cast.cu",)
REPLICA_SOURCES = ("dp_replicas.cu", "step_math.cuh")


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id, self.proc, self.lines = gpu_id, None, []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        time.sleep(0.15)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---- the CPU oracle (the CPU baseline leg and the reference arm) --------------------

def oracle_bytes(wl, elems: int) -> int:
    """Host bytes the oracle holds for a sample of ``elems`` parameters: W
    16-bit gradient vectors and their fp64 copies, fp32 master / m / v per
    rank copy (W of them under literal DP replicas), and fp64 temporaries."""
    copies = wl.W if scheme_of(wl) == 0 else 1
    return elems * (wl.W * (2 + 8) + copies * (12 + 2) + 6 * 8)


def check_host_memory(need: int, what: str) -> None:
    """Fail with a clear message, before allocating, when the host cannot hold ``need`` bytes."""
    avail = host_mem_available()
    if avail is None:
        return
    if need > avail:
        raise MemoryError(f"{what} needs about {need / 1e9:.1f} GB of host memory; {avail / 1e9:.1f} GB available")


def oracle_sample_steps(wl, sample_elems: int, dtype: str, budget_s: float = 0.0, max_steps: int = 1):
    """The oracle on a sample of about ``sample_elems`` parameters of ``wl``
    (ZeRO-3: one unit shrunk to that size; otherwise the first sample_elems
    parameters), on synthetic draws: steps t = 1, 2, ... until ``budget_s``
    seconds of oracle time are spent or ``max_steps`` steps are done (at
    least one).  Returns (seconds in the oracle's steps, parameters of the
    sample, steps run); drawing the inputs is not timed."""
    import workloads as wk
    from oracle import zero_oracle as z
    scheme = scheme_of(wl)
    W = wl.W
    sample_elems = max(W, sample_elems // W * W)
    check_host_memory(oracle_bytes(wl, sample_elems), f"the CPU oracle on {sample_elems:,} parameters")
    units = [sample_elems] if scheme != 3 else [min(sample_elems, wl.units()[0])]
    small = wk.scaled(wl, unit_sizes=units, name=wl.name + "_sample") if scheme == 3 else \
        wk.scaled(wl, n=sample_elems, name=wl.name + "_sample")
    theta0 = wk.draw_theta0(small, "cpu").numpy()
    orc = z.make_scheme(scheme, W, theta0, dtype, units if scheme == 3 else None)
    src = wk.GradSource(small, dtype, "cpu")
    total, steps = 0.0, 0
    while steps < max(1, max_steps) and (steps == 0 or total < budget_s):
        grads = [z.place(wk.to_numpy16(g), orc.layout) for g in src.step(steps + 1)]
        t0 = time.perf_counter()
        orc.step(grads, wl.lr, wl.beta1, wl.beta2, wl.eps)
        total += time.perf_counter() - t0
        steps += 1
        del grads
    return total, small.n, steps


def oracle_sample_step_seconds(wl, sample_elems: int, dtype: str):
    """Seconds of one oracle step (t = 1) on a sample (see oracle_sample_steps)."""
    dt, n, _ = oracle_sample_steps(wl, sample_elems, dtype)
    return dt, n


def cpu_cores_note():
    try:
        n = len(os.sched_getaffinity(0))
    except Exception:
        n = os.cpu_count() or 1
    model = ""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        m = re.search(r"Model name:\s*(.+)", out)
        model = m.group(1).strip() if m else ""
    except Exception:
        pass
    return n, model


SAMPLE_CAP = 1 << 24


def calibrate_sample(wl, dtype, budget_s):
    """Sample size whose oracle step takes about budget_s seconds, at most
    2^24 parameters (the oracle's elementwise rate does not depend on the
    size beyond that, and its host memory does: about 220 bytes per
    parameter at W = 16)."""
    dt, n = oracle_sample_step_seconds(wl, 1 << 20, dtype)
    per = dt / n
    return int(max(1 << 18, min(budget_s / per, wl.n, SAMPLE_CAP)))


def cpu_baseline(wl, dtype, budget_s):
    """The oracle as it stands, timed on this host for about ``budget_s``
    seconds: a sample sized so that one step takes about that long (capped
    at the workload, at one unit for ZeRO-3, and at 2^24 parameters), run
    for as many steps as the budget holds (at most 100)."""
    size = calibrate_sample(wl, dtype, budget_s)
    dt, n, steps = oracle_sample_steps(wl, size, dtype, budget_s, max_steps=100)
    host_cores, model = cpu_cores_note()
    what = (f"{steps} step(s) (t = 1..{steps}) of the oracle on {n:,} of the {wl.n:,} parameters "
            + ("(one unit shrunk to that size, full ZeRO-3 schedule)" if scheme_of(wl) == 3 else "(leading slice)")
            + f", W={wl.W}, {dtype} gradients; NumPy elementwise, one thread of {host_cores} host cores"
            + (f" ({model})" if model else ""))
    return {"value": n * steps / dt, "unit": "params/s", "cores": 1, "kind": "oracle", "sample": what,
            "seconds": round(dt, 3), "steps": steps}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    wl = workload(args.workload, args.units, args.params)
    dtype = args.dtype or wl.dtypes[0]
    budget = max(0.05, args.reference_seconds / max(1, args.steps + args.warmup))
    size = calibrate_sample(wl, dtype, budget)
    for _ in range(args.warmup):
        oracle_sample_step_seconds(wl, size, dtype)
    total, elems = 0.0, 0
    for _ in range(args.steps):
        dt, n = oracle_sample_step_seconds(wl, size, dtype)
        total += dt
        elems += n
    value = elems / total
    host_cores, model = cpu_cores_note()
    n_pad, per_launch, units = layout_sizes(wl)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "params/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(wl, dtype, args.gpus),
        "cpu_baseline": {"value": value, "unit": "params/s", "cores": 1, "kind": "oracle",
                         "sample": f"each step: the oracle on {elems // args.steps:,} of {wl.n:,} parameters, "
                                   f"one NumPy thread of {host_cores} host cores ({model})"},
        "e2e": {"value": value, "unit": "params/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def config_of(wl, dtype, gpus):
    n_pad, per_launch, units = layout_sizes(wl)
    fused, gathers = algorithmic_bytes(wl)
    names = {0: "data parallel", 1: "ZeRO-1", 2: "ZeRO-2", 3: "ZeRO-3"}
    scheme = names[scheme_of(wl)] + (f", {wl.W} replicas kept literally" if wl.dp_replicas else "") + \
        (", optimizer state and update on the host CPU" if wl.offload else "")
    return {"workload": wl.name, "scheme": scheme, "W": wl.W, "params": wl.n, "padded": n_pad,
            "units": len(units), "grad_dtype": dtype, "work_dtype": dtype, "master_dtype": "f32",
            "algorithmic_bytes_per_step": fused + gathers,
            "l2": f"inputs larger than L2: {(fused + gathers) / 1e9:.1f} GB touched per step vs "
                  f"{L2_BYTES / 2**20:.0f} MiB of L2",
            "parallelism": "simulated DP ranks in one GPU" + (f"; {gpus} independent replicas" if gpus > 1 else ""),
            "zero3_schedule": ("forward gathers of all units in one launch (equal units); per unit, backward gather "
                               "fused into the update pass (no unit hook registered); the step's launches "
                               "replayed from a CUDA graph (zero_set_graph), its backward passes on two chains of "
                               "alternate units; the per-launch timing pass as ordinary launches on one stream")
            if scheme_of(wl) == 3 else None}


# ---- several GPUs: independent replicas -----------------------------------------------

def max_over_ranks(x: float) -> float:
    """The slowest rank's time (no data-path collective: a scalar reduction
    over the process group that brackets the timing)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return x
    tt = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def whole_job_value(world: int, n: int, steps: int, ms: float) -> float:
    """Parameters updated per second over all replicas: every replica runs
    the full workload (weak scaling), timed by the slowest one."""
    return world * n * steps / (ms / 1e3)


# ---- our arm ------------------------------------------------------------------------

# (workload, gradient format, bucket elements: the step applied bucket by bucket with zero_step_bucket)
ALSO = (("gpt2_1p5b_w16_zero1", None, None), ("zero3_24x50m_w8", None, None),
        ("gpt2_small_124m_w8_zero2", "bf16", None), ("gpt2_small_124m_w8_zero2", "fp16", None),
        ("gpt2_small_124m_w8_zero2", "bf16", 1 << 24), ("gpt2_small_124m_w8_dp_replicas", "bf16", None),
        ("gpt2_small_124m_w8_zero2_offload", "bf16", None))


def device_leg(args, wl, dtype, dev, world, clocks_too: bool = True, bucket_elems=None, variant="auto",
               hook=False):
    """The step with its inputs resident in HBM: warm-up, then ``args.steps``
    timed steps (pass 1, CUDA events around the loop on the update stream),
    then the same steps again with a CUDA event pair around every launch
    (pass 2, zero_enable_timing) for the per-launch roofline; the brackets
    cost about 3% of a ZeRO-3 step, so they stay out of pass 1.  With
    ``bucket_elems`` (DP/Z1/Z2) each step is applied bucket by bucket
    (zero_step_bucket), each bucket reading its range of the gradient
    vectors, as the buckets of a backward pass would arrive.  Returns (the
    ZeroStep, its update stream, the step counter reached, the leg's
    figures)."""
    import torch
    import torch.distributed as dist
    import zero_sharded_mixed_step_gb300 as zs
    import workloads as wk

    scheme = scheme_of(wl)
    n_pad, per_launch, units = layout_sizes(wl)
    su = torch.cuda.Stream(dev)
    sg = torch.cuda.Stream(dev) if scheme == 3 else None
    with torch.cuda.stream(su):
        theta0 = wk.draw_theta0(wl, dev)
        step = zs.ZeroStep(scheme, wl.W, units, dtype, theta0=theta0, device=dev, stream=su, gather_stream=sg,
                           with_grad_buffers=True)
        step.set_variant({"auto": zs.ZERO_VARIANT_AUTO, "vector": zs.ZERO_VARIANT_VECTOR,
                          "bulk": zs.ZERO_VARIANT_BULK}[variant])
        if scheme == 3 and hook:
            step.set_unit_hook(lambda user, phase, unit, buf, stream: None)
        elif scheme == 3:
            step.set_graph(True)     # the step's launches replayed from one captured graph
        del theta0
        for r, d in enumerate(wk.GradSource(wl, dtype, dev).step(1)):
            step.place_(step.grads[r], d)
            del d
    torch.cuda.synchronize()
    hp = (wl.lr, wl.beta1, wl.beta2, wl.eps)
    buckets = None
    if bucket_elems:
        # each bucket's gradient pointers into the W vectors, built once
        buckets = [(lo, min(bucket_elems, n_pad - lo), [g.data_ptr() + 2 * lo for g in step.grads])
                   for lo in range(0, n_pad, bucket_elems)]

    def one_step(t):
        if buckets is None:
            step.step(step.grads, *hp, t)
        else:
            for lo, length, ptrs in buckets:
                zs.zero_step_bucket(step.ctx, lo, length, ptrs, *hp, t, su)

    t = 0
    for _ in range(args.warmup):
        t += 1
        one_step(t)
    torch.cuda.synchronize()

    def timed_pass(instrumented: bool):
        nonlocal t
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        zs.zero_enable_timing(step.ctx, instrumented)
        n0 = step.stat(zs.ZERO_STAT_LAUNCHES)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(su)
        for _ in range(args.steps):
            t += 1
            one_step(t)
        e1.record(su)
        torch.cuda.synchronize()
        zs.zero_enable_timing(step.ctx, False)
        if world > 1:
            dist.barrier()
        return e0.elapsed_time(e1), step.stat(zs.ZERO_STAT_LAUNCHES) - n0

    zs.zero_read_timing(step.ctx, zs.ZERO_KERNEL_FUSED)
    zs.zero_read_timing(step.ctx, zs.ZERO_KERNEL_GATHER)
    if clocks_too:
        with ClockSampler(gpu_uuid(dev)) as clocks:
            ms, launches = timed_pass(False)
        clock_summary = clocks.summary()
    else:
        ms, launches = timed_pass(False)
        clock_summary = None
    ms_instr, _ = timed_pass(True)
    fused_ms, fused_n = zs.zero_read_timing(step.ctx, zs.ZERO_KERNEL_FUSED)
    last_variant = step.stat(zs.ZERO_STAT_LAST_VARIANT)
    gather_ms, gather_n = zs.zero_read_timing(step.ctx, zs.ZERO_KERNEL_GATHER)
    ms = max_over_ranks(ms)
    ms_per_step = ms / args.steps
    value = whole_job_value(world, wl.n, args.steps, ms)
    fused_b, gather_b = algorithmic_bytes(wl)
    step_gbs = (fused_b + gather_b) / (ms_per_step / 1e3) / 1e9

    # roofline of the dominant kernel: the fused pass, per launch.  Without a
    # unit hook a ZeRO-3 update launch also performs its unit's backward
    # gather (2 bytes read + 2 written per element on top of 2 W + 26).
    peak, peak_src = hbm_peak()
    per_elem = 2 * wl.W + 26 + (4 if scheme == 3 and not hook else 0)   # with a hook the gathers are separate
    per_launch_bytes = per_elem * (per_launch[0] if buckets is None else n_pad // len(buckets))
    fused_avg_ms = fused_ms / max(1, fused_n)
    achieved = per_launch_bytes / (fused_avg_ms / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": recorded_traffic(f"fused_step_{wl.name}", FUSED_SOURCES),
                "kernel": "fused_step_bulk" if last_variant == zs.ZERO_VARIANT_BULK else "fused_step_vector",
                "peak_source": f"{peak_src} copy bandwidth", "launch_ms": fused_avg_ms,
                "algorithmic_bytes_per_launch": per_launch_bytes, "bytes_per_element": per_elem,
                "frac_of_8tbs_nominal": achieved / 8000.0,
                "launches_timed": fused_n, "timing_pass_ms_per_step": ms_instr / args.steps}
    gather_info = None
    if gather_n:
        # the forward gathers move 2 bytes in and 2 out per element of every unit
        # (all units in one launch when they have one size, else two per launch;
        # the backward gathers are inside the fused pass); with a hook every
        # gather, forward and backward, is a launch of its own, one unit each
        gather_bytes = (8 if hook else 4) * n_pad * args.steps
        achieved_g = gather_bytes / (gather_ms / 1e3) / 1e9
        kernel = "copy_segments" if hook else gather_kernel(wl)
        gather_info = {"kernel": kernel, "launch_ms": gather_ms / gather_n, "achieved_gbs": achieved_g,
                       "frac": achieved_g / peak, "launches": gather_n,
                       "bytes_per_launch": gather_bytes // gather_n,
                       "traffic": recorded_traffic(f"{kernel}_{wl.name}", COPY_SOURCES),
                       "share_of_bracketed_time": gather_ms / (gather_ms + fused_ms)}
    leg = {"workload": wl.name, "grad_dtype": dtype, "value": value, "unit": "params/s", "ms_per_step": ms_per_step,
           "buckets": None if buckets is None else {"bucket_elems": bucket_elems, "per_step": len(buckets),
                                                    "entry_point": "zero_step_bucket"},
           "steps": args.steps, "warmup": args.warmup, "step_hbm_gbs": step_gbs, "step_frac_of_peak": step_gbs / peak,
           "algorithmic_bytes_per_step": fused_b + gather_b, "roofline": roofline, "gather": gather_info,
           "gpu_launches": launches, "clocks": clock_summary}
    return step, su, t, leg


def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    from zero_sharded_mixed_step_gb300 import build
    build.build()
    import zero_sharded_mixed_step_gb300 as zs

    wl = workload(args.workload, args.units, args.params)
    dtype = args.dtype or wl.dtypes[0]
    if wl.dp_replicas:
        return run_replicas(args, wl, dtype, world, rank, dev)
    if wl.offload:
        return run_offload(args, wl, dtype, world, rank, dev)
    scheme = scheme_of(wl)
    n_pad, per_launch, units = layout_sizes(wl)
    step, su, t, leg = device_leg(args, wl, dtype, dev, world, variant=args.variant, hook=args.hook)
    hp = (wl.lr, wl.beta1, wl.beta2, wl.eps)

    # ---- end to end: gradients from page-locked host memory, working copy read back --
    # through zero_step_host, the C-ABI call that takes host buffers: each step
    # streams the W ranks' gradients over the host link into a two-slot device
    # staging ring and returns the updated 16-bit working copy to host memory,
    # pipelined chunk by chunk (unit by unit for ZeRO-3) on three streams.
    e2e = None
    out_elems = step.n_pad if scheme != 3 else wl.W * step.sizes["shard_store"]
    e2e_room = host_room_for(2 * (wl.W * step.n_pad + out_elems), world)
    if not args.no_e2e and args.e2e_steps > 0 and e2e_room is not None:
        e2e = {"skipped": e2e_room}
    elif not args.no_e2e and args.e2e_steps > 0:
        # host buffers from zero_host_alloc: page-locked on huge pages, where the
        # link holds its full rate (memory from cudaHostAlloc measured slower)
        # one block for the W gradient vectors and the read-back (all 16-bit),
        # so that even vectors smaller than a huge page sit on huge pages
        need = zs.zero_host_staging_bytes(scheme, wl.W, units, 0)
        staging = torch.empty(need, dtype=torch.uint8, device=dev)
        sh, sd = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

        def views_of(block):
            grads_h = [block[r * step.n_pad:(r + 1) * step.n_pad].view(step.grad_torch_dtype) for r in range(wl.W)]
            out_h = block[wl.W * step.n_pad:].view(step.work_torch_dtype)
            for h, g in zip(grads_h, step.grads):
                h.copy_(g)
            return grads_h, out_h

        def probe_of(views):
            grads_h, out_h = views
            if scheme != 3:
                back = [(out_h, step.p16)]
            else:
                S16 = step.sizes["shard_store"]
                back = [(out_h[r * S16:(r + 1) * S16], step.shard16[r]) for r in range(wl.W)]
            return link_probe(list(zip(step.grads, grads_h)), back, sh)

        block_buf, (host_grads, host_out), link, spares = settled_host_block(wl.W * step.n_pad + out_elems,
                                                                             views_of, probe_of)
        host_bufs = [block_buf]

        def host_step():
            nonlocal t
            t += 1
            zs.zero_step_host(step.ctx, scheme, wl.W, wl.n, host_grads, host_out, staging, need, 0, *hp, t, sh, sd)

        for _ in range(2):               # warm the path, untimed
            host_step()
        step.sync()
        if world > 1:
            dist.barrier()
        marks = StepMarks(sd)            # each step ends with its read-back on sd
        h0 = time.perf_counter()
        for _ in range(args.e2e_steps):
            host_step()
            marks.mark()
        step.sync()
        e2e_s = max_over_ranks(time.perf_counter() - h0)
        link["after"] = after_e2e(probe_of, (host_grads, host_out), host_bufs)
        h2d = sum(h.numel() * h.element_size() for h in host_grads)
        d2h = host_out.numel() * host_out.element_size()
        e2e = {"value": whole_job_value(world, wl.n, args.e2e_steps, 1e3 * e2e_s), "unit": "params/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": args.e2e_steps,
               "ms_per_step": 1e3 * e2e_s / args.e2e_steps, "step_ms": marks.spread(), "staging_bytes": need,
               "path": "zero_step_host: host gradients (zero_host_alloc) -> 2-slot device staging ring -> "
                       "fused step -> 16-bit working copy -> host, pipelined over three streams", "link": link}
        del host_grads, host_out, staging
        for b in host_bufs + spares:
            b.close()

    step.close()
    del step
    torch.cuda.empty_cache()

    # the other configurations, on the device only, one at a time (each
    # freed before the next), after the headline's timed regions
    also = {}
    if not args.no_also and args.units is None and args.params is None:
        for name, dt, bucket in ALSO:
            other = workload(name)
            dt = dt or other.dtypes[0]
            if other.name == wl.name and dt == dtype and bucket is None:
                continue
            if other.dp_replicas:
                o_step, o_grads, _, _, o_leg = replicas_leg(args, other, dt, dev, world)
                del o_grads
            elif other.offload:
                o_step, o_grads, _, _, o_leg = offload_leg(args, other, dt, dev, world)
                del o_grads
            else:
                o_step, _, _, o_leg = device_leg(args, other, dt, dev, world, clocks_too=True, bucket_elems=bucket)
            if hasattr(o_step, "close"):        # the replicas hold only tensors
                o_step.close()
            del o_step
            torch.cuda.empty_cache()
            o_leg["config"] = config_of(other, dt, world)
            key = f"{name}_{dt}" if name == "gpt2_small_124m_w8_zero2" else name
            if bucket:
                key += f"_buckets_of_2p{bucket.bit_length() - 1}"
            also[key] = o_leg

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, dtype, args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": leg["value"], "unit": "params/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": leg["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": config_of(wl, dtype, world),
            "step_hbm_gbs": leg["step_hbm_gbs"], "step_frac_of_peak": leg["step_frac_of_peak"],
            "roofline": leg["roofline"], "gather": leg["gather"], "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": leg["gpu_launches"], "clocks": leg["clocks"],
            "also": also or None,
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def link_probe(h2d_pairs, d2h_pairs, stream):
    """The host link's rate right now: the step's own host->device copies
    and its read-back as plain copies, timed on their own, so that an
    end-to-end number can be read against the link it ran on (the link is
    shared with other jobs on the machine and varies between runs).
    Pairs are (destination, source) tensors."""
    import torch
    h2d = sum(src.numel() * src.element_size() for _, src in h2d_pairs)
    d2h = sum(src.numel() * src.element_size() for _, src in d2h_pairs)
    back = torch.cuda.Stream(stream.device)
    with torch.cuda.stream(stream):
        stream.synchronize()
        t0 = time.perf_counter()
        for dst, src in h2d_pairs:
            dst.copy_(src, non_blocking=True)
        stream.synchronize()
        t1 = time.perf_counter()
        for dst, src in d2h_pairs:
            dst.copy_(src, non_blocking=True)
        stream.synchronize()
        t2 = time.perf_counter()
        # both directions at once, as in a step: the link shares its rate between them
        for dst, src in h2d_pairs:
            dst.copy_(src, non_blocking=True)
        with torch.cuda.stream(back):
            for dst, src in d2h_pairs:
                dst.copy_(src, non_blocking=True)
        stream.synchronize()
        back.synchronize()
        t3 = time.perf_counter()
    return {"h2d_gbs": h2d / (t1 - t0) / 1e9, "d2h_gbs": d2h / (t2 - t1) / 1e9, "floor_ms": 1e3 * (t1 - t0),
            "both_directions_ms": 1e3 * (t3 - t2),
            "note": "plain copies of the step's bytes timed just before the end-to-end steps; "
                    "floor = the step's gradients carried in at that rate; both_directions = the "
                    "gradients in and the read-back out issued together on two streams"}


class StepMarks:
    """CUDA events on the stream that ends each end-to-end step: one before
    the first timed step and one after each, so that the steps' own
    durations can be read without a host synchronisation between them."""

    def __init__(self, stream):
        import torch
        self.stream = stream
        self.events = [torch.cuda.Event(enable_timing=True)]
        self.events[0].record(stream)

    def mark(self):
        import torch
        e = torch.cuda.Event(enable_timing=True)
        e.record(self.stream)
        self.events.append(e)

    def spread(self):
        """min / median / max of the marked steps' durations, ms (after a sync)."""
        ms = sorted(a.elapsed_time(b) for a, b in zip(self.events, self.events[1:]))
        if not ms:
            return None
        return {"min": ms[0], "median": ms[len(ms) // 2], "max": ms[-1]}


def after_e2e(probe_of, views, bufs):
    """The link probe and the huge-page share once more, after the timed
    end-to-end steps: a slow run whose link was slow too was slowed by the
    link (shared with other jobs), one whose link was fast by the pipeline."""
    probe = probe_of(views)
    return {"h2d_gbs": probe["h2d_gbs"], "d2h_gbs": probe["d2h_gbs"],
            "host_huge_page_fraction": huge_page_fraction(bufs)}


def settled_host_block(elems16: int, views_of, probe_of, attempts: int = 3):
    """A zero_host_alloc block of ``elems16`` 16-bit elements whose pages are
    still all huge after a first round of the step's copies.

    ``views_of(block_tensor)`` cuts the block into the step's host tensors
    (and fills them); ``probe_of(views)`` times plain copies of the step's
    bytes (link_probe).  On these hosts an earlier process can leave memory
    whose huge pages get split by the first copies into them, and copies out
    of the split pages run at a fraction of the link's rate.  A block that
    comes out of its probe with split pages is kept aside (so that its pages
    are not handed out again) while a new one is taken, at most ``attempts``
    times.  The block that kept the most of its huge pages is used (the
    fastest probe among equals: a block whose pages have begun to split
    goes on splitting under later copies, even when its probe was still
    fast).  The others come back
    as spares for the caller to free once its timed steps are over: freeing
    tens of GB of pinned memory just before them set the kernel splitting the
    chosen block's huge pages while they ran.
    Returns (block, views, probe, spares) with the attempts recorded in the
    probe."""
    import torch
    import zero_sharded_mixed_step_gb300 as zs
    tried = []
    for _ in range(attempts):
        if tried:
            # another block only while the host keeps room for two more for
            # every process on it (several ranks on one host each hold their own)
            avail = host_mem_available()
            local = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
            if avail is not None and avail < 2 * 2 * elems16 * local:
                break
            try:
                hb = zs.HostBuffer(elems16, torch.int16)
            except zs.ZeroError:
                break
        else:
            hb = zs.HostBuffer(elems16, torch.int16)
        at_alloc = huge_page_fraction([hb])
        views = views_of(hb.tensor)
        probe = probe_of(views)
        probe["host_huge_page_fraction_at_alloc"] = at_alloc
        probe["host_huge_page_fraction"] = huge_page_fraction([hb])
        tried.append((hb, views, probe))
        if probe["host_huge_page_fraction"] is None or probe["host_huge_page_fraction"] >= 0.999:
            break
    best = max(tried, key=lambda x: (x[2]["host_huge_page_fraction"] or 0.0, x[2]["h2d_gbs"]))
    best[2]["host_block_attempts"] = len(tried)
    spares = [hb for hb, _, _ in tried if hb is not best[0]]
    return best[0], best[1], best[2], spares


def host_room_for(block_bytes: int, world: int) -> str | None:
    """None when every process on this host can take a page-locked block of
    ``block_bytes`` for the end-to-end leg (with a quarter of the available
    memory to spare), else the reason it cannot.  Decided the same way on
    every rank (a max over ranks), so that all of them run the leg's
    collectives or none does."""
    local = int(os.environ.get("LOCAL_WORLD_SIZE", "1"))
    avail = host_mem_available()
    short = avail is not None and block_bytes * local > 0.75 * avail
    if max_over_ranks(1.0 if short else 0.0) == 0.0:
        return None
    return (f"host memory: the end-to-end leg page-locks {block_bytes / 1e9:.1f} GB per process, "
            f"{local} process(es) per host; this host has {((avail or 0) / 1e9):.1f} GB available"
            + ("" if short else ", another rank's host ran short"))


def host_mem_available() -> int | None:
    """MemAvailable of /proc/meminfo in bytes (None where unreadable)."""
    try:
        for line in open("/proc/meminfo"):
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    except (OSError, ValueError, IndexError):
        pass
    return None


def huge_page_fraction(bufs) -> float | None:
    """Share of the host buffers' mapped bytes that the kernel backs with
    transparent huge pages (from /proc/self/smaps; None where unreadable)."""
    try:
        spans = {}
        cur = None
        for line in open("/proc/self/smaps"):
            head = line.split()
            if head and "-" in head[0] and line[0] in "0123456789abcdef":
                lo, hi = (int(x, 16) for x in head[0].split("-"))
                cur = (lo, hi)
            elif cur and head and head[0] == "AnonHugePages:":
                spans[cur] = int(head[1]) * 1024
        want = got = 0
        for b in bufs:
            for (lo, hi), huge in spans.items():
                if lo <= b.ptr < hi:
                    want += b.nbytes
                    got += min(huge, b.nbytes)
        return got / want if want else None
    except OSError:
        return None


def gpu_uuid(dev):
    import torch
    gpu_id = getattr(torch.cuda.get_device_properties(dev), "uuid", None)
    return f"GPU-{gpu_id}" if gpu_id is not None and not str(gpu_id).startswith("GPU-") else str(gpu_id or dev.index)


def e2e_through_torch_copies(args, world, wl, su, grads, result, run_step, t0, path):
    """End to end for the entry points that take device gradients: every
    step copies the W gradient vectors in from page-locked host memory
    (zero_host_alloc), runs the step, and reads ``result`` (a device tensor)
    back to host memory, all in order on ``su``.  ``run_step(t)`` enqueues one
    step.  Returns (the e2e dict, the last step counter used)."""
    import torch
    import torch.distributed as dist
    # one block for the W gradient vectors and the read-back (all 16-bit), so
    # that even vectors smaller than a huge page sit on huge pages
    n, W = grads[0].numel(), len(grads)
    room = host_room_for(2 * (W * n + result.numel()), world)
    if room is not None:
        return {"skipped": room}, t0

    def views_of(block):
        grads_h = [block[r * n:(r + 1) * n].view(grads[0].dtype) for r in range(W)]
        for h, g in zip(grads_h, grads):
            h.copy_(g)
        return grads_h, block[W * n:].view(result.dtype)

    def probe_of(views):
        grads_h, out_h = views
        return link_probe(list(zip(grads, grads_h)), [(out_h, result)], su)

    block_buf, (host_grads, host_out), link, spares = settled_host_block(W * n + result.numel(), views_of, probe_of)
    host_bufs = [block_buf]
    t = t0

    def host_step():
        nonlocal t
        t += 1
        with torch.cuda.stream(su):
            for g, h in zip(grads, host_grads):
                g.copy_(h, non_blocking=True)
            run_step(t)
            host_out.copy_(result, non_blocking=True)

    for _ in range(2):               # warm the path, untimed
        host_step()
    su.synchronize()
    if world > 1:
        dist.barrier()
    marks = StepMarks(su)
    h0 = time.perf_counter()
    for _ in range(args.e2e_steps):
        host_step()
        marks.mark()
    su.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - h0)
    link["after"] = after_e2e(probe_of, (host_grads, host_out), host_bufs)
    e2e = {"value": whole_job_value(world, wl.n, args.e2e_steps, 1e3 * e2e_s), "unit": "params/s",
           "h2d_bytes_per_step": sum(h.numel() * h.element_size() for h in host_grads),
           "d2h_bytes_per_step": host_out.numel() * host_out.element_size(), "steps": args.e2e_steps,
           "ms_per_step": 1e3 * e2e_s / args.e2e_steps, "step_ms": marks.spread(), "path": path, "link": link}
    del host_grads, host_out
    for b in host_bufs + spares:
        b.close()
    return e2e, t


def replicas_leg(args, wl, dtype, dev, world):
    """Plain data parallelism with the W replicas kept literally
    (zero_step_dp_replicas), its inputs resident in HBM: warm-up, then
    ``args.steps`` timed steps, one kernel per step, and the bitwise check
    that the replicas stayed equal.  Returns (the DpReplicas, the gradient
    buffers, the update stream, the step counter reached, the leg's
    figures)."""
    import torch
    import torch.distributed as dist
    import zero_sharded_mixed_step_gb300 as zs
    import workloads as wk

    su = torch.cuda.Stream(dev)
    with torch.cuda.stream(su):
        theta0 = wk.draw_theta0(wl, dev)
        rep = zs.DpReplicas(wl.W, wl.n, dtype, theta0=theta0, device=dev, stream=su)
        del theta0
        grads = rep.new_grad_buffers()
        for g, d in zip(grads, wk.GradSource(wl, dtype, dev).step(1)):
            g[: wl.n].copy_(d)
            del d
    torch.cuda.synchronize()
    hp = (wl.lr, wl.beta1, wl.beta2, wl.eps)
    t = 0
    for _ in range(args.warmup):
        t += 1
        rep.step(grads, *hp, t)
    torch.cuda.synchronize()

    # timed region: inputs resident in HBM, one kernel launch per step on su,
    # so the events around the loop time the launches themselves
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_uuid(dev)) as clocks:
        e0.record(su)
        for _ in range(args.steps):
            t += 1
            rep.step(grads, *hp, t)
        e1.record(su)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    ms = max_over_ranks(e0.elapsed_time(e1))
    ms_per_step = ms / args.steps
    launches = args.steps
    if rep.mismatches() != 0:
        raise RuntimeError("the DP replicas drifted apart")
    value = whole_job_value(world, wl.n, args.steps, ms)
    per_elem = bytes_per_element(wl)
    step_bytes = per_elem * rep.n_pad
    peak, peak_src = hbm_peak()
    achieved = step_bytes / (ms_per_step / 1e3) / 1e9
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": recorded_traffic(f"dp_replicas_step_{wl.name}", REPLICA_SOURCES),
                "kernel": "dp_replicas_step", "peak_source": f"{peak_src} copy bandwidth",
                "launch_ms": ms_per_step, "algorithmic_bytes_per_launch": step_bytes,
                "bytes_per_element": per_elem, "frac_of_8tbs_nominal": achieved / 8000.0, "launches_timed": launches}
    resident = sum(x.numel() * x.element_size() for x in rep.master + rep.m + rep.v + rep.p16)
    leg = {"workload": wl.name, "grad_dtype": dtype, "value": value, "unit": "params/s", "ms_per_step": ms_per_step,
           "steps": args.steps, "warmup": args.warmup, "step_hbm_gbs": achieved, "step_frac_of_peak": achieved / peak,
           "algorithmic_bytes_per_step": step_bytes, "replicated_state_bytes": resident, "roofline": roofline,
           "gather": None, "gpu_launches": launches, "clocks": clocks.summary(), "replica_mismatches": 0}
    return rep, grads, su, t, leg


def run_replicas(args, wl, dtype, world, rank, dev):
    """Plain data parallelism with the W replicas kept literally
    (zero_step_dp_replicas): every rank's fp32 master, m, v and 16-bit copy
    in HBM, one kernel per step that reads the W gradients once and updates
    all W replicas.  The same line as the sharded workloads, for the cost
    that sharding removes."""
    import torch
    import torch.distributed as dist

    rep, grads, su, t, leg = replicas_leg(args, wl, dtype, dev, world)
    hp = (wl.lr, wl.beta1, wl.beta2, wl.eps)
    e2e = None
    if not args.no_e2e and args.e2e_steps > 0:
        e2e, t = e2e_through_torch_copies(
            args, world, wl, su, grads, rep.p16[0], lambda tt: rep.step(grads, *hp, tt), t,
            "host gradients (zero_host_alloc) -> device gradient buffers (one copy per rank) -> "
            "zero_step_dp_replicas -> replica 0's 16-bit working copy -> host, one stream")

    del rep, grads
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, dtype, args.cpu_seconds)
    if rank == 0:
        config = config_of(wl, dtype, world)
        config["replicated_state_bytes"] = leg["replicated_state_bytes"]
        line = {
            "metric": METRIC, "value": leg["value"], "unit": "params/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": leg["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": config,
            "step_hbm_gbs": leg["step_hbm_gbs"], "step_frac_of_peak": leg["step_frac_of_peak"],
            "roofline": leg["roofline"], "gather": None, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": leg["gpu_launches"], "clocks": leg["clocks"],
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def host_copy_gbs(threads: int, nbytes: int = 1 << 31) -> float:
    """Measured host memory bandwidth: a multi-threaded copy of nbytes
    (read + write bytes per second), the denominator of the host update."""
    import torch
    old = torch.get_num_threads()
    torch.set_num_threads(threads)
    try:
        a = torch.ones(nbytes // 4, dtype=torch.float32)
        b = torch.empty_like(a)
        b.copy_(a)
        best = 0.0
        for _ in range(5):
            t0 = time.perf_counter()
            b.copy_(a)
            best = max(best, 2 * nbytes / (time.perf_counter() - t0) / 1e9)
        return best
    finally:
        torch.set_num_threads(old)


def offload_leg(args, wl, dtype, dev, world):
    """ZeRO-2 with the optimizer on the host (zero_offload_step), its
    gradients resident in HBM: warm-up, then ``args.steps`` timed steps; the
    roofline is that of the host update, which bounds the step.  Returns (the
    ZeroOffload, the gradient buffers, the update stream, the step counter
    reached, the leg's figures)."""
    import torch
    import torch.distributed as dist
    import zero_sharded_mixed_step_gb300 as zs
    import workloads as wk

    su = torch.cuda.Stream(dev)
    with torch.cuda.stream(su):
        theta0 = wk.draw_theta0(wl, dev)
        off = zs.ZeroOffload(wl.W, wl.n, dtype, theta0=theta0.cpu(), device=dev, stream=su)
        del theta0
        grads = off.new_grad_buffers()
        for g, d in zip(grads, wk.GradSource(wl, dtype, dev).step(1)):
            g[: wl.n].copy_(d)
            del d
    torch.cuda.synchronize()
    hp = (wl.lr, wl.beta1, wl.beta2, wl.eps)
    t = 0
    for _ in range(args.warmup):
        t += 1
        off.step(grads, *hp, t)
    torch.cuda.synchronize()

    if world > 1:
        dist.barrier()
    st0 = off.stats()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_uuid(dev)) as clocks:
        e0.record(su)
        for _ in range(args.steps):
            t += 1
            off.step(grads, *hp, t)
        e1.record(su)
        torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    st1 = off.stats()
    ms = max_over_ranks(e0.elapsed_time(e1))
    ms_per_step = ms / args.steps
    value = whole_job_value(world, wl.n, args.steps, ms)
    host_s = (st1["host_seconds"] - st0["host_seconds"]) / args.steps
    host_bytes = 30 * off.n_pad          # read mean 4 + master, m, v 12; write 12 + 16-bit 2
    achieved = host_bytes / host_s / 1e9
    peak = host_copy_gbs(st1["threads"])
    roofline = {"bound": "host_dram", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": None, "kernel": "host Adam (zero_offload_step's host update)",
                "peak_source": f"host copy measured in this run ({st1['threads']} threads, read + write)",
                "host_ms_per_step": 1e3 * host_s, "algorithmic_bytes_per_step": host_bytes, "bytes_per_element": 30,
                "threads": st1["threads"], "host_state_huge_page_fraction": huge_page_fraction(off._bufs)}
    launches = st1["launches"] - st0["launches"]
    link = {"d2h_bytes_per_step": (st1["d2h_bytes"] - st0["d2h_bytes"]) // args.steps,
            "h2d_bytes_per_step": (st1["h2d_bytes"] - st0["h2d_bytes"]) // args.steps}
    leg = {"workload": wl.name, "grad_dtype": dtype, "value": value, "unit": "params/s", "ms_per_step": ms_per_step,
           "steps": args.steps, "warmup": args.warmup,
           "algorithmic_bytes_per_step": (2 * wl.W + 4) * off.n_pad + host_bytes, "offload_link_bytes_per_step": link,
           "roofline": roofline, "gather": None, "gpu_launches": launches, "clocks": clocks.summary()}
    return off, grads, su, t, leg


def run_offload(args, wl, dtype, world, rank, dev):
    """ZeRO-2 with the optimizer on the host (zero_offload_step): the GPU forms
    the mean gradient, host threads run Adam on host-resident fp32 state, the
    16-bit copy streams back.  Same line as the other workloads; the roofline
    is that of the host update, which bounds the step."""
    import torch
    import torch.distributed as dist

    off, grads, su, t, leg = offload_leg(args, wl, dtype, dev, world)
    hp = (wl.lr, wl.beta1, wl.beta2, wl.eps)
    e2e = None
    if not args.no_e2e and args.e2e_steps > 0:
        e2e, t = e2e_through_torch_copies(
            args, world, wl, su, grads, off.p16, lambda tt: off.step(grads, *hp, tt), t,
            "host gradients (zero_host_alloc) -> device gradient buffers -> zero_offload_step "
            "(device mean, host Adam, 16-bit copy back) -> 16-bit working copy -> host")

    off.close()
    del grads
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, dtype, args.cpu_seconds)
    if rank == 0:
        config = config_of(wl, dtype, world)
        config["algorithmic_bytes_per_step"] = leg["algorithmic_bytes_per_step"]
        config["offload_link_bytes_per_step"] = leg["offload_link_bytes_per_step"]
        line = {
            "metric": METRIC, "value": leg["value"], "unit": "params/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": leg["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": config,
            "roofline": leg["roofline"], "gather": None, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": leg["gpu_launches"], "clocks": leg["clocks"],
        }
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
