"""bench.py's host logic without a GPU: the replicas path's max over ranks
and whole-job value on world_size-2 gloo ranks, the reference arm's rank
handling, and the workload arithmetic."""

import io
import json
import os
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.max_over_ranks(10.0 + rank)            # the slowest replica sets the time
    out[rank] = (ms, bench.whole_job_value(world, 1000, 5, ms))
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_take_the_slowest_rank_over_gloo():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = 29500 + os.getpid() % 2000
        procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert out[0] == out[1]
        ms, value = out[0]
        assert ms == 11.0
        assert value == pytest.approx(2 * 1000 * 5 / 0.011)


def test_single_process_max_is_identity():
    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.whole_job_value(1, 10, 2, 1000.0) == 20.0


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"]) == 0
    assert buf.getvalue() == ""


def test_workload_bytes():
    wl = bench.workload("zero3_24x50m_w8")
    fused, gathers = bench.algorithmic_bytes(wl)
    assert fused == 42 * 24 * 50_331_648 and gathers == 8 * 24 * 50_331_648
    small = bench.workload("zero3_24x50m_w8", units=3)
    assert small.n == 3 * 50_331_648 and bench.layout_sizes(small)[1] == [50_331_648] * 3
    xl = bench.workload("gpt2_1p5b_w16_zero1")
    assert bench.algorithmic_bytes(xl) == (58 * 1_557_611_200, 0)


def test_reference_arm_prints_the_contract_line(monkeypatch):
    monkeypatch.delenv("RANK", raising=False)
    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.main(["--impl", "reference", "--steps", "2", "--warmup", "1", "--reference-seconds", "1",
                           "--workload", "gpt2_small_124m_w8_zero2"]) == 0
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "params/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["metric"] == bench.METRIC


def test_oracle_host_memory_check_refuses_what_does_not_fit(monkeypatch):
    """The CPU oracle's host-memory check: a sample that fits passes, one that
    needs more than the host has fails with a message before allocating."""
    import bench
    import workloads as wk
    wl = wk.GPT2_XL
    bench.check_host_memory(bench.oracle_bytes(wl, 1 << 16), "small sample")
    with pytest.raises(MemoryError, match="host memory"):
        bench.check_host_memory(bench.oracle_bytes(wl, wl.n) * 1000, "the whole GPT-2-1.5B vector, 1000 times")
    # literal DP replicas cost the oracle W copies of the state
    assert bench.oracle_bytes(wk.GPT2_SMALL_DP_REPLICAS, 1000) > bench.oracle_bytes(wk.GPT2_SMALL, 1000)


def test_settled_host_block_retries_split_blocks(monkeypatch):
    """A block whose huge pages were split by the probe is kept aside while a
    new one is taken (at most three); the one with the most huge pages (then
    the fastest) is used and the rest come back as spares, still open, for
    the caller to free after its timed steps."""
    import torch
    import zero_sharded_mixed_step_gb300 as zs

    made, closed = [], []

    class FakeBlock:
        def __init__(self, numel, dtype):
            self.tensor = torch.zeros(numel, dtype=dtype)
            self.index = len(made)
            made.append(self)

        def close(self):
            closed.append(self.index)

    fractions = {0: 0.9, 1: 0.96, 2: 1.0}
    rates = {0: 40.0, 1: 120.0, 2: 211.0}
    monkeypatch.setattr(zs, "HostBuffer", FakeBlock)
    monkeypatch.setattr(bench, "huge_page_fraction", lambda bufs: fractions[bufs[0].index])
    probes = []

    def probe_of(views):
        probes.append(views)
        return {"h2d_gbs": rates[len(probes) - 1]}

    block, views, probe, spares = bench.settled_host_block(64, lambda t: ("views", t.numel()), probe_of)
    assert block.index == 2 and probe["host_block_attempts"] == 3 and probe["h2d_gbs"] == 211.0
    assert sorted(b.index for b in spares) == [0, 1] and closed == []
    # a block that keeps its huge pages is taken at once
    made.clear(), closed.clear(), probes.clear()
    fractions[0] = 1.0
    block, views, probe, spares = bench.settled_host_block(64, lambda t: ("views", t.numel()), probe_of)
    assert block.index == 0 and probe["host_block_attempts"] == 1 and spares == [] and closed == []
    # a block whose pages began to split loses to an intact one, however fast its probe
    made.clear(), closed.clear(), probes.clear()
    fractions.update({0: 0.96, 1: 1.0})
    rates.update({0: 211.5, 1: 211.4})
    block, views, probe, spares = bench.settled_host_block(64, lambda t: ("views", t.numel()), probe_of)
    assert block.index == 1 and probe["host_block_attempts"] == 2 and [b.index for b in spares] == [0]


def test_after_e2e_reports_the_link_and_pages_once_more(monkeypatch):
    """The second probe after the timed end-to-end steps carries the link
    rates and the huge-page share at that point."""
    monkeypatch.setattr(bench, "huge_page_fraction", lambda bufs: 0.5)
    seen = []

    def probe_of(views):
        seen.append(views)
        return {"h2d_gbs": 52.0, "d2h_gbs": 15.0, "floor_ms": 1.0, "note": "x"}

    after = bench.after_e2e(probe_of, ("g", "o"), ["block"])
    assert seen == [("g", "o")]
    assert after == {"h2d_gbs": 52.0, "d2h_gbs": 15.0, "host_huge_page_fraction": 0.5}


def test_settled_host_block_stops_retrying_when_memory_runs_short(monkeypatch):
    """A split block is still used when the host has no room for another one,
    or when taking another one fails."""
    import torch
    import zero_sharded_mixed_step_gb300 as zs

    made = []

    class FakeBlock:
        def __init__(self, numel, dtype):
            if fail_next:
                raise zs.ZeroError(zs.ZERO_E_NOMEM, "zero_host_alloc", "mmap failed")
            self.tensor = torch.zeros(numel, dtype=dtype)
            made.append(self)

        def close(self):
            pass

    monkeypatch.setattr(zs, "HostBuffer", FakeBlock)
    monkeypatch.setattr(bench, "huge_page_fraction", lambda bufs: 0.5)
    probe_of = lambda views: {"h2d_gbs": 100.0}   # noqa: E731
    fail_next = False
    monkeypatch.setattr(bench, "host_mem_available", lambda: 3 * 64)      # less than two more blocks of 128 B
    block, _, probe, spares = bench.settled_host_block(64, lambda t: None, probe_of)
    assert probe["host_block_attempts"] == 1 and spares == [] and len(made) == 1
    made.clear()
    monkeypatch.setattr(bench, "host_mem_available", lambda: None)
    real_init = FakeBlock.__init__

    def init_then_fail(self, numel, dtype):
        nonlocal fail_next
        real_init(self, numel, dtype)
        fail_next = True

    monkeypatch.setattr(FakeBlock, "__init__", init_then_fail)
    block, _, probe, spares = bench.settled_host_block(64, lambda t: None, probe_of)
    assert probe["host_block_attempts"] == 1 and spares == [] and len(made) == 1


def _room_rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), LOCAL_WORLD_SIZE=str(world))
    # rank 1's host reports less memory than two 40 GB blocks need; rank 0's is ample
    bench.host_mem_available = (lambda: 90 * 10**9) if rank == 1 else (lambda: 10**12)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    out[rank] = (bench.host_room_for(40 * 10**9, world), bench.host_room_for(10 * 10**9, world))
    dist.barrier()
    dist.destroy_process_group()


def test_end_to_end_leg_is_skipped_on_every_rank_when_one_host_is_short():
    """The end-to-end leg page-locks a block per process; when one rank's
    host cannot hold a block for every local process, all ranks skip the
    leg (so the collectives inside it stay matched) and say why."""
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = 29500 + (os.getpid() + 977) % 2000
        procs = [ctx.Process(target=_room_rank, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        for r in range(2):
            big, small = out[r]
            assert big is not None and "host memory" in big and "2 process(es)" in big
            assert small is None
