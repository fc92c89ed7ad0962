"""The C ABI without a GPU: the library loads, exports every declared symbol,
its accounting and layout equal the oracle's, and every argument check fails
cleanly before any CUDA call."""

import ctypes
import os
import re

import numpy as np
import pytest

import zero_sharded_mixed_step_gb300 as zs
from oracle import zero_oracle as z

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "zero_step.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[a-z_0-9]+\s*\*?\s*(zero_[a-z_0-9]+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(zlib):
    names = declared_functions()
    assert len(names) >= 20, names
    for name in names:
        assert hasattr(zlib, name), name
    assert set(names) == set(zs.SIGNATURES), set(names) ^ set(zs.SIGNATURES)


def test_header_constants_match_binding():
    text = open(HEADER).read()
    consts = dict((k, int(v)) for k, v in re.findall(r"#define\s+(ZERO_[A-Z0-9_]+)\s+(-?\d+)", text))
    for k, v in consts.items():
        assert getattr(zs, k) == v, k


@pytest.mark.parametrize("scheme", [0, 1, 2, 3])
def test_bytes_per_rank_equals_oracle(zlib, scheme):
    for n in (0, 1, 7, 8, 19210, 124_439_808, 1_557_611_200, 7_500_000_000, 1_000_000_000_000):
        for W in (1, 2, 3, 4, 8, 16, 25, 64):
            assert zs.zero_bytes_per_rank(scheme, n, W) == z.bytes_per_rank(scheme, n, W)
            assert zs.zero_comm_bytes_closed_form(scheme, n, W) == z.comm_bytes_closed_form(scheme, n, W)
            for g in (0, 5, 100_663_296):
                assert zs.zero_bytes_per_rank(scheme, n, W, zs.ZERO_PEAK, g) == z.peak_bytes_per_rank(scheme, n, W, g)


def test_accounting_pins_through_the_abi(zlib):
    from tests.oracle_pins import load_accounting_pins
    for row in load_accounting_pins():
        if row["qty"] == "resident":
            assert zs.zero_bytes_per_rank(row["scheme"], row["psi"], row["N"]) == row["exact"], row["id"]
        if row["qty"] == "comm_bytes_step":
            assert zs.zero_comm_bytes_closed_form(row["scheme"], row["psi"], row["N"]) == row["exact"], row["id"]
    assert zs.zero_comm_bytes_closed_form(3, 24 * 50_331_648, 8) == 6_341_787_648


@pytest.mark.parametrize("units,W", [([8], 4), ([37], 4), ([13, 24, 3], 4), ([50_331_648] * 24, 8),
                                     ([1, 0, 5, 17], 8), ([1_557_611_200], 16), ([0], 3)])
def test_layout_equals_oracle(zlib, units, W):
    L = z.Layout(W, list(units))
    off, shard, off16 = zs.zero_layout(W, units)
    assert off == L.off and shard == L.S and off16 == L.off16
    scheme = 3 if len(units) > 1 else 1
    s = zs.zero_buffer_sizes(scheme, W, units)
    assert s["n"] == L.n and s["n_pad"] == L.n_pad and s["units"] == len(units)
    if scheme == 3:
        assert s["shard_store"] == L.S_total and s["unit_buf"] == max(x * W for x in L.S) and s["p16"] == 0
    else:
        assert s["p16"] == L.n_pad and s["shard_store"] == 0


def test_random_layouts_and_accounting_equal_the_oracle(zlib):
    """300 seeded random configurations: unit lists of 1 to 40 units (empty
    ones included) and W from 1 to 64 for the layout; n up to 10^13 for the
    closed-form accounting of every scheme."""
    rng = np.random.default_rng(2024)
    for _ in range(300):
        W = int(rng.integers(1, 65))
        units = [int(x) for x in rng.integers(0, 10_000_000, int(rng.integers(1, 41)))]
        units = [0 if rng.random() < 0.1 else u for u in units]
        L = z.Layout(W, units)
        off, shard, off16 = zs.zero_layout(W, units)
        assert (off, shard, off16) == (L.off, L.S, L.off16), (W, units)
        n = int(rng.integers(0, 10**13))
        gathered = int(rng.integers(0, 10**9))
        for scheme in (0, 1, 2, 3):
            assert zs.zero_bytes_per_rank(scheme, n, W) == z.bytes_per_rank(scheme, n, W), (scheme, n, W)
            assert zs.zero_bytes_per_rank(scheme, n, W, zs.ZERO_PEAK, gathered) == \
                z.peak_bytes_per_rank(scheme, n, W, gathered), (scheme, n, W, gathered)
            assert zs.zero_comm_bytes_closed_form(scheme, n, W) == z.comm_bytes_closed_form(scheme, n, W)


def _err(fn, *args, **kw):
    with pytest.raises(zs.ZeroError) as e:
        fn(*args, **kw)
    return e.value.code


def test_bad_queries(zlib):
    assert _err(zs.zero_buffer_sizes, 4, 8, [10]) == zs.ZERO_E_ARG
    assert _err(zs.zero_buffer_sizes, 1, 0, [10]) == zs.ZERO_E_ARG
    assert _err(zs.zero_buffer_sizes, 1, 65, [10]) == zs.ZERO_E_ARG
    assert _err(zs.zero_buffer_sizes, 1, 8, [10, 10]) == zs.ZERO_E_ARG
    assert _err(zs.zero_buffer_sizes, 3, 8, [10, -1]) == zs.ZERO_E_ARG
    assert _err(zs.zero_buffer_sizes, 3, 8, []) == zs.ZERO_E_ARG
    assert _err(zs.zero_bytes_per_rank, 1, -1, 8) == zs.ZERO_E_ARG
    assert _err(zs.zero_bytes_per_rank, 1, 8, 0) == zs.ZERO_E_ARG
    assert _err(zs.zero_bytes_per_rank, 1, 8, 4, 7) == zs.ZERO_E_ARG
    assert _err(zs.zero_comm_bytes_closed_form, 9, 8, 4) == zs.ZERO_E_ARG
    assert "scheme" in zs.zero_last_error()


# Fake device addresses: zero_init makes no CUDA call, so no GPU is needed.
A = 0x7F0000000000


def fake(k):
    return A + k * (1 << 30)


def make_ctx(scheme=1, W=4, units=(37,), gdt=0, wdt=0):
    n = sum(units)
    if scheme == 3:
        return zs.zero_init(scheme, W, n, list(units), gdt, wdt, fake(1), fake(2), fake(3), None,
                            [fake(10 + r) for r in range(W)], [fake(8), fake(9)])
    return zs.zero_init(scheme, W, n, list(units), gdt, wdt, fake(1), fake(2), fake(3), fake(4))


def test_init_checks(zlib):
    ok = make_ctx()
    zs.zero_destroy(ok)
    assert _err(zs.zero_init, 1, 0, 8, [8], 0, 0, fake(1), fake(2), fake(3), fake(4)) == zs.ZERO_E_ARG
    assert _err(zs.zero_init, 5, 4, 8, [8], 0, 0, fake(1), fake(2), fake(3), fake(4)) == zs.ZERO_E_ARG
    assert _err(zs.zero_init, 1, 4, 8, [8], 2, 0, fake(1), fake(2), fake(3), fake(4)) == zs.ZERO_E_ARG
    assert _err(zs.zero_init, 1, 4, 9, [8], 0, 0, fake(1), fake(2), fake(3), fake(4)) == zs.ZERO_E_ARG
    assert _err(zs.zero_init, 1, 4, 8, [8], 0, 0, None, fake(2), fake(3), fake(4)) == zs.ZERO_E_ARG
    assert _err(zs.zero_init, 1, 4, 8, [8], 0, 0, fake(1) + 4, fake(2), fake(3), fake(4)) == zs.ZERO_E_ALIGN
    assert _err(zs.zero_init, 1, 4, 8, [8], 0, 0, fake(1), fake(2) + 16, fake(3), fake(4)) == zs.ZERO_E_ALIGN
    assert _err(zs.zero_init, 1, 4, 8, [8], 0, 0, fake(1), fake(2), fake(3), fake(4) + 2) == zs.ZERO_E_ALIGN
    assert _err(zs.zero_init, 1, 4, 8, [8], 0, 0, fake(1), fake(2), fake(3), None) == zs.ZERO_E_ARG
    assert _err(zs.zero_init, 1, 4, 8, [4, 4], 0, 0, fake(1), fake(2), fake(3), fake(4)) == zs.ZERO_E_ARG
    # ZeRO-3 keeps no full copy, and needs its shard stores and two unit buffers
    assert _err(zs.zero_init, 3, 2, 8, [8], 0, 0, fake(1), fake(2), fake(3), fake(4),
                [fake(5), fake(6)], [fake(7), fake(8)]) == zs.ZERO_E_ARG
    assert _err(zs.zero_init, 3, 2, 8, [8], 0, 0, fake(1), fake(2), fake(3), None, None, [fake(7), fake(8)]) \
        == zs.ZERO_E_ARG
    assert _err(zs.zero_init, 3, 2, 8, [8], 0, 0, fake(1), fake(2), fake(3), None,
                [fake(5), fake(6) + 8], [fake(7), fake(8)]) == zs.ZERO_E_ALIGN
    assert _err(zs.zero_init, 1, 2, 8, [8], 0, 0, fake(1), fake(2), fake(3), fake(4), [fake(5), fake(6)]) \
        == zs.ZERO_E_ARG
    zs.zero_destroy(None)


def test_step_checks_before_any_launch(zlib):
    c = make_ctx(scheme=2, W=4, units=(37,))
    g = [fake(20 + r) for r in range(4)]
    hp = (1e-3, 0.9, 0.999, 1e-8)
    assert _err(zs.zero_step, c, 1, 4, 37, g, *hp, 1) == zs.ZERO_E_ARG          # scheme differs
    assert _err(zs.zero_step, c, 2, 8, 37, g, *hp, 1) == zs.ZERO_E_ARG          # W differs
    assert _err(zs.zero_step, c, 2, 4, 36, g, *hp, 1) == zs.ZERO_E_ARG          # n differs
    assert _err(zs.zero_step, c, 2, 4, 37, g, *hp, 0) == zs.ZERO_E_STATE        # t starts at 1
    assert _err(zs.zero_step, c, 2, 4, 37, g, *hp, 2) == zs.ZERO_E_STATE        # t must follow
    assert _err(zs.zero_step, c, 2, 4, 37, g, -1.0, 0.9, 0.999, 1e-8, 1) == zs.ZERO_E_ARG
    assert _err(zs.zero_step, c, 2, 4, 37, g, 1e-3, 1.0, 0.999, 1e-8, 1) == zs.ZERO_E_ARG
    assert _err(zs.zero_step, c, 2, 4, 37, g, 1e-3, 0.9, -0.1, 1e-8, 1) == zs.ZERO_E_ARG
    assert _err(zs.zero_step, c, 2, 4, 37, g, 1e-3, 0.9, 0.999, 0.0, 1) == zs.ZERO_E_ARG
    assert _err(zs.zero_step, c, 2, 4, 37, g, float("nan"), 0.9, 0.999, 1e-8, 1) == zs.ZERO_E_ARG
    assert _err(zs.zero_step, c, 2, 4, 37, g[:3] + [None], *hp, 1) == zs.ZERO_E_ARG
    assert _err(zs.zero_step, c, 2, 4, 37, g[:3] + [fake(30) + 2], *hp, 1) == zs.ZERO_E_ALIGN
    # a rank that stopped answering fails the collective before anything launches
    zs.zero_mark_rank(c, 2, False)
    assert _err(zs.zero_step, c, 2, 4, 37, g, *hp, 1) == zs.ZERO_E_RANK
    assert "rank 2" in zs.zero_last_error()
    assert _err(zs.zero_mark_rank, c, 4, False) == zs.ZERO_E_ARG
    assert zs.zero_stat(c, zs.ZERO_STAT_LAUNCHES) == 0
    assert zs.zero_stat(c, zs.ZERO_STAT_T) == 0
    assert zs.zero_comm_bytes_per_rank(c) == 0
    assert _err(zs.zero_stat, c, 99) == zs.ZERO_E_ARG
    assert _err(zs.zero_set_variant, c, 7) == zs.ZERO_E_ARG
    zs.zero_destroy(c)


def test_unit_calls_checks(zlib):
    c = make_ctx(scheme=3, W=4, units=(13, 24, 3))
    g = [fake(20 + r) for r in range(4)]
    assert _err(zs.zero_gather_unit, c, 3, fake(40)) == zs.ZERO_E_ARG          # no unit 3
    assert _err(zs.zero_gather_unit, c, -1, fake(40)) == zs.ZERO_E_ARG
    assert _err(zs.zero_gather_unit, c, 0, fake(40) + 2) == zs.ZERO_E_ALIGN
    assert _err(zs.zero_gather_unit, c, 0, None) == zs.ZERO_E_ARG
    assert _err(zs.zero_release_unit, c, 1) == zs.ZERO_E_STATE                 # not gathered
    assert _err(zs.zero_update_unit, c, 0, g, 1e-3, 0.9, 0.999, 1e-8, 2) == zs.ZERO_E_STATE
    zs.zero_mark_rank(c, 0, False)
    assert _err(zs.zero_gather_unit, c, 0, fake(40)) == zs.ZERO_E_RANK
    assert _err(zs.zero_update_unit, c, 0, g, 1e-3, 0.9, 0.999, 1e-8, 1) == zs.ZERO_E_RANK
    assert zs.zero_stat(c, zs.ZERO_STAT_GATHERS) == 0 and zs.zero_stat(c, zs.ZERO_STAT_LAUNCHES) == 0
    zs.zero_destroy(c)
    d = make_ctx(scheme=1)
    assert _err(zs.zero_gather_unit, d, 0, fake(40)) == zs.ZERO_E_ARG          # not ZeRO-3
    assert _err(zs.zero_update_unit, d, 0, g, 1e-3, 0.9, 0.999, 1e-8, 1) == zs.ZERO_E_ARG
    zs.zero_destroy(d)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(zs, "_lib", None)
    monkeypatch.setattr(zs, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(zs.ZeroLibraryMissing):
        zs.zero_bytes_per_rank(1, 8, 4)


def test_last_error_is_per_thread(zlib):
    import threading
    _err(zs.zero_bytes_per_rank, 9, 8, 4)
    seen = {}

    def other():
        seen["msg"] = zs.zero_last_error()

    th = threading.Thread(target=other)
    th.start()
    th.join()
    assert seen["msg"] == "" and "scheme" in zs.zero_last_error()
    assert isinstance(ctypes.c_int64(zs.zero_comm_bytes_closed_form(0, 8, 4)).value, int)


def test_host_staging_bytes(zlib):
    # two slots x W ranks x round_up((chunk + 8) * 2, 256)
    assert zs.zero_host_staging_bytes(1, 8, [10_000_000], 1 << 20) == 2 * 8 * (((1 << 20) + 8) * 2 + 255) // 256 * 256
    assert zs.zero_host_staging_bytes(1, 4, [100], 0) == 2 * 4 * (((1 << 24) + 8) * 2 + 255) // 256 * 256
    assert zs.zero_host_staging_bytes(2, 8, [100], 13) == 2 * 8 * 256       # chunk rounds up to 16 elements
    # the default chunk: about 24 per step, in multiples of 2^20, between 2^24 and 2^26
    def slots(W, chunk):
        return 2 * W * (((chunk + 8) * 2 + 255) // 256 * 256)
    assert zs.zero_host_staging_bytes(2, 8, [124_439_808], 0) == slots(8, 1 << 24)
    assert zs.zero_host_staging_bytes(1, 16, [1_557_611_200], 0) == slots(16, 62 << 20)   # 64,900,467 rounded up
    assert zs.zero_host_staging_bytes(1, 1, [10**10], 0) == slots(1, 1 << 26)
    units = [50_331_648] * 24
    assert zs.zero_host_staging_bytes(3, 8, units, 0) == 2 * 8 * ((50_331_648 + 8) * 2 + 255) // 256 * 256
    assert _err(zs.zero_host_staging_bytes, 1, 8, [10, 10], 0) == zs.ZERO_E_ARG
    assert _err(zs.zero_host_staging_bytes, 1, 8, [10], -1) == zs.ZERO_E_ARG


def test_step_host_checks_before_any_launch(zlib):
    c = make_ctx(scheme=1, W=4, units=(1000,))
    need = zs.zero_host_staging_bytes(1, 4, [1000], 256)
    hg = [fake(50 + r) for r in range(4)]
    hp = (1e-3, 0.9, 0.999, 1e-8)
    st = fake(60)
    assert _err(zs.zero_step_host, c, 1, 4, 1000, hg, None, st, need - 1, 256, *hp, 1) == zs.ZERO_E_ARG
    assert _err(zs.zero_step_host, c, 1, 4, 1000, hg, None, st + 16, need, 256, *hp, 1) == zs.ZERO_E_ALIGN
    assert _err(zs.zero_step_host, c, 1, 4, 1000, hg, None, None, need, 256, *hp, 1) == zs.ZERO_E_ARG
    assert _err(zs.zero_step_host, c, 1, 4, 1000, hg[:3] + [None], None, st, need, 256, *hp, 1) == zs.ZERO_E_ARG
    assert _err(zs.zero_step_host, c, 2, 4, 1000, hg, None, st, need, 256, *hp, 1) == zs.ZERO_E_ARG
    assert _err(zs.zero_step_host, c, 1, 4, 1000, hg, None, st, need, 256, *hp, 2) == zs.ZERO_E_STATE
    assert _err(zs.zero_step_host, c, 1, 4, 1000, hg, None, st, need, -5, *hp, 1) == zs.ZERO_E_ARG
    zs.zero_mark_rank(c, 1, False)
    assert _err(zs.zero_step_host, c, 1, 4, 1000, hg, None, st, need, 256, *hp, 1) == zs.ZERO_E_RANK
    assert zs.zero_stat(c, zs.ZERO_STAT_LAUNCHES) == 0 and zs.zero_stat(c, zs.ZERO_STAT_T) == 0
    zs.zero_destroy(c)


def test_step_bucket_checks_before_any_launch(zlib):
    c = make_ctx(scheme=2, W=4, units=(1000,))
    b = [fake(70 + r) for r in range(4)]
    hp = (1e-3, 0.9, 0.999, 1e-8)
    assert _err(zs.zero_step_bucket, c, 4, 16, b, *hp, 1) == zs.ZERO_E_ALIGN          # lo not a multiple of 8
    assert _err(zs.zero_step_bucket, c, 0, 0, b, *hp, 1) == zs.ZERO_E_ARG             # empty
    assert _err(zs.zero_step_bucket, c, 992, 16, b, *hp, 1) == zs.ZERO_E_ARG          # past n_pad
    assert _err(zs.zero_step_bucket, c, 0, 16, b[:3] + [None], *hp, 1) == zs.ZERO_E_ARG
    assert _err(zs.zero_step_bucket, c, 0, 16, b[:3] + [fake(80) + 2], *hp, 1) == zs.ZERO_E_ALIGN
    assert _err(zs.zero_step_bucket, c, 0, 16, b, *hp, 2) == zs.ZERO_E_STATE          # t must start the step
    assert _err(zs.zero_step_bucket, c, 0, 16, b, *hp, 0) == zs.ZERO_E_STATE
    assert zs.zero_stat(c, zs.ZERO_STAT_LAUNCHES) == 0
    zs.zero_destroy(c)
    d = make_ctx(scheme=3, W=4, units=(13, 24, 3))
    assert _err(zs.zero_step_bucket, d, 0, 8, b, *hp, 1) == zs.ZERO_E_ARG             # ZeRO-3 goes unit by unit
    zs.zero_destroy(d)


def test_dp_replicas_checks_before_any_launch(zlib):
    """The replica step and the replica check refuse bad arguments before
    touching the GPU (fake addresses, no device needed)."""
    W, n = 3, 1001
    g = [fake(100 + r) for r in range(W)]
    th, m, v, p = ([fake(200 + 10 * k + r) for r in range(W)] for k in range(4))
    hp = (1e-3, 0.9, 0.999, 1e-8)
    step = zs.zero_step_dp_replicas
    assert _err(step, 0, n, 0, 0, g, th, m, v, p, *hp, 1) == zs.ZERO_E_ARG
    assert _err(step, 65, n, 0, 0, g, th, m, v, p, *hp, 1) == zs.ZERO_E_ARG
    assert _err(step, W, -1, 0, 0, g, th, m, v, p, *hp, 1) == zs.ZERO_E_ARG
    assert _err(step, W, n, 2, 0, g, th, m, v, p, *hp, 1) == zs.ZERO_E_ARG
    assert _err(step, W, n, 0, 0, g, th, m, v, p, *hp, 0) == zs.ZERO_E_STATE
    assert _err(step, W, n, 0, 0, g, th, m, v, p, 1e-3, 1.0, 0.999, 1e-8, 1) == zs.ZERO_E_ARG
    assert _err(step, W, n, 0, 0, g, th, m, v, p, 1e-3, 0.9, 0.999, 0.0, 1) == zs.ZERO_E_ARG
    assert _err(step, W, n, 0, 0, g, None, m, v, p, *hp, 1) == zs.ZERO_E_ARG
    assert _err(step, W, n, 0, 0, g, th[:2] + [None], m, v, p, *hp, 1) == zs.ZERO_E_ARG
    assert _err(step, W, n, 0, 0, g, th, m[:1] + [m[1] + 16] + m[2:], v, p, *hp, 1) == zs.ZERO_E_ALIGN
    assert _err(step, W, n, 0, 0, g, th, m, v, p[:2] + [p[2] + 2], *hp, 1) == zs.ZERO_E_ALIGN
    assert _err(step, W, n, 0, 0, [g[0] + 8] + g[1:], th, m, v, p, *hp, 1) == zs.ZERO_E_ALIGN
    # replicas that share memory would be updated twice
    assert _err(step, W, n, 0, 0, g, th, m, [v[0], v[0], v[2]], p, *hp, 1) == zs.ZERO_E_ARG
    assert "overlap" in zs.zero_last_error()
    assert _err(step, W, n, 0, 0, g, th, m, v, [p[0], th[1] + 1024, p[2]], *hp, 1) == zs.ZERO_E_ARG
    # a gradient vector inside a replica buffer
    assert _err(step, W, n, 0, 0, [g[0], th[2] + 32, g[2]], th, m, v, p, *hp, 1) == zs.ZERO_E_ARG
    assert "gradient" in zs.zero_last_error()
    check = zs.zero_dp_replicas_mismatches
    assert _err(check, 0, n, th, m, v, p, fake(300)) == zs.ZERO_E_ARG
    assert _err(check, W, n, th, m, v, p, None) == zs.ZERO_E_ARG
    assert _err(check, W, n, th, m, v, p, fake(300) + 4) == zs.ZERO_E_ALIGN
    assert _err(check, W, n, th, m, None, p, fake(300)) == zs.ZERO_E_ARG
    assert _err(check, W, n, th, m, v, p[:2] + [p[2] + 1], fake(300)) == zs.ZERO_E_ALIGN


def test_host_alloc_checks(zlib):
    assert _err(zs.zero_host_alloc, 0) == zs.ZERO_E_ARG
    assert _err(zs.zero_host_alloc, -5) == zs.ZERO_E_ARG
    assert _err(zs.zero_host_free, 0x1000) == zs.ZERO_E_ARG
    assert "zero_host_alloc" in zs.zero_last_error()
    zs.zero_host_free(None)


def test_graph_mode_checks(zlib):
    """Graph capture is for ZeRO-3 contexts on a created stream only."""
    z1 = make_ctx(scheme=1)
    assert _err(zs.zero_set_graph, z1, True) == zs.ZERO_E_ARG
    zs.zero_set_graph(z1, False)                 # turning it off is always fine
    z3 = make_ctx(scheme=3, W=4, units=(37, 5))
    assert _err(zs.zero_set_graph, z3, True) == zs.ZERO_E_ARG   # no stream: the legacy default stream
    assert "legacy" in zs.zero_last_error()


def declared_prototypes():
    """name -> (return type, [parameter types]) for every function the header declares."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    text = re.sub(r"#.*", "", text)
    protos = {}
    for ret, name, params in re.findall(r"((?:const\s+)?[a-z_0-9]+\s*\**)\s*(zero_[a-z_0-9]+)\s*\(([^;{]*?)\)\s*;", text,
                                        flags=re.S):
        params = " ".join(params.split())
        plist = [] if params in ("", "void") else [p.strip() for p in params.split(",")]
        protos[name] = (" ".join(ret.split()), plist)
    return protos


def _ctype_of(decl: str):
    """The ctypes type a C parameter or return declaration maps to in the binding."""
    m = re.match(r"^(.*?[\s*])([A-Za-z_][A-Za-z_0-9]*)$", decl.strip())   # drop the parameter's name
    base = (m.group(1) if m else decl).replace("const", "").replace(" ", "")
    table = {"int": ctypes.c_int, "int64_t": ctypes.c_int64, "double": ctypes.c_double,
             "int64_t*": ctypes.POINTER(ctypes.c_int64), "double*": ctypes.POINTER(ctypes.c_double),
             "int*": ctypes.POINTER(ctypes.c_int), "char*": ctypes.c_char_p,
             "zero_unit_hook": zs.HOOK, "void**": zs._PP, "float**": zs._PP,
             "zero_ctx**": ctypes.POINTER(ctypes.c_void_p), "zero_offload**": ctypes.POINTER(ctypes.c_void_p)}
    if base in table:
        return table[base]
    if base.endswith("*"):
        return ctypes.c_void_p
    raise AssertionError(f"no mapping for {decl!r}")


def test_binding_signatures_match_the_header():
    """Every wrapper's ctypes argument and return types follow the header's
    prototype, argument by argument (a mismatch would corrupt calls silently)."""
    protos = declared_prototypes()
    assert set(protos) == set(zs.SIGNATURES)
    for name, (ret, params) in protos.items():
        res, args = zs.SIGNATURES[name]
        assert len(args) == len(params), (name, params, args)
        for p, a in zip(params, args):
            # a pointer may also be passed as a raw address (device memory, tensors' data_ptr())
            raw_ok = "*" in p and a is ctypes.c_void_p
            assert raw_ok or _ctype_of(p) == a, (name, p, a)
        assert _ctype_of(ret + " x" if not ret.endswith("*") else ret) == res, (name, ret, res)


def test_strided_tensors_are_refused_by_the_binding(zlib):
    """The library reads dense vectors from a base address: a strided view
    would be read as the wrong elements, so the binding refuses it."""
    import torch
    x = torch.zeros(64)
    with pytest.raises(ValueError):
        zs.zero_adam_host(32, x[::2], x[:32], x[:32], x[:32], torch.zeros(32, dtype=torch.int16), 0,
                          1e-3, 0.9, 0.95, 1e-8, 1)
    assert zs._ptr(x[8:16]) == x.data_ptr() + 32       # a contiguous slice passes with its own address


def test_static_z3_step_checks_before_any_launch(zlib):
    """The ZeRO-3 step without allocations refuses units beyond its fixed
    gather array, before any CUDA call and before any arithmetic on the
    size that could overflow; and refuses the usual bad arguments."""
    hp = (1e-3, 0.9, 0.95, 1e-8)

    def call(W, units, th=None, s16=None, g=None, t=1):
        th = fake(1) if th is None else th
        s16 = [fake(10 + r) for r in range(W)] if s16 is None else s16
        g = [fake(40 + r) for r in range(W)] if g is None else g
        return _err(zs.zero_step_z3_static, W, units, 1, 1, th, fake(2), fake(3), s16, g, *hp, t)

    for W, units in ((1, [8_388_609]), (3, [8_388_607]), (1, [2**63 - 1]), (5, [2**63 - 2]), (2, [17, 2**62]),
                     (7, [8_388_605])):
        assert call(W, units) == zs.ZERO_E_ARG, (W, units)
        assert "static gather buffer" in zs.zero_last_error()
    assert call(0, [10]) == zs.ZERO_E_ARG
    assert call(65, [10]) == zs.ZERO_E_ARG
    assert call(2, [-1]) == zs.ZERO_E_ARG
    assert call(2, [10], t=0) == zs.ZERO_E_STATE
    assert call(2, [10], th=fake(1) + 16) == zs.ZERO_E_ALIGN
    assert call(2, [10], s16=[fake(10), fake(11) + 2]) == zs.ZERO_E_ALIGN
    assert call(2, [10], g=[fake(40), None]) == zs.ZERO_E_ARG
