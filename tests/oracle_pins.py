"""Checks that pin the CPU oracle to something other than itself.

Each ``check_*`` function raises AssertionError when the oracle disagrees
with what the pages print, with a closed form, with a library routine or
with a brute-force restatement.  ``test_oracle_pins.py`` runs them as
tests; ``test_oracle_mutations.py`` plants plausible mistakes in the oracle
and shows that at least one of them fails.
"""

from __future__ import annotations

import math
import os
import struct
from decimal import ROUND_HALF_UP, Decimal

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------------------
# helpers
# --------------------------------------------------------------------------

def tiny_inputs(dtype="fp16", n=8, W=4, steps=5, theta_sigma=1.0, grad_sigma=0.1, seed=1):
    """Seeded inputs for small cases: theta0 (fp32, n) and per-step per-rank
    16-bit gradients as NumPy (float16, or uint16 bits for bf16)."""
    from workloads import FP16, TORCH_DTYPE, to_numpy16
    g0 = torch.Generator().manual_seed(0)
    theta0 = (torch.randn(n, generator=g0) * theta_sigma).numpy().astype(np.float32)
    g = torch.Generator().manual_seed(seed)
    grads = []
    for _t in range(steps):
        per = []
        for _r in range(W):
            x = (torch.randn(n, generator=g) * grad_sigma).to(TORCH_DTYPE[dtype or FP16])
            per.append(to_numpy16(x))
        grads.append(per)
    return theta0, grads


def placed(z, grads_real, layout):
    """Per-step per-rank gradients placed into the padded layout."""
    return [[z.place(g, layout) for g in per] for per in grads_real]


def f32(x: float) -> float:
    return struct.unpack("<f", struct.pack("<f", x))[0]


def f16_bits_scalar(x: float) -> int:
    return struct.unpack("<H", struct.pack("<e", x))[0]


def bf16_bits_scalar(x: float) -> int:
    """Round-to-nearest-even to bf16 written as the comparison of the
    dropped half with one half-ulp (a different formulation from the
    oracle's add-and-truncate)."""
    b = struct.unpack("<I", struct.pack("<f", x))[0]
    hi, lo = b >> 16, b & 0xFFFF
    if lo > 0x8000 or (lo == 0x8000 and (hi & 1) == 1):
        hi += 1
    return hi & 0xFFFF


def decode_scalar(v, dtype) -> float:
    if dtype == "fp16":
        return float(np.float16(v))
    return struct.unpack("<f", struct.pack("<I", int(v) << 16))[0]


# --------------------------------------------------------------------------
# accounting: the numbers the pages print
# --------------------------------------------------------------------------

def load_accounting_pins():
    rows = []
    with open(os.path.join(GOLDEN, "accounting_pins.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            pid, src, qty, scheme, psi, N, printed, unit, exact = [c.strip() for c in line.split("|")]
            rows.append(dict(id=pid, src=src, qty=qty, scheme=int(scheme), psi=int(psi), N=int(N),
                             printed=printed, unit=unit, exact=float(exact) if "." in exact else int(exact)))
    return rows


def _decimals(s: str) -> int:
    return len(s.split(".")[1]) if "." in s else 0


def check_accounting(z):
    rows = load_accounting_pins()
    assert len(rows) >= 30
    for row in rows:
        s, psi, N, qty = row["scheme"], row["psi"], row["N"], row["qty"]
        if qty == "resident":
            got = z.bytes_per_rank(s, psi, N)
        elif qty == "bytes_pp":
            got = z.lab_bytes_per_param(s, N)
        elif qty == "lab_peak_pp":
            got = z.lab_peak_bytes_per_param(s, N)
        elif qty == "comm_elems_collective":
            got = z.ring_bytes_per_rank(N, z.shard_size(psi, N), elem_bytes=1)
        elif qty == "comm_bytes_step":
            got = z.comm_bytes_closed_form(s, psi, N)
        elif qty == "paper_volume":
            got = z.comm_volume_paper(s, psi)
        else:
            raise AssertionError(qty)
        if isinstance(row["exact"], int):
            assert got == row["exact"], (row["id"], got, row["exact"])
        else:
            assert abs(got - row["exact"]) < 1e-12, (row["id"], got, row["exact"])
        # the pages round half up (41.25 GB prints as 41.3): compare in exact decimal arithmetic
        scale = {"B": 1, "GB": 10 ** 9, "elements": 1, "1e9 elements": 10 ** 9}[row["unit"]]
        q = Decimal(1).scaleb(-_decimals(row["printed"]))
        shown = (Decimal(repr(got)) / Decimal(scale)).quantize(q, rounding=ROUND_HALF_UP)
        assert shown == Decimal(row["printed"]), (row["id"], got, row["printed"])


def check_padded_state_bytes(z):
    """``ZeroAdam.state_bytes`` printed by zero_check ("ZeRO and FSDP"):
    19,210 parameters on 4 ranks hold 57,636 bytes of fp32 master + m + v
    per rank (ceil padding), against 230,520 unsharded."""
    n, W = 64 * 256 + 256 + 256 * 10 + 10, 4
    assert n == 19210
    S = z.shard_size(n, W)
    assert z.B_OPT * S == 57636
    assert z.B_OPT * n == 230520
    # the same figure from a live ZeRO-2 oracle's own arrays
    o = z.ZeRO2(W, np.zeros(n, np.float32), "fp16")
    assert sum(a.nbytes for a in (o.master[1], o.m[1], o.v[1])) == 57636


def check_traffic_from_events(z):
    """Traffic counted from the collectives each scheme ran equals the
    closed forms: 2(W-1)/W and 3(W-1)/W of 2 n_pad bytes per step."""
    for n, W in ((8, 4), (37, 4), (100, 8), (5, 8)):
        theta0, grads = tiny_inputs(n=n, W=W, steps=2)
        for scheme in (z.DP, z.ZERO1, z.ZERO2, z.ZERO3):
            units = [n] if scheme != z.ZERO3 else None
            o = z.make_scheme(scheme, W, theta0, "fp16", units)
            for per in placed(z, grads, o.layout):
                o.step(per, 1e-2, 0.9, 0.999, 1e-8)
            want = 2 * z.comm_bytes_closed_form(scheme, n, W)
            assert o.comm_bytes() == want, (scheme, n, W, o.comm_bytes(), want)
    # ZeRO-3 over several units: three collectives of every unit per step
    n_units = [13, 24, 3]
    theta0, grads = tiny_inputs(n=sum(n_units), W=4, steps=3)
    o = z.ZeRO3(4, theta0, "fp16", n_units)
    for per in placed(z, grads, o.layout):
        o.step(per, 1e-2, 0.9, 0.999, 1e-8)
    per_step = sum(3 * (4 - 1) * 2 * s for s in o.layout.S)
    assert o.comm_bytes() == 3 * per_step
    # ratio to data parallel is 3/2 exactly when nothing is padded
    assert z.comm_bytes_closed_form(z.ZERO3, 1024, 8) * 2 == z.comm_bytes_closed_form(z.DP, 1024, 8) * 3


def check_layer_unit_traffic(z):
    """Traffic of the 24-unit ZeRO-3 workload (24 x 50,331,648 parameters,
    8 ranks): 3 (N-1)/N 2 Psi = 6,341,787,648 bytes per step, and
    2 (N-1)/N 2 Psi = 4,227,858,432 for a schedule that kept the gathered copy."""
    L = z.Layout(8, [50_331_648] * 24)
    per_coll = sum(z.ring_bytes_per_rank(8, s) for s in L.S)
    assert 3 * per_coll == 6_341_787_648
    assert 2 * per_coll == 4_227_858_432
    assert z.comm_bytes_closed_form(z.ZERO3, 24 * 50_331_648, 8) == 6_341_787_648


# --------------------------------------------------------------------------
# arithmetic
# --------------------------------------------------------------------------

def _run(z, scheme, W, theta0, grads_real, dtype, units=None, hp=(1e-2, 0.9, 0.999, 1e-8)):
    o = z.make_scheme(scheme, W, theta0, dtype, units)
    states = []
    for per in placed(z, grads_real, o.layout):
        o.step(per, *hp)
        idx = o.layout.real_index()
        states.append((o.full_master()[idx].view(np.uint32).copy(), o.full_m()[idx].view(np.uint32).copy(),
                       o.full_v()[idx].view(np.uint32).copy(), o.working_copy()[idx].copy()))
    return o, states


def check_scheme_invariance(z):
    """Data parallel, ZeRO-1, ZeRO-2 and ZeRO-3 give bit-identical master,
    m, v and 16-bit copies at every step, equal to one unsharded replica
    ("The four schemes": the same step for every scheme; "ZeRO, annotated"
    section 2)."""
    cases = [(8, 4, None, "fp16"), (8, 4, None, "bf16"), (37, 4, [13, 24], "fp16"),
             (37, 4, [13, 24], "bf16"), (61, 8, [5, 40, 16], "bf16")]
    for n, W, units, dtype in cases:
        theta0, grads = tiny_inputs(dtype, n=n, W=W, steps=5)
        runs = [_run(z, s, W, theta0, grads, dtype, units)[1] for s in (z.DP, z.ZERO1, z.ZERO2, z.ZERO3)]
        ref = z.SingleReplica(theta0, dtype)
        for t, per in enumerate(grads):
            ref.step(per, 1e-2, 0.9, 0.999, 1e-8)
            want = (ref.master.view(np.uint32), ref.m.view(np.uint32), ref.v.view(np.uint32), ref.working_copy())
            for run in runs:
                for a, b in zip(run[t], want):
                    assert np.array_equal(a, b), (n, W, units, dtype, t)


def check_first_step(z):
    """At t = 1 the bias corrections cancel: m_hat = g and v_hat = g^2, so
    each parameter moves by -lr g / (|g| + eps), i.e. by lr sign(g) up to
    lr eps / (|g| + eps), and not at all where g = 0."""
    rng = np.random.default_rng(7)
    for dtype in ("fp16", "bf16"):
        n, W, lr, eps = 4096, 8, 1e-3, 1e-8
        theta0 = rng.normal(0, 0.02, n).astype(np.float32)
        scales = np.array([1e-3, 1e-6, 1e-8, 3e-9])[rng.integers(0, 4, n)]
        grads = []
        for _w in range(W):
            g = rng.normal(0, 1, n) * scales
            g[rng.random(n) < 0.05] = 0.0
            if dtype == "fp16":
                grads.append(g.astype(np.float16))
            else:
                grads.append(z.round_fp32_to_bf16_bits(g.astype(np.float32)))
        gbar = np.zeros(n)
        for w in range(W):
            gbar += z.decode16(grads[w], dtype)
        gbar /= W
        o = z.SingleReplica(theta0, dtype)
        o.step(grads, lr, 0.9, 0.999, eps)
        d = o.master.astype(np.float64) - theta0.astype(np.float64)
        ulp = np.spacing(np.abs(o.master)).astype(np.float64)
        bound = lr * eps / (np.abs(gbar) + eps) + ulp
        assert np.all(np.abs(d + lr * np.sign(gbar)) <= bound), dtype
        assert np.all(d[gbar == 0] == 0)
        big = np.abs(gbar) > 1e-4
        assert np.all(np.abs(np.abs(d[big]) - lr) < 1e-3 * lr)


def check_vs_torch_adam(z):
    """The textbook special case: one replica's update equals
    ``torch.optim.Adam`` (single-tensor path, fp32) on the mean gradient,
    as "ZeRO and FSDP"'s zero_check compares against it."""
    for W in (1, 4):
        theta0, grads = tiny_inputs("fp16", n=257, W=W, steps=10, theta_sigma=0.5, grad_sigma=0.01)
        for (lr, b1, b2, eps) in ((1e-2, 0.9, 0.999, 1e-8), (3e-4, 0.8, 0.95, 1e-6)):
            o = z.SingleReplica(theta0, "fp16")
            p = torch.nn.Parameter(torch.from_numpy(theta0.copy()))
            opt = torch.optim.Adam([p], lr=lr, betas=(b1, b2), eps=eps, foreach=False, fused=False)
            for per in grads:
                o.step(per, lr, b1, b2, eps)
                mean = np.mean([np.asarray(g, np.float64) for g in per], axis=0)
                p.grad = torch.from_numpy(mean.astype(np.float32))
                opt.step()
            ref = p.detach().numpy().astype(np.float64)
            err = np.abs(o.master.astype(np.float64) - ref)
            assert np.all(err <= 1e-6 * np.abs(ref) + 1e-9), (W, lr, err.max())
            st = opt.state[p]
            # torch keeps m and v in fp32 between its operations, so where m nearly
            # cancels its relative error is large: the floor scales with max |m|
            for mine, theirs in ((o.m, st["exp_avg"].numpy()), (o.v, st["exp_avg_sq"].numpy())):
                assert np.all(np.abs(mine - theirs) <= 1e-6 * np.abs(theirs) + 1e-6 * np.abs(theirs).max())


def check_brute_force(z):
    """Psi = 8 on 4 ranks for 5 steps, parameter by parameter in Python
    floats with no arrays, no shards and no padding: bit-identical to every
    scheme of the oracle."""
    lr, b1, b2, eps = 1e-2, 0.9, 0.999, 1e-8
    for dtype in ("fp16", "bf16"):
        theta0, grads = tiny_inputs(dtype)
        n, W = 8, 4
        th = [float(x) for x in theta0]
        m = [0.0] * n
        v = [0.0] * n
        hist = []
        for t, per in enumerate(grads, start=1):
            for i in range(n):
                acc = 0.0
                for w in range(W):
                    acc += decode_scalar(per[w][i], dtype)
                g = acc / W
                m1 = b1 * m[i] + (1 - b1) * g
                v1 = b2 * v[i] + (1 - b2) * g * g
                th1 = th[i] - lr * (m1 / (1 - b1 ** t)) / (math.sqrt(v1 / (1 - b2 ** t)) + eps)
                m[i], v[i], th[i] = f32(m1), f32(v1), f32(th1)
            cast = f16_bits_scalar if dtype == "fp16" else bf16_bits_scalar
            hist.append(([struct.unpack("<I", struct.pack("<f", x))[0] for x in th], [cast(x) for x in th]))
        for scheme in (z.DP, z.ZERO1, z.ZERO2, z.ZERO3):
            _o, states = _run(z, scheme, W, theta0, grads, dtype, [8] if scheme == z.ZERO3 else None,
                              (lr, b1, b2, eps))
            for (th_bits, p16), st in zip(hist, states):
                assert list(st[0]) == th_bits, (dtype, scheme)
                assert list(st[3]) == p16, (dtype, scheme)


def check_padding_stays_zero(z):
    """With n not a multiple of W the padded entries get a zero gradient,
    so m = v = 0 and the update 0 / (0 + eps) = 0 leaves them exactly 0."""
    n_units = [13, 24, 3, 3]
    theta0, grads = tiny_inputs("bf16", n=sum(n_units), W=4, steps=4)
    for scheme, units in ((z.ZERO1, None), (z.DP, None), (z.ZERO3, n_units)):
        o = z.make_scheme(scheme, 4, theta0, "bf16", units)
        pad = np.setdiff1d(np.arange(o.layout.n_pad), o.layout.real_index())
        assert pad.size > 0
        for per in placed(z, grads, o.layout):
            o.step(per, 1e-2, 0.9, 0.999, 1e-8)
            assert np.all(o.full_master()[pad] == 0) and np.all(o.full_m()[pad] == 0)
            assert np.all(o.full_v()[pad] == 0) and np.all(o.working_copy()[pad] == 0)


def _rounding_patterns(rng, per_exponent=2):
    """Every sign and exponent, two top-mantissa halves each (one of them
    all ones, so the carry into the exponent is exercised), crossed with
    every one of the 65,536 low halves; NaNs removed."""
    hi = []
    for s in (0, 1):
        for e in range(256):
            tops = [0x7F, int(rng.integers(0, 0x7F))][:per_exponent]
            for top in tops:
                hi.append((s << 15) | (e << 7) | top)
    hi = np.array(hi, dtype=np.uint64)
    lo = np.arange(1 << 16, dtype=np.uint64)
    bits = ((hi[:, None] << np.uint64(16)) | lo[None, :]).ravel().astype(np.uint32)
    x = bits.view(np.float32)
    return x[~np.isnan(x)]


def check_rounding(z, per_exponent=2):
    """bf16: the oracle's rounding equals torch's fp32 -> bf16 conversion
    (round to nearest even) on every sign, exponent and low half; fp16: the
    NumPy cast equals torch's.  Plus exact tie cases worked by hand."""
    x = _rounding_patterns(np.random.default_rng(3), per_exponent)
    for lo in range(0, x.size, 1 << 24):
        xs = x[lo:lo + (1 << 24)]
        t = torch.from_numpy(xs)
        want_bf = t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(z.cast16(xs, "bf16"), want_bf)
        want_h = t.to(torch.float16).view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(z.bits16(z.cast16(xs, "fp16"), "fp16"), want_h)
    # ties: 1 + 2^-8 is half way between bf16 1 and 1 + 2^-7: goes to even 1.0;
    # 1 + 3 * 2^-8 is half way between 1 + 2^-7 and 1 + 2^-6: goes to even 1 + 2^-6.
    cases = {1.0 + 2 ** -8: 0x3F80, 1.0 + 3 * 2 ** -8: 0x3F82, -(1.0 + 2 ** -8): 0xBF80,
             1.0 + 2 ** -8 + 2 ** -20: 0x3F81,
             (2 - 2 ** -7) * 2.0 ** 127: 0x7F7F, (2 - 2 ** -8) * 2.0 ** 127: 0x7F80}
    for val, bits in cases.items():
        assert int(z.cast16(np.array([val], np.float32), "bf16")[0]) == bits, val
    hcases = {1.0 + 2 ** -11: 0x3C00, 1.0 + 3 * 2 ** -11: 0x3C02, 65520.0: 0x7C00, 65519.0: 0x7BFF}
    for val, bits in hcases.items():
        assert int(z.bits16(z.cast16(np.array([val], np.float32), "fp16"), "fp16")[0]) == bits, val


def check_zero_check_example(z):
    """The worked check of "ZeRO and FSDP" (zero_check): a 64-256-10 MLP
    (19,210 parameters), a 32-sample batch split over 4 ranks, Adam lr 1e-2
    for 3 steps; the sharded update must stay within 1e-5 of single-process
    ``torch.optim.Adam`` on the full batch.  Model and data are this test's
    own (seeded here), all in fp32 as on that page."""
    torch.manual_seed(11)
    ref = torch.nn.Sequential(torch.nn.Linear(64, 256), torch.nn.GELU(), torch.nn.Linear(256, 10))
    mdl = torch.nn.Sequential(torch.nn.Linear(64, 256), torch.nn.GELU(), torch.nn.Linear(256, 10))
    mdl.load_state_dict(ref.state_dict())
    gen = torch.Generator().manual_seed(5)
    X = torch.randn(32, 64, generator=gen)
    Y = torch.randint(0, 10, (32,), generator=gen)
    loss_fn = torch.nn.CrossEntropyLoss()
    params = list(mdl.parameters())
    n = sum(p.numel() for p in params)
    assert n == 19210
    theta0 = torch.cat([p.detach().flatten() for p in params]).numpy().copy()
    W = 4
    o = z.ZeRO2(W, theta0, "fp16", grad_dtype="fp32")
    opt_ref = torch.optim.Adam(ref.parameters(), lr=1e-2)
    for _ in range(3):
        opt_ref.zero_grad()
        loss_fn(ref(X), Y).backward()
        opt_ref.step()
        theta = o.full_master()[:n]
        off = 0
        with torch.no_grad():
            for p in params:
                p.copy_(torch.from_numpy(theta[off:off + p.numel()]).view_as(p))
                off += p.numel()
        per = []
        for r in range(W):
            mdl.zero_grad()
            sl = slice(r * 32 // W, (r + 1) * 32 // W)
            loss_fn(mdl(X[sl]), Y[sl]).backward()
            per.append(z.place(torch.cat([p.grad.flatten() for p in params]).numpy().copy(), o.layout))
        o.step(per, 1e-2, 0.9, 0.999, 1e-8)
    want = torch.cat([p.detach().flatten() for p in ref.parameters()]).numpy()
    diff = np.abs(o.full_master()[:n] - want).max()
    assert diff < 1e-5, diff


def check_zero3_schedule(z):
    """ZeRO-3 ("ZeRO and FSDP", ZeRO-3 and FSDP; "ZeRO, annotated" section 7):
    every step gathers each unit for the forward pass in unit order and
    releases it, gathers it again for the backward pass in reverse order,
    then reduce-scatters it; the gathered values are the 16-bit cast of the
    current master; at most one unit is live; traffic is three collectives."""
    units = [13, 24, 3, 9]
    W, steps = 4, 3
    theta0, grads = tiny_inputs("bf16", n=sum(units), W=W, steps=steps)
    seen = []
    o = z.ZeRO3(W, theta0, "bf16", units, observer=lambda ph, u, bits: seen.append((ph, u, bits.copy())))
    ref = z.SingleReplica(theta0, "bf16")
    L = o.layout
    idx = L.real_index()
    U = L.U
    for t, per in enumerate(placed(z, grads, L), start=1):
        before = z.place(ref.master, L)
        seen.clear()
        n_ev = len(o.events)
        o.step(per, 1e-2, 0.9, 0.999, 1e-8)
        ref.step([g[idx] for g in per], 1e-2, 0.9, 0.999, 1e-8)
        ev = o.events[n_ev:]
        want_ev = [("all_gather", u, "fwd") for u in range(U)]
        for u in reversed(range(U)):
            want_ev += [("all_gather", u, "bwd"), ("reduce_scatter", u, "bwd")]
        assert ev == want_ev, ev
        assert [(ph, u) for ph, u, _ in seen] == [("fwd", u) for u in range(U)] + \
            [("bwd", u) for u in reversed(range(U))]
        cast_before = z.cast16(before, "bf16")
        for ph, u, bits in seen:
            lo, hi = L.off[u], L.off[u] + L.S[u] * W
            assert np.array_equal(bits, cast_before[lo:hi]), (t, ph, u)
        assert o.live == 0
    assert o.peak_live_elems == max(s * W for s in L.S)
    assert o.comm_bytes() == steps * 3 * sum((W - 1) * 2 * s for s in L.S)


def load_peak_pins():
    rows = []
    with open(os.path.join(GOLDEN, "peak_pins.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            pid, where, psi, N, S, gathered, peak, elems, printed = [x.strip() for x in line.split("|")]
            rows.append(dict(id=pid, where=where, psi=int(psi), N=int(N), S=int(S), gathered=gathered,
                             peak=int(peak), elems=int(elems), printed=printed))
    return rows


def check_peak_bytes(z):
    """Peak bytes of a ZeRO-3 rank against what the pages state: a GPU holds
    at most its own shard and the one layer lent to it ("ZeRO, annotated",
    section 7, stage 3 step by step), and parameters worth 2/64 of the model
    at peak on 64 devices ("One Poem Suffices: ZeRO", section 4.1.4).  The 64-device case runs the oracle's
    ZeRO-3 schedule on the scaled model and takes the gathered values from
    what the schedule held live, not from the row."""
    rows = load_peak_pins()
    assert len(rows) == 3
    for row in rows:
        N, S, psi = row["N"], row["S"], row["psi"]
        if row["gathered"] == "schedule":
            block = psi // 192
            units = [3 * block] * 64
            theta0 = np.linspace(-1.0, 1.0, psi, dtype=np.float32)
            o = z.ZeRO3(N, theta0, "fp16", units)
            assert o.layout.S_total == S, (row["id"], o.layout.S_total)
            grads = [np.full(psi, 0.25 * (r + 1), np.float16) for r in range(N)]
            o.step([z.place(g, o.layout) for g in grads], 1e-3, 0.9, 0.999, 1e-8)
            gathered = o.peak_live_elems
            assert o.live == 0
        else:
            gathered = int(row["gathered"])
        peak = z.peak_bytes_per_rank(z.ZERO3, psi, N, gathered, S=S)
        assert peak == row["peak"], (row["id"], peak, row["peak"])
        # the parameter part of the peak: the rank's own 16-bit shard plus the gathered values
        param_bytes = peak - (z.bytes_per_rank(z.ZERO3, psi, N, S) - z.B_P16 * S)
        assert param_bytes == z.B_P16 * row["elems"], (row["id"], param_bytes)
        if row["printed"].startswith("2/64"):
            assert 64 * row["elems"] == 2 * psi, row["id"]
        else:                                  # the rank's shard and one lent layer of one shard
            assert row["elems"] == 2 * S and gathered == S, row["id"]
        # the other schemes gather nothing: their peak is what they hold
        for scheme in (z.DP, z.ZERO1, z.ZERO2):
            assert z.peak_bytes_per_rank(scheme, psi, N, gathered, S=S) == z.bytes_per_rank(scheme, psi, N, S)


ALL_CHECKS = [
    check_accounting, check_padded_state_bytes, check_traffic_from_events, check_layer_unit_traffic,
    check_scheme_invariance, check_first_step, check_vs_torch_adam, check_brute_force,
    check_padding_stays_zero, check_rounding, check_zero_check_example, check_zero3_schedule,
    check_peak_bytes,
]
