"""CPU oracle for the sharded mixed-precision ZeRO step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
links this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference leg of ``bench.py`` may use it.  It shares no code with
the CUDA library (``zero_sharded_mixed_step_gb300``) and imports nothing
from it.

What it computes, and from where
--------------------------------
The step over a flat parameter vector for W data-parallel ranks simulated
in one process, written the plain and slow way:

* The reduce-scatter is a rank-ordered fp64 sum of the W ranks' 16-bit
  gradients followed by a division by W ("The four schemes", Zero From
  Scratch lab: ``reduce_scatter_mean``; "ZeRO and FSDP", implementing
  ZeRO's Adam from scratch: ``reduce_scatter_tensor`` then ``g /= world``).
* Adam with bias correction on each owned shard, in fp64 from the fp32
  stored master, m and v, each result rounded once to fp32 ("The four
  schemes": ``Base._adam``; "ZeRO and FSDP": ``ZeroAdam.step``).  The step
  counter is 1-based and is advanced before the update.
* The recast of the fp32 master to the 16-bit working copy with
  round-to-nearest-even, gathered into the full vector ("The four schemes":
  the ZeRO-1 step casts after its all-gather).
* For ZeRO-3, the per-unit gather / release / re-gather schedule with the
  backward pass in reverse unit order ("ZeRO and FSDP", section "ZeRO-3 and
  FSDP"; "ZeRO, annotated" section 7, "Stage 3, step by step").
* The integer accounting: resident and peak bytes per rank, and the bytes
  each rank sends per step under ring collectives ("ZeRO, annotated"
  sections 5.1-5.3 and 7; "One Poem Suffices: ZeRO" section 4.1.4 and
  appendix B; "Sharding the States").

Readings taken where the pages leave a step open
------------------------------------------------
* A parameter count that does not divide by W is padded with zeros to
  ``S * W`` with ``S = ceil(n / W)`` ("ZeRO and FSDP": ``ZeroAdam`` pads;
  its printed 57,636 state bytes for 19,210 parameters on 4 ranks is
  ``12 * ceil(19210 / 4)``).  The padded entries see a zero gradient and
  therefore stay exactly zero.
* ZeRO-3 gathers the 16-bit working copy (the pages' prose: the 16-bit
  weights are what stage 3 shards), and each rank refreshes its own 16-bit
  shard from its fp32 master right after its update.  The lab's alternative
  accounting (a gathered fp32 copy) is kept only in ``lab_peak_bytes_per_param``.
* ZeRO-3 units are evenly sharded per unit (each unit padded to a multiple
  of W), FSDP style; the traffic is the same as with owner broadcast.
* Traffic counts bytes sent per rank per collective under the ring
  algorithm: ``(W - 1)`` chunks of the shard, 2 bytes per element.

Every function here is pinned, by the CPU tests, to values the pages print,
closed forms, library routines or brute force; the random draws that feed
it are inputs shared with the CUDA path, not part of the method.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

# Bytes per parameter in each band: 16-bit weight, 16-bit gradient, and the
# fp32 master, first moment and second moment ("The four schemes" band
# constants; "ZeRO, annotated" section 3.1: 2 + 2 + K with K = 12).
B_P16, B_GRAD, B_MASTER, B_M, B_V = 2, 2, 4, 4, 4
B_OPT = B_MASTER + B_M + B_V

DP, ZERO1, ZERO2, ZERO3 = 0, 1, 2, 3
SCHEME_NAMES = {DP: "data parallel", ZERO1: "ZeRO-1", ZERO2: "ZeRO-2", ZERO3: "ZeRO-3"}

# (shard_opt, shard_grad, shard_param) for each scheme ("The four schemes",
# the table of three flags).
SCHEME_FLAGS = {
    DP: (False, False, False),
    ZERO1: (True, False, False),
    ZERO2: (True, True, False),
    ZERO3: (True, True, True),
}

FP16, BF16, FP32 = "fp16", "bf16", "fp32"


# --------------------------------------------------------------------------
# Layout
# --------------------------------------------------------------------------

def shard_size(n: int, W: int) -> int:
    """Elements each rank owns: ceil(n / W) ("ZeRO and FSDP", ``ZeroAdam``)."""
    if W <= 0 or n < 0:
        raise ValueError("need W >= 1 and n >= 0")
    return -(-n // W)


@dataclass
class Layout:
    """Flat padded layout of the parameter vector.

    Units are laid out one after another; unit ``u`` holds ``sizes[u]`` real
    parameters followed by zero padding up to ``S[u] * W``.  Rank ``r`` owns
    ``[off[u] + r * S[u], off[u] + (r + 1) * S[u])`` of every unit.  The
    data-parallel, ZeRO-1 and ZeRO-2 schemes use a single unit.
    """

    W: int
    sizes: list
    S: list = field(default_factory=list)
    off: list = field(default_factory=list)
    off16: list = field(default_factory=list)   # start of unit u inside a rank's 16-bit shard store
    n: int = 0
    n_pad: int = 0
    S_total: int = 0

    def __post_init__(self):
        pos, pos16 = 0, 0
        for sz in self.sizes:
            s = shard_size(sz, self.W)
            self.S.append(s)
            self.off.append(pos)
            self.off16.append(pos16)
            pos += s * self.W
            pos16 += s
        self.n = int(sum(self.sizes))
        self.n_pad = pos
        self.S_total = pos16

    @property
    def U(self) -> int:
        return len(self.sizes)

    def real_index(self) -> np.ndarray:
        """Flat padded index of every real parameter, in parameter order."""
        parts = [np.arange(o, o + sz, dtype=np.int64) for o, sz in zip(self.off, self.sizes)]
        return np.concatenate(parts) if parts else np.zeros(0, dtype=np.int64)


def place(real: np.ndarray, layout: Layout) -> np.ndarray:
    """Put a length-n vector into the padded layout, zeros in the padding."""
    out = np.zeros(layout.n_pad, dtype=real.dtype)
    out[layout.real_index()] = real
    return out


# --------------------------------------------------------------------------
# 16-bit formats
# --------------------------------------------------------------------------

def decode16(x: np.ndarray, dtype: str) -> np.ndarray:
    """16-bit values to fp64.  fp16 arrives as np.float16; bf16 as its raw
    uint16 bit pattern (NumPy has no bf16 type): the top half of an fp32.
    fp32 gradients are accepted too, for the pages' all-fp32 ``zero_check``
    comparison ("ZeRO and FSDP")."""
    if dtype == FP32:
        return np.asarray(x, dtype=np.float32).astype(np.float64)
    if dtype == FP16:
        return np.asarray(x, dtype=np.float16).astype(np.float64)
    if dtype == BF16:
        bits = np.asarray(x, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def round_fp32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 with round-to-nearest-even, on the bit pattern.

    Adding 0x7FFF plus the lowest kept bit and truncating the low 16 bits
    rounds to nearest, and ties go to the even neighbour.  Overflow carries
    into the exponent and gives infinity, as IEEE rounding does.  NaN inputs
    are not expected on this path and are not treated specially.
    """
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    keep_lsb = (u >> np.uint64(16)) & np.uint64(1)
    return ((u + np.uint64(0x7FFF) + keep_lsb) >> np.uint64(16)).astype(np.uint16)


def cast16(x32: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 master to the 16-bit working copy, round-to-nearest-even
    ("The four schemes": ``astype(np.float16)``)."""
    if dtype == FP16:
        with np.errstate(over="ignore"):        # |x| > 65504 rounds to +-inf, as IEEE does
            return np.asarray(x32, dtype=np.float32).astype(np.float16)
    if dtype == BF16:
        return round_fp32_to_bf16_bits(x32)
    raise ValueError(dtype)


def bits16(x: np.ndarray, dtype: str) -> np.ndarray:
    """Raw uint16 pattern of a 16-bit array in either format."""
    if dtype == FP16:
        return np.asarray(x, dtype=np.float16).view(np.uint16)
    return np.asarray(x, dtype=np.uint16)


# --------------------------------------------------------------------------
# The arithmetic of one step
# --------------------------------------------------------------------------

def mean_over_ranks(grads, lo: int, hi: int, dtype: str) -> np.ndarray:
    """Reduce-scatter (mean) of ``[lo, hi)``: add rank 0, rank 1, ... in that
    order in fp64, then divide by W."""
    W = len(grads)
    acc = np.zeros(hi - lo, dtype=np.float64)
    for w in range(W):
        acc = acc + decode16(grads[w][lo:hi], dtype)
    return acc / W


def bias_corrections(beta1: float, beta2: float, t: int):
    """``1 - beta1**t`` and ``1 - beta2**t`` with t counted from 1."""
    if t < 1:
        raise ValueError("the step counter starts at 1")
    return 1.0 - beta1 ** t, 1.0 - beta2 ** t


def adam_update(master, m, v, g, lr, beta1, beta2, eps, t):
    """Adam with bias correction on one shard, in place on fp32 arrays.

    m <- b1 m + (1 - b1) g;  v <- b2 v + (1 - b2) g^2;
    theta <- theta - lr * (m / (1 - b1^t)) / (sqrt(v / (1 - b2^t)) + eps).
    Arithmetic in fp64 from the stored fp32 values; m, v and theta are each
    rounded once to fp32 (round to nearest even).
    """
    bc1, bc2 = bias_corrections(beta1, beta2, t)
    m1 = beta1 * m.astype(np.float64) + (1.0 - beta1) * g
    v1 = beta2 * v.astype(np.float64) + (1.0 - beta2) * g * g
    m_hat = m1 / bc1
    v_hat = v1 / bc2
    th1 = master.astype(np.float64) - lr * m_hat / (np.sqrt(v_hat) + eps)
    m[...] = m1.astype(np.float32)
    v[...] = v1.astype(np.float32)
    master[...] = th1.astype(np.float32)


# --------------------------------------------------------------------------
# Accounting
# --------------------------------------------------------------------------

def bytes_per_rank(scheme: int, n: int, W: int, S: int | None = None) -> int:
    """Bytes of model state a rank holds between steps.

    Each band is held whole, or as the rank's shard of S elements when the
    scheme shards it: 16 n, 4 n + 12 S, 2 n + 14 S, 16 S ("ZeRO, annotated"
    sections 5.1-5.3; "ZeRO and FSDP", the three stages).  S defaults to
    ceil(n / W), the padded shard.
    """
    if S is None:
        S = shard_size(n, W)
    shard_opt, shard_grad, shard_param = SCHEME_FLAGS[scheme]
    p = B_P16 * (S if shard_param else n)
    g = B_GRAD * (S if shard_grad else n)
    o = B_OPT * (S if shard_opt else n)
    return p + g + o


def peak_bytes_per_rank(scheme: int, n: int, W: int, gathered_elems: int = 0,
                        S: int | None = None) -> int:
    """Resident bytes plus the 16-bit copies a ZeRO-3 rank holds gathered at
    its worst moment (``gathered_elems`` elements live at once).  The other
    schemes gather nothing, so their peak is their resident figure."""
    base = bytes_per_rank(scheme, n, W, S)
    return base + (B_P16 * gathered_elems if scheme == ZERO3 else 0)


def lab_bytes_per_param(scheme: int, W: int) -> float:
    """Per-parameter form of ``bytes_per_rank`` (no padding)."""
    shard_opt, shard_grad, shard_param = SCHEME_FLAGS[scheme]
    return (B_P16 / (W if shard_param else 1) + B_GRAD / (W if shard_grad else 1)
            + B_OPT / (W if shard_opt else 1))


def lab_peak_bytes_per_param(scheme: int, W: int) -> float:
    """The lab's peak: its ZeRO-3 holds one gathered fp32 copy of the whole
    vector, 4 more bytes per parameter ("The four schemes", the table of
    resident and peak figures).  Kept only to reproduce that table."""
    return lab_bytes_per_param(scheme, W) + (B_MASTER if scheme == ZERO3 else 0)


def ring_bytes_per_rank(W: int, shard_elems: int, elem_bytes: int = 2) -> int:
    """Bytes one rank sends in one ring reduce-scatter or all-gather: W - 1
    chunks of the shard ("One Poem Suffices: ZeRO", appendix B)."""
    return (W - 1) * shard_elems * elem_bytes


def comm_bytes_closed_form(scheme: int, n: int, W: int, S: int | None = None) -> int:
    """Bytes a rank sends per step: two collectives for data parallel and
    ZeRO-1/2 (all-reduce = reduce-scatter + all-gather), three for ZeRO-3
    (two all-gathers and a reduce-scatter) ("ZeRO and FSDP", the three
    stages; "Sharding the States": (n-1)/n of 4N and of 6N)."""
    if S is None:
        S = shard_size(n, W)
    k = 3 if scheme == ZERO3 else 2
    return k * ring_bytes_per_rank(W, S)


def comm_volume_paper(scheme: int, n: int) -> int:
    """The paper's rounded count in elements: each collective moves Psi
    through a device, so 2 Psi per step for data parallel and ZeRO-1/2 and
    3 Psi for ZeRO-3 ("ZeRO, annotated" section 7)."""
    return (3 if scheme == ZERO3 else 2) * n


# --------------------------------------------------------------------------
# The schemes, with W ranks kept as W separate states
# --------------------------------------------------------------------------

class _Scheme:
    """Common state for the four schemes.  ``theta0`` holds the n real
    parameters (fp32); ``unit_sizes`` splits them into ZeRO-3 units."""

    scheme = None

    def __init__(self, W: int, theta0: np.ndarray, dtype: str, unit_sizes=None,
                 grad_dtype: str | None = None):
        theta0 = np.asarray(theta0, dtype=np.float32)
        n = theta0.size
        if unit_sizes is None or self.scheme != ZERO3:
            unit_sizes = [n]
        if sum(unit_sizes) != n:
            raise ValueError("unit sizes must add up to n")
        self.W, self.dtype, self.t = W, dtype, 0
        self.grad_dtype = grad_dtype or dtype
        self.layout = Layout(W, list(unit_sizes))
        self.events = []           # ("all_reduce" | "reduce_scatter" | "all_gather", unit, phase)
        self.theta0_padded = place(theta0, self.layout)

    # traffic is counted from the collectives that actually ran
    def comm_bytes(self) -> int:
        total = 0
        for kind, u, _phase in self.events:
            S = self.layout.S[u]
            if kind == "all_reduce":
                total += 2 * ring_bytes_per_rank(self.W, S)
            else:
                total += ring_bytes_per_rank(self.W, S)
        return total

    def _shard_bounds(self, u: int, r: int):
        lo = self.layout.off[u] + r * self.layout.S[u]
        return lo, lo + self.layout.S[u]


class DataParallel(_Scheme):
    """Every rank keeps the full fp32 master, m, v and 16-bit copy; the
    gradients are all-reduced (mean) and every rank runs the same update
    ("The four schemes": ``DP.step``)."""

    scheme = DP

    def __init__(self, W, theta0, dtype, unit_sizes=None, grad_dtype=None):
        super().__init__(W, theta0, dtype, None, grad_dtype)
        npad = self.layout.n_pad
        self.master = [self.theta0_padded.copy() for _ in range(W)]
        self.m = [np.zeros(npad, np.float32) for _ in range(W)]
        self.v = [np.zeros(npad, np.float32) for _ in range(W)]
        self.p16 = [cast16(self.master[r], dtype) for r in range(W)]

    def step(self, grads, lr, beta1, beta2, eps):
        self.t += 1
        avg = mean_over_ranks(grads, 0, self.layout.n_pad, self.grad_dtype)
        self.events.append(("all_reduce", 0, "step"))
        for r in range(self.W):
            adam_update(self.master[r], self.m[r], self.v[r], avg, lr, beta1, beta2, eps, self.t)
            self.p16[r] = cast16(self.master[r], self.dtype)
        for r in range(1, self.W):
            # the replicas must never drift apart
            assert np.array_equal(self.master[r].view(np.uint32), self.master[0].view(np.uint32))

    def full_master(self):
        return self.master[0].copy()

    def full_m(self):
        return self.m[0].copy()

    def full_v(self):
        return self.v[0].copy()

    def working_copy(self, r: int = 0):
        return bits16(self.p16[r], self.dtype)


class ZeRO1(_Scheme):
    """Optimizer state sharded: rank r keeps master, m and v of its own
    slice; reduce-scatter (mean), update the own slice, all-gather the fp32
    slices and recast ("The four schemes": ``ZeRO1.step``)."""

    scheme = ZERO1

    def __init__(self, W, theta0, dtype, unit_sizes=None, grad_dtype=None):
        super().__init__(W, theta0, dtype, None, grad_dtype)
        S = self.layout.S[0]
        self.master = [self.theta0_padded[r * S:(r + 1) * S].copy() for r in range(W)]
        self.m = [np.zeros(S, np.float32) for _ in range(W)]
        self.v = [np.zeros(S, np.float32) for _ in range(W)]
        self.p16 = [cast16(self.theta0_padded, dtype) for _ in range(W)]

    def step(self, grads, lr, beta1, beta2, eps):
        self.t += 1
        parts = []
        for r in range(self.W):
            lo, hi = self._shard_bounds(0, r)
            parts.append(mean_over_ranks(grads, lo, hi, self.grad_dtype))
        self.events.append(("reduce_scatter", 0, "step"))
        for r in range(self.W):
            adam_update(self.master[r], self.m[r], self.v[r], parts[r], lr, beta1, beta2, eps, self.t)
        gathered = np.concatenate(self.master)          # every rank receives every slice
        self.events.append(("all_gather", 0, "step"))
        for r in range(self.W):
            self.p16[r] = cast16(gathered, self.dtype)

    def full_master(self):
        return np.concatenate(self.master)

    def full_m(self):
        return np.concatenate(self.m)

    def full_v(self):
        return np.concatenate(self.v)

    def working_copy(self, r: int = 0):
        return bits16(self.p16[r], self.dtype)


class ZeRO2(ZeRO1):
    """ZeRO-1 that keeps only its own gradient slice after the scatter: the
    same arithmetic, a smaller resident figure ("The four schemes":
    ``ZeRO2`` changes one flag and no code)."""

    scheme = ZERO2


class ZeRO3(_Scheme):
    """Parameters sharded too.  Rank r keeps, per unit, its fp32 master, m,
    v and its 16-bit shard.  Each step gathers every unit for the forward
    pass and releases it, gathers it again for the backward pass (units in
    reverse order), reduce-scatters that unit's gradients, updates the own
    shard, refreshes the 16-bit shard and releases the unit.

    ``observer(phase, u, full16)`` sees each gathered unit (the 16-bit
    values in flat order, padding included) while it is live.
    """

    scheme = ZERO3

    def __init__(self, W, theta0, dtype, unit_sizes=None, grad_dtype=None, observer=None):
        super().__init__(W, theta0, dtype, unit_sizes, grad_dtype)
        L = self.layout
        self.master, self.m, self.v, self.shard16 = [], [], [], []
        for r in range(W):
            mr, mm, mv, ms = [], [], [], []
            for u in range(L.U):
                lo, hi = self._shard_bounds(u, r)
                mr.append(self.theta0_padded[lo:hi].copy())
                mm.append(np.zeros(hi - lo, np.float32))
                mv.append(np.zeros(hi - lo, np.float32))
                ms.append(cast16(mr[-1], dtype))
            self.master.append(mr)
            self.m.append(mm)
            self.v.append(mv)
            self.shard16.append(ms)
        self.observer = observer
        self.live = 0
        self.peak_live_elems = 0
        self._live_elems = 0

    def gather(self, u: int, phase: str):
        full = np.concatenate([self.shard16[r][u] for r in range(self.W)])
        self.events.append(("all_gather", u, phase))
        self.live += 1
        self._live_elems += full.size
        self.peak_live_elems = max(self.peak_live_elems, self._live_elems)
        return full

    def release(self, full):
        self.live -= 1
        self._live_elems -= full.size

    def step(self, grads, lr, beta1, beta2, eps):
        self.t += 1
        U = self.layout.U
        for u in range(U):                        # forward
            full = self.gather(u, "fwd")
            if self.observer is not None:
                self.observer("fwd", u, bits16(full, self.dtype))
            self.release(full)
        for u in reversed(range(U)):              # backward, reverse order
            full = self.gather(u, "bwd")
            if self.observer is not None:
                self.observer("bwd", u, bits16(full, self.dtype))
            parts = []
            for r in range(self.W):
                lo, hi = self._shard_bounds(u, r)
                parts.append(mean_over_ranks(grads, lo, hi, self.grad_dtype))
            self.events.append(("reduce_scatter", u, "bwd"))
            for r in range(self.W):
                adam_update(self.master[r][u], self.m[r][u], self.v[r][u], parts[r],
                            lr, beta1, beta2, eps, self.t)
                self.shard16[r][u] = cast16(self.master[r][u], self.dtype)
            self.release(full)

    def _flat(self, per_rank_units):
        L = self.layout
        out = np.zeros(L.n_pad, dtype=per_rank_units[0][0].dtype)
        for u in range(L.U):
            for r in range(self.W):
                lo, hi = self._shard_bounds(u, r)
                out[lo:hi] = per_rank_units[r][u]
        return out

    def full_master(self):
        return self._flat(self.master)

    def full_m(self):
        return self._flat(self.m)

    def full_v(self):
        return self._flat(self.v)

    def working_copy(self, r: int = 0):
        """All ranks' 16-bit shards in flat order (what a gather would give)."""
        return bits16(self._flat(self.shard16), self.dtype)

    def shard_store(self, r: int):
        """Rank r's persistent 16-bit store: its shard of every unit, in unit order."""
        return bits16(np.concatenate(self.shard16[r]), self.dtype)


SCHEME_CLASSES = {DP: DataParallel, ZERO1: ZeRO1, ZERO2: ZeRO2, ZERO3: ZeRO3}


def make_scheme(scheme: int, W: int, theta0, dtype: str, unit_sizes=None, **kw):
    return SCHEME_CLASSES[scheme](W, theta0, dtype, unit_sizes, **kw)


# --------------------------------------------------------------------------
# The plain definition every scheme must reach
# --------------------------------------------------------------------------

class SingleReplica:
    """Mixed-precision Adam of one replica on the mean gradient, with no
    sharding at all.  Sharding must not change a single bit of it ("ZeRO,
    annotated" section 2: the result is the model standard training would
    produce).  Works on any subset of positions, which is how full-size
    runs are checked sample by sample."""

    def __init__(self, theta0, dtype: str, grad_dtype: str | None = None):
        self.master = np.array(theta0, dtype=np.float32, copy=True)
        self.m = np.zeros_like(self.master)
        self.v = np.zeros_like(self.master)
        self.dtype = dtype
        self.grad_dtype = grad_dtype or dtype
        self.t = 0

    def step(self, grads, lr, beta1, beta2, eps):
        self.t += 1
        g = mean_over_ranks(grads, 0, self.master.size, self.grad_dtype)
        adam_update(self.master, self.m, self.v, g, lr, beta1, beta2, eps, self.t)

    def working_copy(self):
        return bits16(cast16(self.master, self.dtype), self.dtype)


def ulp_distance16(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in units in the last place between two arrays of 16-bit
    patterns of the same format (sign-magnitude mapped to a monotone line)."""
    def ordered(x):
        x = np.asarray(x, dtype=np.uint16).astype(np.int64)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), 0x8000 + x)
    return np.abs(ordered(a_bits) - ordered(b_bits))

