"""Plant plausible mistakes in the oracle (on the CPU) and show that the pins
catch each one: a dropped term, a wrong sign, index or operand, a schedule
that keeps the gathered copy."""

import numpy as np
import pytest

from oracle import zero_oracle as z
from tests import oracle_pins as pins

ORIG_ADAM = z.adam_update
ORIG_MEAN = z.mean_over_ranks
ORIG_BC = z.bias_corrections


def _adam_variant(kind):
    def adam(master, m, v, g, lr, beta1, beta2, eps, t):
        bc1, bc2 = ORIG_BC(beta1, beta2, t)
        if kind == "betas_swapped":
            beta1, beta2 = beta2, beta1
        m1 = beta1 * m.astype(np.float64) + (1.0 - beta1) * g
        v1 = beta2 * v.astype(np.float64) + (1.0 - beta2) * (np.abs(g) if kind == "v_without_square" else g * g)
        m_hat = m1 if kind == "no_bias_correction_m" else m1 / (bc2 if kind == "corrections_transposed" else bc1)
        v_hat = v1 / (bc1 if kind == "corrections_transposed" else bc2)
        if kind == "eps_inside_sqrt":
            den = np.sqrt(v_hat + eps)
        else:
            den = np.sqrt(v_hat) + eps
        sign = 1.0 if kind == "sign_flipped" else -1.0
        th1 = master.astype(np.float64) + sign * lr * m_hat / den
        m[...] = m1.astype(np.float32)
        v[...] = v1.astype(np.float32)
        master[...] = th1.astype(np.float32)
    return adam


def _mean_variant(kind):
    def mean(grads, lo, hi, dtype):
        W = len(grads)
        acc = np.zeros(hi - lo)
        ranks = range(W - 1) if kind == "last_rank_dropped" else range(W)
        for w in ranks:
            acc = acc + z.decode16(grads[w][lo:hi], dtype)
        return acc if kind == "sum_not_mean" else acc / W
    return mean


def _keep_gathered_step(self, grads, lr, beta1, beta2, eps):
    # the mistake "The four schemes" warns about: gather once, keep it through both passes
    self.t += 1
    kept = {}
    for u in range(self.layout.U):
        kept[u] = self.gather(u, "fwd")
    for u in reversed(range(self.layout.U)):
        parts = []
        for r in range(self.W):
            lo, hi = self._shard_bounds(u, r)
            parts.append(z.mean_over_ranks(grads, lo, hi, self.grad_dtype))
        self.events.append(("reduce_scatter", u, "bwd"))
        for r in range(self.W):
            z.adam_update(self.master[r][u], self.m[r][u], self.v[r][u], parts[r], lr, beta1, beta2, eps, self.t)
            self.shard16[r][u] = z.cast16(self.master[r][u], self.dtype)
        self.release(kept[u])


def _stale_shard_cast(self, grads, lr, beta1, beta2, eps):
    # the lab's ZeRO-3 never refreshes the 16-bit shards after its update
    saved = [[s.copy() for s in row] for row in self.shard16]
    ORIG_Z3_STEP(self, grads, lr, beta1, beta2, eps)
    self.shard16 = saved


ORIG_Z3_STEP = z.ZeRO3.step
ORIG_BOUNDS = z._Scheme._shard_bounds


def _rotated_bounds(self, u, r):
    return ORIG_BOUNDS(self, u, (r + 1) % self.W)


def _forward_order_backward(self, grads, lr, beta1, beta2, eps):
    self.t += 1
    for u in range(self.layout.U):
        self.release(self.gather(u, "fwd"))
    for u in range(self.layout.U):           # should run in reverse
        full = self.gather(u, "bwd")
        parts = [z.mean_over_ranks(grads, *self._shard_bounds(u, r), self.grad_dtype) for r in range(self.W)]
        self.events.append(("reduce_scatter", u, "bwd"))
        for r in range(self.W):
            z.adam_update(self.master[r][u], self.m[r][u], self.v[r][u], parts[r], lr, beta1, beta2, eps, self.t)
            self.shard16[r][u] = z.cast16(self.master[r][u], self.dtype)
        self.release(full)


def _truncating_bf16(x):
    u = np.asarray(x, dtype=np.float32).view(np.uint32)
    return (u >> np.uint32(16)).astype(np.uint16)


def _place_without_zeroing(real, layout):
    out = np.full(layout.n_pad, 1e-3, dtype=real.dtype)
    out[layout.real_index()] = real
    return out


MUTANTS = {
    "no_bias_correction_m": ("adam_update", _adam_variant("no_bias_correction_m")),
    "corrections_transposed": ("adam_update", _adam_variant("corrections_transposed")),
    "eps_inside_sqrt": ("adam_update", _adam_variant("eps_inside_sqrt")),
    "betas_swapped": ("adam_update", _adam_variant("betas_swapped")),
    "v_without_square": ("adam_update", _adam_variant("v_without_square")),
    "sign_flipped": ("adam_update", _adam_variant("sign_flipped")),
    "sum_not_mean": ("mean_over_ranks", _mean_variant("sum_not_mean")),
    "last_rank_dropped": ("mean_over_ranks", _mean_variant("last_rank_dropped")),
    "step_counter_from_zero": ("bias_corrections", lambda b1, b2, t: ORIG_BC(b1, b2, t + 1)),
    "bf16_truncates": ("round_fp32_to_bf16_bits", _truncating_bf16),
    "padding_not_zero": ("place", _place_without_zeroing),
    "z2_keeps_full_gradients": ("SCHEME_FLAGS", {**z.SCHEME_FLAGS, z.ZERO2: (True, False, False)}),
    "z3_two_collectives": ("comm_bytes_closed_form",
                           lambda s, n, W, S=None: 2 * z.ring_bytes_per_rank(W, S or z.shard_size(n, W))),
    "ring_sends_W_chunks": ("ring_bytes_per_rank", lambda W, s, elem_bytes=2: W * s * elem_bytes),
    "peak_gathers_fp32": ("peak_bytes_per_rank",
                          lambda sc, n, W, g=0, S=None: z.bytes_per_rank(sc, n, W, S) + (4 * g if sc == z.ZERO3 else 0)),
    "peak_without_gathered": ("peak_bytes_per_rank", lambda sc, n, W, g=0, S=None: z.bytes_per_rank(sc, n, W, S)),
    "peak_gathers_in_every_scheme": ("peak_bytes_per_rank",
                                     lambda sc, n, W, g=0, S=None: z.bytes_per_rank(sc, n, W, S) + 2 * g),
}

CLASS_MUTANTS = {
    "z3_keeps_gathered_copy": (z.ZeRO3, "step", _keep_gathered_step),
    "z3_stale_16bit_shards": (z.ZeRO3, "step", _stale_shard_cast),
    "z3_backward_in_forward_order": (z.ZeRO3, "step", _forward_order_backward),
    "shard_index_off_by_one": (z._Scheme, "_shard_bounds", _rotated_bounds),
}


def _some_pin_fails():
    # fast checks first; the rounding sweep last and reduced
    checks = [c for c in pins.ALL_CHECKS if c is not pins.check_rounding]
    for check in checks:
        try:
            check(z)
        except Exception:       # an assertion, or the oracle refusing an impossible state
            return check.__name__
    try:
        pins.check_rounding(z, per_exponent=1)
    except Exception:
        return "check_rounding"
    return None


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_module_mutant_is_caught(name, monkeypatch):
    attr, repl = MUTANTS[name]
    monkeypatch.setattr(z, attr, repl)
    assert _some_pin_fails() is not None, f"no pin catches the planted mistake {name}"


@pytest.mark.parametrize("name", sorted(CLASS_MUTANTS))
def test_scheme_mutant_is_caught(name, monkeypatch):
    cls, attr, repl = CLASS_MUTANTS[name]
    monkeypatch.setattr(cls, attr, repl)
    assert _some_pin_fails() is not None, f"no pin catches the planted mistake {name}"


def test_keep_gathered_traffic_is_two_collectives(monkeypatch):
    """The planted keep-gathered schedule sends 2(N-1)/N 2 Psi, which the
    ZeRO-3 traffic pin rejects."""
    monkeypatch.setattr(z.ZeRO3, "step", _keep_gathered_step)
    units = [16, 16]
    theta0, grads = pins.tiny_inputs("bf16", n=32, W=4, steps=1)
    o = z.ZeRO3(4, theta0, "bf16", units)
    o.step(pins.placed(z, grads, o.layout)[0], 1e-2, 0.9, 0.999, 1e-8)
    assert o.comm_bytes() == z.comm_bytes_closed_form(z.ZERO1, 32, 4)
    assert o.comm_bytes() != z.comm_bytes_closed_form(z.ZERO3, 32, 4)
    with pytest.raises(AssertionError):
        pins.check_zero3_schedule(z)
