"""Shared code of the GPU parity tests: run the CUDA path through the C ABI on
seeded inputs and compare it with the CPU oracle on the same draws.

Tolerances: fp32 master, m and v within |a - b| <= 1e-5 |b| + 1e-7 of the
oracle (the stated gate), and also within 1e-5 |b| + 1e-6 max|b| per array
(the same relative bound with the absolute floor scaled to the array: at
these gradient scales v is ~1e-10 and m ~1e-5, where a fixed 1e-7 floor
would accept anything); accounting integers exact.  The 16-bit working copy is checked two
ways: it must be exactly the round-to-nearest-even of the GPU's own master
(the recast the pages define), and within 1 unit in the last place of the
oracle's rounding of some master value inside the fp32 tolerance band of the
oracle's master.  Away from zero that band lies inside one 16-bit ulp, so
this is the plain 1-ulp bound; where the update cancels the master to
~1e-9, fp32 and fp64 arithmetic differ by far less than the fp32 tolerance
but by several 16-bit ulps of that tiny value, and the band says so.
"""

from __future__ import annotations

import numpy as np
import torch

import zero_sharded_mixed_step_gb300 as zs
import workloads as wk
from oracle import zero_oracle as z

RTOL, ATOL = 1e-5, 1e-7


def assert_f32_close(got: np.ndarray, ref: np.ndarray, what: str):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = np.abs(got - ref)
    bad = err > RTOL * np.abs(ref) + ATOL
    if bad.any():
        i = int(np.argmax(bad))
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; first at {i}: "
                             f"got {got[i]!r} want {ref[i]!r}")


def diagnostic_error(got: np.ndarray, ref: np.ndarray) -> float:
    """Worst error against 1e-5 |ref| + 1e-6 max|ref| (1 = at the bound)."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    floor = 1e-6 * (np.abs(ref).max() if ref.size else 0.0) + 1e-30
    return float(np.max(np.abs(got - ref) / (RTOL * np.abs(ref) + floor))) if ref.size else 0.0


def assert_f32_parity(got: np.ndarray, ref: np.ndarray, what: str) -> float:
    """Both fp32 gates: the stated tolerance, and the array-scaled one
    (diagnostic_error <= 1).  Returns the diagnostic error."""
    assert_f32_close(got, ref, what)
    d = diagnostic_error(got, ref)
    assert d <= 1.0, f"{what}: error {d:.3g} x (1e-5 |ref| + 1e-6 max|ref|)"
    return d


def band_width_ulps(ref_master: np.ndarray, dtype: str) -> np.ndarray:
    """16-bit ulps between the roundings of the two ends of each element's
    fp32 tolerance band: <= 1 where the band reading of the 1-ulp bound is
    the plain 1-ulp bound."""
    ref = np.asarray(ref_master, np.float64)
    tol = RTOL * np.abs(ref) + ATOL
    lo = _ordered16(z.bits16(z.cast16((ref - tol).astype(np.float32), dtype), dtype))
    hi = _ordered16(z.bits16(z.cast16((ref + tol).astype(np.float32), dtype), dtype))
    return hi - lo


def assert_strict_ulp16(got_bits: np.ndarray, ref_master: np.ndarray, ref_bits: np.ndarray, dtype: str,
                        what: str) -> tuple[int, int]:
    """The plain 1-ulp bound against the oracle's own rounding, asserted at
    every element whose tolerance band spans at most one 16-bit ulp; the
    elements where it spans more (masters cancelled to ~1e-9, where fp32
    and fp64 round to different tiny values) are counted, not gated.
    Returns (misses where gated (always 0), misses where not gated)."""
    miss = z.ulp_distance16(got_bits, ref_bits) > 1
    gated = band_width_ulps(ref_master, dtype) <= 1
    bad = miss & gated
    if bad.any():
        i = int(np.argmax(bad))
        raise AssertionError(f"{what}: {int(bad.sum())} 16-bit values more than 1 ulp from the oracle's rounding "
                             f"where the tolerance band is within one ulp; first at {i}: {int(got_bits[i]):#06x} "
                             f"vs {int(ref_bits[i]):#06x}")
    return 0, int((miss & ~gated).sum())


def assert_ulp16(got_bits: np.ndarray, ref_bits: np.ndarray, what: str, max_ulp: int = 1):
    d = z.ulp_distance16(got_bits, ref_bits)
    if (d > max_ulp).any():
        i = int(np.argmax(d))
        raise AssertionError(f"{what}: {int((d > max_ulp).sum())} 16-bit values more than {max_ulp} ulp off; "
                             f"first at {i}: {int(got_bits[i]):#06x} vs {int(ref_bits[i]):#06x}")


def _ordered16(bits: np.ndarray) -> np.ndarray:
    x = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    return np.where(x & 0x8000, 0x8000 - (x & 0x7FFF), 0x8000 + x)


def assert_16bit_band(got_bits: np.ndarray, ref_master: np.ndarray, dtype: str, what: str):
    """got within 1 ulp of cast16 of [ref - tol, ref + tol], tol the fp32 tolerance."""
    ref = np.asarray(ref_master, np.float64)
    tol = RTOL * np.abs(ref) + ATOL
    lo = _ordered16(z.bits16(z.cast16((ref - tol).astype(np.float32), dtype), dtype)) - 1
    hi = _ordered16(z.bits16(z.cast16((ref + tol).astype(np.float32), dtype), dtype)) + 1
    g = _ordered16(got_bits)
    bad = (g < lo) | (g > hi)
    if bad.any():
        i = int(np.argmax(bad))
        raise AssertionError(f"{what}: {int(bad.sum())} 16-bit values outside the band; first at {i}: "
                             f"{int(got_bits[i]):#06x} for master {ref[i]!r}")


def bits_of(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def sample_real_indices(n: int, W: int, units, k: int = 4096, seed: int = 0) -> np.ndarray:
    """Random real-parameter indices plus the edges: both ends, every rank
    boundary of every unit, every unit boundary."""
    rng = np.random.default_rng(seed)
    idx = set(rng.integers(0, n, size=min(k, n)).tolist()) if n else set()
    pos = 0
    for sz in units:
        S = -(-sz // W) if sz else 0
        for r in range(W + 1):
            for d in (-1, 0, 1):
                q = r * S + d
                if 0 <= q < sz:
                    idx.add(pos + q)
        for d in (0, 1, sz - 2, sz - 1):
            if 0 <= d < sz:
                idx.add(pos + d)
        pos += sz
    return np.array(sorted(idx), dtype=np.int64)


class Run:
    """One configuration on the GPU with the oracle alongside (all positions
    or a sample of them)."""

    def __init__(self, wl: wk.Workload, scheme: int, dtype: str, units=None, sample=None,
                 gather_stream: bool = True, work_dtype: str | None = None, variant: int = 0):
        self.wl, self.scheme, self.dtype = wl, scheme, dtype
        self.work_dtype = work_dtype or dtype
        self.units = list(units) if units is not None else (wl.units() if scheme == zs.ZERO_SCHEME_Z3 else [wl.n])
        dev = torch.device("cuda")
        theta0 = wk.draw_theta0(wl, dev)
        self.gs = torch.cuda.Stream() if gather_stream and scheme == zs.ZERO_SCHEME_Z3 else None
        self.zs = zs.ZeroStep(scheme, wl.W, self.units, dtype, self.work_dtype, theta0=theta0, device=dev,
                              gather_stream=self.gs, with_grad_buffers=True)
        self.zs.set_variant(variant)
        self.src = wk.GradSource(wl, dtype, dev)
        self.real_idx = self.zs.real_index()
        self.full = sample is None
        self.sample_real = np.arange(wl.n) if self.full else np.asarray(sample)
        self.sample_flat = self.real_idx[torch.from_numpy(self.sample_real).to(dev)]
        self.oracle = z.SingleReplica(theta0.cpu().numpy()[self.sample_real], self.work_dtype, grad_dtype=dtype)
        self.t = 0
        del theta0

    def step(self):
        self.t += 1
        draws = self.src.step(self.t)
        for r, d in enumerate(draws):
            self.zs.place_(self.zs.grads[r], d)
        del draws
        grads_np = [wk.to_numpy16(g[self.sample_flat]) for g in self.zs.grads]
        wl = self.wl
        self.zs.step(self.zs.grads, wl.lr, wl.beta1, wl.beta2, wl.eps, self.t)
        self.oracle.step(grads_np, wl.lr, wl.beta1, wl.beta2, wl.eps)

    def gpu_state(self):
        f = self.sample_flat
        wc = self.zs.working_copy()
        return (self.zs.master[f].cpu().numpy(), self.zs.m[f].cpu().numpy(), self.zs.v[f].cpu().numpy(),
                bits_of(wc[f]))

    def compare(self, what=""):
        torch.cuda.synchronize()
        th, m, v, p16 = self.gpu_state()
        o = self.oracle
        tag = f"{self.wl.name} scheme {self.scheme} {self.dtype} t={self.t} {what}"
        errs = dict(master=assert_f32_parity(th, o.master, f"{tag} master"),
                    m=assert_f32_parity(m, o.m, f"{tag} m"),
                    v=assert_f32_parity(v, o.v, f"{tag} v"))
        assert_16bit_band(p16, o.master, self.work_dtype, f"{tag} 16-bit copy")
        own = bits_of(self.zs.master[self.sample_flat].to(self.zs.work_torch_dtype))
        assert np.array_equal(p16, own), f"{tag}: 16-bit copy is not the RNE of the GPU master"
        _, self.strict_ulp_misses = assert_strict_ulp16(p16, o.master, o.working_copy(), self.work_dtype,
                                                        f"{tag} 16-bit copy")
        return errs

    def padding_is_zero(self):
        n_pad = self.zs.n_pad
        mask = torch.ones(n_pad, dtype=torch.bool, device=self.real_idx.device)
        mask[self.real_idx] = False
        if not mask.any():
            return True
        wc = self.zs.working_copy()
        return all(bool((x[mask] == 0).all()) for x in (self.zs.master, self.zs.m, self.zs.v, wc))

    def close(self):
        self.zs.close()
        del self.zs
        torch.cuda.empty_cache()
