"""Python binding of libzero_gb300.so, the ZeRO step on one GB300.

Argument marshalling only: every function below calls the C entry point of
the same name (declared in ``include/zero_step.h``) and turns a negative
status into :class:`ZeroError`.  Tensors may be passed wherever the C call
takes a device pointer (their ``data_ptr()`` is used) and torch streams
wherever it takes a ``cudaStream_t``.  All arithmetic runs in the library's
CUDA kernels; there is no fallback: if the library has not been built,
every call raises :class:`ZeroLibraryMissing`.

:class:`ZeroStep` is a convenience owner: it allocates the buffers a
configuration needs with PyTorch (the library itself allocates nothing),
places theta0 in the padded layout and creates the context.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libzero_gb300.so")

# constants of include/zero_step.h
ZERO_OK, ZERO_E_ARG, ZERO_E_ALIGN, ZERO_E_CUDA, ZERO_E_RANK, ZERO_E_TIMEOUT, ZERO_E_STATE = 0, -1, -2, -3, -4, -5, -6
ZERO_E_NOMEM = -7
ZERO_SCHEME_DP, ZERO_SCHEME_Z1, ZERO_SCHEME_Z2, ZERO_SCHEME_Z3 = 0, 1, 2, 3
ZERO_FP16, ZERO_BF16 = 0, 1
ZERO_RESIDENT, ZERO_PEAK = 0, 1
ZERO_VARIANT_AUTO, ZERO_VARIANT_VECTOR, ZERO_VARIANT_BULK = 0, 1, 2
(ZERO_STAT_COMM_BYTES, ZERO_STAT_LAUNCHES, ZERO_STAT_GATHERS, ZERO_STAT_SCATTERS, ZERO_STAT_LIVE_ELEMS,
 ZERO_STAT_PEAK_LIVE_ELEMS, ZERO_STAT_T, ZERO_STAT_DEVICE_ERRORS, ZERO_STAT_LAST_VARIANT) = range(9)
ZERO_MAX_RANKS = 64
ZERO_KERNEL_FUSED, ZERO_KERNEL_GATHER, ZERO_KERNEL_CAST = 0, 1, 2
ZERO_DEBUG_POISON_RELEASED = 1

ERROR_NAMES = {ZERO_E_ARG: "ZERO_E_ARG", ZERO_E_ALIGN: "ZERO_E_ALIGN", ZERO_E_CUDA: "ZERO_E_CUDA",
               ZERO_E_RANK: "ZERO_E_RANK", ZERO_E_TIMEOUT: "ZERO_E_TIMEOUT", ZERO_E_STATE: "ZERO_E_STATE",
               ZERO_E_NOMEM: "ZERO_E_NOMEM"}

# every symbol the header declares, with (restype, argtypes)
_P, _I, _L, _D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
_PP = ctypes.POINTER(ctypes.c_void_p)
_LP = ctypes.POINTER(ctypes.c_int64)
HOOK = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p)
SIGNATURES = {
    "zero_buffer_sizes": (_I, [_I, _I, _L, _LP, _LP]),
    "zero_layout": (_I, [_I, _L, _LP, _LP, _LP, _LP]),
    "zero_bytes_per_rank": (_L, [_I, _L, _I, _I, _L]),
    "zero_comm_bytes_closed_form": (_L, [_I, _L, _I]),
    "zero_init": (_I, [ctypes.POINTER(_P), _I, _I, _L, _L, _LP, _I, _I, _P, _P, _P, _P, _PP, _PP, _P, _P]),
    "zero_destroy": (_I, [_P]),
    "zero_refresh_working_copy": (_I, [_P]),
    "zero_step": (_I, [_P, _I, _I, _L, _PP, _D, _D, _D, _D, _L]),
    "zero_set_unit_hook": (_I, [_P, HOOK, _P]),
    "zero_step_bucket": (_I, [_P, _L, _L, _PP, _D, _D, _D, _D, _L, _P]),
    "zero_host_staging_bytes": (_L, [_I, _I, _L, _LP, _L]),
    "zero_step_host": (_I, [_P, _I, _I, _L, _PP, _P, _P, _L, _L, _D, _D, _D, _D, _L, _P, _P]),
    "zero_offload_staging_bytes": (_L, [_L]),
    "zero_offload_init": (_I, [ctypes.POINTER(_P), _I, _L, _I, _I, _P, _P, _P, _P, _P, _P, _P, _L, _L, _I, _P]),
    "zero_offload_step": (_I, [_P, _PP, _D, _D, _D, _D, _L]),
    "zero_offload_stats": (_I, [_P, _LP, ctypes.POINTER(ctypes.c_double), _LP, _LP, _LP,
                                ctypes.POINTER(ctypes.c_int)]),
    "zero_offload_destroy": (_I, [_P]),
    "zero_offload_set_step": (_I, [_P, _L]),
    "zero_adam_host": (_I, [_L, _P, _P, _P, _P, _P, _I, _D, _D, _D, _D, _L, _I, _I]),
    "zero_host_alloc": (_I, [_L, ctypes.POINTER(_P)]),
    "zero_host_free": (_I, [_P]),
    "zero_gather_unit": (_I, [_P, _L, _P, _P]),
    "zero_release_unit": (_I, [_P, _L]),
    "zero_update_unit": (_I, [_P, _L, _PP, _D, _D, _D, _D, _L, _P]),
    "zero_get_state": (_I, [_P, _P, _P, _P, _LP]),
    "zero_set_state": (_I, [_P, _P, _P, _P, _L]),
    "zero_comm_bytes_per_rank": (_L, [_P]),
    "zero_stat": (_L, [_P, _I]),
    "zero_sync": (_I, [_P, _I]),
    "zero_enable_timing": (_I, [_P, _I]),
    "zero_read_timing": (_I, [_P, _I, ctypes.POINTER(ctypes.c_double), _LP]),
    "zero_set_variant": (_I, [_P, _I]),
    "zero_set_graph": (_I, [_P, _I]),
    "zero_inject_stall": (_I, [_P, _L]),
    "zero_set_debug": (_I, [_P, _I]),
    "zero_mark_rank": (_I, [_P, _I, _I]),
    "zero_step_z3_static": (_I, [_I, _L, _LP, _I, _I, _P, _P, _P, _PP, _PP, _D, _D, _D, _D, _L, HOOK, _P, _P]),
    "zero_step_dp_replicas": (_I, [_I, _L, _I, _I, _PP, _PP, _PP, _PP, _PP, _D, _D, _D, _D, _L, _P]),
    "zero_dp_replicas_mismatches": (_I, [_I, _L, _PP, _PP, _PP, _PP, _P, _P]),
    "zero_last_error": (ctypes.c_char_p, []),
}


class ZeroLibraryMissing(ImportError):
    pass


class ZeroError(RuntimeError):
    def __init__(self, code: int, func: str, message: str):
        super().__init__(f"{func}: {ERROR_NAMES.get(code, code)}: {message}")
        self.code = code


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded library (loaded on first use; raises if it is not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ZeroLibraryMissing(
                f"{LIB_PATH} is not built; build it with `python -m zero_sharded_mixed_step_gb300.build`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _check(name: str, rc: int) -> int:
    if rc < 0:
        raise ZeroError(rc, name, lib().zero_last_error().decode())
    return rc


def _ptr(x):
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        # the library reads and writes dense vectors from this address
        if hasattr(x, "is_contiguous") and not x.is_contiguous():
            raise ValueError("a tensor passed to the library must be contiguous")
        return x.data_ptr()
    return int(x)


def _stream(s):
    if s is None:
        return None
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream or None
    return int(s) or None


def _ptr_array(xs):
    if xs is None:
        return None
    return (ctypes.c_void_p * len(xs))(*[_ptr(x) for x in xs])


def _i64_array(xs):
    return (ctypes.c_int64 * len(xs))(*[int(x) for x in xs])


# ---- the entry points, same names as the C ABI --------------------------------

def zero_last_error() -> str:
    return lib().zero_last_error().decode()


def zero_buffer_sizes(scheme: int, W: int, unit_sizes) -> dict:
    out = (ctypes.c_int64 * 6)()
    _check("zero_buffer_sizes", lib().zero_buffer_sizes(scheme, W, len(unit_sizes), _i64_array(unit_sizes), out))
    return dict(n=out[0], n_pad=out[1], p16=out[2], shard_store=out[3], unit_buf=out[4], units=out[5])


def zero_layout(W: int, unit_sizes):
    U = len(unit_sizes)
    off, shard, off16 = (ctypes.c_int64 * U)(), (ctypes.c_int64 * U)(), (ctypes.c_int64 * U)()
    _check("zero_layout", lib().zero_layout(W, U, _i64_array(unit_sizes), off, shard, off16))
    return list(off), list(shard), list(off16)


def zero_bytes_per_rank(scheme: int, n: int, W: int, kind: int = ZERO_RESIDENT, gathered_elems: int = 0) -> int:
    return _check("zero_bytes_per_rank", lib().zero_bytes_per_rank(scheme, n, W, kind, gathered_elems))


def zero_comm_bytes_closed_form(scheme: int, n: int, W: int) -> int:
    return _check("zero_comm_bytes_closed_form", lib().zero_comm_bytes_closed_form(scheme, n, W))


def zero_init(scheme, W, n, unit_sizes, grad_dtype, work_dtype, master, m, v, p16=None, shard16=None,
              unit_bufs=None, stream_update=None, stream_gather=None) -> int:
    ctx = ctypes.c_void_p()
    _check("zero_init", lib().zero_init(
        ctypes.byref(ctx), scheme, W, n, len(unit_sizes), _i64_array(unit_sizes), grad_dtype, work_dtype,
        _ptr(master), _ptr(m), _ptr(v), _ptr(p16), _ptr_array(shard16), _ptr_array(unit_bufs),
        _stream(stream_update), _stream(stream_gather)))
    return ctx.value


def zero_destroy(ctx) -> None:
    _check("zero_destroy", lib().zero_destroy(ctx))


def zero_refresh_working_copy(ctx) -> None:
    _check("zero_refresh_working_copy", lib().zero_refresh_working_copy(ctx))


def zero_step(ctx, scheme, W, n, grads, lr, beta1, beta2, eps, t) -> None:
    _check("zero_step", lib().zero_step(ctx, scheme, W, n, _ptr_array(grads), lr, beta1, beta2, eps, t))


def zero_step_bucket(ctx, lo, length, bucket_grads, lr, beta1, beta2, eps, t, stream=None) -> None:
    _check("zero_step_bucket", lib().zero_step_bucket(ctx, lo, length, _ptr_array(bucket_grads), lr, beta1, beta2, eps,
                                                      t, _stream(stream)))


def zero_host_staging_bytes(scheme, W, unit_sizes, chunk_elems=0) -> int:
    return _check("zero_host_staging_bytes", lib().zero_host_staging_bytes(
        scheme, W, len(unit_sizes), _i64_array(unit_sizes), chunk_elems))


def zero_step_host(ctx, scheme, W, n, host_grads, host_out, staging, staging_bytes, chunk_elems,
                   lr, beta1, beta2, eps, t, stream_h2d=None, stream_d2h=None) -> None:
    """host_grads: W host buffers (tensors or addresses); host_out: host buffer or None."""
    _check("zero_step_host", lib().zero_step_host(
        ctx, scheme, W, n, _ptr_array(host_grads), _ptr(host_out), _ptr(staging), staging_bytes, chunk_elems,
        lr, beta1, beta2, eps, t, _stream(stream_h2d), _stream(stream_d2h)))


def zero_host_alloc(nbytes: int) -> int:
    """Page-locked host memory on huge pages for the host-fed step; returns its address."""
    p = ctypes.c_void_p()
    _check("zero_host_alloc", lib().zero_host_alloc(int(nbytes), ctypes.byref(p)))
    return p.value


def zero_host_free(ptr) -> None:
    _check("zero_host_free", lib().zero_host_free(ptr))


def zero_offload_staging_bytes(chunk_elems: int = 0) -> int:
    return _check("zero_offload_staging_bytes", lib().zero_offload_staging_bytes(chunk_elems))


def zero_offload_init(W, n, grad_dtype, work_dtype, host_master, host_m, host_v, host_grad, host_p16, p16,
                      staging, staging_bytes, chunk_elems=0, threads=0, stream=None):
    ctx = ctypes.c_void_p()
    _check("zero_offload_init", lib().zero_offload_init(
        ctypes.byref(ctx), W, n, grad_dtype, work_dtype, _ptr(host_master), _ptr(host_m), _ptr(host_v),
        _ptr(host_grad), _ptr(host_p16), _ptr(p16), _ptr(staging), staging_bytes, chunk_elems, threads,
        _stream(stream)))
    return ctx


def zero_offload_step(ctx, grads, lr, beta1, beta2, eps, t) -> None:
    _check("zero_offload_step", lib().zero_offload_step(ctx, _ptr_array(grads), lr, beta1, beta2, eps, t))


def zero_offload_stats(ctx) -> dict:
    t, d2h, h2d, launches = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    secs, threads = ctypes.c_double(), ctypes.c_int()
    _check("zero_offload_stats", lib().zero_offload_stats(ctx, ctypes.byref(t), ctypes.byref(secs),
                                                          ctypes.byref(d2h), ctypes.byref(h2d),
                                                          ctypes.byref(launches), ctypes.byref(threads)))
    return {"t": t.value, "host_seconds": secs.value, "d2h_bytes": d2h.value, "h2d_bytes": h2d.value,
            "launches": launches.value, "threads": threads.value}


def zero_offload_set_step(ctx, t: int) -> None:
    _check("zero_offload_set_step", lib().zero_offload_set_step(ctx, t))


def zero_offload_destroy(ctx) -> None:
    _check("zero_offload_destroy", lib().zero_offload_destroy(ctx))


def zero_adam_host(n, grad, master, m, v, out16, work_dtype, lr, beta1, beta2, eps, t, W=1, threads=0) -> None:
    """The offloaded step's host update on host tensors (no GPU needed)."""
    _check("zero_adam_host", lib().zero_adam_host(n, _ptr(grad), _ptr(master), _ptr(m), _ptr(v), _ptr(out16),
                                                  work_dtype, lr, beta1, beta2, eps, t, W, threads))


class HostBuffer:
    """A zero_host_alloc block seen as a CPU tensor of ``numel`` values of
    ``dtype`` (the tensor shares the memory; keep this object alive while it
    or any copy in flight uses it, then ``close()``)."""

    def __init__(self, numel: int, dtype):
        import torch
        itemsize = torch.empty(0, dtype=dtype).element_size()
        self.nbytes = max(1, int(numel) * itemsize)
        self.ptr = zero_host_alloc(self.nbytes)
        raw = (ctypes.c_uint8 * self.nbytes).from_address(self.ptr)
        self.tensor = torch.frombuffer(raw, dtype=torch.uint8)[: int(numel) * itemsize].view(dtype)

    def close(self):
        if self.ptr:
            self.tensor = None
            zero_host_free(self.ptr)
            self.ptr = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def zero_set_unit_hook(ctx, fn, user=None):
    """``fn(user, phase, unit, unit_buf, stream)``; returns the ctypes callback,
    which the caller must keep alive while it is registered."""
    cb = HOOK(fn) if fn is not None else HOOK()
    _check("zero_set_unit_hook", lib().zero_set_unit_hook(ctx, cb, user))
    return cb


def zero_gather_unit(ctx, unit, dst, stream=None) -> None:
    _check("zero_gather_unit", lib().zero_gather_unit(ctx, unit, _ptr(dst), _stream(stream)))


def zero_release_unit(ctx, unit) -> None:
    _check("zero_release_unit", lib().zero_release_unit(ctx, unit))


def zero_update_unit(ctx, unit, grads, lr, beta1, beta2, eps, t, stream=None) -> None:
    _check("zero_update_unit", lib().zero_update_unit(ctx, unit, _ptr_array(grads), lr, beta1, beta2, eps, t,
                                                      _stream(stream)))


def zero_get_state(ctx, master=None, m=None, v=None) -> int:
    t = ctypes.c_int64()
    _check("zero_get_state", lib().zero_get_state(ctx, _ptr(master), _ptr(m), _ptr(v), ctypes.byref(t)))
    return t.value


def zero_set_state(ctx, master, m, v, t) -> None:
    _check("zero_set_state", lib().zero_set_state(ctx, _ptr(master), _ptr(m), _ptr(v), t))


def zero_comm_bytes_per_rank(ctx) -> int:
    return _check("zero_comm_bytes_per_rank", lib().zero_comm_bytes_per_rank(ctx))


def zero_stat(ctx, which: int) -> int:
    return _check("zero_stat", lib().zero_stat(ctx, which))


def zero_sync(ctx, timeout_ms: int = -1) -> None:
    _check("zero_sync", lib().zero_sync(ctx, timeout_ms))


def zero_enable_timing(ctx, on: bool) -> None:
    _check("zero_enable_timing", lib().zero_enable_timing(ctx, 1 if on else 0))


def zero_read_timing(ctx, kernel: int):
    """(total milliseconds, launches) of the timed launches of ``kernel`` since the last read."""
    ms, k = ctypes.c_double(), ctypes.c_int64()
    _check("zero_read_timing", lib().zero_read_timing(ctx, kernel, ctypes.byref(ms), ctypes.byref(k)))
    return ms.value, k.value


def zero_set_variant(ctx, variant: int) -> None:
    _check("zero_set_variant", lib().zero_set_variant(ctx, variant))


def zero_set_graph(ctx, on: bool) -> None:
    _check("zero_set_graph", lib().zero_set_graph(ctx, 1 if on else 0))


def zero_set_debug(ctx, flags: int) -> None:
    _check("zero_set_debug", lib().zero_set_debug(ctx, flags))


def zero_inject_stall(ctx, tile: int) -> None:
    _check("zero_inject_stall", lib().zero_inject_stall(ctx, tile))


def zero_mark_rank(ctx, rank: int, available: bool) -> None:
    _check("zero_mark_rank", lib().zero_mark_rank(ctx, rank, 1 if available else 0))


def zero_step_z3_static(W, unit_sizes, grad_dtype, work_dtype, master, m, v, shard16, grads,
                        lr, beta1, beta2, eps, t, hook=None, stream=None) -> None:
    """The ZeRO-3 step for callers that cannot allocate device memory: its
    gather buffer is the library's own fixed array (units up to 8,388,608
    padded 16-bit values); no context."""
    cb = HOOK(hook) if hook is not None else HOOK()
    _check("zero_step_z3_static", lib().zero_step_z3_static(
        W, len(unit_sizes), _i64_array(unit_sizes), grad_dtype, work_dtype, _ptr(master), _ptr(m), _ptr(v),
        _ptr_array(shard16), _ptr_array(grads), lr, beta1, beta2, eps, t, cb, None, _stream(stream)))


def zero_step_dp_replicas(W, n, grad_dtype, work_dtype, grads, master, m, v, p16, lr, beta1, beta2, eps, t,
                          stream=None) -> None:
    """One DP step over W literal replicas (lists of W device buffers each);
    no context, the caller keeps t."""
    _check("zero_step_dp_replicas", lib().zero_step_dp_replicas(
        W, n, grad_dtype, work_dtype, _ptr_array(grads), _ptr_array(master), _ptr_array(m), _ptr_array(v),
        _ptr_array(p16), lr, beta1, beta2, eps, t, _stream(stream)))


def zero_dp_replicas_mismatches(W, n, master, m, v, p16, mismatches, stream=None) -> None:
    """Enqueue the bitwise comparison of every replica with replica 0; the
    count lands in the device int64 ``mismatches``."""
    _check("zero_dp_replicas_mismatches", lib().zero_dp_replicas_mismatches(
        W, n, _ptr_array(master), _ptr_array(m), _ptr_array(v), _ptr_array(p16), _ptr(mismatches),
        _stream(stream)))


# ---- convenience owners ---------------------------------------------------------

_DT = {"fp16": ZERO_FP16, "bf16": ZERO_BF16, ZERO_FP16: ZERO_FP16, ZERO_BF16: ZERO_BF16}


class ZeroStep:
    """Buffers for one configuration, allocated with PyTorch on ``device``,
    plus the library context that uses them.

    ``theta0`` (n fp32 values, any device) is written to the real positions
    of the padded master; m and v start at zero; the 16-bit working copy is
    cast from the master before the first step.  ``alloc(numel, dtype)``, if
    given, supplies every device buffer instead of ``torch.zeros`` (a
    zero-filled tensor on ``device``, e.g. from the caller's own pool).
    """

    def __init__(self, scheme, W, unit_sizes, grad_dtype="fp16", work_dtype=None, theta0=None,
                 device="cuda", stream=None, gather_stream=None, with_grad_buffers=False, alloc=None):
        import torch
        self.torch = torch
        self.scheme, self.W = int(scheme), int(W)
        self.unit_sizes = [int(s) for s in unit_sizes]
        self.gdt = _DT[grad_dtype]
        self.wdt = _DT[work_dtype if work_dtype is not None else grad_dtype]
        self.sizes = zero_buffer_sizes(self.scheme, self.W, self.unit_sizes)
        self.n, self.n_pad = self.sizes["n"], self.sizes["n_pad"]
        self.off, self.shard, self.off16 = zero_layout(self.W, self.unit_sizes)
        self.device = torch.device(device)
        t16 = {ZERO_FP16: torch.float16, ZERO_BF16: torch.bfloat16}
        self.grad_torch_dtype, self.work_torch_dtype = t16[self.gdt], t16[self.wdt]
        self._alloc = alloc or (lambda numel, dtype: torch.zeros(numel, dtype=dtype, device=self.device))
        f32, w16 = torch.float32, self.work_torch_dtype
        self.master = self._alloc(self.n_pad, f32)
        self.m = self._alloc(self.n_pad, f32)
        self.v = self._alloc(self.n_pad, f32)
        self.p16 = self._alloc(self.sizes["p16"], w16) if self.scheme != ZERO_SCHEME_Z3 else None
        self.shard16 = ([self._alloc(self.sizes["shard_store"], w16) for _ in range(self.W)]
                        if self.scheme == ZERO_SCHEME_Z3 else None)
        self.unit_bufs = ([self._alloc(self.sizes["unit_buf"], w16) for _ in range(2)]
                          if self.scheme == ZERO_SCHEME_Z3 else None)
        if theta0 is not None:
            self.place_(self.master, theta0)
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        self.gather_stream = gather_stream
        self.ctx = zero_init(self.scheme, self.W, self.n, self.unit_sizes, self.gdt, self.wdt, self.master,
                             self.m, self.v, self.p16, self.shard16, self.unit_bufs, self.stream, gather_stream)
        self._hook = None
        zero_refresh_working_copy(self.ctx)
        self.grads = self.new_grad_buffers() if with_grad_buffers else None

    # layout helpers (marshalling between the caller's n values and the padded layout)
    def real_index(self):
        torch = self.torch
        parts = [torch.arange(o, o + s, device=self.device) for o, s in zip(self.off, self.unit_sizes)]
        return torch.cat(parts) if parts else torch.zeros(0, dtype=torch.int64, device=self.device)

    def place_(self, dst, real):
        real = self.torch.as_tensor(real).to(device=dst.device, dtype=dst.dtype)
        if len(self.unit_sizes) == 1:
            dst[: self.n].copy_(real)
        else:
            pos = 0
            for o, s in zip(self.off, self.unit_sizes):
                dst[o:o + s].copy_(real[pos:pos + s])
                pos += s
        return dst

    def new_grad_buffers(self):
        return [self._alloc(self.n_pad, self.grad_torch_dtype) for _ in range(self.W)]

    def working_copy(self):
        """The full 16-bit vector in flat order (Z3: every rank's shards interleaved back)."""
        if self.scheme != ZERO_SCHEME_Z3:
            return self.p16
        out = self.torch.empty(self.n_pad, dtype=self.work_torch_dtype, device=self.device)
        for u, (o, s, o16) in enumerate(zip(self.off, self.shard, self.off16)):
            for r in range(self.W):
                out[o + r * s:o + (r + 1) * s].copy_(self.shard16[r][o16:o16 + s])
        return out

    def step(self, grads, lr, beta1, beta2, eps, t):
        zero_step(self.ctx, self.scheme, self.W, self.n, grads, lr, beta1, beta2, eps, t)

    def set_unit_hook(self, fn):
        self._hook = zero_set_unit_hook(self.ctx, fn)

    def set_variant(self, variant):
        zero_set_variant(self.ctx, variant)

    def set_graph(self, on=True):
        zero_set_graph(self.ctx, on)

    def set_debug(self, flags):
        zero_set_debug(self.ctx, flags)

    def stat(self, which):
        return zero_stat(self.ctx, which)

    def sync(self, timeout_ms=-1):
        zero_sync(self.ctx, timeout_ms)

    def close(self):
        if getattr(self, "ctx", None):
            zero_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class DpReplicas:
    """W literal DP replicas allocated with PyTorch on ``device``: per replica
    an fp32 master, m and v and a 16-bit working copy, n_pad values each.

    ``theta0`` (n fp32 values) is written into every replica's master; m and
    v start at zero.  Each 16-bit working copy is written by the step (it
    holds zeros before the first one).  The step and the replica check run
    in the library.  ``alloc`` as for :class:`ZeroStep`.
    """

    def __init__(self, W, n, grad_dtype="fp16", work_dtype=None, theta0=None, device="cuda", stream=None,
                 alloc=None):
        import torch
        self.torch = torch
        self.W, self.n = int(W), int(n)
        self.gdt = _DT[grad_dtype]
        self.wdt = _DT[work_dtype if work_dtype is not None else grad_dtype]
        self.n_pad = zero_buffer_sizes(ZERO_SCHEME_DP, self.W, [self.n])["n_pad"]
        self.device = torch.device(device)
        t16 = {ZERO_FP16: torch.float16, ZERO_BF16: torch.bfloat16}
        self.grad_torch_dtype, self.work_torch_dtype = t16[self.gdt], t16[self.wdt]
        need = self.W * self.n_pad * (12 + 2)
        if self.device.type == "cuda":
            free, _ = torch.cuda.mem_get_info(self.device)
            if need > free:
                raise MemoryError(f"{self.W} replicas of {self.n_pad} parameters need {need} bytes of device "
                                  f"memory; {free} are free")
        self._alloc = alloc or (lambda numel, dtype: torch.zeros(numel, dtype=dtype, device=self.device))
        self.master = [self._alloc(self.n_pad, torch.float32) for _ in range(self.W)]
        self.m = [self._alloc(self.n_pad, torch.float32) for _ in range(self.W)]
        self.v = [self._alloc(self.n_pad, torch.float32) for _ in range(self.W)]
        self.p16 = [self._alloc(self.n_pad, self.work_torch_dtype) for _ in range(self.W)]
        if theta0 is not None:
            th = torch.as_tensor(theta0).to(device=self.device, dtype=torch.float32)
            for r in range(self.W):
                self.master[r][: self.n].copy_(th)
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        self._count = self._alloc(1, torch.int64)

    def new_grad_buffers(self):
        return [self._alloc(self.n_pad, self.grad_torch_dtype) for _ in range(self.W)]

    def step(self, grads, lr, beta1, beta2, eps, t):
        zero_step_dp_replicas(self.W, self.n, self.gdt, self.wdt, grads, self.master, self.m, self.v, self.p16,
                              lr, beta1, beta2, eps, t, self.stream)

    def mismatches(self) -> int:
        """Elements, over replicas 1..W-1, that differ bitwise from replica 0 (waits)."""
        zero_dp_replicas_mismatches(self.W, self.n, self.master, self.m, self.v, self.p16, self._count,
                                    self.stream)
        self.stream.synchronize()
        return int(self._count.item())


def _itemsize(dtype) -> int:
    import torch
    return torch.empty(0, dtype=dtype).element_size()


def _round4k(nbytes: int) -> int:
    return -(-int(nbytes) // 4096) * 4096


class ZeroOffload:
    """ZeRO-2 with the optimizer on the host: fp32 master, m and v in host
    memory (the 16-bit working copy and the gradients on ``device``), the
    fp32 means and 16-bit results crossing the link through page-locked
    buffers from ``zero_host_alloc``.  ``theta0`` (n values) seeds the
    master; the device working copy is written by each step.  ``alloc`` as
    for :class:`ZeroStep`; ``host_alloc(numel, dtype)``, if given, supplies
    the five host buffers (zero-filled CPU tensors, best page-locked)
    instead of ``zero_host_alloc``."""

    def __init__(self, W, n, grad_dtype="fp16", work_dtype=None, theta0=None, device="cuda", stream=None,
                 chunk_elems=0, threads=0, alloc=None, host_alloc=None):
        import torch
        self.torch = torch
        self.W, self.n = int(W), int(n)
        self.gdt = _DT[grad_dtype]
        self.wdt = _DT[work_dtype if work_dtype is not None else grad_dtype]
        self.n_pad = zero_buffer_sizes(ZERO_SCHEME_Z2, self.W, [self.n])["n_pad"]
        self.device = torch.device(device)
        t16 = {ZERO_FP16: torch.float16, ZERO_BF16: torch.bfloat16}
        self.grad_torch_dtype, self.work_torch_dtype = t16[self.gdt], t16[self.wdt]
        self._bufs = []
        specs = [(self.n_pad, torch.float32)] * 4 + [(self.n_pad, self.work_torch_dtype)]
        if host_alloc is None:
            # one zero_host_alloc block for all five: each vector alone can be
            # smaller than a huge page, and such blocks stay on base pages, over
            # which the host pass and the link copies both measured slower
            block = HostBuffer(max(1, sum(_round4k(numel * _itemsize(d)) for numel, d in specs)), torch.uint8)
            self._bufs.append(block)
            views, pos = [], 0
            for numel, dtype in specs:
                nbytes = numel * _itemsize(dtype)
                views.append(block.tensor[pos:pos + nbytes].view(dtype))
                pos += _round4k(nbytes)
        else:
            views = [host_alloc(numel, dtype) for numel, dtype in specs]
        self.master, self.m, self.v, self.host_grad, self.host_p16 = views
        if theta0 is not None:
            self.master[: self.n].copy_(torch.as_tensor(theta0, dtype=torch.float32).cpu())
        self._alloc = alloc or (lambda numel, dtype: torch.zeros(numel, dtype=dtype, device=self.device))
        self.p16 = self._alloc(self.n_pad, self.work_torch_dtype)
        self.staging_bytes = zero_offload_staging_bytes(chunk_elems)
        self.staging = self._alloc(self.staging_bytes, torch.uint8)
        self.stream = stream if stream is not None else torch.cuda.current_stream(self.device)
        self.ctx = zero_offload_init(self.W, self.n, self.gdt, self.wdt, self.master, self.m, self.v,
                                     self.host_grad, self.host_p16, self.p16, self.staging, self.staging_bytes,
                                     chunk_elems, threads, self.stream)

    def new_grad_buffers(self):
        return [self._alloc(self.n_pad, self.grad_torch_dtype) for _ in range(self.W)]

    def step(self, grads, lr, beta1, beta2, eps, t):
        zero_offload_step(self.ctx, grads, lr, beta1, beta2, eps, t)

    def stats(self):
        return zero_offload_stats(self.ctx)

    def set_step(self, t):
        """Resume at step t: the host master, m and v must hold the state after step t."""
        zero_offload_set_step(self.ctx, t)

    def close(self):
        if getattr(self, "ctx", None):
            zero_offload_destroy(self.ctx)
            self.ctx = None
        for b in getattr(self, "_bufs", []):
            b.close()
        self._bufs = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
