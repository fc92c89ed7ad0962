// The ZeRO-3 step for callers that cannot allocate device memory.
//
// zero_step needs two caller-allocated unit buffers for ZeRO-3: the place
// each unit is gathered into before its forward and backward passes.  Some
// callers cannot provide them: code that runs where cudaMalloc is not
// allowed or not wanted, e.g. inside a host callback, under a memory pool
// that is already fully reserved, or in a process whose allocator belongs
// to another framework.  zero_step_z3_static runs the same step with its
// gather buffer in a fixed array of device memory that belongs to this
// library (kStaticUnitElems 16-bit values, 16 MiB), so the caller passes
// only the state it already owns.
//
// The array is a file-scope __device__ variable: every GPU on which the
// library's code is loaded holds it until the process exits, and every
// call shares it.  In host code its name is only a host-side stand-in, so
// each call looks up the device address with cudaGetSymbolAddress, with the
// caller's device current, and hands that address to the kernels.  The
// lookup is not cached: after cudaDeviceReset (or any teardown of the
// device's context) the module is loaded again and the array may sit at
// another address, and a cached one would then point at freed memory.
//
// The update runs the register kernel (ZERO_VARIANT_VECTOR), which has no
// device-side waits.  The bulk-staged kernel bounds its waits and reports one
// that runs out through a per-context counter, and this entry point has no
// context to report it through.

#include <cuda_runtime.h>

#include <cstdint>

#include "zero_internal.h"
#include "zero_step.h"

namespace {

// The most 16-bit values one gathered unit (S_u * W) may hold.
constexpr int64_t kStaticUnitElems = int64_t(8) << 20;

static __device__ __align__(256) uint16_t g_static_unit[kStaticUnitElems];

// errors are reported through zero_last_error(), like every other entry point
int set_error(int code, const char* msg) { return zero::record_error(code, msg); }

// Device address of g_static_unit on the current device, looked up on every
// call (cheap next to the step, and never stale: see the top of the file).
int unit_scratch(void** out) {
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_static_unit);
  if (e != cudaSuccess || p == nullptr)
    return set_error(ZERO_E_CUDA, e != cudaSuccess ? cudaGetErrorString(e) : "no device address for the scratch");
  *out = p;
  return ZERO_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

extern "C" int zero_step_z3_static(int W, int64_t n_units, const int64_t* unit_sizes, int grad_dtype,
                                   int work_dtype, float* master, float* m, float* v, void* const* shard16,
                                   const void* const* grads, double lr, double beta1, double beta2, double eps,
                                   int64_t t, zero_unit_hook hook, void* user, void* stream) {
  if (W < 1 || W > ZERO_MAX_RANKS) return set_error(ZERO_E_ARG, "W outside [1, ZERO_MAX_RANKS]");
  if (n_units < 1 || unit_sizes == nullptr) return set_error(ZERO_E_ARG, "need at least one unit");
  if ((grad_dtype != ZERO_FP16 && grad_dtype != ZERO_BF16) || (work_dtype != ZERO_FP16 && work_dtype != ZERO_BF16))
    return set_error(ZERO_E_ARG, "16-bit formats must be ZERO_FP16 or ZERO_BF16");
  int rc = zero::check_adam_args(lr, beta1, beta2, eps, t);
  if (rc) return rc;
  // the same layout as every ZeRO-3 context: units padded to S_u * W, one
  // after another (walked forward here, and backward for the backward pass)
  int64_t pos = 0, pos16 = 0;
  for (int64_t u = 0; u < n_units; ++u) {
    if (unit_sizes[u] < 0) return set_error(ZERO_E_ARG, "negative unit size");
    // bounded before any arithmetic, so that padding cannot overflow
    if (unit_sizes[u] > kStaticUnitElems ||
        (unit_sizes[u] + W - 1) / W * W > kStaticUnitElems)
      return set_error(ZERO_E_ARG,
                       "a unit is larger than the static gather buffer (8,388,608 16-bit values after padding); "
                       "use zero_step with caller-allocated unit buffers");
    const int64_t S = (unit_sizes[u] + W - 1) / W;
    pos += S * W;
    pos16 += S;
  }
  const bool any = pos > 0;
  if (any && (!master || !m || !v || !shard16 || !grads)) return set_error(ZERO_E_ARG, "a required pointer is NULL");
  if (!aligned(master, 32) || !aligned(m, 32) || !aligned(v, 32))
    return set_error(ZERO_E_ALIGN, "master, m and v must be 32-byte aligned");
  for (int r = 0; any && r < W; ++r) {
    if (!shard16[r] || !grads[r]) return set_error(ZERO_E_ARG, "a shard store or gradient pointer is NULL");
    if (!aligned(shard16[r], 16) || !aligned(grads[r], 16))
      return set_error(ZERO_E_ALIGN, "shard stores and gradients must be 16-byte aligned");
  }
  void* buf = nullptr;
  if ((rc = unit_scratch(&buf))) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  zero::FusedLaunch a{};
  a.W = W;
  a.grad_dtype = grad_dtype;
  a.work_dtype = work_dtype;
  for (int r = 0; r < W; ++r) a.grads[r] = grads[r];
  a.master = master;
  a.m = m;
  a.v = v;
  a.variant = ZERO_VARIANT_VECTOR;   // no device-side waits (see the top of the file)
  a.coef = zero::adam_coef(lr, beta1, beta2, eps, t, W);
  int64_t launches = 0;
  // One stream and one buffer: each gather waits, in stream order, for the
  // work that used the previous unit.  Without a hook nothing runs between a
  // unit's backward gather and its update, so the update pass does both: it
  // copies each 16-bit value into the buffer before overwriting it.
  auto unit = [&](int64_t u, int64_t off, int64_t off16, int phase) -> int {
    const int64_t S = (unit_sizes[u] + W - 1) / W;
    if (S == 0) {
      if (hook) hook(user, phase, u, buf, stream);
      return ZERO_OK;
    }
    const bool fused_gather = phase == 1 && hook == nullptr;
    cudaError_t e = cudaSuccess;
    if (!fused_gather) {
      zero::CopySeg segs[zero::kMaxCopySegs];
      for (int r = 0; r < W; ++r)
        segs[r] = {static_cast<const char*>(shard16[r]) + off16 * 2, static_cast<char*>(buf) + r * S * 2, S * 2};
      e = zero::launch_copy(segs, W, s, &launches);
      if (e != cudaSuccess) return set_error(ZERO_E_CUDA, cudaGetErrorString(e));
      if (hook) hook(user, phase, u, buf, stream);
    }
    if (phase == 1) {
      a.nseg = W;
      for (int r = 0; r < W; ++r)
        a.segs[r] = {off + r * S, S, static_cast<char*>(shard16[r]) + off16 * 2,
                     fused_gather ? static_cast<char*>(buf) + r * S * 2 : nullptr};
      e = zero::launch_fused_step(a, s, &launches);
      if (e != cudaSuccess) return set_error(ZERO_E_CUDA, cudaGetErrorString(e));
    }
    return ZERO_OK;
  };
  int64_t off = 0, off16 = 0;
  for (int64_t u = 0; u < n_units; ++u) {
    if ((rc = unit(u, off, off16, 0))) return rc;
    const int64_t S = (unit_sizes[u] + W - 1) / W;
    off += S * W;
    off16 += S;
  }
  for (int64_t u = n_units - 1; u >= 0; --u) {
    const int64_t S = (unit_sizes[u] + W - 1) / W;
    off -= S * W;
    off16 -= S;
    if ((rc = unit(u, off, off16, 1))) return rc;
  }
  return ZERO_OK;
}
