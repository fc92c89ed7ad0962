// Data parallelism with its W replicas kept literally, on one GPU.
//
// Under plain data parallelism every rank holds the whole model state: the
// 16-bit working copy, its gradients, and the fp32 master, m and v, 16 bytes
// per parameter on every rank ("The four schemes": the DP baseline; "ZeRO,
// annotated": the redundancy that the three ZeRO stages partition away).
// After the all-reduce every rank holds the same mean gradient and runs the
// same Adam step on its own replica, so the replicas stay bit-identical, which
// the lab's DP class asserts after every step.
//
// zero_step keeps one copy for DP, because the W copies are equal by
// construction.  zero_step_dp_replicas materialises all W of them.  One pass
// reads the W gradient vectors once and forms their rank-ordered mean, the
// all-reduce's result, identical on every rank; it then updates every
// replica's master, m and v and writes every replica's 16-bit copy.  Per
// parameter that moves 2 W + 26 W bytes, where the sharded step moves
// 2 W + 26, and keeps 14 W bytes of replicated state: the cost that
// sharding removes, measured instead of counted.
//
// zero_dp_replicas_mismatches is the lab's assertion: it counts, bit for
// bit, where a replica differs from replica 0.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <utility>
#include <vector>

#include "step_math.cuh"
#include "zero_internal.h"
#include "zero_step.h"

namespace zero {
namespace {

using namespace dev;

// Launch shape, measured on GB300 for 8 replicas of 124M parameters: one
// replica's master, m and v in flight per thread at a time, with 512
// resident threads per SM, moved 98% of the measured copy bandwidth.  Two
// replicas' loads issued together gained nothing at their best occupancy
// (384 threads per SM) and lost 3% at 512 or more; four lost 4%.
constexpr int kThreads = 128;
constexpr int kThreadsPerSm = 512;
constexpr int kCompareThreads = 256;

struct ReplicaArgs {
  int W;
  int64_t n;                        // values per replica vector (n_pad)
  const void* grads[kMaxRanks];     // rank w's 16-bit gradients
  float* master[kMaxRanks];         // replica r's fp32 state ...
  float* m[kMaxRanks];
  float* v[kMaxRanks];
  void* p16[kMaxRanks];             // ... and its 16-bit working copy
  AdamCoef coef;
};

struct CompareArgs {
  int W;
  int vec;                        // every replica 32-byte (fp32) and 16-byte (16-bit) aligned
  int64_t n;
  const float* master[kMaxRanks];
  const float* m[kMaxRanks];
  const float* v[kMaxRanks];
  const uint16_t* p16[kMaxRanks];
  unsigned long long* mismatches;
};

// The rank-ordered fp32 sum of the W gradients of the 8 elements at i (WC > 0:
// W fixed at compile time, all W loads in flight; WC == 0: 8 ranks at a time).
template <typename GT, int WC>
__device__ __forceinline__ void rank_sum8(const ReplicaArgs& a, int64_t i, int W, float (&sum)[8]) {
  if constexpr (WC > 0) {
    uint4 raw[WC];
#pragma unroll
    for (int w = 0; w < WC; ++w) raw[w] = ld_16B(static_cast<const GT*>(a.grads[w]) + i);
    Fmt<GT>::unpack8(raw[0], sum);
#pragma unroll
    for (int w = 1; w < WC; ++w) {
      float f[8];
      Fmt<GT>::unpack8(raw[w], f);
#pragma unroll
      for (int k = 0; k < 8; ++k) sum[k] = __fadd_rn(sum[k], f[k]);
    }
  } else {
    for (int w0 = 0; w0 < W; w0 += 8) {
      uint4 raw[8];
      const int nb = min(8, W - w0);
#pragma unroll
      for (int w = 0; w < 8; ++w)
        if (w < nb) raw[w] = ld_16B(static_cast<const GT*>(a.grads[w0 + w]) + i);
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        if (w < nb) {
          float f[8];
          Fmt<GT>::unpack8(raw[w], f);
#pragma unroll
          for (int k = 0; k < 8; ++k) sum[k] = (w0 + w == 0) ? f[k] : __fadd_rn(sum[k], f[k]);
        }
      }
    }
  }
}

// Adam on replica r for the 8 elements at i, mean gradient g.
template <typename OT>
__device__ __forceinline__ void update_replica(const ReplicaArgs& a, int64_t i, int r, const float (&g)[8]) {
  float th[8], m[8], v[8];
  ld_32B(a.master[r] + i, th);
  ld_32B(a.m[r] + i, m);
  ld_32B(a.v[r] + i, v);
#pragma unroll
  for (int k = 0; k < 8; ++k) adam_element(g[k], th[k], m[k], v[k], a.coef);
  st_32B(a.master[r] + i, th);
  st_32B(a.m[r] + i, m);
  st_32B(a.v[r] + i, v);
  st_16B(static_cast<OT*>(a.p16[r]) + i, Fmt<OT>::pack8(th));
}

template <typename GT, typename OT, int WC>
__global__ void __launch_bounds__(kThreads) dp_replicas_step(const __grid_constant__ ReplicaArgs a) {
  const int W = WC > 0 ? WC : a.W;
  const bool pow2 = (W & (W - 1)) == 0;
  const int64_t groups = a.n >> 3;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t gi = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; gi < groups; gi += nthreads) {
    const int64_t i = gi << 3;
    float g[8];
    rank_sum8<GT, WC>(a, i, W, g);
#pragma unroll
    for (int k = 0; k < 8; ++k) g[k] = rank_mean(g[k], W, a.coef.inv_w, pow2);
    for (int r = 0; r < W; ++r) update_replica<OT>(a, i, r, g);
  }
  // the last n mod 8 values of every vector
  if (blockIdx.x == 0) {
    for (int64_t e = (groups << 3) + threadIdx.x; e < a.n; e += blockDim.x) {
      float sum = Fmt<GT>::load1(a.grads[0], e);
      for (int w = 1; w < W; ++w) sum = __fadd_rn(sum, Fmt<GT>::load1(a.grads[w], e));
      const float g = rank_mean(sum, W, a.coef.inv_w, pow2);
      for (int r = 0; r < W; ++r) {
        float th = a.master[r][e], m = a.m[r][e], v = a.v[r][e];
        adam_element(g, th, m, v, a.coef);
        a.master[r][e] = th;
        a.m[r][e] = m;
        a.v[r][e] = v;
        Fmt<OT>::store1(a.p16[r], e, th);
      }
    }
  }
}

// Counts the (replica r >= 1, element e) pairs where any of master, m, v or
// the 16-bit copy of replica r differs bitwise from replica 0.
// Groups of 8 elements per thread where every replica allows it (32-byte
// loads of master, m and v, 16-byte loads of the 16-bit copy), the rest one
// element at a time; each comparison is a bitwise XOR of the words, with no
// early exit, so that all of a replica's loads are in flight together.
__global__ void __launch_bounds__(kCompareThreads) dp_replicas_compare(const __grid_constant__ CompareArgs a) {
  unsigned long long local = 0;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  int64_t done = 0;
  if (a.vec) {
    const int64_t groups = a.n >> 3;
    for (int64_t g = tid; g < groups; g += nthreads) {
      const int64_t i = g << 3;
      float t0[8], m0[8], v0[8];
      ld_32B(a.master[0] + i, t0);
      ld_32B(a.m[0] + i, m0);
      ld_32B(a.v[0] + i, v0);
      const uint4 p0 = ld_16B(a.p16[0] + i);
      for (int r = 1; r < a.W; ++r) {
        float t[8], m[8], v[8];
        ld_32B(a.master[r] + i, t);
        ld_32B(a.m[r] + i, m);
        ld_32B(a.v[r] + i, v);
        const uint4 p = ld_16B(a.p16[r] + i);
        const uint32_t pd[4] = {p.x ^ p0.x, p.y ^ p0.y, p.z ^ p0.z, p.w ^ p0.w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint32_t d = (__float_as_uint(t[k]) ^ __float_as_uint(t0[k])) |
                             (__float_as_uint(m[k]) ^ __float_as_uint(m0[k])) |
                             (__float_as_uint(v[k]) ^ __float_as_uint(v0[k])) |
                             ((pd[k >> 1] >> (16 * (k & 1))) & 0xFFFFu);   // element k's half of its word
          local += d != 0u ? 1u : 0u;
        }
      }
    }
    done = groups << 3;
  }
  for (int64_t e = done + tid; e < a.n; e += nthreads) {
    const uint32_t t0 = __float_as_uint(a.master[0][e]), m0 = __float_as_uint(a.m[0][e]);
    const uint32_t v0 = __float_as_uint(a.v[0][e]);
    const uint32_t p0 = a.p16[0][e];
    for (int r = 1; r < a.W; ++r) {
      const uint32_t d = (__float_as_uint(a.master[r][e]) ^ t0) | (__float_as_uint(a.m[r][e]) ^ m0) |
                         (__float_as_uint(a.v[r][e]) ^ v0) | (static_cast<uint32_t>(a.p16[r][e]) ^ p0);
      local += d != 0u ? 1u : 0u;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) local += __shfl_down_sync(0xffffffffu, local, o);
  if ((threadIdx.x & 31) == 0 && local != 0) atomicAdd(a.mismatches, local);
}

using StepFn = void (*)(const ReplicaArgs);

template <typename GT, typename OT>
StepFn pick_w(int W) {
  switch (W) {
    case 1: return dp_replicas_step<GT, OT, 1>;
    case 2: return dp_replicas_step<GT, OT, 2>;
    case 4: return dp_replicas_step<GT, OT, 4>;
    case 8: return dp_replicas_step<GT, OT, 8>;
    case 16: return dp_replicas_step<GT, OT, 16>;
    default: return dp_replicas_step<GT, OT, 0>;
  }
}

StepFn pick(int gdt, int wdt, int W) {
  if (gdt == kF16) return wdt == kF16 ? pick_w<__half, __half>(W) : pick_w<__half, __nv_bfloat16>(W);
  return wdt == kF16 ? pick_w<__nv_bfloat16, __half>(W) : pick_w<__nv_bfloat16, __nv_bfloat16>(W);
}

int fail(int code, const char* msg) { return record_error(code, msg); }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// false when any two of the byte ranges overlap
bool disjoint(std::vector<std::pair<uintptr_t, uintptr_t>> r) {
  std::sort(r.begin(), r.end());
  for (size_t k = 1; k < r.size(); ++k)
    if (r[k].first < r[k - 1].second) return false;
  return true;
}

int check_shape(int W, int64_t n, int64_t* n_pad) {
  if (W < 1 || W > kMaxRanks) return fail(ZERO_E_ARG, "W outside [1, ZERO_MAX_RANKS]");
  if (n < 0) return fail(ZERO_E_ARG, "negative parameter count");
  *n_pad = (n + W - 1) / W * W;
  return ZERO_OK;
}

}  // namespace
}  // namespace zero

extern "C" int zero_step_dp_replicas(int W, int64_t n, int grad_dtype, int work_dtype, const void* const* grads,
                                     float* const* master, float* const* m, float* const* v, void* const* p16,
                                     double lr, double beta1, double beta2, double eps, int64_t t, void* stream) {
  using namespace zero;
  int64_t n_pad = 0;
  int rc = check_shape(W, n, &n_pad);
  if (rc) return rc;
  if ((grad_dtype != ZERO_FP16 && grad_dtype != ZERO_BF16) || (work_dtype != ZERO_FP16 && work_dtype != ZERO_BF16))
    return fail(ZERO_E_ARG, "16-bit formats must be ZERO_FP16 or ZERO_BF16");
  if ((rc = check_adam_args(lr, beta1, beta2, eps, t))) return rc;
  if (n_pad == 0) return ZERO_OK;
  if (!grads || !master || !m || !v || !p16) return fail(ZERO_E_ARG, "a pointer array is NULL");
  std::vector<std::pair<uintptr_t, uintptr_t>> outputs;
  for (int r = 0; r < W; ++r) {
    if (!grads[r] || !master[r] || !m[r] || !v[r] || !p16[r]) return fail(ZERO_E_ARG, "a replica pointer is NULL");
    if (!aligned(master[r], 32) || !aligned(m[r], 32) || !aligned(v[r], 32))
      return fail(ZERO_E_ALIGN, "every replica's master, m and v must be 32-byte aligned");
    if (!aligned(p16[r], 16) || !aligned(grads[r], 16))
      return fail(ZERO_E_ALIGN, "16-bit copies and gradients must be 16-byte aligned");
    const uintptr_t f = static_cast<uintptr_t>(n_pad) * 4, h = static_cast<uintptr_t>(n_pad) * 2;
    for (const void* p : {static_cast<const void*>(master[r]), static_cast<const void*>(m[r]),
                          static_cast<const void*>(v[r])})
      outputs.emplace_back(reinterpret_cast<uintptr_t>(p), reinterpret_cast<uintptr_t>(p) + f);
    outputs.emplace_back(reinterpret_cast<uintptr_t>(p16[r]), reinterpret_cast<uintptr_t>(p16[r]) + h);
  }
  if (!disjoint(outputs)) return fail(ZERO_E_ARG, "replica buffers overlap one another");
  for (int r = 0; r < W; ++r) {
    std::vector<std::pair<uintptr_t, uintptr_t>> with = outputs;
    with.emplace_back(reinterpret_cast<uintptr_t>(grads[r]),
                      reinterpret_cast<uintptr_t>(grads[r]) + static_cast<uintptr_t>(n_pad) * 2);
    if (!disjoint(with)) return fail(ZERO_E_ARG, "a gradient vector overlaps a replica buffer");
  }

  ReplicaArgs a{};
  a.W = W;
  a.n = n_pad;
  for (int r = 0; r < W; ++r) {
    a.grads[r] = grads[r];
    a.master[r] = master[r];
    a.m[r] = m[r];
    a.v[r] = v[r];
    a.p16[r] = p16[r];
  }
  a.coef = adam_coef(lr, beta1, beta2, eps, t, W);
  const StepFn fn = pick(grad_dtype, work_dtype, W);
  int per_sm = 0;
  cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, 0);
  if (err != cudaSuccess) return fail(ZERO_E_CUDA, cudaGetErrorString(err));
  per_sm = std::max(1, std::min(per_sm, kThreadsPerSm / kThreads));
  const int64_t needed = (n_pad / 8 + kThreads) / kThreads;
  const int64_t blocks = std::max<int64_t>(1, std::min<int64_t>(static_cast<int64_t>(sm_count()) * per_sm, needed));
  fn<<<static_cast<unsigned>(blocks), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
  err = cudaGetLastError();
  return err == cudaSuccess ? ZERO_OK : fail(ZERO_E_CUDA, cudaGetErrorString(err));
}

extern "C" int zero_dp_replicas_mismatches(int W, int64_t n, const float* const* master, const float* const* m,
                                           const float* const* v, const void* const* p16, int64_t* mismatches,
                                           void* stream) {
  using namespace zero;
  int64_t n_pad = 0;
  int rc = check_shape(W, n, &n_pad);
  if (rc) return rc;
  if (!mismatches) return fail(ZERO_E_ARG, "the mismatch counter is NULL");
  if (!aligned(mismatches, 8)) return fail(ZERO_E_ALIGN, "the mismatch counter must be 8-byte aligned");
  const bool work = n_pad > 0 && W > 1;
  CompareArgs a{};
  a.W = W;
  a.n = n_pad;
  a.mismatches = reinterpret_cast<unsigned long long*>(mismatches);
  if (work && (!master || !m || !v || !p16)) return fail(ZERO_E_ARG, "a pointer array is NULL");
  for (int r = 0; work && r < W; ++r) {
    if (!master[r] || !m[r] || !v[r] || !p16[r]) return fail(ZERO_E_ARG, "a replica pointer is NULL");
    if (!aligned(master[r], 4) || !aligned(m[r], 4) || !aligned(v[r], 4) || !aligned(p16[r], 2))
      return fail(ZERO_E_ALIGN, "replica buffers must be aligned to their element size");
    a.master[r] = master[r];
    a.m[r] = m[r];
    a.v[r] = v[r];
    a.p16[r] = static_cast<const uint16_t*>(p16[r]);
  }
  a.vec = 1;
  for (int r = 0; work && r < W; ++r)
    if (!aligned(master[r], 32) || !aligned(m[r], 32) || !aligned(v[r], 32) || !aligned(p16[r], 16)) a.vec = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err = cudaMemsetAsync(mismatches, 0, sizeof(int64_t), s);
  if (err != cudaSuccess) return fail(ZERO_E_CUDA, cudaGetErrorString(err));
  if (!work) return ZERO_OK;
  const int64_t per_thread = a.vec ? 8 : 1;
  const int64_t needed = (n_pad / per_thread + kCompareThreads) / kCompareThreads;
  int per_sm = 0;   // one resident wave
  err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dp_replicas_compare, kCompareThreads, 0);
  if (err != cudaSuccess) return fail(ZERO_E_CUDA, cudaGetErrorString(err));
  const int64_t blocks =
      std::max<int64_t>(1, std::min<int64_t>(static_cast<int64_t>(sm_count()) * std::max(per_sm, 1), needed));
  dp_replicas_compare<<<static_cast<unsigned>(blocks), kCompareThreads, 0, s>>>(a);
  err = cudaGetLastError();
  return err == cudaSuccess ? ZERO_OK : fail(ZERO_E_CUDA, cudaGetErrorString(err));
}
