// The GPU half of the offloaded step: the mean reduce-scatter alone.
//
// With the optimizer offloaded to the host ("ZeRO and FSDP", ZeRO-3 and
// FSDP: offloading puts the optimizer state in CPU memory, trading link
// bandwidth for device memory; "ZeRO, annotated" section 11: ZeRO-Offload
// moves the optimizer's data and computation to the CPU), the device keeps
// the ranks' 16-bit gradients and working copy only.  This kernel forms, for
// one stretch of the flat vector, the rank-ordered fp32 mean of the W
// ranks' gradients, which the host's Adam consumes.  It is the same sum and
// the same division as the fused step's, from the same header, so the
// offloaded step is bit-identical to it.  Per element it reads 2 W bytes and
// writes 4.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "step_math.cuh"
#include "zero_internal.h"

namespace zero {
namespace {

using namespace dev;

constexpr int kThreads = 128;
constexpr int kThreadsPerSm = 512;

template <typename GT, int WC>
__global__ void __launch_bounds__(kThreads) rank_mean_kernel(const __grid_constant__ MeanLaunch a) {
  const int W = WC > 0 ? WC : a.W;
  const bool pow2 = (W & (W - 1)) == 0;
  const int64_t groups = a.len >> 3;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t gi = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; gi < groups; gi += nthreads) {
    const int64_t i = a.lo + (gi << 3);
    float sum[8];
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
      for (int w = 0; w < W; ++w) {
        float f[8];
        Fmt<GT>::unpack8(ld_16B(static_cast<const GT*>(a.grads[w]) + i), f);
#pragma unroll
        for (int k = 0; k < 8; ++k) sum[k] = w == 0 ? f[k] : __fadd_rn(sum[k], f[k]);
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) sum[k] = rank_mean(sum[k], W, a.inv_w, pow2);
    st_32B(a.out + (gi << 3), sum);
  }
  if (blockIdx.x == 0) {
    for (int64_t e = (groups << 3) + threadIdx.x; e < a.len; e += blockDim.x) {
      float s = Fmt<GT>::load1(a.grads[0], a.lo + e);
      for (int w = 1; w < W; ++w) s = __fadd_rn(s, Fmt<GT>::load1(a.grads[w], a.lo + e));
      a.out[e] = rank_mean(s, W, a.inv_w, pow2);
    }
  }
}

using MeanFn = void (*)(const MeanLaunch);

template <typename GT>
MeanFn pick_w(int W) {
  switch (W) {
    case 1: return rank_mean_kernel<GT, 1>;
    case 2: return rank_mean_kernel<GT, 2>;
    case 4: return rank_mean_kernel<GT, 4>;
    case 8: return rank_mean_kernel<GT, 8>;
    case 16: return rank_mean_kernel<GT, 16>;
    default: return rank_mean_kernel<GT, 0>;
  }
}

}  // namespace

cudaError_t launch_rank_mean(const MeanLaunch& a, cudaStream_t stream, int64_t* launches) {
  if (a.len <= 0) return cudaSuccess;
  if ((a.lo & 7) != 0 || (reinterpret_cast<uintptr_t>(a.out) & 31u) != 0) return cudaErrorInvalidValue;
  const MeanFn fn = a.grad_dtype == kF16 ? pick_w<__half>(a.W) : pick_w<__nv_bfloat16>(a.W);
  const int64_t needed = (a.len / 8 + kThreads) / kThreads;
  const int64_t blocks =
      std::max<int64_t>(1, std::min<int64_t>(static_cast<int64_t>(sm_count()) * (kThreadsPerSm / kThreads), needed));
  fn<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(a);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace zero
