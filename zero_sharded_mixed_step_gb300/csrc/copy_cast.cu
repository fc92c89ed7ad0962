// The ZeRO-3 all-gather of one unit, done inside one GPU's memory, and the
// fp32 -> 16-bit recast of the working copy.
//
// Gather ("ZeRO and FSDP", ZeRO-3 and FSDP: every unit's parameters are
// all-gathered before its forward and again before its backward pass): rank
// r's 16-bit shard of unit u, S_u values, lands at [r S_u, (r + 1) S_u) of the
// unit buffer.  One launch copies all W shards, one grid row per shard,
// 16-byte vectors (four per thread in flight) wherever source and
// destination share their alignment; 2 bytes read and 2 written per element.
//
// Cast: round-to-nearest-even of the fp32 master into the 16-bit copy, used
// when the working copy is (re)built from the master (first step, restored
// state); the step itself recasts inside the fused kernel.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "zero_internal.h"

namespace zero {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

struct CopyArgs {
  CopySeg segs[kMaxCopySegs];
};

__global__ void __launch_bounds__(kCopyThreads) copy_segments(const __grid_constant__ CopyArgs a) {
  const CopySeg& s = a.segs[blockIdx.y];
  const char* src = static_cast<const char*>(s.src);
  char* dst = static_cast<char*>(s.dst);
  const int64_t n = s.count;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const uintptr_t sa = reinterpret_cast<uintptr_t>(src), da = reinterpret_cast<uintptr_t>(dst);
  if (((sa ^ da) & 15u) == 0) {
    // bytes before the first 16-byte boundary, then whole vectors, then the rest
    int64_t head = static_cast<int64_t>((16u - (da & 15u)) & 15u);
    if (head > n) head = n;
    const int64_t nvec = (n - head) >> 4;
    const uint4* vs = reinterpret_cast<const uint4*>(src + head);
    uint4* vd = reinterpret_cast<uint4*>(dst + head);
    int64_t k = tid;
    for (; k + (kCopyUnroll - 1) * nthreads < nvec; k += kCopyUnroll * nthreads) {
      uint4 r[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) r[u] = __ldcs(vs + k + u * nthreads);
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) vd[k + u * nthreads] = r[u];
    }
    for (; k < nvec; k += nthreads) vd[k] = __ldcs(vs + k);
    const int64_t tail = head + (nvec << 4);
    if (blockIdx.x == 0) {
      for (int64_t b = threadIdx.x; b < head; b += blockDim.x) dst[b] = src[b];
      for (int64_t b = tail + threadIdx.x; b < n; b += blockDim.x) dst[b] = src[b];
    }
  } else if (((sa ^ da) & 1u) == 0 && ((sa & 1u) == 0) && (n & 1) == 0) {
    // 16-bit elements whose ends do not share a 16-byte alignment
    const uint16_t* hs = reinterpret_cast<const uint16_t*>(src);
    uint16_t* hd = reinterpret_cast<uint16_t*>(dst);
    for (int64_t k = tid; k < (n >> 1); k += nthreads) hd[k] = hs[k];
  } else {
    for (int64_t k = tid; k < n; k += nthreads) dst[k] = src[k];
  }
}

template <typename OT>
__device__ __forceinline__ OT to16(float x);
template <>
__device__ __forceinline__ __half to16<__half>(float x) {
  return __float2half_rn(x);
}
template <>
__device__ __forceinline__ __nv_bfloat16 to16<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

template <typename OT>
__global__ void __launch_bounds__(kCopyThreads) cast_segments(const __grid_constant__ CopyArgs a) {
  const CopySeg& s = a.segs[blockIdx.y];
  const float* src = static_cast<const float*>(s.src);
  OT* dst = static_cast<OT*>(s.dst);
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < s.count; k += nthreads)
    dst[k] = to16<OT>(src[k]);
}

dim3 grid_for(const CopySeg* segs, int nseg, int64_t per_thread) {
  int64_t longest = 0;
  for (int i = 0; i < nseg; ++i) longest = segs[i].count > longest ? segs[i].count : longest;
  const int64_t total = static_cast<int64_t>(sm_count()) * 8;   // 8 blocks of 256 fill an SM
  int64_t bx = (total + nseg - 1) / nseg;
  const int64_t needed = (longest / per_thread + kCopyThreads) / kCopyThreads;
  if (bx > needed) bx = needed;
  if (bx < 1) bx = 1;
  return dim3(static_cast<unsigned>(bx), static_cast<unsigned>(nseg));
}

__global__ void __launch_bounds__(kCopyThreads) fill16(uint16_t* dst, int64_t n, uint16_t value) {
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t k = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; k < n; k += nthreads) dst[k] = value;
}

}  // namespace

cudaError_t launch_fill16(void* dst, int64_t count, uint16_t value, cudaStream_t stream, int64_t* launches) {
  if (count <= 0) return cudaSuccess;
  int64_t blocks = (count + kCopyThreads - 1) / kCopyThreads;
  const int64_t cap = static_cast<int64_t>(sm_count()) * 8;
  if (blocks > cap) blocks = cap;
  fill16<<<static_cast<unsigned>(blocks), kCopyThreads, 0, stream>>>(static_cast<uint16_t*>(dst), count, value);
  ++*launches;
  return cudaGetLastError();
}

const void* copy_kernel() { return reinterpret_cast<const void*>(copy_segments); }

cudaError_t launch_copy(const CopySeg* segs, int nseg, cudaStream_t stream, int64_t* launches) {
  if (nseg <= 0) return cudaSuccess;
  if (nseg > kMaxCopySegs) return cudaErrorInvalidValue;
  CopyArgs a;
  for (int i = 0; i < nseg; ++i) a.segs[i] = segs[i];
  copy_segments<<<grid_for(segs, nseg, 16 * kCopyUnroll), kCopyThreads, 0, stream>>>(a);
  ++*launches;
  return cudaGetLastError();
}

cudaError_t launch_cast(const CopySeg* segs, int nseg, int work_dtype, cudaStream_t stream, int64_t* launches) {
  if (nseg <= 0) return cudaSuccess;
  if (nseg > kMaxCopySegs) return cudaErrorInvalidValue;
  CopyArgs a;
  for (int i = 0; i < nseg; ++i) a.segs[i] = segs[i];
  const dim3 grid = grid_for(segs, nseg, 4);
  if (work_dtype == kF16)
    cast_segments<__half><<<grid, kCopyThreads, 0, stream>>>(a);
  else
    cast_segments<__nv_bfloat16><<<grid, kCopyThreads, 0, stream>>>(a);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace zero
