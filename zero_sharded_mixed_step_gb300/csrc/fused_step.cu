// Fused reduce-scatter + Adam + recast over a flat parameter vector.
//
// For every element i of a segment of the flat vector:
//   g     = (G_0[i] + G_1[i] + ... + G_{W-1}[i]) / W     (ranks in order, fp32)
//   m[i]  = b1 m[i] + (1 - b1) g
//   v[i]  = b2 v[i] + (1 - b2) g g
//   th[i] = th[i] - (lr / (1 - b1^t)) m[i] / (sqrt(v[i]) / sqrt(1 - b2^t) + eps)
//   out   = round_to_nearest_even_16bit(th[i])
// which is, for the rank that owns i, the mean reduce-scatter, the
// bias-corrected Adam update and the recast of the 16-bit working copy
// ("The four schemes", Zero From Scratch lab: reduce_scatter_mean, Base._adam
// and the fp16 recast after the all-gather; "ZeRO and FSDP": ZeroAdam.step).
// Writing `out` straight to its slot of the full 16-bit vector is the
// all-gather; for ZeRO-3 the slot is the owning rank's 16-bit shard.
//
// The pass is HBM-bound: per element it reads 2 W + 12 bytes and writes 14,
// at about one flop per byte, with no contraction anywhere.  Each thread
// handles groups of 8 consecutive elements: W 16-byte gradient loads, one
// 32-byte load each of master, m and v (Blackwell's 256-bit global access),
// all issued before any arithmetic; the same widths for the stores.
//
// The grid is persistent and grid-strides.  How many threads each SM keeps
// resident matters more than anything else here: measured on GB300, DRAM
// throughput peaks sharply at 512 resident threads per SM for W <= 8 and at
// 640 for W = 16 (about 5% above both fewer threads, which leave latency
// exposed, and the full 1024, which overloads the memory system with
// requests).  Blocks are 128 threads so the count can be set finely (and
// the kernel carries no minimum-blocks bound: asking the compiler for one
// changed its register allocation and cost 6%).  Plain
// (default-policy) loads and stores measured 3-5% faster than the same
// accesses with the streaming (.cs) hint.
//
// The arithmetic uses explicit round-to-nearest intrinsics (no contraction
// left to the compiler) so that every scheme and every launch shape gives
// bit-identical results.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>
#include <mutex>

#include "zero_internal.h"

namespace zero {

// Bounded device-side waits that gave up (none in the vector variant).
__device__ unsigned int g_wait_timeouts = 0;

namespace {

constexpr int kThreads = 128;

// Resident threads per SM that measured fastest for each rank count.
int threads_per_sm(int W) { return W >= 16 ? 640 : 512; }

// ---- wide global accesses -----------------------------------------------------

__device__ __forceinline__ uint4 ld_16B(const void* p) {
  uint4 r;
  asm volatile("ld.global.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

__device__ __forceinline__ void ld_32B(const float* p, float (&a)[8]) {
  asm volatile("ld.global.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=f"(a[0]), "=f"(a[1]), "=f"(a[2]), "=f"(a[3]), "=f"(a[4]), "=f"(a[5]), "=f"(a[6]),
                 "=f"(a[7])
               : "l"(p));
}

__device__ __forceinline__ void st_32B(float* p, const float (&a)[8]) {
  asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "f"(a[0]), "f"(a[1]), "f"(a[2]),
               "f"(a[3]), "f"(a[4]), "f"(a[5]), "f"(a[6]), "f"(a[7])
               : "memory");
}

__device__ __forceinline__ void st_16B(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// ---- 16-bit formats ----------------------------------------------------------

template <typename T>
struct Fmt;

template <>
struct Fmt<__half> {
  static __device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
    const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 t = __half22float2(h[k]);
      f[2 * k] = t.x;
      f[2 * k + 1] = t.y;
    }
  }
  static __device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint4 u;
    __half2* h = reinterpret_cast<__half2*>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) h[k] = __floats2half2_rn(f[2 * k], f[2 * k + 1]);
    return u;
  }
  static __device__ __forceinline__ float load1(const void* p, int64_t i) {
    return __half2float(static_cast<const __half*>(p)[i]);
  }
  static __device__ __forceinline__ void store1(void* p, int64_t i, float x) {
    static_cast<__half*>(p)[i] = __float2half_rn(x);
  }
};

template <>
struct Fmt<__nv_bfloat16> {
  static __device__ __forceinline__ void unpack8(const uint4& u, float (&f)[8]) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 t = __bfloat1622float2(h[k]);
      f[2 * k] = t.x;
      f[2 * k + 1] = t.y;
    }
  }
  static __device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    uint4 u;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) h[k] = __floats2bfloat162_rn(f[2 * k], f[2 * k + 1]);
    return u;
  }
  static __device__ __forceinline__ float load1(const void* p, int64_t i) {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  }
  static __device__ __forceinline__ void store1(void* p, int64_t i, float x) {
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(x);
  }
};

// ---- the element update (shared by every path) ------------------------------

// Mean of the rank sum: W a power of two divides exactly by multiplying.
__device__ __forceinline__ float rank_mean(float sum, int W, float inv_w, bool pow2) {
  return pow2 ? __fmul_rn(sum, inv_w) : __fdiv_rn(sum, static_cast<float>(W));
}

__device__ __forceinline__ void adam_element(float g, float& th, float& m, float& v, const AdamCoef& c) {
  m = __fmaf_rn(c.b1, m, __fmul_rn(c.omb1, g));
  v = __fmaf_rn(c.b2, v, __fmul_rn(__fmul_rn(c.omb2, g), g));
  const float den = __fmaf_rn(__fsqrt_rn(v), c.rsqrt_bc2, c.eps);
  th = __fsub_rn(th, __fdiv_rn(__fmul_rn(c.step_size, m), den));
}

// ---- scalar path: segment heads and tails not covering a full group ---------

template <typename GT, typename OT, bool PRE>
__device__ void scalar_elements(const FusedLaunch& a, const Seg& seg, int64_t e_lo, int64_t e_hi, bool pow2) {
  for (int64_t e = e_lo + threadIdx.x; e < e_hi; e += blockDim.x) {
    if (PRE) static_cast<uint16_t*>(seg.pre_out)[e - seg.lo] = static_cast<const uint16_t*>(seg.out)[e - seg.lo];
    float sum = Fmt<GT>::load1(a.grads[0], e);
    for (int w = 1; w < a.W; ++w) sum = __fadd_rn(sum, Fmt<GT>::load1(a.grads[w], e));
    const float g = rank_mean(sum, a.W, a.coef.inv_w, pow2);
    float th = a.master[e], m = a.m[e], v = a.v[e];
    adam_element(g, th, m, v, a.coef);
    a.master[e] = th;
    a.m[e] = m;
    a.v[e] = v;
    Fmt<OT>::store1(seg.out, e - seg.lo, th);
  }
}

// ---- the vector kernel ---------------------------------------------------------

// WC > 0: W known at compile time (all W gradient loads in flight at once);
// WC == 0: any W, gradients read in batches of 8 ranks.  PRE: every segment
// also copies its old 16-bit values to pre_out before overwriting them.
template <typename GT, typename OT, int WC, bool PRE>
__global__ void __launch_bounds__(kThreads) fused_step_vector(const __grid_constant__ FusedLaunch a) {
  const Seg& seg = a.segs[blockIdx.y];
  const int W = WC > 0 ? WC : a.W;
  const bool pow2 = (W & (W - 1)) == 0;
  const int64_t lo = seg.lo, hi = seg.lo + seg.len;
  const int64_t g_begin = (lo + 7) >> 3;   // first whole group of 8 inside [lo, hi)
  const int64_t g_end = hi >> 3;           // one past the last whole group
  // Whether the 16-bit destination of a whole group is 16-byte aligned (the
  // same for every group of the segment).
  const bool out_vec = ((reinterpret_cast<uintptr_t>(seg.out) - static_cast<uintptr_t>(lo) * 2u) & 15u) == 0;
  OT* const out = static_cast<OT*>(seg.out);
  const bool pre_vec =
      PRE && out_vec && ((reinterpret_cast<uintptr_t>(seg.pre_out) - static_cast<uintptr_t>(lo) * 2u) & 15u) == 0;

  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t g = g_begin + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; g < g_end;
       g += stride) {
    const int64_t i = g << 3;
    float sum[8], th[8], m[8], v[8];
    if constexpr (WC > 0) {
      uint4 raw[WC];
#pragma unroll
      for (int w = 0; w < WC; ++w) raw[w] = ld_16B(static_cast<const GT*>(a.grads[w]) + i);
      ld_32B(a.master + i, th);
      ld_32B(a.m + i, m);
      ld_32B(a.v + i, v);
      Fmt<GT>::unpack8(raw[0], sum);
#pragma unroll
      for (int w = 1; w < WC; ++w) {
        float f[8];
        Fmt<GT>::unpack8(raw[w], f);
#pragma unroll
        for (int k = 0; k < 8; ++k) sum[k] = __fadd_rn(sum[k], f[k]);
      }
    } else {
      ld_32B(a.master + i, th);
      ld_32B(a.m + i, m);
      ld_32B(a.v + i, v);
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
    if (PRE) {
      // the gather of this unit: its 16-bit values as they are before the update
      if (pre_vec) {
        st_16B(static_cast<uint16_t*>(seg.pre_out) + (i - lo), ld_16B(out + (i - lo)));
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k)
          static_cast<uint16_t*>(seg.pre_out)[i - lo + k] = reinterpret_cast<const uint16_t*>(out)[i - lo + k];
      }
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float gk = rank_mean(sum[k], W, a.coef.inv_w, pow2);
      adam_element(gk, th[k], m[k], v[k], a.coef);
    }
    st_32B(a.master + i, th);
    st_32B(a.m + i, m);
    st_32B(a.v + i, v);
    if (out_vec) {
      st_16B(out + (i - lo), Fmt<OT>::pack8(th));
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) Fmt<OT>::store1(out, i - lo + k, th[k]);
    }
  }

  if (blockIdx.x == 0) {
    if (g_begin >= g_end) {
      scalar_elements<GT, OT, PRE>(a, seg, lo, hi, pow2);
    } else {
      scalar_elements<GT, OT, PRE>(a, seg, lo, g_begin << 3, pow2);
      scalar_elements<GT, OT, PRE>(a, seg, g_end << 3, hi, pow2);
    }
  }
}

using KernelFn = void (*)(const FusedLaunch);

template <typename GT, typename OT, bool PRE>
KernelFn pick_w(int W) {
  switch (W) {
    case 1: return fused_step_vector<GT, OT, 1, PRE>;
    case 2: return fused_step_vector<GT, OT, 2, PRE>;
    case 4: return fused_step_vector<GT, OT, 4, PRE>;
    case 8: return fused_step_vector<GT, OT, 8, PRE>;
    case 16: return fused_step_vector<GT, OT, 16, PRE>;
    default: return fused_step_vector<GT, OT, 0, PRE>;
  }
}

template <bool PRE>
KernelFn pick_t(int gdt, int wdt, int W) {
  if (gdt == kF16) return wdt == kF16 ? pick_w<__half, __half, PRE>(W) : pick_w<__half, __nv_bfloat16, PRE>(W);
  return wdt == kF16 ? pick_w<__nv_bfloat16, __half, PRE>(W) : pick_w<__nv_bfloat16, __nv_bfloat16, PRE>(W);
}

KernelFn pick(int gdt, int wdt, int W, bool pre) { return pre ? pick_t<true>(gdt, wdt, W) : pick_t<false>(gdt, wdt, W); }

}  // namespace

int sm_count() {
  static int count = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev);
    if (count <= 0) count = 1;
  });
  return count;
}

cudaError_t launch_fused_step(const FusedLaunch& a, cudaStream_t stream, int64_t* launches) {
  if (a.nseg <= 0) return cudaSuccess;
  // every segment copies its old values, or none does
  const bool pre = a.segs[0].pre_out != nullptr;
  for (int s = 1; s < a.nseg; ++s)
    if ((a.segs[s].pre_out != nullptr) != pre) return cudaErrorInvalidValue;
  const KernelFn fn = pick(a.grad_dtype, a.work_dtype, a.W, pre);
  int per_sm = 0;
  cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, 0);
  if (err != cudaSuccess) return err;
  const int wanted = threads_per_sm(a.W) / kThreads;
  if (per_sm > wanted) per_sm = wanted;
  if (per_sm < 1) per_sm = 1;
  int64_t max_groups = 0;
  for (int s = 0; s < a.nseg; ++s) max_groups = a.segs[s].len / 8 + 1 > max_groups ? a.segs[s].len / 8 + 1 : max_groups;
  // a persistent grid: every SM full, the segments sharing it evenly
  int64_t bx = (static_cast<int64_t>(sm_count()) * per_sm + a.nseg - 1) / a.nseg;
  const int64_t needed = (max_groups + kThreads - 1) / kThreads;
  if (bx > needed) bx = needed;
  if (bx < 1) bx = 1;
  dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(a.nseg));
  fn<<<grid, kThreads, 0, stream>>>(a);
  ++*launches;
  return cudaGetLastError();
}

cudaError_t read_device_errors(unsigned int* out) {
  return cudaMemcpyFromSymbol(out, g_wait_timeouts, sizeof(unsigned int));
}

}  // namespace zero
