// Device-side building blocks shared by the step kernels: wide global
// accesses, the two 16-bit formats, and the element update (mean of the rank
// sum, bias-corrected Adam) in explicit round-to-nearest operations, so that
// every kernel that includes this computes bit-identical results.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "zero_internal.h"

namespace zero {
namespace dev {

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

}  // namespace dev
}  // namespace zero
