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

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "step_math.cuh"
#include "zero_internal.h"
#include "zero_step.h"

namespace zero {

// Bounded device-side waits that gave up, per context slot (only the
// bulk-staged kernel waits on the device).
__device__ unsigned int g_wait_timeouts[kErrSlots];

namespace {

using namespace dev;

constexpr int kThreads = 128;

// Resident threads per SM that measured fastest for each rank count.
int threads_per_sm(int W) { return W >= 16 ? 640 : 512; }

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

// ---- one group of 8 elements through registers ---------------------------------

// Loads of the group at flat index i: the W ranks' gradients summed in rank
// order, and master, m, v.  WC > 0: W known at compile time (all W gradient
// loads in flight at once); WC == 0: any W, read 8 ranks at a time.
template <typename GT, int WC>
__device__ __forceinline__ void load_group(const FusedLaunch& a, int64_t i, int W, float (&sum)[8], float (&th)[8],
                                           float (&m)[8], float (&v)[8]) {
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
}

// The rest of a group once its inputs are in registers: the optional copy
// of the old 16-bit values (PRE), the mean, Adam, and the stores.
template <typename OT, bool PRE>
__device__ __forceinline__ void finish_group(const FusedLaunch& a, const Seg& seg, int64_t i, int W, bool pow2,
                                             bool out_vec, bool pre_vec, float (&sum)[8], float (&th)[8],
                                             float (&m)[8], float (&v)[8]) {
  OT* const out = static_cast<OT*>(seg.out);
  const int64_t j = i - seg.lo;
  if (PRE) {
    // the gather of this unit: its 16-bit values as they are before the update
    if (pre_vec) {
      st_16B(static_cast<uint16_t*>(seg.pre_out) + j, ld_16B(out + j));
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k)
        static_cast<uint16_t*>(seg.pre_out)[j + k] = reinterpret_cast<const uint16_t*>(out)[j + k];
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
    st_16B(out + j, Fmt<OT>::pack8(th));
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) Fmt<OT>::store1(out, j + k, th[k]);
  }
}

// Whether the 16-bit destinations of whole groups of a segment are 16-byte
// aligned (the same for every group of the segment).
__device__ __forceinline__ bool vec16(const void* p, int64_t lo) {
  return ((reinterpret_cast<uintptr_t>(p) - static_cast<uintptr_t>(lo) * 2u) & 15u) == 0;
}

// Groups [g0, g1) of a segment, strided over `threads` threads starting at
// `first`, then the scalar head [lo, head_end) and tail [tail_begin, hi) by
// the caller's choice.
template <typename GT, typename OT, int WC, bool PRE>
__device__ __forceinline__ void groups_through_registers(const FusedLaunch& a, const Seg& seg, int64_t g0, int64_t g1,
                                                         int64_t first, int64_t threads, int W, bool pow2) {
  const bool out_vec = vec16(seg.out, seg.lo);
  const bool pre_vec = PRE && out_vec && vec16(seg.pre_out, seg.lo);
  for (int64_t g = g0 + first; g < g1; g += threads) {
    const int64_t i = g << 3;
    float sum[8], th[8], m[8], v[8];
    load_group<GT, WC>(a, i, W, sum, th, m, v);
    finish_group<OT, PRE>(a, seg, i, W, pow2, out_vec, pre_vec, sum, th, m, v);
  }
}

// ---- the vector kernel -------------------------------------------------------------

// PRE: every segment also copies its old 16-bit values to pre_out before
// overwriting them.
template <typename GT, typename OT, int WC, bool PRE>
__global__ void __launch_bounds__(kThreads) fused_step_vector(const __grid_constant__ FusedLaunch a) {
  const Seg& seg = a.segs[blockIdx.y];
  const int W = WC > 0 ? WC : a.W;
  const bool pow2 = (W & (W - 1)) == 0;
  const int64_t lo = seg.lo, hi = seg.lo + seg.len;
  const int64_t g_begin = (lo + 7) >> 3;   // first whole group of 8 inside [lo, hi)
  const int64_t g_end = hi >> 3;           // one past the last whole group
  groups_through_registers<GT, OT, WC, PRE>(a, seg, g_begin, g_end,
                                            static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x,
                                            static_cast<int64_t>(gridDim.x) * blockDim.x, W, pow2);
  if (blockIdx.x == 0) {
    if (g_begin >= g_end) {
      scalar_elements<GT, OT, PRE>(a, seg, lo, hi, pow2);
    } else {
      scalar_elements<GT, OT, PRE>(a, seg, lo, g_begin << 3, pow2);
      scalar_elements<GT, OT, PRE>(a, seg, g_end << 3, hi, pow2);
    }
  }
}

// ---- the bulk-staged kernel ---------------------------------------------------------
//
// The same pass with every input stream staged through shared memory by the
// Tensor Memory Accelerator's 1-D bulk copies (cp.async.bulk, completion on
// an mbarrier): one persistent CTA per SM, tiles of kTile elements, a ring of
// kStages stages.  Thread 0 issues the W + 3 bulk copies of tile k + 1 while
// all threads compute tile k from shared memory and store the results with
// 256-bit global stores.  The streams are contiguous, so the 1-D form needs
// no tensor map.  Measured on GB300 this moves 1-1.5% more bytes per second
// than the register version at its best occupancy (two stages of 2048
// elements beat three or four, and one CTA per SM beats two).
//
// Every wait is bounded: a stage that has not landed after ~2^31 SM cycles
// (about a second; a real wait is microseconds) makes the CTA count a device
// error, wait (again bounded) for the copies it issued, and return.

constexpr int kTile = 2048;
constexpr int kStages = 2;
constexpr int kBulkThreads = kTile / 8;
constexpr long long kWaitCycles = 1LL << 31;
constexpr int64_t kBulkMinTilesPerCta = 8;

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// false when the phase has not completed within kWaitCycles
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity))
    if (clock64() - t0 > kWaitCycles) return false;
  return true;
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_addr(dst)),
               "l"(src), "r"(bytes), "r"(smem_addr(bar))
               : "memory");
}

// One stage: W gradient tiles, master, m, v, and (PRE) the old 16-bit values.
template <int W, bool PRE>
__host__ __device__ constexpr uint32_t stage_bytes() {
  return static_cast<uint32_t>(W) * kTile * 2 + 3u * kTile * 4 + (PRE ? kTile * 2u : 0u);
}

template <typename GT, typename OT, int W, bool PRE>
__global__ void __launch_bounds__(kBulkThreads) fused_step_bulk(const __grid_constant__ FusedLaunch a) {
  constexpr uint32_t kStageBytes = stage_bytes<W, PRE>();
  constexpr uint32_t kOldOffset = stage_bytes<W, false>();   // where the old 16-bit values land (PRE)
  extern __shared__ __align__(128) unsigned char ring[];
  __shared__ __align__(8) uint64_t full[kStages];
  const Seg& seg = a.segs[blockIdx.y];
  constexpr bool pow2 = (W & (W - 1)) == 0;
  const int64_t lo = seg.lo, hi = seg.lo + seg.len;
  const int64_t body = (lo + 7) & ~int64_t(7);                 // 16-byte aligned start of the tiles
  const int64_t ntiles = hi > body ? (hi - body) / kTile : 0;
  const int tid = threadIdx.x;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&full[s]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // tile j of this CTA's sequence goes to stage j % kStages, phase j / kStages
  auto issue = [&](int64_t j) -> bool {
    const int64_t tile = blockIdx.x + j * gridDim.x;
    if (tile >= ntiles) return false;
    if (a.inject_stall && blockIdx.x == 0 && blockIdx.y == 0 && j == a.stall_tile) return true;   // never loaded
    unsigned char* st = ring + (j % kStages) * kStageBytes;
    uint64_t* bar = &full[j % kStages];
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_expect_tx(bar, kStageBytes);
    const int64_t e0 = body + tile * kTile;
#pragma unroll
    for (int w = 0; w < W; ++w) bulk_load(st + w * kTile * 2, static_cast<const GT*>(a.grads[w]) + e0, kTile * 2, bar);
    bulk_load(st + W * kTile * 2, a.master + e0, kTile * 4, bar);
    bulk_load(st + W * kTile * 2 + kTile * 4, a.m + e0, kTile * 4, bar);
    bulk_load(st + W * kTile * 2 + 2 * kTile * 4, a.v + e0, kTile * 4, bar);
    if (PRE) bulk_load(st + kOldOffset, static_cast<const OT*>(seg.out) + (e0 - lo), kTile * 2, bar);
    return true;
  };

  int64_t issued = 0;
  if (tid == 0)
    for (int64_t j = 0; j < kStages - 1; ++j)
      if (issue(j)) issued = j + 1;
  for (int64_t k = 0;; ++k) {
    const int64_t tile = blockIdx.x + k * gridDim.x;
    if (tile >= ntiles) break;
    if (tid == 0 && issue(k + kStages - 1)) issued = k + kStages;
    const int s = static_cast<int>(k % kStages);
    const bool landed = mbar_wait_bounded(&full[s], static_cast<uint32_t>((k / kStages) & 1));
    if (__syncthreads_or(!landed)) {
      if (tid == 0) {
        atomicAdd(&g_wait_timeouts[a.err_slot], 1u);
        for (int64_t j = k; j < issued; ++j)
          mbar_wait_bounded(&full[j % kStages], static_cast<uint32_t>((j / kStages) & 1));
      }
      __syncthreads();
      return;
    }
    const unsigned char* st = ring + s * kStageBytes;
    const int64_t i = body + tile * kTile + tid * 8;
    float sum[8], th[8], m[8], v[8];
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const uint4 raw = *reinterpret_cast<const uint4*>(st + w * kTile * 2 + tid * 16);
      if (w == 0) {
        Fmt<GT>::unpack8(raw, sum);
      } else {
        float f[8];
        Fmt<GT>::unpack8(raw, f);
#pragma unroll
        for (int q = 0; q < 8; ++q) sum[q] = __fadd_rn(sum[q], f[q]);
      }
    }
    const float4* ps = reinterpret_cast<const float4*>(st + W * kTile * 2 + tid * 32);
    const float4* pm = reinterpret_cast<const float4*>(st + W * kTile * 2 + kTile * 4 + tid * 32);
    const float4* pv = reinterpret_cast<const float4*>(st + W * kTile * 2 + 2 * kTile * 4 + tid * 32);
    const float4 t0 = ps[0], t1 = ps[1], m0 = pm[0], m1 = pm[1], v0 = pv[0], v1 = pv[1];
    th[0] = t0.x; th[1] = t0.y; th[2] = t0.z; th[3] = t0.w; th[4] = t1.x; th[5] = t1.y; th[6] = t1.z; th[7] = t1.w;
    m[0] = m0.x; m[1] = m0.y; m[2] = m0.z; m[3] = m0.w; m[4] = m1.x; m[5] = m1.y; m[6] = m1.z; m[7] = m1.w;
    v[0] = v0.x; v[1] = v0.y; v[2] = v0.z; v[3] = v0.w; v[4] = v1.x; v[5] = v1.y; v[6] = v1.z; v[7] = v1.w;
    if (PRE) {
      // the unit's gather: its old 16-bit values, staged with the rest of the tile
      st_16B(static_cast<uint16_t*>(seg.pre_out) + (i - lo), *reinterpret_cast<const uint4*>(st + kOldOffset + tid * 16));
    }
    // the host launches this kernel only when the segment's 16-bit slots are 16-byte aligned
    finish_group<OT, false>(a, seg, i, W, pow2, true, false, sum, th, m, v);
    __syncthreads();   // every thread is done with stage s before it is refilled
  }

  // what the tiles do not cover: the head up to the aligned start and the
  // tail after the last whole tile, through registers, by the first CTA
  if (blockIdx.x == 0) {
    const int64_t rest = body + ntiles * kTile;
    if (rest < hi) {
      groups_through_registers<GT, OT, W, PRE>(a, seg, rest >> 3, hi >> 3, tid, blockDim.x, W, pow2);
      scalar_elements<GT, OT, PRE>(a, seg, max(rest, hi & ~int64_t(7)), hi, pow2);
    }
    scalar_elements<GT, OT, PRE>(a, seg, lo, min(body, hi), pow2);
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

struct BulkKernel {
  KernelFn fn;
  int smem;
};

template <typename GT, typename OT, bool PRE>
BulkKernel pick_bulk_w(int W) {
  switch (W) {
    case 1: return {fused_step_bulk<GT, OT, 1, PRE>, kStages * static_cast<int>(stage_bytes<1, PRE>())};
    case 2: return {fused_step_bulk<GT, OT, 2, PRE>, kStages * static_cast<int>(stage_bytes<2, PRE>())};
    case 4: return {fused_step_bulk<GT, OT, 4, PRE>, kStages * static_cast<int>(stage_bytes<4, PRE>())};
    case 8: return {fused_step_bulk<GT, OT, 8, PRE>, kStages * static_cast<int>(stage_bytes<8, PRE>())};
    case 16: return {fused_step_bulk<GT, OT, 16, PRE>, kStages * static_cast<int>(stage_bytes<16, PRE>())};
    default: return {nullptr, 0};
  }
}

template <bool PRE>
BulkKernel pick_bulk_t(int gdt, int wdt, int W) {
  if (gdt == kF16) return wdt == kF16 ? pick_bulk_w<__half, __half, PRE>(W) : pick_bulk_w<__half, __nv_bfloat16, PRE>(W);
  return wdt == kF16 ? pick_bulk_w<__nv_bfloat16, __half, PRE>(W) : pick_bulk_w<__nv_bfloat16, __nv_bfloat16, PRE>(W);
}

bool vec16_host(const void* p, int64_t lo) {
  return ((reinterpret_cast<uintptr_t>(p) - static_cast<uintptr_t>(lo) * 2u) & 15u) == 0;
}

thread_local int g_last_variant = ZERO_VARIANT_VECTOR;

}  // namespace

int last_fused_variant() { return g_last_variant; }

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
  int64_t longest = 0;
  bool aligned = true;
  for (int s = 0; s < a.nseg; ++s) {
    if ((a.segs[s].pre_out != nullptr) != pre) return cudaErrorInvalidValue;
    longest = a.segs[s].len > longest ? a.segs[s].len : longest;
    aligned = aligned && vec16_host(a.segs[s].out, a.segs[s].lo) && (!pre || vec16_host(a.segs[s].pre_out, a.segs[s].lo));
  }
  // The bulk-staged kernel needs a compile-time W and 16-byte aligned 16-bit
  // slots.  Left to choose, it is used where it measured no slower: W of 8 or
  // 16 and at least kBulkMinTilesPerCta tiles for each CTA (with fewer, the
  // ring's fill and drain dominate: at 2^20 elements the register kernel
  // took 15 us against 17).
  const BulkKernel bulk = pre ? pick_bulk_t<true>(a.grad_dtype, a.work_dtype, a.W)
                              : pick_bulk_t<false>(a.grad_dtype, a.work_dtype, a.W);
  const bool bulk_ok = bulk.fn != nullptr && aligned && a.variant != ZERO_VARIANT_VECTOR;
  const int64_t bulk_ctas = (static_cast<int64_t>(sm_count()) + a.nseg - 1) / a.nseg;   // one CTA per SM in all
  const int64_t tiles = longest / kTile;
  const bool use_bulk =
      bulk_ok && (a.variant == ZERO_VARIANT_BULK || (a.W >= 8 && tiles >= kBulkMinTilesPerCta * bulk_ctas));
  if (use_bulk) {
    cudaError_t err = cudaFuncSetAttribute(bulk.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bulk.smem);
    if (err != cudaSuccess) return err;
    const int64_t bx = std::max<int64_t>(1, std::min(bulk_ctas, tiles));
    dim3 grid(static_cast<unsigned>(bx), static_cast<unsigned>(a.nseg));
    bulk.fn<<<grid, kBulkThreads, bulk.smem, stream>>>(a);
    ++*launches;
    g_last_variant = ZERO_VARIANT_BULK;
    return cudaGetLastError();
  }
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
  g_last_variant = ZERO_VARIANT_VECTOR;
  return cudaGetLastError();
}

cudaError_t reset_device_errors(int slot, cudaStream_t stream) {
  if (slot < 0 || slot >= kErrSlots) return cudaErrorInvalidValue;
  void* base = nullptr;
  cudaError_t err = cudaGetSymbolAddress(&base, g_wait_timeouts);
  if (err != cudaSuccess) return err;
  return cudaMemsetAsync(static_cast<unsigned int*>(base) + slot, 0, sizeof(unsigned int), stream);
}

cudaError_t read_device_errors(int slot, unsigned int* out) {
  if (slot < 0 || slot >= kErrSlots) return cudaErrorInvalidValue;
  return cudaMemcpyFromSymbol(out, g_wait_timeouts, sizeof(unsigned int), slot * sizeof(unsigned int));
}

}  // namespace zero
