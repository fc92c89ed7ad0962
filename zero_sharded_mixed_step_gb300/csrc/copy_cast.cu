// The ZeRO-3 all-gather of one unit, done inside one GPU's memory, and the
// fp32 -> 16-bit recast of the working copy.
//
// Gather ("ZeRO and FSDP", ZeRO-3 and FSDP: every unit's parameters are
// all-gathered before its forward and again before its backward pass): rank
// r's 16-bit shard of unit u, S_u values, lands at [r S_u, (r + 1) S_u) of the
// unit buffer.  One launch copies all W shards, one grid row per shard,
// 16-byte vectors (four per thread in flight, plain loads: the streaming
// hint measured 5% slower and doubled the registers) wherever source and
// destination share their alignment, on a grid of one resident wave; 2
// bytes read and 2 written per element.
//
// All forward gathers of a ZeRO-3 step in one launch (gather_units), for
// steps with nothing to run between them; see launch_gather_units.
//
// Cast: round-to-nearest-even of the fp32 master into the 16-bit copy, used
// when the working copy is (re)built from the master (first step, restored
// state); the step itself recasts inside the fused kernel.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "step_math.cuh"
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
      for (int u = 0; u < kCopyUnroll; ++u) r[u] = vs[k + u * nthreads];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) vd[k + u * nthreads] = r[u];
    }
    for (; k < nvec; k += nthreads) vd[k] = vs[k];
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

// Eight elements per thread: one 32-byte load of fp32 values, eight
// round-to-nearest-even conversions, one 16-byte store, wherever the source
// is 32-byte aligned and the destination 16-byte aligned at the same
// element (elements before the source's first 32-byte boundary, and those
// after the last whole group, one at a time); 4 bytes read and 2 written per
// element.
template <typename OT>
__global__ void __launch_bounds__(kCopyThreads) cast_segments(const __grid_constant__ CopyArgs a) {
  const CopySeg& s = a.segs[blockIdx.y];
  const float* src = static_cast<const float*>(s.src);
  OT* dst = static_cast<OT*>(s.dst);
  const int64_t n = s.count;
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthreads = static_cast<int64_t>(gridDim.x) * blockDim.x;
  const uintptr_t sa = reinterpret_cast<uintptr_t>(src), da = reinterpret_cast<uintptr_t>(dst);
  int64_t head = static_cast<int64_t>(((32u - (sa & 31u)) & 31u) >> 2);
  if (head > n) head = n;
  const bool vec = (sa & 3u) == 0 && ((da + static_cast<uintptr_t>(head) * 2u) & 15u) == 0;
  int64_t done = 0;   // elements [0, done) go through the vector loop, past the head
  if (vec) {
    const int64_t groups = (n - head) >> 3;
    for (int64_t k = tid; k < groups; k += nthreads) {
      float f[8];
      dev::ld_32B(src + head + 8 * k, f);
      dev::st_16B(dst + head + 8 * k, dev::Fmt<OT>::pack8(f));
    }
    done = head + (groups << 3);
  } else {
    head = 0;
  }
  // the head (vector case) and everything after the vector part, one at a time
  for (int64_t k = tid; k < head; k += nthreads) dev::Fmt<OT>::store1(dst, k, src[k]);
  for (int64_t k = (vec ? done : 0) + tid; k < n; k += nthreads) dev::Fmt<OT>::store1(dst, k, src[k]);
}

// ---- every forward gather of a ZeRO-3 step in one launch ------------------------------
//
// Unit u goes into buffer u % 2, as in the schedule that gathers two units
// per launch (units 2k and 2k + 1 are pair k), and every unit has the same
// shard size S.  The launch walks the pairs in order; for each pair every
// CTA copies the same tiles of the two buffers, so each 32-byte position
// of a buffer is always written by the same thread, pair after pair, in unit
// order: the buffers end as they do after the separate launches.  Between
// two writes of one position the whole pair (2 S W values each way) passes
// through the memory system, far more than L2 holds, so every unit's bytes
// reach DRAM as they would launch by launch (2 read and 2 written per
// gathered value); what goes away is the fixed cost of each launch boundary
// (ramp-up and drain, some microseconds each on GB300), which is what kept a
// two-unit launch below the copy rate.
constexpr int kGatherThreads = 256;
constexpr int kGatherVec = 32;     // bytes per access
constexpr int kGatherUnroll = 3;   // accesses in flight per thread

struct UnitGatherArgs {
  const void* shard[kMaxRanks];   // rank r's store; unit u's shard at u * S values
  void* buf[2];
  int64_t units;
  int64_t S;                      // values per rank per unit
  int64_t nvec;                   // 32-byte vectors per rank per unit
  int64_t tiles_per_rank;         // tiles of kGatherThreads * kGatherUnroll vectors per rank slice
  int W;
  int nbuf;
};

__global__ void __launch_bounds__(kGatherThreads) gather_units(const __grid_constant__ UnitGatherArgs g) {
  const int64_t per_buf = static_cast<int64_t>(g.W) * g.tiles_per_rank;
  const int64_t tiles = per_buf * g.nbuf;
  const int64_t unit_bytes = g.S * 2;   // from one unit's shard to the next, in a store
  const int64_t pairs = (g.units + 1) / 2;
  for (int64_t pair = 0; pair < pairs; ++pair) {
    for (int64_t tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
      const int b = static_cast<int>(tile / per_buf);
      const int64_t u = 2 * pair + b;
      if (u >= g.units) continue;   // an odd count: the last pair has no unit for buffer 1
      const int64_t rem = tile - b * per_buf;
      const int r = static_cast<int>(rem / g.tiles_per_rank);
      const int64_t k0 = (rem - r * g.tiles_per_rank) * (kGatherThreads * kGatherUnroll) + threadIdx.x;
      const char* src = static_cast<const char*>(g.shard[r]) + u * unit_bytes;
      char* dst = static_cast<char*>(g.buf[b]) + r * unit_bytes;
      float x[kGatherUnroll][8];
#pragma unroll
      for (int i = 0; i < kGatherUnroll; ++i) {
        const int64_t k = k0 + i * kGatherThreads;
        if (k < g.nvec) dev::ld_32B(reinterpret_cast<const float*>(src + k * kGatherVec), x[i]);
      }
#pragma unroll
      for (int i = 0; i < kGatherUnroll; ++i) {
        const int64_t k = k0 + i * kGatherThreads;
        if (k < g.nvec) dev::st_32B(reinterpret_cast<float*>(dst + k * kGatherVec), x[i]);
      }
    }
  }
}

// Blocks of 256 threads for the segments: as many as fit on the device at
// once (blocks_per_sm per SM), split evenly among the segments, and no more
// than the longest segment needs.
dim3 grid_for(const CopySeg* segs, int nseg, int64_t per_thread, int blocks_per_sm = 8) {
  int64_t longest = 0;
  for (int i = 0; i < nseg; ++i) longest = segs[i].count > longest ? segs[i].count : longest;
  const int64_t total = static_cast<int64_t>(sm_count()) * blocks_per_sm;
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

bool is_gather_kernel(const void* fn) {
  return fn == reinterpret_cast<const void*>(copy_segments) || fn == reinterpret_cast<const void*>(gather_units);
}

bool gather_units_applies(const void* const* shard, int W, void* const* bufs, int64_t units, int64_t S) {
  if (units < 1 || S <= 0 || W < 1 || W > kMaxRanks || (S * 2) % kGatherVec != 0) return false;
  for (int r = 0; r < W; ++r)
    if (shard[r] == nullptr || (reinterpret_cast<uintptr_t>(shard[r]) % kGatherVec) != 0) return false;
  for (int b = 0; b < (units >= 2 ? 2 : 1); ++b)
    if (bufs[b] == nullptr || (reinterpret_cast<uintptr_t>(bufs[b]) % kGatherVec) != 0) return false;
  return true;
}

cudaError_t launch_gather_units(const void* const* shard, int W, void* const* bufs, int64_t units, int64_t S,
                                cudaStream_t stream, int64_t* launches) {
  if (!gather_units_applies(shard, W, bufs, units, S)) return cudaErrorInvalidValue;
  UnitGatherArgs g;
  for (int r = 0; r < W; ++r) g.shard[r] = shard[r];
  g.buf[0] = bufs[0];
  g.buf[1] = units >= 2 ? bufs[1] : nullptr;
  g.units = units;
  g.S = S;
  g.nvec = S * 2 / kGatherVec;
  g.tiles_per_rank = (g.nvec + kGatherThreads * kGatherUnroll - 1) / (kGatherThreads * kGatherUnroll);
  g.W = W;
  g.nbuf = units >= 2 ? 2 : 1;
  // Blocks of 256 threads, between 1.5 and 2 per SM, as many as split each
  // pair's tiles evenly (every block the same number, so that none finishes
  // a tile behind the others pair after pair); two per SM when no count in
  // that range does.  Measured on GB300 over the 24 x 50,331,648-value
  // units (W = 8): 3 accesses of 32 bytes per thread on 256 blocks (32 tiles
  // each per pair) took 704 us; 3 accesses on 304 blocks 735 us, and 2 or 4
  // accesses on 256 to 768 blocks 728-814 us.
  const int64_t total = g.tiles_per_rank * W * g.nbuf;
  const int64_t sms = sm_count();
  int64_t blocks = 0;
  for (int64_t b = 2 * sms; b >= (3 * sms + 1) / 2 && blocks == 0; --b)
    if (total % b == 0) blocks = b;
  if (blocks == 0) blocks = 2 * sms;
  if (blocks > total) blocks = total;
  gather_units<<<static_cast<unsigned>(blocks), kGatherThreads, 0, stream>>>(g);
  ++*launches;
  return cudaGetLastError();
}

cudaError_t launch_copy(const CopySeg* segs, int nseg, cudaStream_t stream, int64_t* launches) {
  if (nseg <= 0) return cudaSuccess;
  if (nseg > kMaxCopySegs) return cudaErrorInvalidValue;
  CopyArgs a;
  for (int i = 0; i < nseg; ++i) a.segs[i] = segs[i];
  // one wave: the blocks that are resident at once on every SM
  int per_sm = 0;
  cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, copy_segments, kCopyThreads, 0);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  copy_segments<<<grid_for(segs, nseg, 16 * kCopyUnroll, per_sm), kCopyThreads, 0, stream>>>(a);
  ++*launches;
  return cudaGetLastError();
}

cudaError_t launch_cast(const CopySeg* segs, int nseg, int work_dtype, cudaStream_t stream, int64_t* launches) {
  if (nseg <= 0) return cudaSuccess;
  if (nseg > kMaxCopySegs) return cudaErrorInvalidValue;
  CopyArgs a;
  for (int i = 0; i < nseg; ++i) a.segs[i] = segs[i];
  const dim3 grid = grid_for(segs, nseg, 8);
  if (work_dtype == kF16)
    cast_segments<__half><<<grid, kCopyThreads, 0, stream>>>(a);
  else
    cast_segments<__nv_bfloat16><<<grid, kCopyThreads, 0, stream>>>(a);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace zero
