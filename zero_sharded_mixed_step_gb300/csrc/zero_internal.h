// Internal interface between the host side of the library (zero_api.cpp)
// and its CUDA kernels (fused_step.cu, copy_cast.cu).  Not part of the ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace zero {

constexpr int kMaxRanks = 64;     // simulated ranks per context
constexpr int kMaxSegs = 64;      // output segments per fused launch (one per rank at most)
constexpr int kMaxCopySegs = 64;  // segments per copy / cast launch

enum Dtype : int { kF16 = 0, kBF16 = 1 };

// fp32 coefficients of one Adam step, derived on the host in fp64 from
// (lr, beta1, beta2, eps, t) and rounded once each:
//   m <- b1 m + omb1 g;  v <- b2 v + omb2 g g;
//   theta <- theta - step_size m / (sqrt(v) rsqrt_bc2 + eps)
// with step_size = lr / (1 - beta1^t) and rsqrt_bc2 = 1 / sqrt(1 - beta2^t),
// which is the bias-corrected update theta - lr m_hat / (sqrt(v_hat) + eps).
struct AdamCoef {
  float b1, omb1, b2, omb2, step_size, rsqrt_bc2, eps, inv_w;
};

// One contiguous stretch of the flat vector whose 16-bit results go to one
// contiguous destination: elements [lo, lo + len) of master / m / v and of
// every rank's gradient vector; out points at the 16-bit slot of element lo.
// When pre_out is set, the 16-bit value held at out before the update is
// first copied to pre_out (the ZeRO-3 backward gather of the same unit).
struct Seg {
  int64_t lo;
  int64_t len;
  void* out;
  void* pre_out;
};

struct FusedLaunch {
  int W;
  int grad_dtype, work_dtype;
  const void* grads[kMaxRanks];   // rank w's gradient vector (flat, 16-bit)
  float* master;
  float* m;
  float* v;
  Seg segs[kMaxSegs];
  int nseg;
  AdamCoef coef;
  int variant;                    // ZERO_VARIANT_*
  // Testing the bounded waits: with inject_stall set, the bulk-staged kernel's
  // first CTA never loads its tile number stall_tile, so its wait runs out.
  int inject_stall;
  int64_t stall_tile;
  // Counter slot that bounded waits which give up increment (0: no context).
  int err_slot;
};

// Device-side counters of bounded waits that gave up, one slot per context.
constexpr int kErrSlots = 1024;

// Which fused kernel a launch used (ZERO_VARIANT_VECTOR or ZERO_VARIANT_BULK).
int last_fused_variant();

// The rank-ordered fp32 mean of the W ranks' 16-bit gradients over
// elements [lo, lo + len) of the flat vector, written to out[0, len).
// lo must be a multiple of 8 and out 32-byte aligned.
struct MeanLaunch {
  int W;
  int grad_dtype;
  const void* grads[kMaxRanks];
  int64_t lo, len;
  float* out;
  float inv_w;
};

cudaError_t launch_rank_mean(const MeanLaunch& a, cudaStream_t stream, int64_t* launches);

// A byte range to copy, or a float range to cast.
struct CopySeg {
  const void* src;
  void* dst;
  int64_t count;                  // bytes (copy) or elements (cast)
};

// Fused reduce-scatter + Adam + recast over the given segments.
// Returns the CUDA error of the launch; *launches counts kernels started.
cudaError_t launch_fused_step(const FusedLaunch& a, cudaStream_t stream, int64_t* launches);

// Gather: copy each segment's bytes (16-byte vectors where both ends allow).
cudaError_t launch_copy(const CopySeg* segs, int nseg, cudaStream_t stream, int64_t* launches);

// Whether a kernel function is one of the gather kernels (to tell the nodes
// of a captured graph apart from the fused kernels').
bool is_gather_kernel(const void* fn);

// Every forward gather of a ZeRO-3 step in one launch: unit u (of `units`,
// each with shard size S, unit u's shard at u * S in every rank's store)
// into bufs[u % 2].  Applies (gather_units_applies) when S * 2 is a multiple
// of 32 bytes and the stores and buffers are 32-byte aligned; otherwise the
// launch returns cudaErrorInvalidValue.
bool gather_units_applies(const void* const* shard, int W, void* const* bufs, int64_t units, int64_t S);
cudaError_t launch_gather_units(const void* const* shard, int W, void* const* bufs, int64_t units, int64_t S,
                                cudaStream_t stream, int64_t* launches);

// Fill count 16-bit values with `value` (debug poisoning of released units).
cudaError_t launch_fill16(void* dst, int64_t count, uint16_t value, cudaStream_t stream, int64_t* launches);

// Cast fp32 -> 16-bit (round to nearest even) for each segment.
cudaError_t launch_cast(const CopySeg* segs, int nseg, int work_dtype, cudaStream_t stream, int64_t* launches);

// Clear a context's counter slot, in order on `stream` (asynchronous).
cudaError_t reset_device_errors(int slot, cudaStream_t stream);

// Read a counter slot (synchronous; call after the work has finished).
cudaError_t read_device_errors(int slot, unsigned int* out);

// Streaming multiprocessors of the current device.
int sm_count();

// Set the calling thread's zero_last_error() message; returns code.
int record_error(int code, const char* msg);

// Check Adam's hyper-parameters and the step counter t >= 1; on failure
// records the message and returns ZERO_E_ARG or ZERO_E_STATE.
int check_adam_args(double lr, double beta1, double beta2, double eps, int64_t t);

// The fp32 coefficients of Adam step t for W ranks, derived in fp64.
AdamCoef adam_coef(double lr, double beta1, double beta2, double eps, int64_t t, int W);

}  // namespace zero
