// Internal to the host side of the library: the context behind zero_ctx and
// what the files implementing its entry points share (zero_api.cpp,
// host_step.cpp, bucket_step.cpp).  Not part of the ABI.
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdint>
#include <cstdio>
#include <map>
#include <utility>
#include <vector>

#include "zero_internal.h"
#include "zero_step.h"

namespace zero {
namespace host {

// Set the calling thread's zero_last_error() message (printf format); returns code.
int fail(int code, const char* fmt, ...);
int cuda_fail(cudaError_t e, const char* what);

// Return ZERO_E_CUDA, with the call's text in the message, if a CUDA call fails.
#define ZERO_CUDA(call)                                               \
  do {                                                                \
    cudaError_t e_ = (call);                                          \
    if (e_ != cudaSuccess) return ::zero::host::cuda_fail(e_, #call); \
  } while (0)

// NVTX range on the host timeline (a no-op unless a profiler is attached)
struct Range {
  explicit Range(const char* name) { nvtxRangePushA(name); }
  Range(const char* fmt, long long a) {
    char buf[96];
    snprintf(buf, sizeof buf, fmt, a);
    nvtxRangePushA(buf);
  }
  ~Range() { nvtxRangePop(); }
  Range(const Range&) = delete;
  Range& operator=(const Range&) = delete;
};

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// master, m and v are read and written 32 bytes at a time
inline bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline bool valid_scheme(int s) { return s >= ZERO_SCHEME_DP && s <= ZERO_SCHEME_Z3; }
inline bool valid_dtype(int d) { return d == ZERO_FP16 || d == ZERO_BF16; }

// Flat padded layout of the units ("ZeRO and FSDP": even split, zero padding
// to a multiple of W; each unit split on its own for ZeRO-3).
struct Layout {
  std::vector<int64_t> size, off, shard, off16;
  int64_t n = 0, n_pad = 0, shard_total = 0, unit_max = 0;
};

int make_layout(int W, int64_t n_units, const int64_t* sizes, Layout* L);

// Bytes one rank sends in one ring reduce-scatter or all-gather of a unit
// whose shard is S values of 2 bytes: W - 1 chunks ("One Poem Suffices:
// ZeRO", appendix B).
inline int64_t ring_bytes(int W, int64_t S) { return int64_t(W - 1) * S * 2; }

inline int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

}  // namespace host
}  // namespace zero

struct zero_ctx {
  int scheme = 0, W = 0, gdt = 0, wdt = 0;
  zero::host::Layout L;
  float* master = nullptr;
  float* m = nullptr;
  float* v = nullptr;
  void* p16 = nullptr;
  std::vector<void*> shard16;
  void* ubuf[2] = {nullptr, nullptr};
  cudaStream_t su = nullptr, sg = nullptr;
  bool cuda_ready = false;
  cudaEvent_t ev_begin = nullptr, ev_gathered[2] = {nullptr, nullptr}, ev_free[2] = {nullptr, nullptr};
  cudaEvent_t ev_landed[2] = {nullptr, nullptr}, ev_slot_free[2] = {nullptr, nullptr};
  cudaEvent_t ev_updated[2] = {nullptr, nullptr}, ev_out_done = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;   // the two backward chains of a captured step
  cudaStream_t s_alt = nullptr;                       // the second chain's stream (owned)
  bool capturing = false;                             // a ZeRO-3 step is being captured
  std::vector<cudaStream_t> touched;
  int variant = ZERO_VARIANT_AUTO;
  int64_t t = 0;
  int64_t comm = 0, launches = 0, gathers = 0, scatters = 0, live_elems = 0, peak_live = 0;
  std::vector<char> live;
  std::vector<char> rank_up;
  zero_unit_hook hook = nullptr;
  void* hook_user = nullptr;
  bool timing = false;
  bool stall_pending = false;
  int64_t stall_tile = -1;
  int err_slot = 0;            // this context's device error counter slot
  bool err_slot_ready = false; // cleared on the device (at the first fused launch)
  int64_t dev_err_seen = 0;    // count at the last zero_sync
  int last_variant = 0;
  // a step being done bucket by bucket: the ranges covered so far (lo -> hi)
  int debug = 0;
  std::vector<void*> live_buf;          // where the caller gathered each live unit
  std::vector<cudaStream_t> live_stream;
  bool bucket_open = false;
  std::map<int64_t, int64_t> covered;
  int64_t covered_elems = 0;
  std::vector<cudaEvent_t> event_pool;
  std::vector<std::pair<cudaEvent_t, cudaEvent_t>> timed[3];
  // ZeRO-3 steps replayed from a CUDA graph (zero_set_graph): the captured
  // step, its fused-kernel nodes with their launch arguments, and what one
  // step adds to the counters
  bool graph_on = false;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t graph_exec = nullptr;
  std::vector<std::pair<cudaGraphNode_t, zero::FusedLaunch>> graph_fused;
  int64_t graph_comm = 0, graph_launches = 0, graph_gathers = 0, graph_scatters = 0;
};

namespace zero {
namespace host {

// CUDA events of the context, created at its first GPU work.
int ensure_cuda(zero_ctx* c);

// An event from the context's pool (timing brackets).
int take_event(zero_ctx* c, cudaEvent_t* e);

// Timing brackets: an event before and after a launch, on its stream.
struct Bracket {
  zero_ctx* c;
  int kind;
  cudaStream_t s;
  cudaEvent_t a = nullptr, b = nullptr;
  int open() {
    if (!c->timing) return ZERO_OK;
    int rc = take_event(c, &a);
    if (rc == ZERO_OK) rc = take_event(c, &b);
    if (rc) return rc;
    ZERO_CUDA(cudaEventRecord(a, s));
    return ZERO_OK;
  }
  int close() {
    if (!c->timing) return ZERO_OK;
    ZERO_CUDA(cudaEventRecord(b, s));
    c->timed[kind].push_back({a, b});
    return ZERO_OK;
  }
};

// Remember a stream the context has enqueued work on (zero_sync waits on all of them).
void touch(zero_ctx* c, cudaStream_t s);

// Argument and state checks shared by the step entry points.
int check_ranks_up(const zero_ctx* c);
int check_grads(const zero_ctx* c, const void* const* grads);
int check_no_open_bucket_step(const zero_ctx* c);
int check_hyper(double lr, double b1, double b2, double eps, int64_t t);

// The fp32 coefficients of Adam step t.
AdamCoef make_coef(double lr, double b1, double b2, double eps, int64_t t, int W);

// The fused pass over unit u (or, for DP/Z1/Z2, [lo, lo + len) of the flat
// vector; len < 0: all of it); with gather_dst set (ZeRO-3), the pass first
// copies the unit's current 16-bit shards into gather_dst: its gather.
int launch_update(zero_ctx* c, int64_t u, const void* const* grads, const AdamCoef& coef, cudaStream_t stream,
                  void* gather_dst = nullptr, int64_t lo = 0, int64_t len = -1);

// Gather unit u's 16-bit shards into dst, in flat order; launch_gathers does
// `count` units (each into its own buffer) in one launch.
int launch_gather(zero_ctx* c, int64_t u, void* dst, cudaStream_t stream);
int launch_gathers(zero_ctx* c, const int64_t* units, void* const* dsts, int count, cudaStream_t stream);

// Counters: gathers, reduce-scatters and traffic, gathered elements live.
void count_gather(zero_ctx* c, int64_t u);
void count_scatter(zero_ctx* c, int64_t u);
void live_add(zero_ctx* c, int64_t elems);

}  // namespace host
}  // namespace zero
