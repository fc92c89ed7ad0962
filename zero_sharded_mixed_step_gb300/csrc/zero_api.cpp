// Host side of libzero_gb300: argument checks, layout and accounting, the
// context, and the ZeRO-3 unit scheduler that drives the kernels on CUDA
// streams.  The step fed from host memory is in host_step.cpp and the
// bucketed step in bucket_step.cpp.  See include/zero_step.h for the
// contract of every entry point.

#include "zero_step.h"

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include "zero_context.h"
#include "zero_internal.h"

static_assert(ZERO_MAX_RANKS == zero::kMaxRanks, "rank limit must match the kernels'");

namespace {

thread_local std::string g_last_error;

}  // namespace

namespace zero {
namespace host {

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(ZERO_E_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

int make_layout(int W, int64_t n_units, const int64_t* sizes, Layout* L) {
  if (W < 1 || W > ZERO_MAX_RANKS) return fail(ZERO_E_ARG, "W=%d outside [1, %d]", W, ZERO_MAX_RANKS);
  if (n_units < 1 || sizes == nullptr) return fail(ZERO_E_ARG, "need at least one unit");
  if (n_units > (int64_t(1) << 24)) return fail(ZERO_E_ARG, "too many units (%lld)", (long long)n_units);
  L->size.assign(sizes, sizes + n_units);
  int64_t pos = 0, pos16 = 0;
  for (int64_t u = 0; u < n_units; ++u) {
    if (sizes[u] < 0) return fail(ZERO_E_ARG, "unit %lld has negative size", (long long)u);
    if (sizes[u] > (int64_t(1) << 46)) return fail(ZERO_E_ARG, "unit %lld too large", (long long)u);
    const int64_t s = ceil_div(sizes[u], W);
    L->off.push_back(pos);
    L->shard.push_back(s);
    L->off16.push_back(pos16);
    pos += s * W;
    pos16 += s;
    L->n += sizes[u];
    if (s * W > L->unit_max) L->unit_max = s * W;
  }
  L->n_pad = pos;
  L->shard_total = pos16;
  return ZERO_OK;
}

int ensure_cuda(zero_ctx* c) {
  if (c->cuda_ready) return ZERO_OK;
  ZERO_CUDA(cudaEventCreateWithFlags(&c->ev_begin, cudaEventDisableTiming));
  for (int b = 0; b < 2; ++b) {
    ZERO_CUDA(cudaEventCreateWithFlags(&c->ev_gathered[b], cudaEventDisableTiming));
    ZERO_CUDA(cudaEventCreateWithFlags(&c->ev_free[b], cudaEventDisableTiming));
    ZERO_CUDA(cudaEventCreateWithFlags(&c->ev_landed[b], cudaEventDisableTiming));
    ZERO_CUDA(cudaEventCreateWithFlags(&c->ev_slot_free[b], cudaEventDisableTiming));
    ZERO_CUDA(cudaEventCreateWithFlags(&c->ev_updated[b], cudaEventDisableTiming));
  }
  ZERO_CUDA(cudaEventCreateWithFlags(&c->ev_out_done, cudaEventDisableTiming));
  ZERO_CUDA(cudaEventCreateWithFlags(&c->ev_fork, cudaEventDisableTiming));
  ZERO_CUDA(cudaEventCreateWithFlags(&c->ev_join, cudaEventDisableTiming));
  c->cuda_ready = true;
  return ZERO_OK;
}

int take_event(zero_ctx* c, cudaEvent_t* e) {
  if (!c->event_pool.empty()) {
    *e = c->event_pool.back();
    c->event_pool.pop_back();
    return ZERO_OK;
  }
  ZERO_CUDA(cudaEventCreate(e));
  return ZERO_OK;
}

void touch(zero_ctx* c, cudaStream_t s) {
  for (cudaStream_t x : c->touched)
    if (x == s) return;
  c->touched.push_back(s);
}

int check_ranks_up(const zero_ctx* c) {
  for (int r = 0; r < c->W; ++r)
    if (!c->rank_up[r]) return fail(ZERO_E_RANK, "simulated rank %d is unavailable", r);
  return ZERO_OK;
}

int check_grads(const zero_ctx* c, const void* const* grads) {
  if (grads == nullptr) return fail(ZERO_E_ARG, "grads is NULL");
  for (int w = 0; w < c->W; ++w) {
    if (grads[w] == nullptr && c->L.n_pad > 0) return fail(ZERO_E_ARG, "gradient pointer of rank %d is NULL", w);
    if (!aligned16(grads[w])) return fail(ZERO_E_ALIGN, "gradient pointer of rank %d is not 16-byte aligned", w);
  }
  return ZERO_OK;
}

// A step done bucket by bucket must be complete before any other step starts.
int check_no_open_bucket_step(const zero_ctx* c) {
  if (c->bucket_open)
    return fail(ZERO_E_STATE, "step %lld is being done bucket by bucket and %lld of %lld elements are still missing",
                (long long)c->t, (long long)(c->L.n_pad - c->covered_elems), (long long)c->L.n_pad);
  return ZERO_OK;
}

int check_hyper(double lr, double b1, double b2, double eps, int64_t t) {
  if (!std::isfinite(lr) || lr < 0) return fail(ZERO_E_ARG, "lr must be finite and >= 0");
  if (!(b1 >= 0 && b1 < 1) || !(b2 >= 0 && b2 < 1)) return fail(ZERO_E_ARG, "betas must lie in [0, 1)");
  if (!std::isfinite(eps) || !(eps > 0)) return fail(ZERO_E_ARG, "eps must be finite and > 0");
  if (t < 1) return fail(ZERO_E_STATE, "the step counter starts at 1 (got %lld)", (long long)t);
  // The update runs in fp32: eps must stay a positive fp32 value (an eps that
  // rounds to 0 makes 0 / 0 of every element without gradient history), and
  // the step size lr / (1 - beta1^t) a finite one (inf times a zero m is NaN).
  const float eps32 = static_cast<float>(eps);
  if (!(eps32 > 0) || !std::isfinite(eps32))
    return fail(ZERO_E_ARG, "eps %g is not a positive finite fp32 value", eps);
  const double step_size = lr / (1.0 - std::pow(b1, static_cast<double>(t)));
  if (!std::isfinite(static_cast<float>(step_size)))
    return fail(ZERO_E_ARG, "lr / (1 - beta1^t) = %g overflows fp32", step_size);
  return ZERO_OK;
}

zero::AdamCoef make_coef(double lr, double b1, double b2, double eps, int64_t t, int W) {
  const double bc1 = 1.0 - std::pow(b1, static_cast<double>(t));
  const double bc2 = 1.0 - std::pow(b2, static_cast<double>(t));
  zero::AdamCoef c;
  c.b1 = static_cast<float>(b1);
  c.omb1 = static_cast<float>(1.0 - b1);
  c.b2 = static_cast<float>(b2);
  c.omb2 = static_cast<float>(1.0 - b2);
  c.step_size = static_cast<float>(lr / bc1);
  c.rsqrt_bc2 = static_cast<float>(1.0 / std::sqrt(bc2));
  c.eps = static_cast<float>(eps);
  c.inv_w = static_cast<float>(1.0 / W);
  return c;
}

// The fused pass over unit u (or, for DP/Z1/Z2, the whole vector).  With
// gather_dst set (ZeRO-3 only), the same pass first copies unit u's current
// 16-bit shards into gather_dst, in flat order: the unit's gather.
// For DP/Z1/Z2, [lo, lo + len) limits the pass to part of the flat vector
// (len < 0: all of it).
int launch_update(zero_ctx* c, int64_t u, const void* const* grads, const zero::AdamCoef& coef,
                  cudaStream_t stream, void* gather_dst, int64_t lo, int64_t len) {
  zero::FusedLaunch a;
  std::memset(&a, 0, sizeof a);
  a.W = c->W;
  a.grad_dtype = c->gdt;
  a.work_dtype = c->wdt;
  for (int w = 0; w < c->W; ++w) a.grads[w] = grads[w];
  a.master = c->master;
  a.m = c->m;
  a.v = c->v;
  a.coef = coef;
  a.variant = c->variant;
  if (c->stall_pending) {
    a.inject_stall = 1;
    a.stall_tile = c->stall_tile;
    c->stall_pending = false;
  }
  a.err_slot = c->err_slot;
  if (!c->err_slot_ready) {
    cudaError_t e0 = zero::reset_device_errors(c->err_slot, stream);
    if (e0 != cudaSuccess) return cuda_fail(e0, "clearing the device error counter");
    c->err_slot_ready = true;
  }
  const int64_t S = c->L.shard[u], off = c->L.off[u];
  if (c->scheme != ZERO_SCHEME_Z3) {
    // one stretch: the recast goes straight to its place in the full vector
    if (len < 0) {
      lo = 0;
      len = c->L.n_pad;
    }
    a.nseg = len > 0 ? 1 : 0;
    a.segs[0] = {lo, len, static_cast<char*>(c->p16) + lo * 2, nullptr};
  } else {
    // rank r's slice of the unit goes to r's own 16-bit shard store
    a.nseg = 0;
    for (int r = 0; r < c->W; ++r) {
      if (S == 0) break;
      char* dst = static_cast<char*>(c->shard16[r]) + c->L.off16[u] * 2;
      void* pre = gather_dst ? static_cast<char*>(gather_dst) + r * S * 2 : nullptr;
      a.segs[a.nseg++] = {off + r * S, S, dst, pre};
    }
  }
  Bracket br{c, ZERO_KERNEL_FUSED, stream};
  int rc = br.open();
  if (rc) return rc;
  cudaError_t e = zero::launch_fused_step(a, stream, &c->launches);
  if (e != cudaSuccess) return cuda_fail(e, "fused reduce-scatter/Adam/recast launch");
  c->last_variant = zero::last_fused_variant();
  touch(c, stream);
  return br.close();
}

int launch_gather(zero_ctx* c, int64_t u, void* dst, cudaStream_t stream) {
  return launch_gathers(c, &u, &dst, 1, stream);
}

int launch_gathers(zero_ctx* c, const int64_t* units, void* const* dsts, int count, cudaStream_t stream) {
  std::vector<zero::CopySeg> segs;
  for (int k = 0; k < count; ++k) {
    const int64_t u = units[k], S = c->L.shard[u];
    for (int r = 0; r < c->W && S > 0; ++r) {
      const char* src = static_cast<const char*>(c->shard16[r]) + c->L.off16[u] * 2;
      segs.push_back({src, static_cast<char*>(dsts[k]) + r * S * 2, S * 2});
    }
  }
  if (segs.empty()) return ZERO_OK;
  Bracket br{c, ZERO_KERNEL_GATHER, stream};
  int rc = br.open();
  if (rc) return rc;
  cudaError_t e = zero::launch_copy(segs.data(), static_cast<int>(segs.size()), stream, &c->launches);
  if (e != cudaSuccess) return cuda_fail(e, "unit gather launch");
  touch(c, stream);
  return br.close();
}

void count_gather(zero_ctx* c, int64_t u) {
  c->gathers += 1;
  c->comm += ring_bytes(c->W, c->L.shard[u]);
}

void count_scatter(zero_ctx* c, int64_t u) {
  c->scatters += 1;
  c->comm += ring_bytes(c->W, c->L.shard[u]);
}

void live_add(zero_ctx* c, int64_t elems) {
  c->live_elems += elems;
  if (c->live_elems > c->peak_live) c->peak_live = c->live_elems;
}

}  // namespace host
}  // namespace zero

using namespace zero::host;

namespace {

constexpr uint16_t kPoison16 = 0x7FFF;   // a NaN in both fp16 and bf16

int64_t resident_bytes(int scheme, int64_t n, int64_t S) {
  // bands: 2 (16-bit weight) + 2 (16-bit gradient) + 12 (fp32 master, m, v)
  const bool so = scheme >= ZERO_SCHEME_Z1, sg = scheme >= ZERO_SCHEME_Z2, sp = scheme >= ZERO_SCHEME_Z3;
  return 2 * (sp ? S : n) + 2 * (sg ? S : n) + 12 * (so ? S : n);
}

// Counter slots for bounded device waits: slot 0 belongs to no context, the
// others are handed to contexts while they live; when all are taken, new
// contexts share the last one.
std::mutex g_slot_mu;
bool g_slot_used[zero::kErrSlots] = {true};

int take_slot() {
  std::lock_guard<std::mutex> lock(g_slot_mu);
  for (int i = 1; i < zero::kErrSlots; ++i)
    if (!g_slot_used[i]) {
      g_slot_used[i] = true;
      return i;
    }
  return zero::kErrSlots - 1;
}

void give_slot(int i) {
  std::lock_guard<std::mutex> lock(g_slot_mu);
  if (i > 0 && i < zero::kErrSlots - 1) g_slot_used[i] = false;
}

int poison_unit(zero_ctx* c, int64_t u, void* buf, cudaStream_t s) {
  if (!(c->debug & ZERO_DEBUG_POISON_RELEASED)) return ZERO_OK;
  cudaError_t e = zero::launch_fill16(buf, c->L.shard[u] * c->W, kPoison16, s, &c->launches);
  if (e != cudaSuccess) return cuda_fail(e, "poisoning a released unit");
  return ZERO_OK;
}

// ZeRO-3 step: forward gathers in unit order, backward gathers in reverse
// order each followed by the unit's update, two gather buffers in turn.  The
// gather of the next unit (stream G) waits only for the buffer it reuses to
// be released by stream A, so it overlaps the current unit's work (the
// prefetch of "ZeRO and FSDP").  That overlap is there to hide a gather
// behind the caller's compute on the unit before it, so it is used when a
// unit hook is registered; with no hook the only work on stream A is the
// memory-bound update, and running the gathers beside it on GB300 measured
// slower than running everything in order on stream A.  Without a hook the
// forward gathers go in one launch when every unit has the same shard size
// (zero::launch_gather_units: pair after pair of units, each buffer position
// receiving its units in unit order), else two units per launch (one into
// each buffer), and each backward gather is done by its unit's update pass.
// A unit counts as live from its gather until its buffer is taken by a later
// gather (or the step ends): at most two units are live.
int run_zero3_step(zero_ctx* c, const void* const* grads, const zero::AdamCoef& coef) {
  int rc = ensure_cuda(c);
  if (rc) return rc;
  cudaStream_t su = c->su;
  const bool two_streams = c->sg != su && c->hook != nullptr;
  cudaStream_t sg = two_streams ? c->sg : su;
  if (two_streams) {
    ZERO_CUDA(cudaEventRecord(c->ev_begin, su));
    ZERO_CUDA(cudaStreamWaitEvent(sg, c->ev_begin, 0));
  }
  const int64_t U = static_cast<int64_t>(c->L.size.size());
  bool used[2] = {false, false};
  int64_t held[2] = {0, 0};
  int64_t seq = 0;
  // the stream of the fused backward pass (without a hook): su, or the
  // second chain of a captured step (see below)
  cudaStream_t s_upd = su;
  auto unit = [&](int64_t u, int phase) -> int {
    Range range(phase == 0 ? "zero3 forward unit %lld" : "zero3 backward unit %lld", static_cast<long long>(u));
    const int b = static_cast<int>(seq++ & 1);
    void* buf = c->ubuf[b];
    if (used[b] && two_streams) ZERO_CUDA(cudaStreamWaitEvent(sg, c->ev_free[b], 0));
    c->live_elems -= held[b];
    held[b] = c->L.shard[u] * c->W;
    live_add(c, held[b]);
    count_gather(c, u);
    int r = ZERO_OK;
    if (phase == 1 && c->hook == nullptr) {
      // nothing runs between this unit's gather and its update, so one pass
      // does both: it copies the pre-update 16-bit values out, then updates
      r = launch_update(c, u, grads, coef, s_upd, buf);
      if (r) return r;
      count_scatter(c, u);
      if ((r = poison_unit(c, u, buf, s_upd))) return r;
      used[b] = true;
      return ZERO_OK;
    }
    r = launch_gather(c, u, buf, sg);
    if (r) return r;
    if (two_streams) {
      ZERO_CUDA(cudaEventRecord(c->ev_gathered[b], sg));
      ZERO_CUDA(cudaStreamWaitEvent(su, c->ev_gathered[b], 0));
    }
    if (c->hook) c->hook(c->hook_user, phase, u, buf, static_cast<void*>(su));
    if (phase == 1) {
      r = launch_update(c, u, grads, coef, su);
      if (r) return r;
      count_scatter(c, u);
    }
    if ((r = poison_unit(c, u, buf, su))) return r;
    if (two_streams) ZERO_CUDA(cudaEventRecord(c->ev_free[b], su));
    used[b] = true;
    return ZERO_OK;
  };
  bool equal_units = U > 0 && c->debug == 0;
  for (int64_t u = 1; u < U && equal_units; ++u) equal_units = c->L.shard[u] == c->L.shard[0];
  if (c->hook == nullptr && equal_units &&
      zero::gather_units_applies(c->shard16.data(), c->W, c->ubuf, U, c->L.shard[0])) {
    // Nothing runs between the forward gathers and every unit has the same
    // shard size: all of them in one launch, pair after pair, each buffer
    // position receiving its units in unit order (the buffers end as after
    // the separate launches, and the same bytes move).
    for (int64_t u = 0; u < U; ++u) {
      const int b = static_cast<int>(seq++ & 1);
      c->live_elems -= held[b];
      held[b] = c->L.shard[u] * c->W;
      live_add(c, held[b]);
      count_gather(c, u);
      used[b] = true;
    }
    Range range("zero3 forward units 0..%lld", static_cast<long long>(U - 1));
    Bracket br{c, ZERO_KERNEL_GATHER, su};
    if ((rc = br.open())) return rc;
    const cudaError_t e = zero::launch_gather_units(c->shard16.data(), c->W, c->ubuf, U, c->L.shard[0], su,
                                                    &c->launches);
    if (e != cudaSuccess) return cuda_fail(e, "forward unit gathers launch");
    touch(c, su);
    if ((rc = br.close())) return rc;
  } else if (c->hook == nullptr && 2 * c->W <= zero::kMaxCopySegs) {
    // Nothing runs between the forward gathers, so two units (one into each
    // buffer) go in one launch: the same copies in half the launches.
    for (int64_t u = 0; u < U; u += 2) {
      Range range("zero3 forward units %lld+", static_cast<long long>(u));
      const int count = U - u >= 2 ? 2 : 1;
      int64_t us[2];
      void* dsts[2];
      for (int k = 0; k < count; ++k) {
        const int b = static_cast<int>(seq++ & 1);
        c->live_elems -= held[b];
        held[b] = c->L.shard[u + k] * c->W;
        live_add(c, held[b]);
        count_gather(c, u + k);
        us[k] = u + k;
        dsts[k] = c->ubuf[b];
        used[b] = true;
      }
      if ((rc = launch_gathers(c, us, dsts, count, su))) return rc;
      for (int k = 0; k < count; ++k)
        if ((rc = poison_unit(c, us[k], dsts[k], su))) return rc;
    }
  } else {
    for (int64_t u = 0; u < U; ++u) {
      rc = unit(u, 0);
      if (rc) return rc;
    }
  }
  // Backward.  While a step is being captured (no hook, no poisoning), the
  // fused passes go on two chains: backward units k = 0, 2, 4, ... on su and
  // k = 1, 3, ... on a second stream, both after the forward gathers.  A
  // unit's pass writes only its own range of the state, its shard slots and
  // its unit buffer, and the units that share a buffer (k and k + 2) are on
  // one chain, in order; so the graph orders exactly what must be ordered,
  // and a unit's CTAs can take the SMs that the one before it frees instead
  // of waiting for all of them.
  const bool chains = c->capturing && c->s_alt != nullptr && c->hook == nullptr && c->debug == 0;
  if (chains) {
    ZERO_CUDA(cudaEventRecord(c->ev_fork, su));
    ZERO_CUDA(cudaStreamWaitEvent(c->s_alt, c->ev_fork, 0));
  }
  for (int64_t u = U - 1, k = 0; u >= 0; --u, ++k) {
    s_upd = chains && (k & 1) ? c->s_alt : su;
    if ((rc = unit(u, 1))) break;
  }
  if (chains) {   // joined even after a failed launch, so that the capture ends cleanly
    ZERO_CUDA(cudaEventRecord(c->ev_join, c->s_alt));
    ZERO_CUDA(cudaStreamWaitEvent(su, c->ev_join, 0));
  }
  if (rc) return rc;
  c->live_elems -= held[0] + held[1];
  return ZERO_OK;
}

// ---- ZeRO-3 steps replayed from a CUDA graph ----------------------------------------
//
// A ZeRO-3 step without a hook is a fixed set of launches: the forward
// gathers, then one update per unit (on two chains in the graph, see
// run_zero3_step).  Captured once, it is replayed as one graph launch, which
// saves the launch gaps between its kernels; only the fused kernels' Adam
// coefficients and gradient pointers change from step to step, and they are
// set on the graph's nodes before each replay.

void drop_graph(zero_ctx* c) {
  if (c->graph_exec) cudaGraphExecDestroy(c->graph_exec);
  if (c->graph) cudaGraphDestroy(c->graph);
  c->graph_exec = nullptr;
  c->graph = nullptr;
  c->graph_fused.clear();
}

// Whether this step may run from the graph: anything that adds or changes
// work (a hook, timing brackets, poisoning, an injected stall) runs the
// ordinary launches instead.
bool graph_applies(const zero_ctx* c) {
  return c->graph_on && c->scheme == ZERO_SCHEME_Z3 && c->hook == nullptr && !c->timing && c->debug == 0 &&
         !c->stall_pending;
}

// Capture one step's launches into c->graph (nothing runs) and remember what
// the step adds to the counters.
int capture_zero3(zero_ctx* c, const void* const* grads, const zero::AdamCoef& coef) {
  int rc = ensure_cuda(c);
  if (rc) return rc;
  if (!c->err_slot_ready) {   // the counter reset stays outside the graph
    const cudaError_t e0 = zero::reset_device_errors(c->err_slot, c->su);
    if (e0 != cudaSuccess) return cuda_fail(e0, "clearing the device error counter");
    c->err_slot_ready = true;
  }
  // the stream of the second backward chain (created once, outside the capture)
  if (c->s_alt == nullptr) ZERO_CUDA(cudaStreamCreateWithFlags(&c->s_alt, cudaStreamNonBlocking));
  const int64_t comm = c->comm, launches = c->launches, gathers = c->gathers, scatters = c->scatters;
  const int64_t live = c->live_elems, peak = c->peak_live;
  ZERO_CUDA(cudaStreamBeginCapture(c->su, cudaStreamCaptureModeThreadLocal));
  c->capturing = true;
  rc = run_zero3_step(c, grads, coef);
  c->capturing = false;
  cudaGraph_t g = nullptr;
  const cudaError_t e = cudaStreamEndCapture(c->su, &g);
  c->graph_comm = c->comm - comm;
  c->graph_launches = c->launches - launches;
  c->graph_gathers = c->gathers - gathers;
  c->graph_scatters = c->scatters - scatters;
  c->comm = comm;               // the captured work has not run yet
  c->launches = launches;
  c->gathers = gathers;
  c->scatters = scatters;
  if (rc || e != cudaSuccess) {
    // a step that failed part way leaves the unit counters as they were
    c->live_elems = live;
    c->peak_live = peak;
    if (g) cudaGraphDestroy(g);
    return rc ? rc : cuda_fail(e, "capturing the ZeRO-3 step");
  }
  c->graph = g;
  size_t count = 0;
  cudaError_t e1 = cudaGraphGetNodes(g, nullptr, &count);
  std::vector<cudaGraphNode_t> nodes(count);
  if (e1 == cudaSuccess && count) e1 = cudaGraphGetNodes(g, nodes.data(), &count);
  for (size_t k = 0; e1 == cudaSuccess && k < count; ++k) {
    cudaGraphNodeType type;
    e1 = cudaGraphNodeGetType(nodes[k], &type);
    if (e1 != cudaSuccess || type != cudaGraphNodeTypeKernel) continue;
    cudaKernelNodeParams p;
    e1 = cudaGraphKernelNodeGetParams(nodes[k], &p);
    if (e1 == cudaSuccess && !zero::is_gather_kernel(p.func))
      c->graph_fused.emplace_back(nodes[k], *static_cast<const zero::FusedLaunch*>(p.kernelParams[0]));
  }
  if (e1 == cudaSuccess) e1 = cudaGraphInstantiate(&c->graph_exec, g, 0);
  if (e1 != cudaSuccess) {
    drop_graph(c);
    return cuda_fail(e1, "building the ZeRO-3 step graph");
  }
  int64_t updates = 0;
  for (int64_t u = 0; u < static_cast<int64_t>(c->L.size.size()); ++u) updates += c->L.shard[u] > 0;
  if (static_cast<int64_t>(c->graph_fused.size()) != updates) {
    drop_graph(c);
    return fail(ZERO_E_CUDA, "the captured ZeRO-3 step has %zu update launches, expected %lld",
                c->graph_fused.size(), static_cast<long long>(updates));
  }
  return ZERO_OK;
}

// One step from the graph: this step's coefficients and gradients on the
// fused nodes, then one graph launch on the update stream.
int replay_zero3(zero_ctx* c, const void* const* grads, const zero::AdamCoef& coef) {
  for (auto& node : c->graph_fused) {
    zero::FusedLaunch a = node.second;
    a.coef = coef;
    for (int w = 0; w < c->W; ++w) a.grads[w] = grads[w];
    cudaKernelNodeParams p;
    ZERO_CUDA(cudaGraphKernelNodeGetParams(node.first, &p));
    void* args[] = {&a};
    p.kernelParams = args;
    p.extra = nullptr;
    ZERO_CUDA(cudaGraphExecKernelNodeSetParams(c->graph_exec, node.first, &p));
  }
  ZERO_CUDA(cudaGraphLaunch(c->graph_exec, c->su));
  c->comm += c->graph_comm;
  c->launches += c->graph_launches;
  c->gathers += c->graph_gathers;
  c->scatters += c->graph_scatters;
  touch(c, c->su);
  return ZERO_OK;
}

}  // namespace

int zero::record_error(int code, const char* msg) { return fail(code, "%s", msg); }

int zero::check_adam_args(double lr, double beta1, double beta2, double eps, int64_t t) {
  return check_hyper(lr, beta1, beta2, eps, t);
}

zero::AdamCoef zero::adam_coef(double lr, double beta1, double beta2, double eps, int64_t t, int W) {
  return make_coef(lr, beta1, beta2, eps, t, W);
}

extern "C" {

const char* zero_last_error(void) { return g_last_error.c_str(); }

int zero_buffer_sizes(int scheme, int W, int64_t n_units, const int64_t* unit_sizes, int64_t* out) {
  if (!valid_scheme(scheme)) return fail(ZERO_E_ARG, "scheme %d is not one of DP/Z1/Z2/Z3", scheme);
  if (out == nullptr) return fail(ZERO_E_ARG, "out is NULL");
  if (scheme != ZERO_SCHEME_Z3 && n_units != 1)
    return fail(ZERO_E_ARG, "data parallel, ZeRO-1 and ZeRO-2 take exactly one unit");
  Layout L;
  int rc = make_layout(W, n_units, unit_sizes, &L);
  if (rc) return rc;
  const bool z3 = scheme == ZERO_SCHEME_Z3;
  out[0] = L.n;
  out[1] = L.n_pad;
  out[2] = z3 ? 0 : L.n_pad;
  out[3] = z3 ? L.shard_total : 0;
  out[4] = z3 ? L.unit_max : 0;
  out[5] = n_units;
  return ZERO_OK;
}

int zero_layout(int W, int64_t n_units, const int64_t* unit_sizes, int64_t* off, int64_t* shard, int64_t* off16) {
  Layout L;
  int rc = make_layout(W, n_units, unit_sizes, &L);
  if (rc) return rc;
  for (int64_t u = 0; u < n_units; ++u) {
    if (off) off[u] = L.off[u];
    if (shard) shard[u] = L.shard[u];
    if (off16) off16[u] = L.off16[u];
  }
  return ZERO_OK;
}

int64_t zero_bytes_per_rank(int scheme, int64_t n, int W, int kind, int64_t gathered_elems) {
  if (!valid_scheme(scheme)) return fail(ZERO_E_ARG, "scheme %d is not one of DP/Z1/Z2/Z3", scheme);
  if (W < 1 || n < 0 || gathered_elems < 0) return fail(ZERO_E_ARG, "need W >= 1, n >= 0, gathered >= 0");
  if (kind != ZERO_RESIDENT && kind != ZERO_PEAK) return fail(ZERO_E_ARG, "kind must be resident or peak");
  if (n > (int64_t(1) << 58) / 16) return fail(ZERO_E_ARG, "n too large");
  const int64_t S = ceil_div(n, W);
  int64_t b = resident_bytes(scheme, n, S);
  if (kind == ZERO_PEAK && scheme == ZERO_SCHEME_Z3) b += 2 * gathered_elems;
  return b;
}

int64_t zero_comm_bytes_closed_form(int scheme, int64_t n, int W) {
  if (!valid_scheme(scheme)) return fail(ZERO_E_ARG, "scheme %d is not one of DP/Z1/Z2/Z3", scheme);
  if (W < 1 || n < 0) return fail(ZERO_E_ARG, "need W >= 1 and n >= 0");
  if (n > (int64_t(1) << 58) / 16) return fail(ZERO_E_ARG, "n too large");
  const int64_t k = scheme == ZERO_SCHEME_Z3 ? 3 : 2;
  return k * ring_bytes(W, ceil_div(n, W));
}

int zero_init(zero_ctx** out, int scheme, int W, int64_t n, int64_t n_units, const int64_t* unit_sizes,
              int grad_dtype, int work_dtype, float* master, float* m, float* v, void* p16,
              void* const* shard16, void* const* unit_bufs, void* stream_update, void* stream_gather) {
  if (out == nullptr) return fail(ZERO_E_ARG, "out is NULL");
  *out = nullptr;
  if (!valid_scheme(scheme)) return fail(ZERO_E_ARG, "scheme %d is not one of DP/Z1/Z2/Z3", scheme);
  if (!valid_dtype(grad_dtype) || !valid_dtype(work_dtype))
    return fail(ZERO_E_ARG, "16-bit formats must be ZERO_FP16 or ZERO_BF16");
  if (scheme != ZERO_SCHEME_Z3 && n_units != 1)
    return fail(ZERO_E_ARG, "data parallel, ZeRO-1 and ZeRO-2 take exactly one unit");
  Layout L;
  int rc = make_layout(W, n_units, unit_sizes, &L);
  if (rc) return rc;
  if (L.n != n) return fail(ZERO_E_ARG, "unit sizes add up to %lld, not n=%lld", (long long)L.n, (long long)n);
  // empty buffers (nothing to hold) may be NULL
  const bool any = L.n_pad > 0;
  if (any && (!master || !m || !v)) return fail(ZERO_E_ARG, "master, m and v are required");
  if (!aligned32(master) || !aligned32(m) || !aligned32(v))
    return fail(ZERO_E_ALIGN, "master, m and v must be 32-byte aligned");
  auto* c = new zero_ctx();
  c->scheme = scheme;
  c->W = W;
  c->gdt = grad_dtype;
  c->wdt = work_dtype;
  c->L = L;
  c->master = master;
  c->m = m;
  c->v = v;
  if (scheme == ZERO_SCHEME_Z3) {
    if (p16 != nullptr) {
      delete c;
      return fail(ZERO_E_ARG, "ZeRO-3 keeps no full 16-bit copy: p16 must be NULL");
    }
    if (shard16 == nullptr || unit_bufs == nullptr) {
      delete c;
      return fail(ZERO_E_ARG, "ZeRO-3 needs shard16 (W pointers) and unit_bufs (2 pointers)");
    }
    for (int r = 0; r < W; ++r) {
      if ((shard16[r] == nullptr && L.shard_total > 0) || !aligned16(shard16[r])) {
        delete c;
        return fail(shard16[r] ? ZERO_E_ALIGN : ZERO_E_ARG, "16-bit shard store of rank %d is NULL or unaligned", r);
      }
      c->shard16.push_back(shard16[r]);
    }
    for (int b = 0; b < 2; ++b) {
      if ((unit_bufs[b] == nullptr && L.unit_max > 0) || !aligned16(unit_bufs[b])) {
        delete c;
        return fail(unit_bufs[b] ? ZERO_E_ALIGN : ZERO_E_ARG, "unit buffer %d is NULL or unaligned", b);
      }
      c->ubuf[b] = unit_bufs[b];
    }
  } else {
    if ((p16 == nullptr && any) || !aligned16(p16)) {
      delete c;
      return fail(p16 ? ZERO_E_ALIGN : ZERO_E_ARG, "p16 is NULL or not 16-byte aligned");
    }
    if (shard16 != nullptr || unit_bufs != nullptr) {
      delete c;
      return fail(ZERO_E_ARG, "shard16 and unit_bufs are for ZeRO-3 only");
    }
    c->p16 = p16;
  }
  c->su = static_cast<cudaStream_t>(stream_update);
  c->sg = stream_gather ? static_cast<cudaStream_t>(stream_gather) : c->su;
  c->live.assign(static_cast<size_t>(n_units), 0);
  c->live_buf.assign(static_cast<size_t>(n_units), nullptr);
  c->live_stream.assign(static_cast<size_t>(n_units), nullptr);
  c->rank_up.assign(static_cast<size_t>(W), 1);
  c->err_slot = take_slot();
  *out = c;
  return ZERO_OK;
}

int zero_destroy(zero_ctx* c) {
  if (c == nullptr) return ZERO_OK;
  int rc = ZERO_OK;
  if (!c->touched.empty()) rc = zero_sync(c, -1);
  for (auto& list : c->timed)
    for (auto& pr : list) {
      cudaEventDestroy(pr.first);
      cudaEventDestroy(pr.second);
    }
  for (cudaEvent_t e : c->event_pool) cudaEventDestroy(e);
  drop_graph(c);
  give_slot(c->err_slot);
  if (c->cuda_ready) {
    cudaEventDestroy(c->ev_begin);
    for (int b = 0; b < 2; ++b) {
      cudaEventDestroy(c->ev_gathered[b]);
      cudaEventDestroy(c->ev_free[b]);
      cudaEventDestroy(c->ev_landed[b]);
      cudaEventDestroy(c->ev_slot_free[b]);
      cudaEventDestroy(c->ev_updated[b]);
    }
    cudaEventDestroy(c->ev_out_done);
    cudaEventDestroy(c->ev_fork);
    cudaEventDestroy(c->ev_join);
  }
  if (c->s_alt) cudaStreamDestroy(c->s_alt);
  delete c;
  return rc;
}

int zero_refresh_working_copy(zero_ctx* c) {
  if (c == nullptr) return fail(ZERO_E_ARG, "ctx is NULL");
  std::vector<zero::CopySeg> segs;
  if (c->scheme != ZERO_SCHEME_Z3) {
    if (c->L.n_pad > 0) segs.push_back({c->master, c->p16, c->L.n_pad});
    Bracket br{c, ZERO_KERNEL_CAST, c->su};
    int rc = br.open();
    if (rc) return rc;
    cudaError_t e = zero::launch_cast(segs.data(), static_cast<int>(segs.size()), c->wdt, c->su, &c->launches);
    if (e != cudaSuccess) return cuda_fail(e, "working-copy cast launch");
    if ((rc = br.close())) return rc;
  } else {
    for (size_t u = 0; u < c->L.size.size(); ++u) {
      segs.clear();
      const int64_t S = c->L.shard[u];
      for (int r = 0; r < c->W && S > 0; ++r)
        segs.push_back({c->master + c->L.off[u] + r * S, static_cast<char*>(c->shard16[r]) + c->L.off16[u] * 2, S});
      if (segs.empty()) continue;
      Bracket br{c, ZERO_KERNEL_CAST, c->su};
      int rc = br.open();
      if (rc) return rc;
      cudaError_t e = zero::launch_cast(segs.data(), static_cast<int>(segs.size()), c->wdt, c->su, &c->launches);
      if (e != cudaSuccess) return cuda_fail(e, "shard cast launch");
      if ((rc = br.close())) return rc;
    }
  }
  touch(c, c->su);
  return ZERO_OK;
}

int zero_step(zero_ctx* c, int scheme, int W, int64_t n, const void* const* grads, double lr, double beta1,
              double beta2, double eps, int64_t t) {
  if (c == nullptr) return fail(ZERO_E_ARG, "ctx is NULL");
  if (scheme != c->scheme || W != c->W || n != c->L.n)
    return fail(ZERO_E_ARG, "scheme/W/n (%d/%d/%lld) differ from the context's (%d/%d/%lld)", scheme, W,
                (long long)n, c->scheme, c->W, (long long)c->L.n);
  int rc = check_hyper(lr, beta1, beta2, eps, t);
  if (rc) return rc;
  if (t != c->t + 1)
    return fail(ZERO_E_STATE, "step counter %lld does not follow %lld", (long long)t, (long long)c->t);
  if ((rc = check_no_open_bucket_step(c))) return rc;
  if ((rc = check_grads(c, grads)) || (rc = check_ranks_up(c))) return rc;
  for (size_t u = 0; u < c->live.size(); ++u)
    if (c->live[u]) return fail(ZERO_E_STATE, "unit %zu is still gathered by the caller", u);
  const zero::AdamCoef coef = make_coef(lr, beta1, beta2, eps, t, W);
  Range range("zero_step %lld", static_cast<long long>(t));
  if (c->scheme != ZERO_SCHEME_Z3) {
    rc = launch_update(c, 0, grads, coef, c->su);
    if (rc) return rc;
    // all-reduce (DP) or reduce-scatter + all-gather (Z1/Z2): two collectives
    count_scatter(c, 0);
    c->gathers += 1;
    c->comm += ring_bytes(c->W, c->L.shard[0]);
  } else if (graph_applies(c)) {
    if (!c->graph_exec && (rc = capture_zero3(c, grads, coef))) return rc;
    if ((rc = replay_zero3(c, grads, coef))) return rc;
  } else {
    rc = run_zero3_step(c, grads, coef);
    if (rc) return rc;
  }
  c->t = t;
  return ZERO_OK;
}

int zero_set_unit_hook(zero_ctx* c, zero_unit_hook fn, void* user) {
  if (c == nullptr) return fail(ZERO_E_ARG, "ctx is NULL");
  c->hook = fn;
  c->hook_user = fn ? user : nullptr;
  return ZERO_OK;
}

int zero_gather_unit(zero_ctx* c, int64_t unit, void* dst, void* stream) {
  if (c == nullptr) return fail(ZERO_E_ARG, "ctx is NULL");
  if (c->scheme != ZERO_SCHEME_Z3) return fail(ZERO_E_ARG, "only ZeRO-3 gathers units");
  if (unit < 0 || unit >= static_cast<int64_t>(c->L.size.size()))
    return fail(ZERO_E_ARG, "unit %lld out of range", (long long)unit);
  if (dst == nullptr || !aligned16(dst)) return fail(dst ? ZERO_E_ALIGN : ZERO_E_ARG, "dst is NULL or unaligned");
  int rc = check_ranks_up(c);
  if (rc) return rc;
  if (c->live[unit]) return fail(ZERO_E_STATE, "unit %lld is already gathered; release it first", (long long)unit);
  cudaStream_t s = stream ? static_cast<cudaStream_t>(stream) : c->sg;
  rc = launch_gather(c, unit, dst, s);
  if (rc) return rc;
  c->live[unit] = 1;
  c->live_buf[unit] = dst;
  c->live_stream[unit] = s;
  live_add(c, c->L.shard[unit] * c->W);
  count_gather(c, unit);
  return ZERO_OK;
}

int zero_release_unit(zero_ctx* c, int64_t unit) {
  if (c == nullptr) return fail(ZERO_E_ARG, "ctx is NULL");
  if (c->scheme != ZERO_SCHEME_Z3) return fail(ZERO_E_ARG, "only ZeRO-3 releases units");
  if (unit < 0 || unit >= static_cast<int64_t>(c->L.size.size()))
    return fail(ZERO_E_ARG, "unit %lld out of range", (long long)unit);
  if (!c->live[unit]) return fail(ZERO_E_STATE, "unit %lld is not gathered", (long long)unit);
  int rc = poison_unit(c, unit, c->live_buf[unit], c->live_stream[unit]);
  if (rc) return rc;
  c->live[unit] = 0;
  c->live_elems -= c->L.shard[unit] * c->W;
  return ZERO_OK;
}

int zero_update_unit(zero_ctx* c, int64_t unit, const void* const* grads, double lr, double beta1, double beta2,
                     double eps, int64_t t, void* stream) {
  if (c == nullptr) return fail(ZERO_E_ARG, "ctx is NULL");
  if (c->scheme != ZERO_SCHEME_Z3) return fail(ZERO_E_ARG, "zero_update_unit is for ZeRO-3; use zero_step");
  if (unit < 0 || unit >= static_cast<int64_t>(c->L.size.size()))
    return fail(ZERO_E_ARG, "unit %lld out of range", (long long)unit);
  int rc = check_hyper(lr, beta1, beta2, eps, t);
  if (rc) return rc;
  if (t != c->t && t != c->t + 1)
    return fail(ZERO_E_STATE, "step counter %lld is neither %lld nor the next", (long long)t, (long long)c->t);
  if ((rc = check_grads(c, grads)) || (rc = check_ranks_up(c))) return rc;
  cudaStream_t s = stream ? static_cast<cudaStream_t>(stream) : c->su;
  rc = launch_update(c, unit, grads, make_coef(lr, beta1, beta2, eps, t, c->W), s);
  if (rc) return rc;
  count_scatter(c, unit);
  c->t = t;
  return ZERO_OK;
}

int zero_get_state(zero_ctx* c, float* master, float* m, float* v, int64_t* t) {
  if (c == nullptr) return fail(ZERO_E_ARG, "ctx is NULL");
  int rc = zero_sync(c, -1);
  if (rc) return rc;
  const size_t bytes = static_cast<size_t>(c->L.n_pad) * sizeof(float);
  if (master) ZERO_CUDA(cudaMemcpyAsync(master, c->master, bytes, cudaMemcpyDefault, c->su));
  if (m) ZERO_CUDA(cudaMemcpyAsync(m, c->m, bytes, cudaMemcpyDefault, c->su));
  if (v) ZERO_CUDA(cudaMemcpyAsync(v, c->v, bytes, cudaMemcpyDefault, c->su));
  ZERO_CUDA(cudaStreamSynchronize(c->su));
  if (t) *t = c->t;
  return ZERO_OK;
}

int zero_set_state(zero_ctx* c, const float* master, const float* m, const float* v, int64_t t) {
  if (c == nullptr) return fail(ZERO_E_ARG, "ctx is NULL");
  if (int rb = check_no_open_bucket_step(c)) return rb;
  if (!master || !m || !v) return fail(ZERO_E_ARG, "master, m and v are required");
  if (t < 0) return fail(ZERO_E_ARG, "step counter must be >= 0");
  int rc = zero_sync(c, -1);
  if (rc) return rc;
  const size_t bytes = static_cast<size_t>(c->L.n_pad) * sizeof(float);
  ZERO_CUDA(cudaMemcpyAsync(c->master, master, bytes, cudaMemcpyDefault, c->su));
  ZERO_CUDA(cudaMemcpyAsync(c->m, m, bytes, cudaMemcpyDefault, c->su));
  ZERO_CUDA(cudaMemcpyAsync(c->v, v, bytes, cudaMemcpyDefault, c->su));
  rc = zero_refresh_working_copy(c);
  if (rc) return rc;
  ZERO_CUDA(cudaStreamSynchronize(c->su));
  c->t = t;
  return ZERO_OK;
}

int64_t zero_comm_bytes_per_rank(const zero_ctx* c) {
  if (c == nullptr) return fail(ZERO_E_ARG, "ctx is NULL");
  return c->comm;
}

int64_t zero_stat(const zero_ctx* c, int which) {
  if (c == nullptr) return fail(ZERO_E_ARG, "ctx is NULL");
  switch (which) {
    case ZERO_STAT_COMM_BYTES: return c->comm;
    case ZERO_STAT_LAUNCHES: return c->launches;
    case ZERO_STAT_GATHERS: return c->gathers;
    case ZERO_STAT_SCATTERS: return c->scatters;
    case ZERO_STAT_LIVE_ELEMS: return c->live_elems;
    case ZERO_STAT_PEAK_LIVE_ELEMS: return c->peak_live;
    case ZERO_STAT_T: return c->t;
    case ZERO_STAT_DEVICE_ERRORS: {
      if (!c->err_slot_ready) return 0;
      unsigned int n = 0;
      cudaError_t e = zero::read_device_errors(c->err_slot, &n);
      if (e != cudaSuccess) return cuda_fail(e, "reading the device error counter");
      return static_cast<int64_t>(n);
    }
    case ZERO_STAT_LAST_VARIANT: return c->last_variant;
    default: return fail(ZERO_E_ARG, "unknown statistic %d", which);
  }
}

int zero_sync(zero_ctx* c, int timeout_ms) {
  if (c == nullptr) return fail(ZERO_E_ARG, "ctx is NULL");
  if (c->touched.empty()) return ZERO_OK;
  std::vector<cudaEvent_t> evs;
  for (cudaStream_t s : c->touched) {
    cudaEvent_t e = nullptr;
    cudaError_t err = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
    if (err == cudaSuccess) err = cudaEventRecord(e, s);
    if (err != cudaSuccess) {
      if (e) cudaEventDestroy(e);
      for (cudaEvent_t x : evs) cudaEventDestroy(x);
      return cuda_fail(err, "recording a completion event");
    }
    evs.push_back(e);
  }
  const auto deadline = std::chrono::steady_clock::now() + std::chrono::milliseconds(timeout_ms < 0 ? 0 : timeout_ms);
  int rc = ZERO_OK;
  for (cudaEvent_t e : evs) {
    for (;;) {
      cudaError_t q = cudaEventQuery(e);
      if (q == cudaSuccess) break;
      if (q != cudaErrorNotReady) {
        rc = cuda_fail(q, "work enqueued by the context failed");
        break;
      }
      if (timeout_ms >= 0 && std::chrono::steady_clock::now() >= deadline) {
        rc = fail(ZERO_E_TIMEOUT, "work still running after %d ms", timeout_ms);
        break;
      }
      std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
    if (rc) break;
  }
  for (cudaEvent_t e : evs) cudaEventDestroy(e);
  if (rc) return rc;
  if (!c->err_slot_ready) return ZERO_OK;   // nothing of ours has run a bounded wait
  unsigned int nerr = 0;
  cudaError_t e = zero::read_device_errors(c->err_slot, &nerr);
  if (e != cudaSuccess) return cuda_fail(e, "reading the device error counter");
  if (static_cast<int64_t>(nerr) > c->dev_err_seen) {
    const int64_t fresh = static_cast<int64_t>(nerr) - c->dev_err_seen;
    c->dev_err_seen = nerr;
    return fail(ZERO_E_STATE, "%lld bounded device waits gave up; the work they belonged to is incomplete",
                (long long)fresh);
  }
  return ZERO_OK;
}

int zero_enable_timing(zero_ctx* c, int on) {
  if (c == nullptr) return fail(ZERO_E_ARG, "ctx is NULL");
  c->timing = on != 0;
  return ZERO_OK;
}

int zero_read_timing(zero_ctx* c, int kernel, double* total_ms, int64_t* launches) {
  if (c == nullptr) return fail(ZERO_E_ARG, "ctx is NULL");
  if (kernel < ZERO_KERNEL_FUSED || kernel > ZERO_KERNEL_CAST) return fail(ZERO_E_ARG, "unknown kernel %d", kernel);
  double sum = 0.0;
  int64_t count = 0;
  auto& list = c->timed[kernel];
  for (auto& pr : list) {
    ZERO_CUDA(cudaEventSynchronize(pr.second));
    float ms = 0.f;
    ZERO_CUDA(cudaEventElapsedTime(&ms, pr.first, pr.second));
    sum += ms;
    ++count;
  }
  for (auto& pr : list) {
    c->event_pool.push_back(pr.first);
    c->event_pool.push_back(pr.second);
  }
  list.clear();
  if (total_ms) *total_ms = sum;
  if (launches) *launches = count;
  return ZERO_OK;
}

int zero_set_variant(zero_ctx* c, int variant) {
  if (c == nullptr) return fail(ZERO_E_ARG, "ctx is NULL");
  if (variant != ZERO_VARIANT_AUTO && variant != ZERO_VARIANT_VECTOR && variant != ZERO_VARIANT_BULK)
    return fail(ZERO_E_ARG, "unknown variant %d", variant);
  if (variant != c->variant) drop_graph(c);   // the captured launches used the old choice
  c->variant = variant;
  return ZERO_OK;
}

int zero_set_graph(zero_ctx* c, int on) {
  if (c == nullptr) return fail(ZERO_E_ARG, "ctx is NULL");
  if (on && c->scheme != ZERO_SCHEME_Z3)
    return fail(ZERO_E_ARG, "only ZeRO-3 steps launch more than one kernel; there is nothing to capture");
  if (on && c->su == nullptr)
    return fail(ZERO_E_ARG, "graph capture needs a created update stream, not the legacy default stream");
  c->graph_on = on != 0;
  if (!c->graph_on) drop_graph(c);
  return ZERO_OK;
}

int zero_set_debug(zero_ctx* c, int flags) {
  if (c == nullptr) return fail(ZERO_E_ARG, "ctx is NULL");
  if (flags & ~ZERO_DEBUG_POISON_RELEASED) return fail(ZERO_E_ARG, "unknown debug flags %d", flags);
  c->debug = flags;
  return ZERO_OK;
}

int zero_inject_stall(zero_ctx* c, int64_t tile) {
  if (c == nullptr) return fail(ZERO_E_ARG, "ctx is NULL");
  c->stall_pending = tile >= 0;
  c->stall_tile = tile;
  return ZERO_OK;
}

int zero_mark_rank(zero_ctx* c, int rank, int available) {
  if (c == nullptr) return fail(ZERO_E_ARG, "ctx is NULL");
  if (rank < 0 || rank >= c->W) return fail(ZERO_E_ARG, "rank %d out of range", rank);
  c->rank_up[rank] = available ? 1 : 0;
  return ZERO_OK;
}

}  // extern "C"
