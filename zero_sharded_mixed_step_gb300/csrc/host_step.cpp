// The ZeRO step fed from host memory (zero_step_host): the W ranks'
// gradients cross the host link chunk by chunk (unit by unit for ZeRO-3)
// into a two-slot device staging ring while earlier chunks are updated and
// their 16-bit results return to host memory, on three streams.  The
// staging ring has a constant size, the constant buffers of "One Poem
// Suffices: ZeRO" section 4.2.2.

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <vector>

#include "zero_context.h"
#include "zero_internal.h"
#include "zero_step.h"

using namespace zero::host;

namespace {

// The default chunk: about kDefaultJobs chunks per step, between 2^24 and
// 2^26 elements, in whole multiples of 2^20.  Every chunk costs W copies
// across the host link, and each copy has a fixed cost, so long vectors want
// long chunks; short ones want enough chunks to overlap the copies with the
// updates.  Measured on GB300 with 16 ranks: the 1,557,611,200-element vector
// took 244.1 / 241.9 / 240.7 / 241.1 ms per step at 2^24 / 2^25 / 2^26 /
// 2^27, and the 124,439,808-element one was fastest at 2^24.
constexpr int64_t kDefaultJobs = 24;
constexpr int64_t kMinDefaultChunk = int64_t(1) << 24;
constexpr int64_t kMaxDefaultChunk = int64_t(1) << 26;

int64_t default_chunk(int64_t n_pad) {
  const int64_t c = round_up((n_pad + kDefaultJobs - 1) / kDefaultJobs, int64_t(1) << 20);
  return c < kMinDefaultChunk ? kMinDefaultChunk : (c > kMaxDefaultChunk ? kMaxDefaultChunk : c);
}

// Elements of the largest chunk (DP/Z1/Z2: the chunk, rounded up to 8;
// ZeRO-3: the largest padded unit) and the bytes of one rank's slot.
void staging_geometry(int scheme, int W, const Layout& L, int64_t chunk_elems, int64_t* chunk, int64_t* slot) {
  if (scheme == ZERO_SCHEME_Z3) {
    *chunk = L.unit_max;
  } else {
    *chunk = round_up(chunk_elems > 0 ? chunk_elems : default_chunk(L.n_pad), 8);
  }
  *slot = round_up((*chunk + 8) * 2, 256);
  (void)W;
}

struct HostJob {
  int64_t lo, len, unit;   // flat range; unit for ZeRO-3 (else 0)
};

int run_host_step(zero_ctx* c, const void* const* host_grads, void* host_out, char* staging, int64_t chunk,
                  int64_t slot, const zero::AdamCoef& coef, cudaStream_t sh, cudaStream_t sd) {
  int rc = ensure_cuda(c);
  if (rc) return rc;
  cudaStream_t su = c->su;
  const int W = c->W;
  const bool z3 = c->scheme == ZERO_SCHEME_Z3;
  std::vector<HostJob> jobs;
  if (z3) {
    for (int64_t u = static_cast<int64_t>(c->L.size.size()) - 1; u >= 0; --u)
      jobs.push_back({c->L.off[u], c->L.shard[u] * W, u});
  } else {
    for (int64_t lo = 0; lo < c->L.n_pad; lo += chunk) jobs.push_back({lo, std::min(chunk, c->L.n_pad - lo), 0});
  }
  const int64_t J = static_cast<int64_t>(jobs.size());
  // the staging slots were last read by earlier work on the update stream
  ZERO_CUDA(cudaEventRecord(c->ev_begin, su));
  if (sh != su) ZERO_CUDA(cudaStreamWaitEvent(sh, c->ev_begin, 0));
  if (sd != su) ZERO_CUDA(cudaStreamWaitEvent(sd, c->ev_begin, 0));
  auto slot_base = [&](int64_t k, int w) { return staging + ((k & 1) * W + w) * slot; };
  auto h2d = [&](int64_t k) -> int {
    const HostJob& j = jobs[k];
    if (k >= 2) ZERO_CUDA(cudaStreamWaitEvent(sh, c->ev_slot_free[k & 1], 0));
    const int64_t slack = j.lo & 7;
    for (int w = 0; w < W && j.len > 0; ++w)
      ZERO_CUDA(cudaMemcpyAsync(slot_base(k, w) + slack * 2, static_cast<const char*>(host_grads[w]) + j.lo * 2,
                                static_cast<size_t>(j.len) * 2, cudaMemcpyHostToDevice, sh));
    ZERO_CUDA(cudaEventRecord(c->ev_landed[k & 1], sh));
    return ZERO_OK;
  };
  for (int64_t k = 0; k < std::min<int64_t>(2, J); ++k)
    if ((rc = h2d(k))) return rc;
  touch(c, sh);
  touch(c, sd);

  // ZeRO-3: the forward gathers need no gradients and run while they arrive
  int64_t seq = 0, held[2] = {0, 0};
  if (z3) {
    for (size_t u = 0; u < c->L.size.size(); ++u) {
      const int b = static_cast<int>(seq++ & 1);
      c->live_elems -= held[b];
      held[b] = c->L.shard[u] * W;
      live_add(c, held[b]);
      count_gather(c, static_cast<int64_t>(u));
      if ((rc = launch_gather(c, static_cast<int64_t>(u), c->ubuf[b], su))) return rc;
    }
  }
  for (int64_t k = 0; k < J; ++k) {
    const HostJob& j = jobs[k];
    ZERO_CUDA(cudaStreamWaitEvent(su, c->ev_landed[k & 1], 0));
    const void* g[zero::kMaxRanks];
    for (int w = 0; w < W; ++w) g[w] = slot_base(k, w) + (j.lo & 7) * 2 - j.lo * 2;
    if (z3) {
      const int b = static_cast<int>(seq++ & 1);
      c->live_elems -= held[b];
      held[b] = c->L.shard[j.unit] * W;
      live_add(c, held[b]);
      count_gather(c, j.unit);
      if ((rc = launch_update(c, j.unit, g, coef, su, c->ubuf[b]))) return rc;
      count_scatter(c, j.unit);
    } else {
      if ((rc = launch_update(c, 0, g, coef, su, nullptr, j.lo, j.len))) return rc;
    }
    ZERO_CUDA(cudaEventRecord(c->ev_slot_free[k & 1], su));
    ZERO_CUDA(cudaEventRecord(c->ev_updated[k & 1], su));
    if (host_out != nullptr && j.len > 0) {
      if (sd != su) ZERO_CUDA(cudaStreamWaitEvent(sd, c->ev_updated[k & 1], 0));
      char* out = static_cast<char*>(host_out);
      if (z3) {
        const int64_t S = c->L.shard[j.unit], o16 = c->L.off16[j.unit];
        for (int r = 0; r < W; ++r)
          ZERO_CUDA(cudaMemcpyAsync(out + (r * c->L.shard_total + o16) * 2,
                                    static_cast<const char*>(c->shard16[r]) + o16 * 2, static_cast<size_t>(S) * 2,
                                    cudaMemcpyDeviceToHost, sd));
      } else {
        ZERO_CUDA(cudaMemcpyAsync(out + j.lo * 2, static_cast<const char*>(c->p16) + j.lo * 2,
                                  static_cast<size_t>(j.len) * 2, cudaMemcpyDeviceToHost, sd));
      }
    }
    if (k + 2 < J && (rc = h2d(k + 2))) return rc;
  }
  if (z3) c->live_elems -= held[0] + held[1];
  else {
    // the all-reduce of DP, or the reduce-scatter + all-gather of ZeRO-1/2
    count_scatter(c, 0);
    c->gathers += 1;
    c->comm += ring_bytes(c->W, c->L.shard[0]);
  }
  // later work on the update stream comes after the read-back too
  if (sd != su) {
    ZERO_CUDA(cudaEventRecord(c->ev_out_done, sd));
    ZERO_CUDA(cudaStreamWaitEvent(su, c->ev_out_done, 0));
  }
  return ZERO_OK;
}

}  // namespace

extern "C" {

int64_t zero_host_staging_bytes(int scheme, int W, int64_t n_units, const int64_t* unit_sizes, int64_t chunk_elems) {
  if (!valid_scheme(scheme)) return fail(ZERO_E_ARG, "scheme %d is not one of DP/Z1/Z2/Z3", scheme);
  if (scheme != ZERO_SCHEME_Z3 && n_units != 1)
    return fail(ZERO_E_ARG, "data parallel, ZeRO-1 and ZeRO-2 take exactly one unit");
  if (chunk_elems < 0 || chunk_elems > (int64_t(1) << 40)) return fail(ZERO_E_ARG, "chunk_elems out of range");
  Layout L;
  int rc = make_layout(W, n_units, unit_sizes, &L);
  if (rc) return rc;
  int64_t chunk = 0, slot = 0;
  staging_geometry(scheme, W, L, chunk_elems, &chunk, &slot);
  return 2 * W * slot;
}

int zero_step_host(zero_ctx* c, int scheme, int W, int64_t n, const void* const* host_grads, void* host_out,
                   void* staging, int64_t staging_bytes, int64_t chunk_elems, double lr, double beta1, double beta2,
                   double eps, int64_t t, void* stream_h2d, void* stream_d2h) {
  if (c == nullptr) return fail(ZERO_E_ARG, "ctx is NULL");
  if (scheme != c->scheme || W != c->W || n != c->L.n)
    return fail(ZERO_E_ARG, "scheme/W/n (%d/%d/%lld) differ from the context's (%d/%d/%lld)", scheme, W,
                (long long)n, c->scheme, c->W, (long long)c->L.n);
  int rc = check_hyper(lr, beta1, beta2, eps, t);
  if (rc) return rc;
  if (t != c->t + 1)
    return fail(ZERO_E_STATE, "step counter %lld does not follow %lld", (long long)t, (long long)c->t);
  if (chunk_elems < 0 || chunk_elems > (int64_t(1) << 40)) return fail(ZERO_E_ARG, "chunk_elems out of range");
  if ((rc = check_no_open_bucket_step(c))) return rc;
  if (host_grads == nullptr) return fail(ZERO_E_ARG, "host_grads is NULL");
  for (int w = 0; w < W; ++w)
    if (host_grads[w] == nullptr && c->L.n_pad > 0) return fail(ZERO_E_ARG, "host gradients of rank %d are NULL", w);
  int64_t chunk = 0, slot = 0;
  staging_geometry(c->scheme, W, c->L, chunk_elems, &chunk, &slot);
  const int64_t need = 2 * W * slot;
  if (c->L.n_pad > 0) {
    if (staging == nullptr) return fail(ZERO_E_ARG, "staging is NULL");
    if ((reinterpret_cast<uintptr_t>(staging) & 255u) != 0) return fail(ZERO_E_ALIGN, "staging must be 256-byte aligned");
    if (staging_bytes < need)
      return fail(ZERO_E_ARG, "staging holds %lld bytes; this configuration needs %lld", (long long)staging_bytes,
                  (long long)need);
  }
  if ((rc = check_ranks_up(c))) return rc;
  for (size_t u = 0; u < c->live.size(); ++u)
    if (c->live[u]) return fail(ZERO_E_STATE, "unit %zu is still gathered by the caller", u);
  const zero::AdamCoef coef = make_coef(lr, beta1, beta2, eps, t, W);
  cudaStream_t sh = stream_h2d ? static_cast<cudaStream_t>(stream_h2d) : c->su;
  cudaStream_t sd = stream_d2h ? static_cast<cudaStream_t>(stream_d2h) : c->su;
  Range range("zero_step_host %lld", static_cast<long long>(t));
  if (c->L.n_pad > 0) {
    rc = run_host_step(c, host_grads, host_out, static_cast<char*>(staging), chunk, slot, coef, sh, sd);
    if (rc) return rc;
  }
  c->t = t;
  return ZERO_OK;
}

}  // extern "C"
