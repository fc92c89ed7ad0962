// The ZeRO step with the optimizer offloaded to the host CPU.
//
// "ZeRO and FSDP" (ZeRO-3 and FSDP) and "Sharding the States" describe
// offloading as putting the optimizer states in CPU memory, paying in link
// bandwidth for device memory; "ZeRO, annotated" (section 11) lists
// ZeRO-Offload, which moves the optimizer's computation to the CPU as well.
// Here the fp32 master, m and v live in host memory and Adam runs on the host
// cores; the device keeps only the W ranks' 16-bit gradients and the 16-bit
// working copy, 2 W + 2 bytes per parameter instead of 2 W + 14.
//
// One step, chunk by chunk along the flat vector:
//   GPU     the rank-ordered fp32 mean of the W gradients of the chunk
//           (offload_mean.cu) into one slot of a two-slot device staging ring;
//   D2H     the chunk's mean into host memory (4 bytes per element);
//   host    Adam on the chunk's master, m, v, and the round-to-nearest-even
//           16-bit copy, on a pool of threads;
//   H2D     the chunk's 16-bit values into the device working copy (the
//           all-gather, streamed).
// The GPU and copy work for every chunk is enqueued up front.  The host
// threads then take pieces of the flat vector in order, with no barrier at
// chunk boundaries: a chunk is updated as soon as its mean has landed, and
// its return copy is enqueued as soon as its last piece is done, so the
// copies of one chunk overlap the host arithmetic of its neighbours.
//
// The host arithmetic is the device kernel's operation for operation: fused
// multiply-adds where the kernel fuses, separate products where it does not,
// IEEE square root and division, no contraction by the compiler (this file
// is built with -ffp-contract=off), so the offloaded step gives the same bits
// as zero_step.  This is the only arithmetic of the library that runs on the
// host, by design of the offloaded step; no GPU entry point falls back to it.

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <condition_variable>
#include <cstdint>
#include <cstring>
#include <functional>
#include <memory>
#include <mutex>
#include <string>
#include <thread>
#include <utility>
#include <vector>

#include "zero_internal.h"
#include "zero_step.h"

namespace {

// ---- a fixed pool of host threads ----------------------------------------------

class ThreadPool {
 public:
  explicit ThreadPool(int n) : size_(std::max(1, n)) {
    for (int i = 1; i < size_; ++i) workers_.emplace_back([this] { loop(); });
  }

  ~ThreadPool() {
    {
      std::lock_guard<std::mutex> lk(mu_);
      stop_ = true;
      ++generation_;
    }
    cv_.notify_all();
    for (auto& t : workers_) t.join();
  }

  int size() const { return size_; }

  // f(lo, hi) over [0, n) in pieces of `grain`, on every thread including the
  // caller's; returns when all pieces are done.
  void run(int64_t n, int64_t grain, const std::function<void(int64_t, int64_t)>& f) {
    if (n <= 0) return;
    {
      std::lock_guard<std::mutex> lk(mu_);
      job_ = &f;
      n_ = n;
      grain_ = std::max<int64_t>(1, grain);
      next_.store(0);
      pending_ = static_cast<int>(workers_.size());
      ++generation_;
    }
    cv_.notify_all();
    work();
    std::unique_lock<std::mutex> lk(mu_);
    done_.wait(lk, [this] { return pending_ == 0; });
    job_ = nullptr;
  }

 private:
  void work() {
    for (;;) {
      const int64_t lo = next_.fetch_add(grain_);
      if (lo >= n_) return;
      (*job_)(lo, std::min(n_, lo + grain_));
    }
  }

  void loop() {
    uint64_t seen = 0;
    std::unique_lock<std::mutex> lk(mu_);
    for (;;) {
      cv_.wait(lk, [&] { return generation_ != seen; });
      seen = generation_;
      if (stop_) return;
      lk.unlock();
      work();
      lk.lock();
      if (--pending_ == 0) done_.notify_one();
    }
  }

  int size_;
  std::vector<std::thread> workers_;
  std::mutex mu_;
  std::condition_variable cv_, done_;
  uint64_t generation_ = 0;
  bool stop_ = false;
  const std::function<void(int64_t, int64_t)>* job_ = nullptr;
  int64_t n_ = 0, grain_ = 1;
  std::atomic<int64_t> next_{0};
  int pending_ = 0;
};

int default_threads() {
  const unsigned hw = std::thread::hardware_concurrency();
  return hw ? static_cast<int>(hw) : 1;
}

// ---- the host Adam -----------------------------------------------------------------

// Round to nearest even, fp32 -> bf16 (the upper 16 bits, rounded); NaN stays NaN.
inline uint16_t to_bf16(float x) {
  uint32_t u;
  std::memcpy(&u, &x, sizeof u);
  if ((u & 0x7fffffffu) > 0x7f800000u) return static_cast<uint16_t>((u >> 16) | 0x0040u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}

// Round to nearest even, fp32 -> IEEE binary16 (the compiler's conversion).
inline uint16_t to_fp16(float x) {
  const _Float16 h = static_cast<_Float16>(x);
  uint16_t b;
  std::memcpy(&b, &h, sizeof b);
  return b;
}

// Adam on [0, n) of the given arrays with mean gradient g; the order of
// operations is that of the device kernel's element update.  The recast runs
// as a second loop over each tile of kTile elements (still in cache), so
// that both loops vectorise at full width.
constexpr int64_t kTile = 2048;

template <bool BF16>
void adam_range(const float* __restrict g, float* __restrict th, float* __restrict m, float* __restrict v,
                uint16_t* __restrict out, int64_t n, const zero::AdamCoef c) {
  for (int64_t t0 = 0; t0 < n; t0 += kTile) {
    const int64_t t1 = std::min(n, t0 + kTile);
    for (int64_t i = t0; i < t1; ++i) {
      const float gi = g[i];
      const float mi = std::fma(c.b1, m[i], c.omb1 * gi);
      const float vi = std::fma(c.b2, v[i], (c.omb2 * gi) * gi);
      const float den = std::fma(std::sqrt(vi), c.rsqrt_bc2, c.eps);
      m[i] = mi;
      v[i] = vi;
      th[i] = th[i] - (c.step_size * mi) / den;
    }
    for (int64_t i = t0; i < t1; ++i) out[i] = BF16 ? to_bf16(th[i]) : to_fp16(th[i]);
  }
}

constexpr int64_t kGrain = 1 << 16;   // elements per piece handed to a thread

void adam_parallel(ThreadPool& pool, const float* g, float* th, float* m, float* v, uint16_t* out, int64_t n,
                   const zero::AdamCoef& c, int work_dtype) {
  pool.run(n, kGrain, [&](int64_t lo, int64_t hi) {
    if (work_dtype == ZERO_BF16)
      adam_range<true>(g + lo, th + lo, m + lo, v + lo, out + lo, hi - lo, c);
    else
      adam_range<false>(g + lo, th + lo, m + lo, v + lo, out + lo, hi - lo, c);
  });
}

int fail(int code, const std::string& msg) { return zero::record_error(code, msg.c_str()); }

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

constexpr int64_t kDefaultChunk = int64_t(4) << 20;
constexpr double kWaitSeconds = 60.0;

int64_t chunk_of(int64_t chunk_elems) {
  const int64_t c = chunk_elems > 0 ? chunk_elems : kDefaultChunk;
  return (c + 7) / 8 * 8;
}

// Wait for an event with a deadline, sleeping between polls.  Returns
// ZERO_OK, or an error code with *why set (nothing is recorded: the caller
// may be a pool thread whose error message would not reach the user).
int poll_event(cudaEvent_t e, const char** why) {
  const auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    const cudaError_t r = cudaEventQuery(e);
    if (r == cudaSuccess) return ZERO_OK;
    if (r != cudaErrorNotReady) {
      *why = cudaGetErrorString(r);
      return ZERO_E_CUDA;
    }
    if (std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count() > kWaitSeconds) {
      *why = "a chunk's mean gradient did not reach host memory within 60 s";
      return ZERO_E_TIMEOUT;
    }
    std::this_thread::sleep_for(std::chrono::microseconds(20));
  }
}

// The first error of a parallel phase (code and message), kept for the caller.
struct FirstError {
  std::atomic<int> code{ZERO_OK};
  std::mutex mu;
  std::string msg;
  void note(int c, const char* m) {
    int expected = ZERO_OK;
    if (code.compare_exchange_strong(expected, c)) {
      std::lock_guard<std::mutex> lk(mu);
      msg = m;
    }
  }
};

}  // namespace

struct zero_offload {
  int W = 0;
  int64_t n = 0, n_pad = 0, chunk = 0, n_chunks = 0;
  int grad_dtype = 0, work_dtype = 0;
  float *master = nullptr, *m = nullptr, *v = nullptr, *host_grad = nullptr;
  uint16_t* host_p16 = nullptr;
  void* p16 = nullptr;
  float* slots[2] = {nullptr, nullptr};
  cudaStream_t stream = nullptr, d2h = nullptr, h2d = nullptr;
  std::vector<cudaEvent_t> mean_done, landed;
  cudaEvent_t returned = nullptr;
  std::unique_ptr<ThreadPool> pool;
  int64_t t = 0;
  int64_t launches = 0;
  double host_seconds = 0.0;
  int64_t d2h_bytes = 0, h2d_bytes = 0;
};

namespace {

void release(zero_offload* c) {
  if (!c) return;
  if (c->stream) cudaStreamSynchronize(c->stream);
  if (c->d2h) cudaStreamSynchronize(c->d2h);
  if (c->h2d) cudaStreamSynchronize(c->h2d);
  for (cudaEvent_t e : c->mean_done) cudaEventDestroy(e);
  for (cudaEvent_t e : c->landed) cudaEventDestroy(e);
  if (c->returned) cudaEventDestroy(c->returned);
  if (c->d2h) cudaStreamDestroy(c->d2h);
  if (c->h2d) cudaStreamDestroy(c->h2d);
  delete c;
}

}  // namespace

extern "C" int64_t zero_offload_staging_bytes(int64_t chunk_elems) { return 2 * chunk_of(chunk_elems) * 4; }

extern "C" int zero_offload_init(zero_offload** out, int W, int64_t n, int grad_dtype, int work_dtype,
                                 float* host_master, float* host_m, float* host_v, float* host_grad,
                                 void* host_p16, void* p16, void* staging, int64_t staging_bytes,
                                 int64_t chunk_elems, int threads, void* stream) {
  if (!out) return fail(ZERO_E_ARG, "out is NULL");
  *out = nullptr;
  if (W < 1 || W > ZERO_MAX_RANKS) return fail(ZERO_E_ARG, "W outside [1, ZERO_MAX_RANKS]");
  if (n < 0) return fail(ZERO_E_ARG, "negative parameter count");
  if ((grad_dtype != ZERO_FP16 && grad_dtype != ZERO_BF16) || (work_dtype != ZERO_FP16 && work_dtype != ZERO_BF16))
    return fail(ZERO_E_ARG, "16-bit formats must be ZERO_FP16 or ZERO_BF16");
  if (!host_master || !host_m || !host_v || !host_grad || !host_p16 || !p16 || !staging)
    return fail(ZERO_E_ARG, "a buffer pointer is NULL");
  if (!aligned(p16, 16)) return fail(ZERO_E_ALIGN, "the device working copy must be 16-byte aligned");
  if (!aligned(staging, 256)) return fail(ZERO_E_ALIGN, "the staging buffer must be 256-byte aligned");
  if (!aligned(host_master, 4) || !aligned(host_m, 4) || !aligned(host_v, 4) || !aligned(host_grad, 4) ||
      !aligned(host_p16, 2))
    return fail(ZERO_E_ALIGN, "host buffers must be aligned to their element size");
  const int64_t chunk = chunk_of(chunk_elems);
  if (staging_bytes < zero_offload_staging_bytes(chunk_elems))
    return fail(ZERO_E_ARG, "staging is smaller than zero_offload_staging_bytes(chunk_elems)");
  {
    // the host buffers are all written: none may share memory with another
    const uintptr_t np = static_cast<uintptr_t>((n + W - 1) / W * W);
    std::vector<std::pair<uintptr_t, uintptr_t>> r;
    for (const void* p : {static_cast<const void*>(host_master), static_cast<const void*>(host_m),
                          static_cast<const void*>(host_v), static_cast<const void*>(host_grad)})
      r.emplace_back(reinterpret_cast<uintptr_t>(p), reinterpret_cast<uintptr_t>(p) + 4 * np);
    r.emplace_back(reinterpret_cast<uintptr_t>(host_p16), reinterpret_cast<uintptr_t>(host_p16) + 2 * np);
    std::sort(r.begin(), r.end());
    for (size_t k = 1; k < r.size(); ++k)
      if (np > 0 && r[k].first < r[k - 1].second) return fail(ZERO_E_ARG, "host buffers overlap one another");
  }
  auto* c = new zero_offload;
  c->W = W;
  c->n = n;
  c->n_pad = (n + W - 1) / W * W;
  c->chunk = chunk;
  c->n_chunks = (c->n_pad + chunk - 1) / chunk;
  c->grad_dtype = grad_dtype;
  c->work_dtype = work_dtype;
  c->master = host_master;
  c->m = host_m;
  c->v = host_v;
  c->host_grad = host_grad;
  c->host_p16 = static_cast<uint16_t*>(host_p16);
  c->p16 = p16;
  c->slots[0] = static_cast<float*>(staging);
  c->slots[1] = static_cast<float*>(staging) + chunk;
  c->stream = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamCreateWithFlags(&c->d2h, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c->h2d, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&c->returned, cudaEventDisableTiming);
  for (int64_t k = 0; e == cudaSuccess && k < c->n_chunks; ++k) {
    cudaEvent_t a = nullptr, b = nullptr;
    e = cudaEventCreateWithFlags(&a, cudaEventDisableTiming);
    if (e == cudaSuccess) c->mean_done.push_back(a);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&b, cudaEventDisableTiming);
    if (e == cudaSuccess) c->landed.push_back(b);
  }
  if (e != cudaSuccess) {
    release(c);
    return fail(ZERO_E_CUDA, cudaGetErrorString(e));
  }
  c->pool = std::make_unique<ThreadPool>(threads > 0 ? threads : default_threads());
  *out = c;
  return ZERO_OK;
}

extern "C" int zero_offload_destroy(zero_offload* ctx) {
  release(ctx);
  return ZERO_OK;
}

extern "C" int zero_offload_step(zero_offload* c, const void* const* grads, double lr, double beta1, double beta2,
                                 double eps, int64_t t) {
  if (!c) return fail(ZERO_E_ARG, "context is NULL");
  int rc = zero::check_adam_args(lr, beta1, beta2, eps, t);
  if (rc) return rc;
  if (t != c->t + 1) return fail(ZERO_E_STATE, "the step counter must follow the last one");
  if (!grads) return fail(ZERO_E_ARG, "grads is NULL");
  zero::MeanLaunch a{};
  a.W = c->W;
  a.grad_dtype = c->grad_dtype;
  for (int r = 0; r < c->W; ++r) {
    if (!grads[r]) return fail(ZERO_E_ARG, "a gradient pointer is NULL");
    if (!aligned(grads[r], 16)) return fail(ZERO_E_ALIGN, "gradients must be 16-byte aligned");
    a.grads[r] = grads[r];
  }
  const zero::AdamCoef coef = zero::adam_coef(lr, beta1, beta2, eps, t, c->W);
  a.inv_w = coef.inv_w;
  // NVTX ranges on the host timeline: the whole step, and its host phase
  struct Range {
    explicit Range(const char* name) { nvtxRangePushA(name); }
    ~Range() { nvtxRangePop(); }
  } step_range("zero_offload_step");
  cudaError_t e = cudaSuccess;
  // everything on the device side, up front
  for (int64_t k = 0; k < c->n_chunks && e == cudaSuccess; ++k) {
    const int64_t lo = k * c->chunk, len = std::min(c->chunk, c->n_pad - lo);
    float* slot = c->slots[k & 1];
    if (k >= 2) e = cudaStreamWaitEvent(c->stream, c->landed[k - 2], 0);   // the slot has been copied out
    a.lo = lo;
    a.len = len;
    a.out = slot;
    if (e == cudaSuccess) e = zero::launch_rank_mean(a, c->stream, &c->launches);
    if (e == cudaSuccess) e = cudaEventRecord(c->mean_done[k], c->stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(c->d2h, c->mean_done[k], 0);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(c->host_grad + lo, slot, len * 4, cudaMemcpyDeviceToHost, c->d2h);
    if (e == cudaSuccess) e = cudaEventRecord(c->landed[k], c->d2h);
    c->d2h_bytes += len * 4;
  }
  if (e != cudaSuccess) return fail(ZERO_E_CUDA, cudaGetErrorString(e));
  // The host half.  Every host thread takes pieces of kGrain elements in flat
  // order, with no barrier between chunks: the first thread to reach a chunk
  // waits for its mean to land, and the thread that finishes a chunk's last
  // piece sends the chunk's 16-bit values back to the device.
  const int64_t per_chunk = (c->chunk + kGrain - 1) / kGrain;
  const int64_t last_len = c->n_pad - (c->n_chunks - 1) * c->chunk;
  const int64_t pieces = c->n_chunks > 0 ? (c->n_chunks - 1) * per_chunk + (last_len + kGrain - 1) / kGrain : 0;
  std::vector<std::atomic<int>> ready(c->n_chunks);
  std::vector<std::atomic<int64_t>> left(c->n_chunks);
  for (int64_t k = 0; k < c->n_chunks; ++k) {
    ready[k].store(0);
    const int64_t len = std::min(c->chunk, c->n_pad - k * c->chunk);
    left[k].store((len + kGrain - 1) / kGrain);
  }
  FirstError err;
  uint16_t* const dev16 = static_cast<uint16_t*>(c->p16);
  const auto t0 = std::chrono::steady_clock::now();
  nvtxRangePushA("zero_offload_step host update");
  c->pool->run(pieces, 1, [&](int64_t p0, int64_t p1) {
    for (int64_t p = p0; p < p1; ++p) {
      if (err.code.load() != ZERO_OK) return;
      const int64_t k = p / per_chunk;
      const int64_t clo = k * c->chunk, clen = std::min(c->chunk, c->n_pad - clo);
      const int64_t lo = clo + (p % per_chunk) * kGrain, hi = std::min(clo + clen, lo + kGrain);
      if (!ready[k].load(std::memory_order_acquire)) {
        const char* why = "";
        const int rc2 = poll_event(c->landed[k], &why);
        if (rc2 != ZERO_OK) {
          err.note(rc2, why);
          return;
        }
        ready[k].store(1, std::memory_order_release);
      }
      if (c->work_dtype == ZERO_BF16)
        adam_range<true>(c->host_grad + lo, c->master + lo, c->m + lo, c->v + lo, c->host_p16 + lo, hi - lo, coef);
      else
        adam_range<false>(c->host_grad + lo, c->master + lo, c->m + lo, c->v + lo, c->host_p16 + lo, hi - lo, coef);
      if (left[k].fetch_sub(1) == 1) {
        const cudaError_t e2 =
            cudaMemcpyAsync(dev16 + clo, c->host_p16 + clo, clen * 2, cudaMemcpyHostToDevice, c->h2d);
        if (e2 != cudaSuccess) {
          err.note(ZERO_E_CUDA, cudaGetErrorString(e2));
          return;
        }
      }
    }
  });
  nvtxRangePop();
  c->host_seconds += std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
  if (err.code.load() != ZERO_OK) return fail(err.code.load(), err.msg);
  c->h2d_bytes += c->n_pad * 2;
  // later work on the caller's stream sees the new working copy
  e = cudaEventRecord(c->returned, c->h2d);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(c->stream, c->returned, 0);
  if (e != cudaSuccess) return fail(ZERO_E_CUDA, cudaGetErrorString(e));
  c->t = t;
  return ZERO_OK;
}

extern "C" int zero_offload_set_step(zero_offload* c, int64_t t) {
  if (!c) return fail(ZERO_E_ARG, "context is NULL");
  if (t < 0) return fail(ZERO_E_ARG, "the step counter cannot be negative");
  c->t = t;
  return ZERO_OK;
}

extern "C" int zero_offload_stats(const zero_offload* c, int64_t* t, double* host_seconds, int64_t* d2h_bytes,
                                  int64_t* h2d_bytes, int64_t* launches, int* threads) {
  if (!c) return fail(ZERO_E_ARG, "context is NULL");
  if (t) *t = c->t;
  if (host_seconds) *host_seconds = c->host_seconds;
  if (d2h_bytes) *d2h_bytes = c->d2h_bytes;
  if (h2d_bytes) *h2d_bytes = c->h2d_bytes;
  if (launches) *launches = c->launches;
  if (threads) *threads = c->pool->size();
  return ZERO_OK;
}

extern "C" int zero_adam_host(int64_t n, const float* grad, float* master, float* m, float* v, void* out16,
                              int work_dtype, double lr, double beta1, double beta2, double eps, int64_t t, int W,
                              int threads) {
  if (n < 0) return fail(ZERO_E_ARG, "negative element count");
  if (W < 1 || W > ZERO_MAX_RANKS) return fail(ZERO_E_ARG, "W outside [1, ZERO_MAX_RANKS]");
  if (work_dtype != ZERO_FP16 && work_dtype != ZERO_BF16)
    return fail(ZERO_E_ARG, "the 16-bit format must be ZERO_FP16 or ZERO_BF16");
  int rc = zero::check_adam_args(lr, beta1, beta2, eps, t);
  if (rc) return rc;
  if (n == 0) return ZERO_OK;
  if (!grad || !master || !m || !v || !out16) return fail(ZERO_E_ARG, "a buffer pointer is NULL");
  ThreadPool pool(threads > 0 ? threads : default_threads());
  adam_parallel(pool, grad, master, m, v, static_cast<uint16_t*>(out16), n,
                zero::adam_coef(lr, beta1, beta2, eps, t, W), work_dtype);
  return ZERO_OK;
}
