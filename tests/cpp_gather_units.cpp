// The one-launch forward gather of a ZeRO-3 step (zero::launch_gather_units),
// driven directly: after the launch, buffer b must hold, at every position,
// the last unit of parity b (unit u goes to buffer u % 2, in unit order), and
// nothing around the buffers may be written.  In a whole step the backward
// pass overwrites both buffers, so this is where the forward result is
// checked bit for bit.  Also checks when the launch applies.  Exit 0 on
// success.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <vector>

#include "zero_internal.h"

#define CHECK(cond, ...)             \
  do {                               \
    if (!(cond)) {                   \
      fprintf(stderr, __VA_ARGS__);  \
      fprintf(stderr, "\n");         \
      std::exit(1);                  \
    }                                \
  } while (0)
#define CUDA(x) CHECK((x) == cudaSuccess, "%s failed", #x)

static uint16_t value(int r, int64_t u, int64_t j) {
  uint64_t h = (static_cast<uint64_t>(r) * 1000003u + static_cast<uint64_t>(u)) * 2654435761u + static_cast<uint64_t>(j);
  h ^= h >> 17;
  return static_cast<uint16_t>(h * 0x9E3779B97F4A7C15ull >> 48);
}

int main() {
  const int64_t kGuard = 4096;   // 16-bit values of guard on each side of a buffer
  const uint16_t kFill = 0xA5A5;
  int cases = 0;
  for (int W : {1, 3, 8}) {
    for (int64_t U : {1, 2, 3, 7}) {
      for (int64_t S : {16, 48, 8208}) {
        std::vector<void*> shard(W);
        for (int r = 0; r < W; ++r) {
          std::vector<uint16_t> h(static_cast<size_t>(U * S));
          for (int64_t u = 0; u < U; ++u)
            for (int64_t j = 0; j < S; ++j) h[u * S + j] = value(r, u, j);
          CUDA(cudaMalloc(&shard[r], h.size() * 2));
          CUDA(cudaMemcpy(shard[r], h.data(), h.size() * 2, cudaMemcpyHostToDevice));
        }
        const int64_t len = W * S, total = len + 2 * kGuard;
        uint16_t* raw[2];
        void* bufs[2];
        std::vector<uint16_t> fill(static_cast<size_t>(total), kFill);
        for (int b = 0; b < 2; ++b) {
          CUDA(cudaMalloc(reinterpret_cast<void**>(&raw[b]), total * 2));
          CUDA(cudaMemcpy(raw[b], fill.data(), total * 2, cudaMemcpyHostToDevice));
          bufs[b] = raw[b] + kGuard;   // 8,192 bytes in: 32-byte aligned
        }
        CHECK(zero::gather_units_applies(shard.data(), W, bufs, U, S), "W=%d U=%lld S=%lld should apply", W,
              (long long)U, (long long)S);
        int64_t launches = 0;
        CUDA(zero::launch_gather_units(shard.data(), W, bufs, U, S, nullptr, &launches));
        CUDA(cudaDeviceSynchronize());
        CHECK(launches == 1, "one launch, counted");
        for (int b = 0; b < 2; ++b) {
          std::vector<uint16_t> got(static_cast<size_t>(total));
          CUDA(cudaMemcpy(got.data(), raw[b], total * 2, cudaMemcpyDeviceToHost));
          for (int64_t i = 0; i < kGuard; ++i)
            CHECK(got[i] == kFill && got[kGuard + len + i] == kFill, "W=%d U=%lld S=%lld: guard of buffer %d written",
                  W, (long long)U, (long long)S, b);
          const int64_t last = (U - 1 - b) >= 0 ? ((U - 1 - b) / 2) * 2 + b : -1;   // last unit of parity b
          for (int r = 0; r < W; ++r)
            for (int64_t j = 0; j < S; ++j) {
              const uint16_t want = last >= 0 ? value(r, last, j) : kFill;
              CHECK(got[kGuard + r * S + j] == want, "W=%d U=%lld S=%lld: buffer %d rank %d value %lld", W,
                    (long long)U, (long long)S, b, r, (long long)j);
            }
        }
        for (int r = 0; r < W; ++r) CUDA(cudaFree(shard[r]));
        for (int b = 0; b < 2; ++b) CUDA(cudaFree(raw[b]));
        ++cases;
      }
    }
  }
  // where it does not apply: shard sizes off the 32-byte grain, misaligned
  // stores or buffers, no units
  void* p = nullptr;
  CUDA(cudaMalloc(&p, 1 << 20));
  char* base = static_cast<char*>(p);
  void* st[2] = {base, base + 4096};
  void* bf[2] = {base + 8192, base + 65536};
  CHECK(zero::gather_units_applies(st, 2, bf, 3, 16), "aligned case applies");
  CHECK(!zero::gather_units_applies(st, 2, bf, 3, 8), "S = 8 (16 bytes) must not apply");
  CHECK(!zero::gather_units_applies(st, 2, bf, 3, 24), "S = 24 (48 bytes) must not apply");
  CHECK(!zero::gather_units_applies(st, 2, bf, 0, 16), "no units must not apply");
  void* st_bad[2] = {base, base + 4112};
  CHECK(!zero::gather_units_applies(st_bad, 2, bf, 3, 16), "a store off 32 bytes must not apply");
  void* bf_bad[2] = {base + 8192, base + 65552};
  CHECK(!zero::gather_units_applies(st, 2, bf_bad, 3, 16), "a buffer off 32 bytes must not apply");
  CHECK(zero::gather_units_applies(st, 2, bf_bad, 1, 16), "one unit uses only the first buffer");
  int64_t launches = 0;
  CHECK(zero::launch_gather_units(st, 2, bf, 3, 24, nullptr, &launches) == cudaErrorInvalidValue && launches == 0,
        "a launch that does not apply is refused before launching");
  CUDA(cudaFree(p));
  printf("gather_units: %d configurations, every buffer position holds the last unit of its parity\n", cases);
  return 0;
}
