/*
 * The ZeRO-3 step that allocates nothing (zero_step_z3_static), across a
 * device reset, from plain C.
 *
 * Pass 1 runs one ZeRO-3 step twice on the same inputs: through a context
 * (zero_step, with its two caller-allocated unit buffers) and through
 * zero_step_z3_static (gathering into the library's own device array), and
 * requires the same bits.  Then cudaDeviceReset tears the device's context
 * down - every allocation is freed and the library's device code, with the
 * array, is unloaded - and pass 2 allocates everything again, restores
 * pass 1's state and runs step 2 the same two ways.  The array's device
 * address is looked up on every call, so pass 2 finds it wherever the
 * reloaded module put it.  This program and the library must share one CUDA
 * runtime (both link the shared libcudart).  Exit status 0 on success.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "zero_step.h"

#define CHECK(cond, ...)             \
  do {                               \
    if (!(cond)) {                   \
      fprintf(stderr, __VA_ARGS__);  \
      fprintf(stderr, "\n");         \
      exit(1);                       \
    }                                \
  } while (0)
#define CUDA(x) CHECK((x) == cudaSuccess, "%s: %s", #x, cudaGetErrorString(cudaGetLastError()))

enum { W = 4, U = 4 };
static const int64_t units[U] = {1000, 37, 0, 4096};

/* a deterministic bf16 gradient around 1e-3 (a test input, not the method) */
static uint16_t grad_bits(uint64_t* state) {
  *state = *state * 6364136223846793005ULL + 1442695040888963407ULL;
  const double u = (double)(*state >> 11) / 9007199254740992.0;
  float g = (float)((u - 0.5) * 2e-3);
  uint32_t bits;
  memcpy(&bits, &g, sizeof bits);
  return (uint16_t)(bits >> 16);
}

static int hook_calls;
static void count_hook(void* user, int phase, int64_t unit, void* buf, void* stream) {
  (void)user, (void)phase, (void)unit, (void)buf, (void)stream;
  ++hook_calls;
}

int main(void) {
  int64_t sz[6];
  CHECK(zero_buffer_sizes(ZERO_SCHEME_Z3, W, U, units, sz) == ZERO_OK, "sizes: %s", zero_last_error());
  int64_t n = 0;
  for (int u = 0; u < U; ++u) n += units[u];
  const int64_t n_pad = sz[1], s16 = sz[3], ubuf = sz[4];
  float* h_master = calloc((size_t)n_pad, 4);
  float* h_m = calloc((size_t)n_pad, 4);
  float* h_v = calloc((size_t)n_pad, 4);
  float* got = calloc((size_t)n_pad, 4);
  uint16_t* h16a = calloc((size_t)s16 + 1, 2);
  uint16_t* h16b = calloc((size_t)s16 + 1, 2);
  uint16_t* h_grads = calloc((size_t)(W * n_pad), 2);
  for (int64_t i = 0; i < n_pad; ++i) h_master[i] = 0.02f * (float)((i * 7919) % 2001 - 1000) / 1000.0f;
  uint64_t state = 99;
  const double lr = 3e-4, b1 = 0.9, b2 = 0.95, eps = 1e-8;

  for (int pass = 1; pass <= 2; ++pass) {
    const int64_t t = pass;
    float *master, *m, *v, *sm, *smm, *sv;
    void *shard[W], *sshard[W], *grads[W], *ub[2];
    CUDA(cudaMalloc((void**)&master, n_pad * 4));
    CUDA(cudaMalloc((void**)&m, n_pad * 4));
    CUDA(cudaMalloc((void**)&v, n_pad * 4));
    CUDA(cudaMalloc((void**)&sm, n_pad * 4));
    CUDA(cudaMalloc((void**)&smm, n_pad * 4));
    CUDA(cudaMalloc((void**)&sv, n_pad * 4));
    for (int r = 0; r < W; ++r) {
      CUDA(cudaMalloc(&shard[r], s16 * 2 + 16));
      CUDA(cudaMalloc(&sshard[r], s16 * 2 + 16));
      CUDA(cudaMalloc(&grads[r], n_pad * 2));
    }
    for (int b = 0; b < 2; ++b) CUDA(cudaMalloc(&ub[b], ubuf * 2 + 16));
    CUDA(cudaMemcpy(master, h_master, n_pad * 4, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(m, h_m, n_pad * 4, cudaMemcpyHostToDevice));
    CUDA(cudaMemcpy(v, h_v, n_pad * 4, cudaMemcpyHostToDevice));

    zero_ctx* ctx = NULL;
    CHECK(zero_init(&ctx, ZERO_SCHEME_Z3, W, n, U, units, ZERO_BF16, ZERO_BF16, master, m, v, NULL, shard, ub, NULL,
                    NULL) == ZERO_OK,
          "init: %s", zero_last_error());
    CHECK(zero_set_state(ctx, h_master, h_m, h_v, t - 1) == ZERO_OK, "set_state: %s", zero_last_error());
    CUDA(cudaDeviceSynchronize());
    /* the caller's own copy of the same state, for the step without allocations */
    CUDA(cudaMemcpy(sm, master, n_pad * 4, cudaMemcpyDeviceToDevice));
    CUDA(cudaMemcpy(smm, m, n_pad * 4, cudaMemcpyDeviceToDevice));
    CUDA(cudaMemcpy(sv, v, n_pad * 4, cudaMemcpyDeviceToDevice));
    for (int r = 0; r < W; ++r) CUDA(cudaMemcpy(sshard[r], shard[r], s16 * 2, cudaMemcpyDeviceToDevice));

    memset(h_grads, 0, (size_t)(W * n_pad) * 2);
    int64_t off = 0;
    for (int u = 0; u < U; ++u) {   /* real positions only; the padding stays zero */
      const int64_t S = (units[u] + W - 1) / W;
      for (int w = 0; w < W; ++w)
        for (int64_t i = 0; i < units[u]; ++i) h_grads[w * n_pad + off + i] = grad_bits(&state);
      off += S * W;
    }
    for (int r = 0; r < W; ++r)
      CUDA(cudaMemcpy(grads[r], h_grads + r * n_pad, n_pad * 2, cudaMemcpyHostToDevice));

    CHECK(zero_step(ctx, ZERO_SCHEME_Z3, W, n, (const void* const*)grads, lr, b1, b2, eps, t) == ZERO_OK,
          "step: %s", zero_last_error());
    CHECK(zero_sync(ctx, 60000) == ZERO_OK, "sync: %s", zero_last_error());
    hook_calls = 0;
    CHECK(zero_step_z3_static(W, U, units, ZERO_BF16, ZERO_BF16, sm, smm, sv, sshard, (const void* const*)grads, lr,
                              b1, b2, eps, t, pass == 2 ? count_hook : NULL, NULL, NULL) == ZERO_OK,
          "static step (pass %d): %s", pass, zero_last_error());
    CUDA(cudaDeviceSynchronize());
    CHECK(pass == 1 || hook_calls == 2 * U, "hook ran %d times", hook_calls);

    float* pairs[3][2] = {{master, sm}, {m, smm}, {v, sv}};
    float* keep[3] = {h_master, h_m, h_v};
    for (int k = 0; k < 3; ++k) {
      CUDA(cudaMemcpy(keep[k], pairs[k][0], n_pad * 4, cudaMemcpyDeviceToHost));
      CUDA(cudaMemcpy(got, pairs[k][1], n_pad * 4, cudaMemcpyDeviceToHost));
      CHECK(memcmp(got, keep[k], (size_t)n_pad * 4) == 0, "pass %d: state %d differs from zero_step's", pass, k);
    }
    for (int r = 0; r < W; ++r) {
      CUDA(cudaMemcpy(h16a, shard[r], s16 * 2, cudaMemcpyDeviceToHost));
      CUDA(cudaMemcpy(h16b, sshard[r], s16 * 2, cudaMemcpyDeviceToHost));
      CHECK(memcmp(h16a, h16b, (size_t)s16 * 2) == 0, "pass %d: shard store %d differs", pass, r);
    }
    int moved = 0;
    for (int64_t i = 0; i < n_pad; ++i) moved += h_m[i] != 0.0f;
    CHECK(moved > n / 2, "pass %d: the step moved almost nothing (%d)", pass, moved);
    CHECK(zero_destroy(ctx) == ZERO_OK, "destroy: %s", zero_last_error());
    if (pass == 1) {
      /* frees every allocation above and unloads the library's device code */
      CUDA(cudaDeviceReset());
    }
  }
  printf("static ZeRO-3 step matches zero_step before and after cudaDeviceReset\n");
  return 0;
}
