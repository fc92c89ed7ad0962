/*
 * A plain C client of libzero_gb300.so: no Python, no torch.  It sizes and
 * allocates the buffers of a ZeRO-2 configuration with the CUDA runtime, runs
 * the first step, and checks the first-step closed form of bias-corrected
 * Adam on every parameter: at t = 1, m_hat = g and v_hat = g^2, so each
 * parameter moves by -lr g / (|g| + eps) - by lr sign(g) up to
 * lr eps / (|g| + eps) - and not at all where g = 0.  It also checks that an
 * out-of-order step counter is refused with ZERO_E_STATE, and runs the same
 * step with the optimizer on the host (zero_offload_*, link buffers from
 * zero_host_alloc), which must give the same master bit for bit.  Exit
 * status 0 on success.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "zero_step.h"

#define CHECK(cond, ...)                   \
  do {                                     \
    if (!(cond)) {                         \
      fprintf(stderr, __VA_ARGS__);        \
      fprintf(stderr, "\n");               \
      return 1;                            \
    }                                      \
  } while (0)

/* bf16 value of a bit pattern: the top half of an fp32 */
static float bf16_value(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* a deterministic pseudo-random bf16 gradient around 1e-3 (a test input, not the method) */
static uint16_t grad_bits(uint64_t* state) {
  *state = *state * 6364136223846793005ULL + 1442695040888963407ULL;
  const double u = (double)(*state >> 11) / 9007199254740992.0;
  float g = (float)((u - 0.5) * 2e-3);
  if ((*state >> 60) == 0) g = 0.0f; /* some exact zeros */
  uint32_t bits;
  memcpy(&bits, &g, sizeof bits);
  return (uint16_t)(bits >> 16);
}

int main(void) {
  const int W = 4;
  const int64_t n = 1001;
  const int64_t units[1] = {n};
  int64_t sz[6];
  CHECK(zero_buffer_sizes(ZERO_SCHEME_Z2, W, 1, units, sz) == ZERO_OK, "sizes: %s", zero_last_error());
  const int64_t n_pad = sz[1];
  CHECK(n_pad == 1004, "n_pad %lld", (long long)n_pad);

  float* h_theta = calloc((size_t)n_pad, sizeof(float));
  float* h_out = calloc((size_t)n_pad, sizeof(float));
  uint16_t* h_grads[4];
  uint64_t state = 12345;
  for (int64_t i = 0; i < n; ++i) h_theta[i] = 0.02f * (float)sin((double)i);
  for (int w = 0; w < W; ++w) {
    h_grads[w] = calloc((size_t)n_pad, sizeof(uint16_t));
    for (int64_t i = 0; i < n; ++i) h_grads[w][i] = grad_bits(&state);
  }

  float *master, *m, *v;
  void* p16;
  void* grads[4];
  CHECK(cudaMalloc((void**)&master, n_pad * 4) == cudaSuccess, "cudaMalloc");
  CHECK(cudaMalloc((void**)&m, n_pad * 4) == cudaSuccess, "cudaMalloc");
  CHECK(cudaMalloc((void**)&v, n_pad * 4) == cudaSuccess, "cudaMalloc");
  CHECK(cudaMalloc(&p16, n_pad * 2) == cudaSuccess, "cudaMalloc");
  cudaMemcpy(master, h_theta, n_pad * 4, cudaMemcpyHostToDevice);
  cudaMemset(m, 0, n_pad * 4);
  cudaMemset(v, 0, n_pad * 4);
  for (int w = 0; w < W; ++w) {
    CHECK(cudaMalloc(&grads[w], n_pad * 2) == cudaSuccess, "cudaMalloc");
    cudaMemcpy(grads[w], h_grads[w], n_pad * 2, cudaMemcpyHostToDevice);
  }

  zero_ctx* ctx = NULL;
  CHECK(zero_init(&ctx, ZERO_SCHEME_Z2, W, n, 1, units, ZERO_BF16, ZERO_BF16, master, m, v, p16, NULL, NULL, NULL,
                  NULL) == ZERO_OK,
        "init: %s", zero_last_error());
  CHECK(zero_refresh_working_copy(ctx) == ZERO_OK, "refresh: %s", zero_last_error());
  const double lr = 1e-3, b1 = 0.9, b2 = 0.999, eps = 1e-8;
  CHECK(zero_step(ctx, ZERO_SCHEME_Z2, W, n, (const void* const*)grads, lr, b1, b2, eps, 3) == ZERO_E_STATE,
        "an out-of-order step counter must be refused");
  CHECK(strlen(zero_last_error()) > 0, "no message for the refused step");
  CHECK(zero_step(ctx, ZERO_SCHEME_Z2, W, n, (const void* const*)grads, lr, b1, b2, eps, 1) == ZERO_OK, "step: %s",
        zero_last_error());
  int64_t t = 0;
  CHECK(zero_get_state(ctx, h_out, NULL, NULL, &t) == ZERO_OK, "get_state: %s", zero_last_error());
  CHECK(t == 1, "t = %lld", (long long)t);
  CHECK(zero_comm_bytes_per_rank(ctx) == zero_comm_bytes_closed_form(ZERO_SCHEME_Z2, n, W), "traffic");

  int bad = 0;
  for (int64_t i = 0; i < n_pad; ++i) {
    double g = 0.0;
    for (int w = 0; w < W; ++w) g += (double)bf16_value(h_grads[w][i]);
    g /= W;
    const double d = (double)h_out[i] - (double)h_theta[i];
    const double ulp = fabs((double)nextafterf(h_out[i], INFINITY) - (double)h_out[i]);
    const double sign = g > 0 ? 1.0 : (g < 0 ? -1.0 : 0.0);
    const double bound = lr * eps / (fabs(g) + eps) + 2 * ulp + 1e-5 * lr;
    if (fabs(d + lr * sign) > bound || (g == 0.0 && d != 0.0)) ++bad;
  }
  CHECK(bad == 0, "%d parameters violate the first-step closed form", bad);
  CHECK(zero_destroy(ctx) == ZERO_OK, "destroy: %s", zero_last_error());

  /* The same step with the optimizer on the host: fp32 state in malloc'd
   * memory, the link buffers from zero_host_alloc; bit-identical master. */
  float* o_master = calloc((size_t)n_pad, sizeof(float));
  float* o_m = calloc((size_t)n_pad, sizeof(float));
  float* o_v = calloc((size_t)n_pad, sizeof(float));
  memcpy(o_master, h_theta, (size_t)n_pad * sizeof(float));
  void *o_grad = NULL, *o_p16 = NULL, *d_p16 = NULL, *staging = NULL;
  CHECK(zero_host_alloc(n_pad * 4, &o_grad) == ZERO_OK, "host alloc: %s", zero_last_error());
  CHECK(zero_host_alloc(n_pad * 2, &o_p16) == ZERO_OK, "host alloc: %s", zero_last_error());
  const int64_t chunk = 64; /* many chunks, to exercise the pipeline */
  const int64_t sbytes = zero_offload_staging_bytes(chunk);
  CHECK(cudaMalloc(&d_p16, n_pad * 2) == cudaSuccess, "cudaMalloc");
  CHECK(cudaMalloc(&staging, sbytes) == cudaSuccess, "cudaMalloc");
  zero_offload* off = NULL;
  CHECK(zero_offload_init(&off, W, n, ZERO_BF16, ZERO_BF16, o_master, o_m, o_v, (float*)o_grad, o_p16, d_p16,
                          staging, sbytes, chunk, 3, NULL) == ZERO_OK,
        "offload init: %s", zero_last_error());
  CHECK(zero_offload_step(off, (const void* const*)grads, lr, b1, b2, eps, 1) == ZERO_OK, "offload step: %s",
        zero_last_error());
  CHECK(cudaDeviceSynchronize() == cudaSuccess, "sync");
  CHECK(memcmp(o_master, h_out, (size_t)n_pad * sizeof(float)) == 0, "offloaded master differs from ZeRO-2");
  uint16_t* dev_copy = malloc((size_t)n_pad * 2);
  cudaMemcpy(dev_copy, d_p16, n_pad * 2, cudaMemcpyDeviceToHost);
  CHECK(memcmp(dev_copy, o_p16, (size_t)n_pad * 2) == 0, "device working copy differs from the host's");
  CHECK(zero_offload_destroy(off) == ZERO_OK, "offload destroy");
  CHECK(zero_host_free(o_grad) == ZERO_OK && zero_host_free(o_p16) == ZERO_OK, "host free");
  printf("c client: ZeRO-2 first step of %lld parameters on %d ranks matches the closed form; "
         "the host-offloaded step gives the same bits\n", (long long)n, W);
  return 0;
}
