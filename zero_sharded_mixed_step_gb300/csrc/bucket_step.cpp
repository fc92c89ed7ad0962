// The bucketed step (zero_step_bucket): DP/Z1/Z2 applied one range of the
// flat vector at a time, as each bucket's gradients become ready during the
// backward pass ("ZeRO and FSDP", the gradient buckets of ZeRO-2; "One Poem
// Suffices: ZeRO" section 4.2.2, constant-size buffers).  The context
// tracks which ranges the open step has covered, refuses overlaps, and
// counts the step's collectives when its last bucket arrives.

#include <cuda_runtime.h>

#include <cstdint>
#include <iterator>
#include <map>

#include "zero_context.h"
#include "zero_internal.h"
#include "zero_step.h"

using namespace zero::host;

extern "C" {

int zero_step_bucket(zero_ctx* c, int64_t lo, int64_t len, const void* const* bucket_grads, double lr,
                     double beta1, double beta2, double eps, int64_t t, void* stream) {
  if (c == nullptr) return fail(ZERO_E_ARG, "ctx is NULL");
  if (c->scheme == ZERO_SCHEME_Z3) return fail(ZERO_E_ARG, "ZeRO-3 updates unit by unit: use zero_update_unit");
  int rc = check_hyper(lr, beta1, beta2, eps, t);
  if (rc) return rc;
  if (len <= 0 || lo < 0 || lo > c->L.n_pad - len)
    return fail(ZERO_E_ARG, "bucket [%lld, %lld) is not inside [0, %lld)", (long long)lo, (long long)(lo + len),
                (long long)c->L.n_pad);
  if (lo % 8 != 0) return fail(ZERO_E_ALIGN, "a bucket must start at a multiple of 8 elements (lo=%lld)", (long long)lo);
  if (bucket_grads == nullptr) return fail(ZERO_E_ARG, "bucket_grads is NULL");
  for (int w = 0; w < c->W; ++w) {
    if (bucket_grads[w] == nullptr) return fail(ZERO_E_ARG, "bucket of rank %d is NULL", w);
    if (!aligned16(bucket_grads[w])) return fail(ZERO_E_ALIGN, "bucket of rank %d is not 16-byte aligned", w);
  }
  const bool new_step = t == c->t + 1;
  if (new_step) {
    if ((rc = check_no_open_bucket_step(c))) return rc;
  } else if (!(t == c->t && c->bucket_open)) {
    return fail(ZERO_E_STATE, "bucket of step %lld: the context is at step %lld%s", (long long)t, (long long)c->t,
                c->bucket_open ? "" : " and no bucketed step is open");
  }
  if (!new_step) {
    // no overlap with what this step has already covered
    auto it = c->covered.upper_bound(lo);
    if (it != c->covered.end() && it->first < lo + len)
      return fail(ZERO_E_STATE, "bucket [%lld, %lld) overlaps one already applied in step %lld", (long long)lo,
                  (long long)(lo + len), (long long)t);
    if (it != c->covered.begin() && std::prev(it)->second > lo)
      return fail(ZERO_E_STATE, "bucket [%lld, %lld) overlaps one already applied in step %lld", (long long)lo,
                  (long long)(lo + len), (long long)t);
  }
  if ((rc = check_ranks_up(c))) return rc;
  for (size_t u = 0; u < c->live.size(); ++u)
    if (c->live[u]) return fail(ZERO_E_STATE, "unit %zu is still gathered by the caller", u);
  // the kernel indexes gradients by flat position: shift each bucket back by lo
  const void* g[zero::kMaxRanks];
  for (int w = 0; w < c->W; ++w) g[w] = static_cast<const char*>(bucket_grads[w]) - lo * 2;
  cudaStream_t s = stream ? static_cast<cudaStream_t>(stream) : c->su;
  rc = launch_update(c, 0, g, make_coef(lr, beta1, beta2, eps, t, c->W), s, nullptr, lo, len);
  if (rc) return rc;
  if (new_step) {
    c->covered.clear();
    c->covered_elems = 0;
    c->bucket_open = true;
    c->t = t;
  }
  // record [lo, lo + len), merging with its neighbours
  int64_t a = lo, b = lo + len;
  auto it = c->covered.lower_bound(a);
  if (it != c->covered.begin() && std::prev(it)->second == a) {
    --it;
    a = it->first;
    it = c->covered.erase(it);
  }
  if (it != c->covered.end() && it->first == b) {
    b = it->second;
    c->covered.erase(it);
  }
  c->covered[a] = b;
  c->covered_elems += len;
  if (c->covered_elems == c->L.n_pad) {
    // the whole vector is done: the step's reduce-scatter and all-gather
    c->bucket_open = false;
    c->covered.clear();
    count_scatter(c, 0);
    c->gathers += 1;
    c->comm += ring_bytes(c->W, c->L.shard[0]);
  }
  return ZERO_OK;
}

}  // extern "C"
