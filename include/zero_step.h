/*
 * zero_step.h - C ABI of libzero_gb300.so, the ZeRO step on one GB300.
 *
 * The data-parallel hot path of ZeRO over a flat parameter vector, for W
 * data-parallel ranks simulated inside one GPU's memory:
 *
 *   (1) reduce-scatter: the mean over the W ranks of their 16-bit gradients,
 *       summed in rank order, for every element of each rank's 1/W shard;
 *   (2) Adam with bias correction on that shard's fp32 master, m and v;
 *   (3) the round-to-nearest-even recast of the master to the 16-bit working
 *       copy, written straight to its place in the full vector (the
 *       all-gather) or, for ZeRO-3, into the owning rank's 16-bit shard;
 *   (4) for ZeRO-3, the per-unit gather / release / re-gather schedule.
 *
 * Sources (page title and section):
 *   "The four schemes" (Zero From Scratch lab): the three flags that define
 *     data parallel and ZeRO-1/2/3, the per-shard Adam update, the step of
 *     each scheme, the resident and peak accounting.
 *   "ZeRO and FSDP" (AI infra handbook): the closed forms 16 Psi,
 *     4 Psi + 12 Psi/N, 2 Psi + 14 Psi/N, 16 Psi/N; the zero-padded even
 *     split of the flat vector; the per-unit ZeRO-3 flow with prefetch.
 *   "ZeRO, annotated" sections 5 and 7, "One Poem Suffices: ZeRO" section
 *     4.1.4 and appendix B, "Sharding the States": traffic per rank under
 *     ring collectives, (N-1)/N of the data per collective.
 *
 * Beside the step itself (zero_step, and zero_gather_unit / zero_update_unit
 * / zero_release_unit for callers that drive ZeRO-3 themselves) the library
 * offers: the step fed from host memory (zero_step_host) with its host
 * allocator (zero_host_alloc); the step applied bucket by bucket
 * (zero_step_bucket); ZeRO-3 steps replayed from a CUDA graph
 * (zero_set_graph); a ZeRO-3 step that allocates nothing
 * (zero_step_z3_static); data parallelism with its replicas kept literally
 * (zero_step_dp_replicas); and ZeRO-2 with the optimizer on the host CPU
 * (zero_offload_*).
 *
 * Layout.  n real parameters are split into units (one unit for data
 * parallel, ZeRO-1 and ZeRO-2; the caller's units, e.g. one per transformer
 * layer, for ZeRO-3).  Unit u holds unit_sizes[u] parameters padded with
 * zeros to S_u * W elements, S_u = ceil(unit_sizes[u] / W); units follow one
 * another in a flat vector of n_pad = sum_u S_u * W elements.  Rank r owns
 * [off_u + r S_u, off_u + (r + 1) S_u) of unit u.  The fp32 master, m and v
 * are n_pad floats each in this flat order; every rank's gradient vector is
 * n_pad 16-bit values in the same order (zeros in the padding).
 *
 * Memory ownership.  The caller allocates and owns every device buffer and
 * every stream; the library keeps non-owning pointers and calls no device
 * allocator.  master, m and v must be 32-byte aligned, every other device
 * pointer 16-byte aligned (ZERO_E_ALIGN otherwise).
 *
 * Errors.  Every function that returns int returns ZERO_OK (0) or a negative
 * ZERO_E_* code; functions returning int64_t return a negative code on error.
 * zero_last_error() gives a message for the calling thread's last error.
 * Arguments are checked on the host before anything is launched: a call that
 * fails a check has enqueued no GPU work.
 *
 * Asynchrony.  zero_step, zero_gather_unit, zero_update_unit and
 * zero_refresh_working_copy enqueue work on the context's streams and return
 * without waiting; zero_sync waits (with a deadline), and zero_get_state /
 * zero_set_state wait for their own copies.
 *
 * Threads.  A context (zero_ctx, zero_offload) is used by one host thread at
 * a time; different contexts may be used from different threads at once.
 * Error messages are kept per thread.
 */
#ifndef ZERO_STEP_H
#define ZERO_STEP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define ZERO_OK          0
#define ZERO_E_ARG      -1  /* an argument is out of range or inconsistent      */
#define ZERO_E_ALIGN    -2  /* a device pointer is not 16-byte aligned           */
#define ZERO_E_CUDA     -3  /* a CUDA runtime call failed                        */
#define ZERO_E_RANK     -4  /* a simulated rank is marked unavailable            */
#define ZERO_E_TIMEOUT  -5  /* zero_sync's deadline passed before the work ended */
#define ZERO_E_STATE    -6  /* call out of order (step counter, unit not live)   */
#define ZERO_E_NOMEM    -7  /* host memory could not be mapped                   */

/* ---- schemes ("The four schemes": shard_opt / shard_grad / shard_param) - */
#define ZERO_SCHEME_DP  0   /* nothing sharded, gradients all-reduced           */
#define ZERO_SCHEME_Z1  1   /* optimizer state sharded                          */
#define ZERO_SCHEME_Z2  2   /* + gradients sharded                              */
#define ZERO_SCHEME_Z3  3   /* + 16-bit parameters sharded, gathered per unit   */

/* ---- 16-bit formats ---------------------------------------------------- */
#define ZERO_FP16       0
#define ZERO_BF16       1

/* ---- accounting kinds --------------------------------------------------- */
#define ZERO_RESIDENT   0
#define ZERO_PEAK       1

/* ---- kernel variants for the fused reduce + Adam + cast pass ------------ */
#define ZERO_VARIANT_AUTO   0  /* the fastest measured variant for the launch     */
#define ZERO_VARIANT_VECTOR 1  /* 256-bit vector loads into registers             */
#define ZERO_VARIANT_BULK   2  /* bulk async copies into a shared-memory ring     */

/* ---- statistics (zero_stat) --------------------------------------------- */
#define ZERO_STAT_COMM_BYTES      0  /* bytes a rank would send, cumulative       */
#define ZERO_STAT_LAUNCHES        1  /* kernels this context launched, cumulative */
#define ZERO_STAT_GATHERS         2  /* unit all-gathers performed                */
#define ZERO_STAT_SCATTERS        3  /* unit reduce-scatters performed            */
#define ZERO_STAT_LIVE_ELEMS      4  /* gathered 16-bit elements live right now   */
#define ZERO_STAT_PEAK_LIVE_ELEMS 5  /* most gathered elements ever live at once  */
#define ZERO_STAT_T               6  /* the last step counter used                */
#define ZERO_STAT_DEVICE_ERRORS   7  /* bounded device waits of this context's
                                        launches that gave up                       */
#define ZERO_STAT_LAST_VARIANT    8  /* kernel of the last fused launch: ZERO_VARIANT_VECTOR
                                        or ZERO_VARIANT_BULK (0 before any)          */

typedef struct zero_ctx zero_ctx;

/*
 * Host hook for ZeRO-3 steps.  zero_step calls it on the host once per
 * gathered unit, after the unit's gather has been enqueued and before the
 * unit is released: phase 0 is the forward pass, 1 the backward pass.
 * unit_buf holds the unit's S_u * W 16-bit values in flat order; work that
 * reads it must be enqueued on `stream` (a cudaStream_t) and must not keep
 * the pointer: the buffer is reused for a later unit once that work ends.
 */
typedef void (*zero_unit_hook)(void* user, int phase, int64_t unit, void* unit_buf, void* stream);

/* ---- pure host queries (no GPU needed) --------------------------------- */

/*
 * Buffer sizes for a configuration.  out[0] = n, out[1] = n_pad (floats in
 * each of master / m / v, 16-bit values in each rank's gradient vector),
 * out[2] = elements of the full 16-bit working copy (n_pad for DP/Z1/Z2,
 * 0 for Z3), out[3] = elements of each rank's 16-bit shard store (Z3:
 * sum_u S_u; else 0), out[4] = elements of one ZeRO-3 unit buffer
 * (max_u S_u * W; else 0), out[5] = number of units.  DP/Z1/Z2 take exactly
 * one unit (unit_sizes[0] = n).  Returns ZERO_E_ARG for W outside
 * [1, ZERO_MAX_RANKS], no units, or a negative unit size.
 */
#define ZERO_MAX_RANKS 64
int zero_buffer_sizes(int scheme, int W, int64_t n_units, const int64_t* unit_sizes, int64_t* out);

/*
 * Per-unit layout: off[u] (flat offset of unit u), shard[u] (S_u) and
 * off16[u] (offset of unit u's shard inside each rank's shard store), for
 * u < n_units.  Any of the three output arrays may be NULL.
 */
int zero_layout(int W, int64_t n_units, const int64_t* unit_sizes, int64_t* off, int64_t* shard, int64_t* off16);

/*
 * Model-state bytes per rank ("ZeRO and FSDP", the three stages; "The four
 * schemes", bytes_per_param): resident = 16 n (DP), 4 n + 12 S (Z1),
 * 2 n + 14 S (Z2), 16 S (Z3) with S = ceil(n / W).  kind ZERO_PEAK adds,
 * for ZeRO-3 only, 2 bytes for each of `gathered_elems` gathered 16-bit
 * values live at once.  Negative on a bad argument.
 */
int64_t zero_bytes_per_rank(int scheme, int64_t n, int W, int kind, int64_t gathered_elems);

/*
 * Bytes one rank sends per step under ring collectives of 2-byte values
 * ("Sharding the States": (n-1)/n of 4 N, and of 6 N for stage 3):
 * 2 (W-1) S 2 for DP/Z1/Z2 and 3 (W-1) S 2 for ZeRO-3, S = ceil(n / W).
 */
int64_t zero_comm_bytes_closed_form(int scheme, int64_t n, int W);

/* ---- context lifetime --------------------------------------------------- */

/*
 * Create a context.  No GPU work and no CUDA call happen here.
 *   scheme            ZERO_SCHEME_*.
 *   W                 simulated ranks, 1..ZERO_MAX_RANKS.
 *   n                 real parameters, = sum of unit_sizes.
 *   n_units, unit_sizes  the units (exactly one for DP/Z1/Z2).
 *   grad_dtype, work_dtype  ZERO_FP16 or ZERO_BF16: the gradients' format and
 *                     the 16-bit working copy's format.
 *   master, m, v      device, n_pad floats each, flat layout.  The caller
 *                     writes theta0 into master (zeros in the padding) and
 *                     zeros into m and v before the first step.
 *   p16               device, n_pad 16-bit values: the full working copy
 *                     (DP/Z1/Z2; must be NULL for Z3).
 *   shard16           host array of W device pointers, each rank's shard
 *                     store of sum_u S_u values (Z3; NULL otherwise).
 *   unit_bufs         host array of 2 device pointers, each max_u S_u * W
 *                     16-bit values: the ping-pong gather buffers zero_step
 *                     uses for ZeRO-3 (Z3; NULL otherwise).
 *   stream_update     cudaStream_t for updates (may be the caller's stream;
 *                     NULL means the legacy default stream).
 *   stream_gather     cudaStream_t for ZeRO-3 gathers, so that with a unit
 *                     hook the next unit's gather overlaps the work on the
 *                     current one; NULL means stream_update (no overlap).
 *                     Work the caller enqueues on different streams itself
 *                     (zero_gather_unit, zero_update_unit) is ordered by the
 *                     caller.
 * On success *out receives the context.  Call zero_refresh_working_copy
 * once after writing theta0, before the first step or gather.
 */
int zero_init(zero_ctx** out, int scheme, int W, int64_t n, int64_t n_units, const int64_t* unit_sizes,
              int grad_dtype, int work_dtype, float* master, float* m, float* v, void* p16,
              void* const* shard16, void* const* unit_bufs, void* stream_update, void* stream_gather);

/* Destroy a context (waits for its work first).  NULL is accepted. */
int zero_destroy(zero_ctx* ctx);

/* ---- the step ------------------------------------------------------------ */

/*
 * Cast the fp32 master to the 16-bit working copy (DP/Z1/Z2: p16; Z3: each
 * rank's shard store), round to nearest even, on stream_update.
 */
int zero_refresh_working_copy(zero_ctx* ctx);

/*
 * One ZeRO step ("The four schemes": the step of each scheme).
 *   scheme, W, n      must equal the context's (else ZERO_E_ARG).
 *   grads             host array of W device pointers; rank w's gradients,
 *                     n_pad values of grad_dtype in flat order, read only.
 *   lr, beta1, beta2, eps  Adam hyper-parameters (0 <= beta < 1, eps > 0).
 *          The update runs in fp32, so eps must also be a positive finite
 *          fp32 value and lr / (1 - beta1^t) finite in fp32 (ZERO_E_ARG).
 *   t                 the step counter, 1-based: must be the context's last
 *                     step counter + 1 (ZERO_E_STATE otherwise).
 * DP/Z1/Z2: one fused pass over the flat vector: mean of the W gradients,
 * Adam, recast into p16.  Traffic counted: 2 (W-1) S 2 bytes.
 * Z3: for u = 0..U-1 gather u, call the hook, release; then for
 * u = U-1..0 gather u, call the hook, update unit u (stream_update),
 * release.  With a hook registered the gathers run on stream_gather, so the
 * next unit's gather overlaps the work on the current one (prefetch); with
 * none, everything runs in order on stream_update (there is no compute to
 * hide a gather behind): the forward pass gathers two units per launch, one
 * into each unit buffer - all the pairs in one launch when every unit has
 * the same shard size, every buffer position receiving its units in unit
 * order, so that the buffers end as after separate gathers - and each
 * backward gather is done by the unit's update pass, which copies the
 * unit's 16-bit values into the unit buffer before overwriting them.  At
 * most two unit buffers are live.  Traffic: 3 (W-1) S_u 2 bytes per unit.
 * The step is ordered after earlier work on stream_update and all its work
 * is finished when work enqueued later on stream_update starts.
 */
int zero_step(zero_ctx* ctx, int scheme, int W, int64_t n, const void* const* grads,
              double lr, double beta1, double beta2, double eps, int64_t t);

/* Register (fn != NULL) or clear the ZeRO-3 unit hook. */
int zero_set_unit_hook(zero_ctx* ctx, zero_unit_hook fn, void* user);

/* ---- the step bucket by bucket --------------------------------------------- */

/*
 * One bucket of a DP/Z1/Z2 step: reduce-scatter (mean) + Adam + recast of
 * the flat range [lo, lo + len), as soon as the ranks' gradients for that
 * range exist ("ZeRO and FSDP": real ZeRO-2 reduce-scatters by bucket during
 * the backward pass; "One Poem Suffices: ZeRO" section 4.2.2: constant-size
 * buffers).  The update is elementwise, so a step done bucket by bucket is
 * bit-identical to zero_step, and the full gradient vectors never need to
 * exist: bucket_grads[w] points at rank w's len gradient values of the range
 * (device, 16-byte aligned; lo must be a multiple of 8).
 *   t      the first bucket of a step passes the context's step counter + 1,
 *          the others the same t.  A step's buckets may arrive in any order but
 *          must cover [0, n_pad) exactly once before the next step (or any
 *          other kind of step) starts: an overlap, or a new step while one is
 *          incomplete, is ZERO_E_STATE.
 *   stream cudaStream_t (NULL: the update stream).
 * Traffic: the step's two collectives are counted when its last bucket
 * arrives.  ZeRO-3 updates unit by unit with zero_update_unit instead.
 */
int zero_step_bucket(zero_ctx* ctx, int64_t lo, int64_t len, const void* const* bucket_grads, double lr,
                     double beta1, double beta2, double eps, int64_t t, void* stream);

/* ---- the step fed from host memory ---------------------------------------- */

/*
 * Device bytes of the staging ring zero_step_host needs: two slots, each
 * holding every rank's gradients for one chunk (DP/Z1/Z2: chunk_elems
 * values, 0 meaning the default: n_pad / 24 rounded up to a multiple of
 * 2^20 and kept between 2^24 and 2^26; ZeRO-3: one unit, max_u S_u * W
 * values), in
 * the gradient format: 2 * W * round_up((chunk + 8) * 2, 256).  The ring
 * stays this size whatever n is: the constant-size buffers of "One Poem
 * Suffices: ZeRO" section 4.2.2 (C_B) instead of W full gradient vectors on
 * the device.  Negative on a bad argument.
 */
int64_t zero_host_staging_bytes(int scheme, int W, int64_t n_units, const int64_t* unit_sizes, int64_t chunk_elems);

/*
 * One ZeRO step whose gradients are in host memory and whose updated 16-bit
 * working copy is written back to host memory.  The step is cut into chunks
 * (DP/Z1/Z2: chunk_elems of the flat vector; ZeRO-3: one unit, backward
 * order) and pipelined over three streams: the gradients of chunk k + 1
 * cross the host link into the staging ring on stream_h2d while chunk k is
 * updated on the context's update stream and chunk k - 1's results return
 * on stream_d2h.  The arithmetic is that of zero_step (bit-identical).
 *   scheme, W, n, lr, beta1, beta2, eps, t   as for zero_step.
 *   host_grads   host array of W host pointers, rank w's n_pad gradient
 *                values in flat order (pinned memory for full speed;
 *                pageable memory works but its copies are synchronous).
 *   host_out     host buffer for the updated working copy, or NULL: DP/Z1/Z2
 *                n_pad values in flat order; ZeRO-3 each rank's shard store,
 *                rank after rank (W * sum_u S_u values).
 *   staging      device buffer of at least zero_host_staging_bytes(...)
 *                bytes, 256-byte aligned; staging_bytes its size.
 *   chunk_elems  as given to zero_host_staging_bytes (ignored for ZeRO-3).
 *   stream_h2d, stream_d2h  cudaStream_t for the two copy directions (NULL
 *                for either: the update stream, without overlap).
 * ZeRO-3 runs the unit schedule of zero_step without a hook: forward gathers,
 * then per unit (reverse order) one pass that gathers and updates.  When the
 * call returns, the work is enqueued; work enqueued later on the update stream
 * runs after all of it, copies included.  ZERO_E_ARG if the staging is too
 * small or misaligned; the other errors as for zero_step.
 */
int zero_step_host(zero_ctx* ctx, int scheme, int W, int64_t n, const void* const* host_grads, void* host_out,
                   void* staging, int64_t staging_bytes, int64_t chunk_elems, double lr, double beta1,
                   double beta2, double eps, int64_t t, void* stream_h2d, void* stream_d2h);

/*
 * Host memory for zero_step_host's gradients and results: `bytes` bytes,
 * page-locked (registered with cudaHostRegister, so copies from and to it
 * run asynchronously at the link's rate), on a private anonymous mapping
 * advised for transparent huge pages and populated before it is returned.
 * The pages do not need to be huge for correctness; they help speed.
 * Measured on GB300 hosts,
 * 1 GB copies out of memory pinned with cudaHostAlloc ran from 38 to 212
 * GB/s, slower in later processes on the same host, while copies out of
 * this memory held 208-212 GB/s.  A block of at least one huge page is
 * mapped as whole huge pages from a huge-page boundary (its last page may
 * extend past `bytes`); a smaller one starts on a page boundary, on base
 * pages.
 * The contents are zero.  For many vectors (e.g. every rank's gradients)
 * one block, sliced, keeps them all on huge pages even when each is
 * smaller than a huge page.  *out receives the address (NULL on
 * failure).  The memory is the caller's until zero_host_free.
 * ZERO_E_ARG for bytes <= 0 or out NULL; ZERO_E_NOMEM if the mapping
 * fails; ZERO_E_CUDA if the registration fails (e.g. no device).
 */
int zero_host_alloc(int64_t bytes, void** out);

/*
 * Release memory from zero_host_alloc (unregister and unmap).  NULL is
 * accepted; any other pointer that zero_host_alloc did not return is
 * ZERO_E_ARG.  No work that uses the memory may still be in flight.
 */
int zero_host_free(void* p);

/* ---- ZeRO-3 driven by the caller ---------------------------------------- */

/*
 * Gather unit `unit` of a ZeRO-3 context: dst (device, S_u * W 16-bit values
 * of work_dtype) receives every rank's shard of the unit in flat order, on
 * `stream` (NULL: stream_gather).  The unit becomes live; gathering a live
 * unit is ZERO_E_STATE.  Traffic counted: (W-1) S_u 2 bytes.
 */
int zero_gather_unit(zero_ctx* ctx, int64_t unit, void* dst, void* stream);

/* Release a live unit (host bookkeeping; the buffer stays the caller's). */
int zero_release_unit(zero_ctx* ctx, int64_t unit);

/*
 * Reduce-scatter + Adam + recast of one ZeRO-3 unit, on `stream` (NULL:
 * stream_update).  grads as in zero_step.  t must be the context's step
 * counter (another unit of the same step) or that + 1 (a new step).
 * Traffic counted: (W-1) S_u 2 bytes.
 */
int zero_update_unit(zero_ctx* ctx, int64_t unit, const void* const* grads,
                     double lr, double beta1, double beta2, double eps, int64_t t, void* stream);

/* ---- state, statistics, waiting ------------------------------------------ */

/*
 * Copy master, m and v (n_pad floats each) out to the caller's buffers
 * (host or device; any of them may be NULL) and the step counter to *t;
 * waits for the copies.
 */
int zero_get_state(zero_ctx* ctx, float* master, float* m, float* v, int64_t* t);

/*
 * Copy master, m and v (n_pad floats each, host or device) into the
 * context's buffers, set the step counter to t (>= 0), and refresh the
 * 16-bit working copy; waits for the copies.
 */
int zero_set_state(zero_ctx* ctx, const float* master, const float* m, const float* v, int64_t t);

/* Cumulative bytes one rank would have sent for the collectives run so far. */
int64_t zero_comm_bytes_per_rank(const zero_ctx* ctx);

/* One of the ZERO_STAT_* counters; negative on a bad argument. */
int64_t zero_stat(const zero_ctx* ctx, int which);

/*
 * Wait until all work the context has enqueued has finished, polling with a
 * host deadline of timeout_ms (< 0: no deadline).  ZERO_E_TIMEOUT when the
 * deadline passes first; the work is left running and a later call may
 * wait again.  ZERO_E_CUDA if the work failed; ZERO_E_STATE if a bounded
 * device-side wait gave up (ZERO_STAT_DEVICE_ERRORS).
 */
int zero_sync(zero_ctx* ctx, int timeout_ms);

/* ---- timing of the context's own kernels ---------------------------------- */
#define ZERO_KERNEL_FUSED   0  /* the fused reduce-scatter + Adam + recast pass */
#define ZERO_KERNEL_GATHER  1  /* ZeRO-3 unit gathers                           */
#define ZERO_KERNEL_CAST    2  /* working-copy casts                            */

/*
 * Per-launch timing on (1) or off (0).  While on, every kernel the context
 * launches is bracketed by two CUDA events recorded on the stream it is
 * launched on; the events come from a pool the context owns.
 */
int zero_enable_timing(zero_ctx* ctx, int on);

/*
 * Wait for the timed launches of `kernel` (ZERO_KERNEL_*) recorded so far,
 * return their summed device time in milliseconds and their number, and
 * start a new tally for that kernel.  Either output may be NULL.
 */
int zero_read_timing(zero_ctx* ctx, int kernel, double* total_ms, int64_t* launches);

/* ---- debugging ----------------------------------------------------------------- */
#define ZERO_DEBUG_POISON_RELEASED 1  /* fill a released ZeRO-3 unit buffer with NaN */

/*
 * Debug flags (ZERO_DEBUG_*, or 0).  With ZERO_DEBUG_POISON_RELEASED, every
 * ZeRO-3 unit buffer is filled with the 16-bit NaN 0x7FFF when its unit is
 * released (zero_release_unit, and each release inside zero_step), in order
 * on the stream that used it: work that reads a unit after its release then
 * sees NaN instead of plausible stale weights.  Costs one fill per release.
 */
int zero_set_debug(zero_ctx* ctx, int flags);

/*
 * Select the fused-pass variant (ZERO_VARIANT_*).  AUTO uses the bulk-staged
 * kernel where it measured no slower (W of 8 or 16, at least 8 2048-element
 * tiles for each CTA) and the vector kernel elsewhere.  BULK asks for the
 * bulk-staged kernel; it still runs the vector kernel where the bulk one
 * cannot (W not in {1, 2, 4, 8, 16}, or 16-bit slots not 16-byte aligned).
 * Both give bit-identical results.  Changing the variant drops a captured
 * step graph (zero_set_graph).
 */
int zero_set_variant(zero_ctx* ctx, int variant);

/*
 * ZeRO-3 steps from a CUDA graph (on != 0) or as ordinary launches (0, the
 * default).  With it on, the first zero_step that runs without a unit hook,
 * timing brackets, debug flags or an injected stall captures its launches
 * (the forward gathers, then U update passes) into a graph; that step and
 * every later one with the same conditions set the fused kernels' Adam
 * coefficients and gradient pointers on the graph and launch it once on the
 * update stream, which saves the gaps between the launches.  In the graph
 * the backward update passes form two chains (alternate units, each chain
 * holding the units that share a unit buffer), so that one unit's pass can
 * take SMs as the other's frees them; the graph orders everything the
 * schedule's data needs.  Steps under other conditions run the ordinary
 * launches; results are bit-identical either way and the counters advance
 * the same.  ZERO_E_ARG for a scheme other than ZeRO-3 (one launch per step:
 * nothing to capture) or a context whose update stream is the legacy default
 * stream (it cannot be captured).  Turning it off frees the graph.
 */
int zero_set_graph(zero_ctx* ctx, int on);

/*
 * Testing the bounded device waits.  The next fused launch of this context,
 * if it runs the bulk-staged kernel, never loads tile `tile` of its first
 * CTA: that CTA's wait for it runs out after about a second, the CTA counts
 * a device error, waits (bounded) for the copies it did issue and returns.
 * zero_sync then returns ZERO_E_STATE and the context stays usable; the
 * values that launch should have written are not valid.  Nothing faults or
 * hangs.  tile < 0 cancels a pending injection.
 */
int zero_inject_stall(zero_ctx* ctx, int64_t tile);

/*
 * Host-side fault injection: mark simulated rank `rank` unavailable
 * (available = 0) or back (1).  While any rank is unavailable, zero_step,
 * zero_gather_unit and zero_update_unit return ZERO_E_RANK before launching
 * anything, as a collective with a missing peer would fail.
 */
int zero_mark_rank(zero_ctx* ctx, int rank, int available);

/*
 * ZeRO-3 step that allocates nothing.  The pages have no counterpart to this
 * entry point; it exists for callers that cannot allocate device memory:
 * code running where cudaMalloc is not allowed or not wanted (a host
 * callback, a memory pool that is already fully reserved, a process whose
 * device allocator belongs to another framework), which therefore cannot
 * hand zero_step the two unit buffers ZeRO-3 gathers into.
 *
 * It runs the same step as zero_step does for a ZeRO-3 context - forward
 * gathers in unit order, backward gathers in reverse order each followed by
 * the unit's reduce-scatter + Adam + recast - all on `stream`, and gathers
 * into a fixed 16 MiB array of device memory that belongs to the library
 * instead of caller buffers.  Layout and arguments are those of zero_init
 * and zero_step for ZeRO-3: master, m, v (n_pad floats, 32-byte aligned),
 * shard16 (W shard stores of sum_u S_u values), grads (W vectors of n_pad
 * values, 16-byte aligned); hook/user as in zero_set_unit_hook (may be
 * NULL), called with the library's buffer.  There is no context: the caller
 * keeps the step counter t, and the shard stores must already hold the
 * 16-bit cast of the master (as zero_refresh_working_copy leaves them).
 *
 * Limits and sharing.  Each unit, padded, may hold at most 8,388,608 16-bit
 * values (S_u * W); larger units return ZERO_E_ARG with a message, before
 * any GPU work.  The array is held by every GPU on which the library is
 * loaded until the process exits.  All calls share it and it keeps the last
 * call's contents (each gather overwrites what it reads, so nothing needs
 * clearing); calls whose work overlaps on the GPU race on it, so issue
 * them on one stream or otherwise serialise them.  Every call looks up the
 * array's device address on the current device (cudaGetSymbolAddress); the
 * address is not kept between calls, so a call after cudaDeviceReset finds
 * the array where the reloaded module put it.  The first call on a device
 * also loads the library's device code there: make that first call before
 * any stream capture.  Nothing here calls cudaMalloc, cudaFree or any other
 * allocator.
 *
 * Without a hook, each unit's backward gather is done by its update pass
 * (the pass copies each 16-bit value into the array before overwriting it),
 * as zero_step does; with a hook the gather is a copy of its own, so that
 * the hook sees the unit before it is updated.  The update runs the register
 * kernel (ZERO_VARIANT_VECTOR): it has no device-side waits, so there is no
 * timed-out wait that this context-free call would have to report.
 */
int zero_step_z3_static(int W, int64_t n_units, const int64_t* unit_sizes, int grad_dtype, int work_dtype,
                        float* master, float* m, float* v, void* const* shard16, const void* const* grads,
                        double lr, double beta1, double beta2, double eps, int64_t t,
                        zero_unit_hook hook, void* user, void* stream);

/* ---- data parallelism with literal replicas ---------------------------------- */

/*
 * One DP step with every rank's replica kept literally ("The four schemes":
 * the DP baseline, every rank holding the 16-bit weights, the gradients and
 * the fp32 master, m and v in full; "ZeRO, annotated": the redundancy the
 * three ZeRO stages remove).  zero_step for ZERO_SCHEME_DP keeps one copy,
 * since the replicas are equal by construction; this call materialises all
 * W of them, to measure what sharding saves.
 *   W, n          ranks (1..ZERO_MAX_RANKS) and real parameters; every vector
 *                 holds n_pad = ceil(n / W) * W values (padded tail zero),
 *                 as zero_buffer_sizes reports for ZERO_SCHEME_DP.
 *   grad_dtype, work_dtype  ZERO_FP16 or ZERO_BF16.
 *   grads         host array of W device pointers: rank w's gradients
 *                 (16-byte aligned), read only.
 *   master, m, v  host arrays of W device pointers: replica r's fp32 state
 *                 (32-byte aligned), read and written in place.
 *   p16           host array of W device pointers: replica r's 16-bit
 *                 working copy (16-byte aligned), written.
 *   lr, beta1, beta2, eps, t  as for zero_step; there is no context, so the
 *                 caller keeps t (t >= 1, else ZERO_E_STATE).
 *   stream        the CUDA stream the one kernel is enqueued on (NULL: the
 *                 legacy default stream); returns without waiting.
 * Every replica receives the rank-ordered mean of the W gradients and the
 * same Adam step, so the replicas stay bit-identical to one another and to
 * zero_step for DP on the same inputs.  Buffers stay the caller's.  Returns
 * ZERO_E_ARG for a NULL pointer, a bad dtype or hyper-parameter, or replica
 * buffers that overlap one another or a gradient vector; ZERO_E_ALIGN for a
 * misaligned pointer; ZERO_E_CUDA if the launch fails.
 */
int zero_step_dp_replicas(int W, int64_t n, int grad_dtype, int work_dtype, const void* const* grads,
                          float* const* master, float* const* m, float* const* v, void* const* p16,
                          double lr, double beta1, double beta2, double eps, int64_t t, void* stream);

/*
 * The lab's DP assertion: count the (replica r >= 1, element e) pairs, over
 * the n_pad values of each vector, where master, m, v or the 16-bit copy of
 * replica r differs bitwise from replica 0.  Arguments as for
 * zero_step_dp_replicas (pointers aligned to their element size);
 * `mismatches` is one int64 of device memory (8-byte aligned, the
 * caller's), set to 0 and then to the count by work enqueued on `stream`;
 * read it after that work finishes.  Returns ZERO_E_ARG / ZERO_E_ALIGN /
 * ZERO_E_CUDA as above.
 */
int zero_dp_replicas_mismatches(int W, int64_t n, const float* const* master, const float* const* m,
                                const float* const* v, const void* const* p16, int64_t* mismatches,
                                void* stream);

/* ---- the optimizer offloaded to the host ------------------------------------ */

/*
 * ZeRO-2 with the optimizer state and its update on the host CPU ("ZeRO and
 * FSDP", ZeRO-3 and FSDP, and "Sharding the States": offloading puts the
 * optimizer states in CPU memory, trading link bandwidth for device memory;
 * "ZeRO, annotated" section 11: ZeRO-Offload moves the optimizer's
 * computation to the CPU too).  The device keeps the W ranks' 16-bit
 * gradients and the 16-bit working copy; the fp32 master, m and v live in
 * host memory.  Per step, chunk by chunk: the GPU forms the rank-ordered fp32
 * mean of the W gradients (the reduce-scatter), copy engines carry it to the
 * host (4 bytes per element), a pool of host threads runs Adam and the
 * round-to-nearest-even recast, and copy engines carry the 16-bit values back
 * into the device working copy (2 bytes per element).  The host arithmetic
 * repeats the device kernel's operations one for one in IEEE single
 * precision, so the result is bit-identical to zero_step.  Only this entry
 * point and zero_adam_host compute on the host; no GPU entry point falls back
 * to them.
 */
typedef struct zero_offload zero_offload;

/* Device staging the offloaded step needs: two chunks of fp32 means
 * (chunk_elems <= 0: the default of 4,194,304 elements; rounded up to a
 * multiple of 8). */
int64_t zero_offload_staging_bytes(int64_t chunk_elems);

/*
 * Create an offloaded-step context.  Layout as for ZERO_SCHEME_Z2 (one unit,
 * n_pad = ceil(n / W) * W values per vector, rank r owning [r S, (r + 1) S)).
 *   host_master, host_m, host_v  host memory, n_pad floats each; master holds
 *                theta0 (padding zero), m and v zeros.  Read and written by the
 *                host threads only.
 *   host_grad    host memory for n_pad fp32 means; host_p16 host memory for
 *                n_pad 16-bit values.  Both should be page-locked (e.g. from
 *                zero_host_alloc) so that their copies run asynchronously.
 *                Slicing all five host vectors from one zero_host_alloc block
 *                puts them on huge pages even where each alone is smaller
 *                than one; the host pass and the copies run faster there.
 *   p16          device, n_pad 16-bit values (work_dtype), 16-byte aligned:
 *                the working copy, overwritten by each step.
 *   staging      device, >= zero_offload_staging_bytes(chunk_elems) bytes,
 *                256-byte aligned.
 *   threads      host threads for Adam (<= 0: all hardware threads).
 *   stream       cudaStream_t the GPU work is enqueued on (NULL: legacy default).
 * All buffers stay the caller's.  The context owns two copy streams, its
 * events and its threads.
 */
int zero_offload_init(zero_offload** out, int W, int64_t n, int grad_dtype, int work_dtype, float* host_master,
                      float* host_m, float* host_v, float* host_grad, void* host_p16, void* p16, void* staging,
                      int64_t staging_bytes, int64_t chunk_elems, int threads, void* stream);

/*
 * One offloaded step.  grads: host array of W device pointers (n_pad values
 * of grad_dtype each, 16-byte aligned).  t must follow the context's last
 * step counter (ZERO_E_STATE otherwise).  The call returns when the host
 * update is done; the copies of the new working copy may still be in
 * flight, and work enqueued later on `stream` runs after them.  A chunk whose
 * mean has not reached host memory within 60 s gives ZERO_E_TIMEOUT.  An
 * error after the argument checks (ZERO_E_CUDA, ZERO_E_TIMEOUT) can leave
 * the host state and the working copy partly updated and the step counter
 * unchanged: restore master, m and v from a saved copy before going on.
 */
int zero_offload_step(zero_offload* ctx, const void* const* grads, double lr, double beta1, double beta2,
                      double eps, int64_t t);

/*
 * Resume: set the context's step counter to t (>= 0), the number of steps
 * already applied to the master, m and v it works on.  The fp32 state lives
 * in the caller's host buffers, so a checkpoint is those three arrays plus t;
 * to resume, copy them back and call this.  The next zero_offload_step takes
 * t + 1.  The device working copy is rewritten by that step.
 */
int zero_offload_set_step(zero_offload* ctx, int64_t t);

/* Cumulative figures of a context (any pointer may be NULL): the last step
 * counter, seconds of the steps' host phases (from the wait for the first
 * chunk's mean to the last piece's update), bytes copied device->host and
 * host->device, kernels launched, host threads. */
int zero_offload_stats(const zero_offload* ctx, int64_t* t, double* host_seconds, int64_t* d2h_bytes,
                       int64_t* h2d_bytes, int64_t* launches, int* threads);

/* Destroy a context (waits for its work). NULL is accepted. */
int zero_offload_destroy(zero_offload* ctx);

/*
 * The offloaded step's host update alone, on host memory: Adam step t for
 * W ranks (W fixes only the mean's 1/W coefficient, unused here) on n
 * elements with mean gradient `grad`, updating master, m and v in place and
 * writing the round-to-nearest-even 16-bit copy (work_dtype) to out16.
 * threads as above.  Needs no GPU.
 */
int zero_adam_host(int64_t n, const float* grad, float* master, float* m, float* v, void* out16, int work_dtype,
                   double lr, double beta1, double beta2, double eps, int64_t t, int W, int threads);

/* Message for the calling thread's last error ("" if none). */
const char* zero_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ZERO_STEP_H */
