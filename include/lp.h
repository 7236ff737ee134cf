/*
 * lp.h: C ABI of liblp, batch-invariant selected-token log-probabilities on
 * GB300 (sm_103a).
 *
 * For every row t of a logits matrix z[T, V] and its selected token y_t the
 * library computes
 *
 *     logp[t]    = z[t, y_t] - log sum_v exp z[t, v]
 *     entropy[t] = -sum_v p[t, v] log p[t, v],   p[t, :] = softmax(z[t, :])
 *
 * in float32 output.  This is the selected-token log-probability that every
 * candidate of the RL-Kernel logprob prior-art report (report.json, kind
 * qwen3_next_logprob_prior_art, field "candidates") computes from shared
 * logits, and the "linear_logp" operator (rlkernel.linear_logp.bitwise.v1 in
 * the backend readbacks of the RL-Kernel H100 PCP evidence record,
 * h100-pcp.json, section "validation") when the logits are the LM-head
 * projection z = H W^T.  The entropy is the per-row quantity the trainer logs
 * as train/entropy_loss (h100-pcp.json, section "comparison").
 *
 * Results are bitwise identical for a given row whatever batch it sits in, at
 * whatever offset, whatever number of vocabulary shards (1, 2 or 4) it is split
 * into, and however often the call is repeated: the properties batch_bitwise,
 * tp4_equals_tp1 and distinct_results_in_repeats == 1 of the prior-art report.
 * The reduction over the vocabulary is cut into four fixed "quarters"
 * [floor(q V / 4), floor((q+1) V / 4)), q = 0..3; each quarter is reduced in a
 * fixed order and the quarters are merged as (Q0 + Q1) + (Q2 + Q3).
 *
 * Conventions for every entry point:
 *  - Memory: every pointer argument is DEVICE memory owned by the caller,
 *    except the array of shard pointers of lp_merge_partials, which lives on
 *    the host (its elements are device pointers).  The library never
 *    allocates or frees memory; the fused path takes a caller-provided
 *    workspace sized by its query function.
 *  - Streams: all work is enqueued on `stream` (a cudaStream_t; NULL is the
 *    legacy default stream).  Calls do not synchronise with the host.
 *  - Errors: argument errors are detected on the host and returned before
 *    anything is enqueued; outputs are then untouched.  A failed launch
 *    returns LP_ERR_CUDA.  Errors found on the device never fault: a target
 *    outside [0, V) gives logp = NaN for that row (its entropy is still
 *    valid); a pipeline wait that exceeds its time bound sets the workspace
 *    error word (read it with lp_get_device_error) and that call's outputs
 *    are NaN.
 *  - Device: the current CUDA device must have compute capability 10.3
 *    (sm_103a).  Any other device gives LP_ERR_UNSUPPORTED_DEVICE; there is no
 *    fallback.
 *  - Types: logits and outputs are float32; H and W are bfloat16 (raw 16-bit
 *    storage, passed as void*); targets are int64.  Strides are in elements.
 */
#ifndef LP_H_
#define LP_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LP_API __attribute__((visibility("default")))
#else
#define LP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum lp_status {
  LP_OK = 0,
  LP_ERR_INVALID_ARGUMENT = 1,   /* null pointer, bad size or stride, bad shard */
  LP_ERR_MISALIGNED = 2,         /* a pointer or stride breaks an alignment rule */
  LP_ERR_UNSUPPORTED_DEVICE = 3, /* current device is not compute capability 10.3 */
  LP_ERR_WORKSPACE_TOO_SMALL = 4,
  LP_ERR_CUDA = 5,               /* a CUDA runtime or driver call failed */
  LP_ERR_TIMEOUT = 6             /* a device-side wait gave up (see lp_get_device_error) */
} lp_status;

/* ------------------------------------------------------------------------
 * Logits given: a bandwidth-bound streaming reduction of fp32 logits.
 * ------------------------------------------------------------------------ */

/*
 * lp_logprob_from_logits: logp and (optionally) entropy of every row of
 * fp32 logits, as the prior-art report's candidates compute them from shared
 * logits (report.json, "candidates", "reference": "shared_logits_fp64").
 *
 *   logits      [T, V] float32, row r at logits + r * ld_logits; 4-byte aligned.
 *               Rows whose start is 16-byte aligned are read with 128-bit loads;
 *               others with scalar loads (same arithmetic, same result).
 *   ld_logits   row stride in elements, >= V.
 *   targets     [T] int64 selected token per row (8-byte aligned).
 *   T           rows, >= 0 (T == 0 returns LP_OK and enqueues nothing).
 *   V           vocabulary size, 1 <= V < 2^31.
 *   logp_out    [T] float32.
 *   entropy_out [T] float32, or NULL to skip the entropy output.
 *   stream      cudaStream_t.
 */
LP_API lp_status lp_logprob_from_logits(const float* logits, int64_t ld_logits,
                                 const int64_t* targets, int64_t T, int64_t V,
                                 float* logp_out, float* entropy_out,
                                 void* stream);

/*
 * lp_vocab_shard_range: the global vocabulary columns [*begin, *end) that
 * shard `shard_index` of `n_shards` (1, 2 or 4) contiguous shards covers:
 * begin = floor(shard_index * V / n_shards).  A shard is a whole number of
 * quarters, so its per-row partial states merge bitwise-identically to the
 * unsharded result (the single-GPU form of the prior-art report's
 * tp4_equals_tp1 property).  Pure host function.
 */
LP_API lp_status lp_vocab_shard_range(int64_t vocab_total, int shard_index, int n_shards,
                               int64_t* begin, int64_t* end);

/*
 * lp_logprob_partials_from_logits: per-row quarter states of one vocabulary
 * shard of fp32 logits.
 *
 *   logits_shard [T, end - begin] float32: the shard's columns only (column 0
 *                is global column `begin`, see lp_vocab_shard_range).  May be
 *                NULL for an empty shard (possible only when vocab_total < 4).
 *   ld_logits    row stride in elements, >= end - begin.
 *   targets      [T] int64 GLOBAL token ids.
 *   vocab_total  V of the unsharded vocabulary.
 *   shard_index, n_shards: which shard (n_shards in {1, 2, 4}).
 *   partials_out [T][4 / n_shards][8] float32 (16-byte aligned): for each row
 *                and quarter of the shard, the 32-byte state
 *                (m, s_hi, s_lo, u, t, tau, 0, 0) of the distribution
 *                softmax(z / tau) (tau = 1 here): the quarter's maximum raw
 *                logit m; s = s_hi + s_lo = sum exp((z - m) / tau), held as an
 *                unevaluated float pair; u = sum exp((z - m) / tau) (z - m) / tau;
 *                the raw target logit t (-inf when the target is not in this
 *                quarter, NaN when it is outside [0, vocab_total)); and tau.
 */
LP_API lp_status lp_logprob_partials_from_logits(const float* logits_shard, int64_t ld_logits,
                                          const int64_t* targets, int64_t T,
                                          int64_t vocab_total, int shard_index,
                                          int n_shards, float* partials_out,
                                          void* stream);

/*
 * lp_merge_partials: merge the quarter states of 1, 2 or 4 shards in the fixed
 * order (Q0 + Q1) + (Q2 + Q3) and finalise logp and entropy.
 *
 *   shard_partials  HOST array of n_shards DEVICE pointers, in shard order;
 *                   element i is shard i's partials_out ([T][4 / n_shards][8]
 *                   float32, 16-byte aligned) from either partials entry point.
 *   n_shards        1, 2 or 4.
 *   logp_out        [T] float32; entropy_out [T] float32 or NULL.
 * The four states of a row are rebased to the row's largest m and summed as
 * (Q0 + Q1) + (Q2 + Q3), and logp = (t - M) / tau - log S,
 * entropy = log S - U / S are formed with float pairs (hi + lo, ~44 bits)
 * and rounded once.  A row whose
 * states carry different tau gives NaN.
 */
LP_API lp_status lp_merge_partials(const float* const* shard_partials, int n_shards,
                            int64_t T, float* logp_out, float* entropy_out,
                            void* stream);

/* ------------------------------------------------------------------------
 * Fused LM-head projection + logprob ("linear_logp"): z = H W^T is formed
 * tile by tile in tensor memory (tcgen05, bf16 inputs, fp32 accumulation) and
 * reduced on the fly; the T x V logits never reach global memory.
 * ------------------------------------------------------------------------ */

/*
 * lp_linear_logprob_workspace_size: bytes of workspace lp_linear_logprob needs
 * for T rows and vocabulary V (d does not change it).  The workspace holds a
 * 256-byte header (the device error word) and one 16-byte state per row and
 * 256-column vocabulary tile.
 */
LP_API size_t lp_linear_logprob_workspace_size(int64_t T, int64_t d, int64_t V);

/*
 * lp_linear_logprob: logp and entropy of softmax(H W^T) per row.
 *
 *   H           [T, d] bfloat16, row r at H + r * ld_h (elements); 16-byte
 *               aligned; ld_h % 8 == 0 and ld_h >= d.
 *   W           [V, d] bfloat16 LM-head weight, row v at W + v * ld_w; 16-byte
 *               aligned; ld_w % 8 == 0 and ld_w >= d.
 *   targets     [T] int64.
 *   T >= 0, 1 <= d < 2^31, 1 <= V < 2^31.
 *   logp_out    [T] float32; entropy_out [T] float32 or NULL.
 *   workspace   device memory, 256-byte aligned, at least
 *               lp_linear_logprob_workspace_size(T, d, V) bytes; its contents
 *               on entry do not matter.  Do not share one workspace between
 *               calls that may run concurrently.
 *
 * H and W are expected to hold finite values.  Non-finite inputs never fault;
 * a row whose logits include NaN or +inf gives NaN, and a row whose logits
 * include -inf may give NaN instead of treating that column as absent.
 */
LP_API lp_status lp_linear_logprob(const void* H, int64_t ld_h, const void* W, int64_t ld_w,
                            const int64_t* targets, int64_t T, int64_t d, int64_t V,
                            float* logp_out, float* entropy_out,
                            void* workspace, size_t workspace_bytes, void* stream);

/*
 * lp_linear_logprob_noalloc: lp_linear_logprob without a caller-provided
 * workspace, for callers that cannot allocate device memory: code hosted by a
 * runtime that owns every byte of device memory through its own pool and does
 * not let plug-ins call cudaMalloc, or code on a latency-critical path where a
 * cudaMalloc (which can synchronise the device) is not acceptable.  The pages
 * this library follows have no counterpart of this call.
 *
 * It allocates nothing: its scratch is a fixed 32 MiB array in device memory
 * that every GPU loading the library holds until the process exits.  Inputs
 * and outputs are as in lp_linear_logprob and are still the caller's.  The
 * results are those of lp_linear_logprob on the same inputs.
 *
 *   Limit: the call needs lp_linear_logprob_workspace_size(T, d, V) <= 32 MiB
 *   (at V = 151936 that is T <= 3518 rows); larger calls return
 *   LP_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.
 *   Set-up: the array's device address belongs to the module as loaded into
 *   one CUDA context.  The first call in each context (each device's primary
 *   context, a context the caller created, or the primary context re-created
 *   after cudaDeviceReset) looks it up with cudaGetSymbolAddress and keeps it
 *   under that context's id; make that first call before any stream capture.
 *   Sharing: all calls in a context share the array, which keeps the last
 *   call's contents (each call clears what must start at zero).  Calls whose
 *   work can overlap on the GPU, e.g. on two unsynchronised streams, race on
 *   the array: order them on one stream.
 *   Errors on the device: the error word lives in the hidden array, so
 *   lp_get_device_error cannot read it; a call whose bounded device-side wait
 *   gave up shows it as NaN in every logp and entropy it writes.
 */
LP_API lp_status lp_linear_logprob_noalloc(const void* H, int64_t ld_h, const void* W,
                                           int64_t ld_w, const int64_t* targets, int64_t T,
                                           int64_t d, int64_t V, float* logp_out,
                                           float* entropy_out, void* stream);

/*
 * lp_linear_logprob_partials_workspace_size: workspace bytes for one shard.
 */
LP_API size_t lp_linear_logprob_partials_workspace_size(int64_t T, int64_t d,
                                                 int64_t vocab_total, int n_shards);

/*
 * lp_linear_logprob_partials: the quarter states of one vocabulary shard of the
 * fused path, to be merged by lp_merge_partials.
 *
 *   W_shard     [end - begin, d] bfloat16: rows [begin, end) of the full W,
 *               (see lp_vocab_shard_range), row 0 = global row `begin`.  A
 *               shard that is empty (possible only when vocab_total < 4) must
 *               still point to one readable row; it contributes nothing.
 *   targets     [T] int64 GLOBAL token ids.
 *   partials_out [T][4 / n_shards][4] float32, layout as in
 *               lp_logprob_partials_from_logits.
 *   Other arguments as in lp_linear_logprob.
 */
LP_API lp_status lp_linear_logprob_partials(const void* H, int64_t ld_h, const void* W_shard,
                                     int64_t ld_w, const int64_t* targets, int64_t T,
                                     int64_t d, int64_t vocab_total, int shard_index,
                                     int n_shards, float* partials_out,
                                     void* workspace, size_t workspace_bytes,
                                     void* stream);

/* ------------------------------------------------------------------------
 * Temperature-scaled variants: softmax(z / tau) instead of softmax(z).  The
 * rollout engine of the RL-Kernel H100 PCP evidence record samples at
 * temperature 0.7 (h100-pcp.json, section "scope"); these return the
 * log-probability and entropy of the tempered distribution.
 *
 * No logit is rounded after scaling: maxima are taken over the raw logits,
 * each difference z - m is multiplied by 1/tau (on the logits path as the
 * float pair fl(1/tau) + fl(1/tau - fl(1/tau)); on the fused path by
 * fl(1/tau)) before its exponential, and the target enters as (t - M) / tau
 * formed with float pairs (~44 bits).  Every invariance above holds for a fixed tau, and
 * tau == 1 gives exactly the bits of the unscaled entry points.  temperature
 * must be finite and > 0 with 1/tau a finite positive float, else
 * LP_ERR_INVALID_ARGUMENT.  All other arguments are those of the unscaled
 * entry point of the same name; partial states from the *_partials_temperature
 * calls carry tau and merge with lp_merge_partials (a row whose states carry
 * different tau gives NaN).
 * ------------------------------------------------------------------------ */

LP_API lp_status lp_logprob_from_logits_temperature(const float* logits, int64_t ld_logits,
                                                    const int64_t* targets, int64_t T,
                                                    int64_t V, float temperature,
                                                    float* logp_out, float* entropy_out,
                                                    void* stream);

LP_API lp_status lp_logprob_partials_from_logits_temperature(
    const float* logits_shard, int64_t ld_logits, const int64_t* targets, int64_t T,
    int64_t vocab_total, int shard_index, int n_shards, float temperature, float* partials_out,
    void* stream);

LP_API lp_status lp_linear_logprob_temperature(const void* H, int64_t ld_h, const void* W,
                                               int64_t ld_w, const int64_t* targets, int64_t T,
                                               int64_t d, int64_t V, float temperature,
                                               float* logp_out, float* entropy_out,
                                               void* workspace, size_t workspace_bytes,
                                               void* stream);

LP_API lp_status lp_linear_logprob_partials_temperature(
    const void* H, int64_t ld_h, const void* W_shard, int64_t ld_w, const int64_t* targets,
    int64_t T, int64_t d, int64_t vocab_total, int shard_index, int n_shards, float temperature,
    float* partials_out, void* workspace, size_t workspace_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Backward of the logits path: the gradient of
 *     L = sum_t grad_logp[t] * logp[t] + grad_entropy[t] * entropy[t]
 * with respect to the logits, for logp and entropy of softmax(z / tau) (the
 * trainer of the RL-Kernel H100 PCP evidence record back-propagates through
 * the log-probabilities it computes; h100-pcp.json, section "comparison").
 * With log p = z / tau - log Z and p = exp(log p):
 *     dL/dz[t, v] = (grad_logp[t] (delta(v, y_t) - p) -
 *                    grad_entropy[t] p (log p + entropy[t])) / tau,
 * a term with p = 0 being 0 and a row whose target is outside [0, V)
 * contributing no logp term.  Rows are independent and every element is
 * computed alone, so the bits do not depend on T or the row's offset.
 * ------------------------------------------------------------------------ */

/*
 * lp_logprob_from_logits_lse: lp_logprob_from_logits_temperature (same bits)
 * that also writes lse_out[t] = log Z = log sum_v exp(z[t, v] / tau) (float32
 * [T]); keep lse_out and entropy_out for lp_logprob_from_logits_backward.
 * All three outputs are required.
 */
LP_API lp_status lp_logprob_from_logits_lse(const float* logits, int64_t ld_logits,
                                            const int64_t* targets, int64_t T, int64_t V,
                                            float temperature, float* logp_out,
                                            float* entropy_out, float* lse_out, void* stream);

/*
 * lp_logprob_from_logits_backward:
 *   logits, ld_logits, targets, T, V, temperature: as in
 *               lp_logprob_from_logits_temperature.
 *   saved_lse, saved_entropy  [T] float32 from lp_logprob_from_logits_lse on
 *               the same logits, targets and temperature (required).
 *   grad_logp, grad_entropy   [T] float32 upstream gradients, each NULL for
 *               zero; at least one must be given.
 *   grad_logits [T, V] float32 output, row stride ld_grad >= V elements; it
 *               must not overlap the logits.  Rows and the logits' rows need
 *               not be 16-byte aligned (aligned rows use 16-byte accesses).
 * One pass over the logits: 8 T V bytes of HBM traffic.  Errors: as the
 * other logits-path calls; an overlap of grad_logits and logits is
 * LP_ERR_INVALID_ARGUMENT.
 */
LP_API lp_status lp_logprob_from_logits_backward(const float* logits, int64_t ld_logits,
                                                 const int64_t* targets, int64_t T, int64_t V,
                                                 float temperature, const float* saved_lse,
                                                 const float* saved_entropy,
                                                 const float* grad_logp,
                                                 const float* grad_entropy, float* grad_logits,
                                                 int64_t ld_grad, void* stream);

/*
 * Vocabulary-parallel training on the logits path.  Each rank merges the
 * all-gathered quarter states with lp_merge_partials_lse, which also writes
 * log Z per row, and then takes the gradient of its own shard of the logits
 * with lp_logprob_partials_from_logits_backward: every element depends only on
 * its logit and the row's log Z and entropy, so the shards' gradients are the
 * columns of the single-GPU gradient, bit for bit, with no further exchange.
 *
 * lp_merge_partials_lse: lp_merge_partials (same bits) that also writes
 *   lse_out[t] = log Z (float32 [T]); all three outputs are required.
 * lp_logprob_partials_from_logits_backward: lp_logprob_from_logits_backward
 *   over the shard lp_vocab_shard_range(vocab_total, shard_index, n_shards) of
 *   the logits; logits_shard and grad_shard are [T, end - begin] (row strides
 *   ld_logits and ld_grad), targets are global vocabulary indices, and
 *   saved_lse / saved_entropy are the merged rows' (lp_merge_partials_lse).
 */
LP_API lp_status lp_merge_partials_lse(const float* const* shard_partials, int n_shards,
                                       int64_t T, float* logp_out, float* entropy_out,
                                       float* lse_out, void* stream);

LP_API lp_status lp_logprob_partials_from_logits_backward(
    const float* logits_shard, int64_t ld_logits, const int64_t* targets, int64_t T,
    int64_t vocab_total, int shard_index, int n_shards, float temperature,
    const float* saved_lse, const float* saved_entropy, const float* grad_logp,
    const float* grad_entropy, float* grad_shard, int64_t ld_grad, void* stream);

/* ------------------------------------------------------------------------
 * Backward of the fused path: gradients of
 *     L = sum_t grad_logp[t] * logp[t] + grad_entropy[t] * entropy[t]
 * with respect to H and W, for logp and entropy of softmax(H W^T / tau).
 * The trainer of the RL-Kernel H100 PCP evidence record back-propagates
 * through these log-probabilities (h100-pcp.json, section "comparison",
 * train/grad_norm).  With p = softmax(z / tau),
 *     G[t, v] = (grad_logp[t] (delta(v, y_t) - p[t, v])
 *                - grad_entropy[t] p[t, v] (log p[t, v] + entropy[t])) / tau,
 *     grad_H = G W,   grad_W = G^T H.
 * G is formed in fp32 from recomputed logits and rounded to bf16 for the two
 * tensor-core products (fp32 accumulation).  Results are deterministic; a row
 * of grad_H depends only on that row's inputs.  A row whose target is outside
 * [0, V) contributes no logp gradient.  grad_H is summed over fixed
 * vocabulary ranges in a fixed order: when V % 64 == 0, seven ranges per
 * quarter of the vocabulary (the quarters of the forward's reduction tree),
 * summed in order, and the quarter sums as (Q0 + Q1) + (Q2 + Q3), which is
 * what lets a vocabulary-parallel backward reproduce it (below); otherwise 19
 * ranges of the whole vocabulary, summed in order.
 * ------------------------------------------------------------------------ */

/* Workspace bytes of lp_linear_logprob_backward: the forward's workspace, the
 * bf16 G [T, V] (2 T V bytes) and the fp32 partial grad_H (28 of T d floats
 * when V % 64 == 0, else 19); 0 for invalid sizes. */
LP_API size_t lp_linear_logprob_backward_workspace_size(int64_t T, int64_t d, int64_t V);

/*
 * lp_linear_logprob_lse: lp_linear_logprob_temperature that also writes, per
 * row, lse_out[t] = log sum_v exp(z[t, v] / tau) (float32 [T], formed as
 * M / tau + log S with float pairs and rounded once).  Keep lse_out
 * and entropy_out from the forward pass and hand them to the backward to skip
 * its forward recomputation.  All three outputs are required.
 */
LP_API lp_status lp_linear_logprob_lse(const void* H, int64_t ld_h, const void* W, int64_t ld_w,
                                       const int64_t* targets, int64_t T, int64_t d, int64_t V,
                                       float temperature, float* logp_out, float* entropy_out,
                                       float* lse_out, void* workspace, size_t workspace_bytes,
                                       void* stream);

/*
 * lp_linear_logprob_backward:
 *   H, ld_h, W, ld_w, targets, T, d, V, temperature: as in
 *               lp_linear_logprob_temperature (temperature 1: no scaling);
 *               T <= 2^24.
 *   saved_lse, saved_entropy  [T] float32 from lp_linear_logprob_lse on the
 *               same inputs and temperature, or both NULL (the backward then
 *               recomputes them; the results are the same bits either way).
 *   grad_logp   [T] float32 upstream gradient of logp, or NULL (zero).
 *   grad_entropy [T] float32 upstream gradient of entropy, or NULL (zero);
 *               at least one of the two must be given.
 *   grad_H      [T, d] float32 output, dense rows (stride d), 16-byte aligned.
 *   grad_W      [V, d] float32 output, dense rows (stride d), 16-byte aligned,
 *               or NULL to skip it.
 *   workspace   device memory, 256-byte aligned, at least
 *               lp_linear_logprob_backward_workspace_size(T, d, V) bytes.
 * If a device-side wait gives up, lp_get_device_error reports it; grad_W is
 * then NaN, and so is grad_H unless the wait was in the grad_W product (the
 * last kernel of the call, whose failure leaves grad_H exact).
 */
LP_API lp_status lp_linear_logprob_backward(const void* H, int64_t ld_h, const void* W,
                                            int64_t ld_w, const int64_t* targets, int64_t T,
                                            int64_t d, int64_t V, float temperature,
                                            const float* saved_lse, const float* saved_entropy,
                                            const float* grad_logp, const float* grad_entropy,
                                            float* grad_H, float* grad_W, void* workspace,
                                            size_t workspace_bytes, void* stream);

/* Element type of grad_W for lp_linear_logprob_backward_ex, and whether it is
 * written or added to. */
typedef enum lp_grad_w_dtype {
  LP_GRAD_W_FLOAT32 = 0,   /* float32 [V, d], written */
  LP_GRAD_W_BFLOAT16 = 1,  /* bfloat16 [V, d], each element the float32 result rounded to
                              nearest even, written */
  LP_GRAD_W_FLOAT32_ACCUMULATE = 2  /* float32 [V, d] that already holds a gradient (a
                              trainer's main gradient): grad_W[v, k] + (G^T H)[v, k] is
                              stored in it, one float32 add per element made by the TMA
                              unit's reduction (round to nearest; the same bits on every
                              run) */
} lp_grad_w_dtype;

/*
 * lp_linear_logprob_backward_ex: lp_linear_logprob_backward with the element
 * type of grad_W chosen by grad_W_dtype (an lp_grad_w_dtype).  With
 * LP_GRAD_W_BFLOAT16, grad_W is [V, d] bfloat16 (dense rows, 16-byte aligned):
 * the same float32 products rounded once to bf16 on the way out, which halves
 * the product's 4 V d bytes of output (the trainer of the RL-Kernel H100 PCP
 * evidence record keeps bf16 weights; its fp32 main gradients can accumulate
 * these).  With LP_GRAD_W_FLOAT32_ACCUMULATE the product is added into the
 * float32 grad_W the caller passes (gradient accumulation over micro-batches
 * without a second pass over 4 V d bytes).  If a device-side wait gives up,
 * grad_W is NaN (also when accumulating: the previous contents are lost).
 * Other arguments as in lp_linear_logprob_backward; an unknown dtype gives
 * LP_ERR_INVALID_ARGUMENT.
 */
LP_API lp_status lp_linear_logprob_backward_ex(const void* H, int64_t ld_h, const void* W,
                                               int64_t ld_w, const int64_t* targets, int64_t T,
                                               int64_t d, int64_t V, float temperature,
                                               const float* saved_lse, const float* saved_entropy,
                                               const float* grad_logp, const float* grad_entropy,
                                               float* grad_H, void* grad_W, int grad_W_dtype,
                                               void* workspace, size_t workspace_bytes,
                                               void* stream);

/*
 * Vocabulary-parallel training on the fused path (the RL-Kernel logprob
 * report grades TP4 against TP1 bit for bit: report.json,
 * candidates.*.tp4_equals_tp1).  W is split by rows into the shards of
 * lp_vocab_shard_range; every rank holds all of H, the targets and the
 * merged rows' log Z and entropy (lp_merge_partials_lse over the all-gathered
 * quarter states of lp_linear_logprob_partials).  Each rank then calls
 * lp_linear_logprob_partials_backward on its shard, which writes
 *   grad_W_shard = G_shard^T H, the rows of the single-GPU grad_W, and
 *   grad_H_partial = the quarter-tree subtree of the shard's quarters
 *                    (Q_i, or Q_i + Q_i+1 for two shards),
 * and the ranks all-gather the partials in shard order and merge them with
 * lp_merge_grad_h_partials (P0, P0 + P1, or (P0 + P1) + (P2 + P3)): grad_H and
 * the concatenated grad_W are the bits of lp_linear_logprob_backward on one
 * GPU.  The exchange moves bytes only (4 T d per rank).
 *
 * lp_linear_logprob_partials_backward:
 *   H, ld_h, targets, T, d, temperature: as in lp_linear_logprob_backward;
 *               targets are global vocabulary indices.
 *   W_shard, ld_w  the shard's rows [end - begin, d] of W.
 *   vocab_total, shard_index, n_shards  the shard (as lp_vocab_shard_range);
 *               n_shards > 1 needs vocab_total % 64 == 0 (the quarters must
 *               start on 16-column boundaries), else LP_ERR_INVALID_ARGUMENT.
 *   saved_lse, saved_entropy  [T] float32 of the merged rows (required).
 *   grad_logp, grad_entropy   as in lp_linear_logprob_backward.
 *   grad_H_partial [T, d] float32 output, dense rows, 16-byte aligned.
 *   grad_W_shard   [end - begin, d] output of grad_W_dtype (an lp_grad_w_dtype:
 *               written as float32 or bfloat16, or added into a float32 main
 *               gradient), dense rows, 16-byte aligned, or NULL to skip it.
 *   workspace   256-byte aligned, at least
 *               lp_linear_logprob_partials_backward_workspace_size(T, d,
 *               vocab_total, n_shards) bytes.
 * With n_shards == 1 it is lp_linear_logprob_backward_ex with saved
 * statistics (same bits).  Device-side timeouts: as lp_linear_logprob_backward
 * (NaN outputs; lp_get_device_error on the workspace).
 */
LP_API size_t lp_linear_logprob_partials_backward_workspace_size(int64_t T, int64_t d,
                                                                 int64_t vocab_total,
                                                                 int n_shards);

LP_API lp_status lp_linear_logprob_partials_backward(
    const void* H, int64_t ld_h, const void* W_shard, int64_t ld_w, const int64_t* targets,
    int64_t T, int64_t d, int64_t vocab_total, int shard_index, int n_shards, float temperature,
    const float* saved_lse, const float* saved_entropy, const float* grad_logp,
    const float* grad_entropy, float* grad_H_partial, void* grad_W_shard, int grad_W_dtype,
    void* workspace, size_t workspace_bytes, void* stream);

/*
 * lp_merge_grad_h_partials: grad_H [T, d] float32 (dense rows) = the n_shards
 * (1, 2 or 4) partials shard_grad_h[i] ([T, d] float32, dense rows, in shard
 * order; a host array of device pointers) added as P0, P0 + P1 or
 * (P0 + P1) + (P2 + P3).  Every pointer 16-byte aligned, d % 8 == 0.  grad_H
 * may be one of the partials.
 */
LP_API lp_status lp_merge_grad_h_partials(const float* const* shard_grad_h, int n_shards,
                                          int64_t T, int64_t d, float* grad_H, void* stream);

/* ------------------------------------------------------------------------
 * Diagnostics and tuning.
 * ------------------------------------------------------------------------ */

/*
 * lp_get_device_error: read the error word of a fused-path workspace after the
 * call that used it (synchronises `stream`).  Returns LP_OK when no
 * device-side wait gave up, LP_ERR_TIMEOUT when one did (then *word_out, if
 * not NULL, holds which pipeline role gave up: bit 0 loader, bit 1 MMA issuer,
 * bit 2 epilogue), LP_ERR_CUDA if the read failed.
 */
LP_API lp_status lp_get_device_error(const void* workspace, size_t workspace_bytes,
                              uint32_t* word_out, void* stream);

/*
 * lp_set_persistent_grid_limit: cap the number of persistent CTAs of the fused
 * kernel (0 = one per SM, the default).  Results do not depend on it: the work
 * is cut into fixed tiles whatever the grid (the single-GPU analogue of the
 * report's nccl_setting_invariant property).  Process-wide setting.
 */
LP_API lp_status lp_set_persistent_grid_limit(int max_ctas);

/*
 * lp_set_kernel_timing_events: diagnostics.  When both are non-NULL, every
 * later fused-path call records `start_event` on its stream immediately before
 * its tensor-core kernel (the dominant kernel) and `stop_event` immediately
 * after it, so a caller can time that kernel alone with cudaEventElapsedTime.
 * Arguments are cudaEvent_t handles owned by the caller; pass NULL, NULL to
 * stop recording.  Process-wide setting; not for concurrent callers.
 */
LP_API lp_status lp_set_kernel_timing_events(void* start_event, void* stop_event);

/*
 * lp_set_fault_injection: tests of the bounded device-side waits.  Mode 1:
 * every later fused forward call withholds one TMA load of its first CTA pair,
 * so that pair's pipeline waits give up after their time bound (about a second
 * each); the call still returns LP_OK, its outputs are NaN and
 * lp_get_device_error returns LP_ERR_TIMEOUT.  Mode 2: the same in the grad_W
 * product of every later backward call (grad_W is NaN, grad_H exact).  No
 * fault is raised on the device and the context stays usable.  Mode 0 (the
 * default) turns it off.  Process-wide setting; not for production use.
 */
LP_API lp_status lp_set_fault_injection(int mode);

/*
 * lp_get_check_word: the index checks of the checked build.  A library built
 * with -DLP_CHECKED (lp_backend_id() then ends in "+checked") tests, in every
 * kernel, the indexes and TMA coordinates it computes against the extents
 * derived from the call's arguments; a failed test skips the access and sets
 * a bit of a check word instead of faulting (bit 0 logit read outside its
 * quarter, 1 row outside [0, T), 2 quarter or tile state outside its buffer,
 * 3 negative TMA load coordinate, 4 store of G outside its buffer, 5 output
 * box outside C, 6 split-sum index, 7 padding or row-copy index).  This call
 * synchronises the device, writes the OR of the check words of every kernel
 * since the previous call to *word_out and clears them.  In the normal build
 * the word is always 0.  LP_ERR_CUDA if the read failed.
 */
LP_API lp_status lp_get_check_word(uint32_t* word_out);

/* Human-readable name of a status code (static storage). */
LP_API const char* lp_status_string(lp_status status);

/* Fixed identifier of this backend, "lp.sm103a.bitwise.v1" ("+checked"
 * appended in the checked build). */
LP_API const char* lp_backend_id(void);

#ifdef __cplusplus
}
#endif

#endif /* LP_H_ */
