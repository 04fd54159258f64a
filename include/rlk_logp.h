/*
 * rlk_logp.h -- C ABI of the strict, batch-invariant token-logprob operator
 * for GB300 (sm_103a).
 *
 * The operator (sources named by page title and section):
 *
 *   "Configurable H100 consistency runs", topology paragraph: the CUDA path
 *   uses a fixed virtual TP8 partition and a padded vocabulary of 152576
 *   columns whatever the physical layout.  Here the real vocabulary is the
 *   first 151936 columns; the 640 padded columns are never read.
 *
 *   "Reproduce and profile the Qwen3-8B TP4/CP2 experiment", section "How
 *   non-default CUDA topology reuses TP4/CP2": every vocabulary shard yields a
 *   summary, and the summaries combine in one fixed order of vocabulary
 *   position.  Here each of
 *   the 8 shards of 19072 columns emits a (max, sum-exp) pair built in a fixed
 *   reduction tree and the pairs merge as a left fold over shard index 0..7.
 *
 *   "Configurable H100 consistency runs", sampling-flags paragraph: float32
 *   temperature scaling after the BF16 logits; temperature 0 is greedy;
 *   top-p in (0, 1]; top-k is -1 (off) or 1..151936; the top-p/top-k support
 *   is computed from the whole real vocabulary.  KL-reference paragraph: the
 *   reference logprob is scaled over the full vocabulary (not truncated)
 *   while the policy logprob keeps its actual top-p/top-k support.
 *
 * Per row i with target t = target[i]:
 *   full[i]    = s_t - log sum_{j < 151936} exp(s_j),  s_j = x_j / tau_i
 *   restr[i]   = s_t - log sum_{j in S} exp(s_j) if t in S, else -inf
 *   support[i] = |S|
 * S is top-k first (every token >= the k-th largest value, ties kept), then
 * top-p on the renormalised top-k distribution (token j kept iff the mass of
 * strictly larger tokens is < p of the top-k mass).  p == 1 together with
 * k == -1 (or k == 151936) disables both filters and restr == full bit for
 * bit, support == 151936.  tau == 0 (greedy): both outputs are 0 at the
 * argmax (lowest column on ties) and -inf elsewhere, support == 1.
 * A NaN or +inf among the real logits, a row that is all -inf, or a scaled
 * maximum that overflows float32 gives NaN outputs and support -1.
 *
 * Results are bit-identical for a row whatever T, the row's position in the
 * batch, or the buffer it sits in: every reduction has a fixed shape that
 * depends only on the column index.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library allocates nothing, frees nothing and never synchronises: work
 *     is enqueued on `stream` (a cudaStream_t passed as void*; NULL is the
 *     legacy default stream) and outputs are ready when the stream reaches
 *     that point.
 *   - Host-checkable faults return a status before anything is enqueued:
 *     RLK_EINVAL for a null required pointer, T < 0, row_stride <
 *     vocab_padded, vocab sizes other than 151936/152576, a scalar parameter
 *     out of its domain (used when the per-row array is NULL), or T too large
 *     for one launch (T > 2^28); RLK_EALIGN for a logits base that is not
 *     16-byte aligned, a row_stride that is not a multiple of 8 elements, or
 *     an int/float array that is not 4-byte aligned.  T == 0 returns RLK_OK
 *     with nothing enqueued.  RLK_ECUDA reports a launch failure.
 *   - Per-row parameter arrays cannot be checked on the host without a
 *     synchronisation: a row whose tau, top_p, top_k or target is out of
 *     domain gets NaN outputs, support -1, and increments *err_count (an
 *     optional device int32).  A shard load or exchange that does not
 *     complete within 0.2 s is treated the same way.
 *   - rlk_last_error() returns a message for the last non-OK status of the
 *     calling host thread.
 */
#ifndef RLK_LOGP_H
#define RLK_LOGP_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RLK_VOCAB_PADDED 152576
#define RLK_VOCAB_REAL 151936
#define RLK_NUM_SHARDS 8
#define RLK_SHARD_WIDTH 19072
#define RLK_ABI_VERSION 5

typedef enum {
  RLK_OK = 0,
  RLK_EINVAL = 1,
  RLK_EALIGN = 2,
  RLK_ECUDA = 3
} rlk_status;

typedef struct rlk_logp_args {
  /* bf16 logits, row-major: row i starts at logits + i * row_stride
   * (elements).  Only columns 0..151935 are read. */
  const void* logits;
  int64_t T;                 /* rows */
  int64_t row_stride;        /* elements between rows; >= vocab_padded, % 8 == 0 */
  int32_t vocab_real;        /* must be RLK_VOCAB_REAL */
  int32_t vocab_padded;      /* must be RLK_VOCAB_PADDED */
  const int32_t* target;     /* [T] target column per row, 0 <= t < vocab_real */
  /* Sampling parameters: a per-row device array [T], or NULL to use the
   * scalar for every row.  top_p/top_k are ignored by rlk_logp_full. */
  const float* temperature;  float temperature_scalar;  /* finite, >= 0 */
  const float* top_p;        float top_p_scalar;        /* (0, 1]      */
  const int32_t* top_k;      int32_t top_k_scalar;      /* -1 or 1..vocab_real */
  int32_t* err_count;        /* optional device counter of rejected rows */
} rlk_logp_args;

/* Per-row record of a resolved row, written by rlk_logp_pair_save and read
 * by rlk_logp_backward_saved (16 bytes, device memory, opaque to most
 * callers):
 *   max_logit      row maximum M of the real logits (a bf16 value);
 *   inv_z          1 / sum_j exp((x_j - M) / tau) over the real vocabulary;
 *                  NaN for a row whose outputs are NaN; 0 for greedy rows;
 *   inv_z_support  1 / the same sum over the support S when the target is in
 *                  S, else 0 (the restricted logprob is then -inf and has no
 *                  gradient);
 *   min_key        lowest bf16 order key in S (0 when S is the whole
 *                  vocabulary).  The order key of a bf16 bit pattern b is
 *                  b | 0x8000 for b >= 0 (and for -0), ~b & 0xFFFF for b < 0. */
typedef struct rlk_row_stats {
  float max_logit;
  float inv_z;
  float inv_z_support;
  int32_t min_key;
} rlk_row_stats;

/* Full-vocabulary logprob of the target (the KL-reference side).
 * out_full: device float[T], required. */
rlk_status rlk_logp_full(const rlk_logp_args* args, float* out_full, void* stream);

/* Top-k-then-top-p restricted, renormalised logprob (the policy side).
 * out_restr: device float[T], required.  out_support: device int32[T] or NULL. */
rlk_status rlk_logp_restricted(const rlk_logp_args* args, float* out_restr,
                               int32_t* out_support, void* stream);

/* Both sides in one pass over the logits.  Each output pointer may be NULL
 * except that at least one of out_full/out_restr must be given. */
rlk_status rlk_logp_pair(const rlk_logp_args* args, float* out_full, float* out_restr,
                         int32_t* out_support, void* stream);

/* Policy pair plus the per-row KL term of the sampled token,
 *   out_kl[i] = full_policy[i] - full_ref[i],
 * where full_ref is the full-vocabulary logprob of the same target under the
 * reference logits (same temperature; "Configurable H100 consistency runs",
 * KL-reference paragraph).  ref_logits follows the same layout rules as
 * args->logits with its own ref_row_stride.  out_full, out_full_ref and
 * out_kl are required; out_restr and out_support may be NULL.  Two launches
 * on `stream`: one cluster launch over 2T rows in which even clusters
 * resolve policy row i (full and restricted) and odd clusters the same
 * row's reference logits (full only), then a small kernel that forms the
 * difference.  Each row's results are bit-identical to rlk_logp_pair
 * followed by rlk_logp_kl_ref.  RLK_EINVAL when T >= 2^27 (the doubled
 * cluster count must stay below 2^31 CTAs). */
rlk_status rlk_logp_kl(const rlk_logp_args* policy, const void* ref_logits,
                       int64_t ref_row_stride, float* out_full, float* out_restr,
                       int32_t* out_support, float* out_full_ref, float* out_kl,
                       void* stream);

/* rlk_logp_kl on inputs that live in host memory, the copies in: the
 * rows go in `chunks` row ranges; the host-to-device copy of range c + 1
 * runs on copy_stream while the passes over range c run on `stream`, and
 * each range's results are copied back on `stream`.  The host link, not
 * the passes, then bounds the call.  Each row's results are bit-identical to
 * rlk_logp_kl on the same logits (the passes only see the rows of a range,
 * and a row's results do not depend on its batch).
 *   policy: as for rlk_logp_kl, except that policy->logits and
 *     policy->target are HOST pointers (pinned memory, or the copies cannot
 *     run beside the passes).  The per-row parameter arrays
 *     (temperature/top_p/top_k) and err_count stay device pointers or NULL.
 *   ref_logits, ref_row_stride: the reference logits in host memory.
 *   out_full, out_restr, out_support, out_full_ref, out_kl: HOST pointers,
 *     required as for rlk_logp_kl; valid once `stream` has completed.
 *   workspace: device scratch of RLK_LOGP_KL_HOST_WORKSPACE_BYTES(T) bytes,
 *     256-byte aligned: both logits tensors (real columns only, 151936 of
 *     each row are copied), the targets and the five outputs.  A call's
 *     first copy waits for the work already queued on `stream`, so
 *     consecutive calls may share one workspace on the same streams.
 *   chunks: number of row ranges, >= 1 (capped at T and at
 *     RLK_KL_HOST_MAX_CHUNKS).
 *   copy_stream: the stream for the host-to-device copies; NULL (or equal
 *     to `stream`) runs everything on `stream`, with no overlap.
 * Asynchronous: no host synchronisation; the library allocates no memory
 * (it creates and releases a few CUDA events).  RLK_EINVAL for missing
 * pointers or chunks < 1, RLK_EALIGN for a misaligned workspace, RLK_ECUDA
 * for a failed copy, event or launch. */
#define RLK_KL_HOST_MAX_CHUNKS 4096
#define RLK_LOGP_KL_HOST_WORKSPACE_BYTES(T) ((size_t)(T) * 610304u + 6u * ((((size_t)(T) * 4u) + 255u) & ~(size_t)255u))
rlk_status rlk_logp_kl_host(const rlk_logp_args* policy, const void* ref_logits,
                            int64_t ref_row_stride, float* out_full, float* out_restr,
                            int32_t* out_support, float* out_full_ref, float* out_kl,
                            void* workspace, int32_t chunks, void* stream, void* copy_stream);

/* The reference half of rlk_logp_kl on its own: the full-vocabulary logprob
 * of each row's target under ref->logits, and out_kl[i] = full_policy[i] -
 * out_full_ref[i] with full_policy an earlier result of rlk_logp_full/pair
 * on the same stream.  ref carries the reference logits, targets and
 * temperatures (top_p/top_k are ignored).  full_policy, out_full_ref and
 * out_kl are required device float[T]. */
rlk_status rlk_logp_kl_ref(const rlk_logp_args* ref, const float* full_policy,
                           float* out_full_ref, float* out_kl, void* stream);

/* Backward: the gradient of  g_full[i] * full[i] + g_restr[i] * restr[i]
 * with respect to the logits, in one pass that also recomputes the forward
 * (the training side differentiates the very logprobs the rollout side
 * scored; "H100 canonical CP backward validation" asks for gradients that are
 * identical whatever the training topology, and this one is a function of
 * the row alone).  With p the softmax of x / tau over the real vocabulary
 * and q the softmax over the support S (0 outside it):
 *   grad[i, j] = ( g_full (1[j == t] - p_j)
 *                + g_restr 1[j in S] (1[j == t] - q_j) ) / tau
 * The support is locally constant: no gradient flows through the
 * thresholds.  The restricted term is 0 when t is not in S (restr is the
 * constant -inf there).  Greedy rows (tau == 0) get a zero gradient; padded
 * columns get 0; a row whose outputs are NaN (non-finite logits, rejected
 * parameters, timeout) gets NaN on every real column.
 *   grad_full, grad_restr: device float[T] upstream gradients; either may be
 *     NULL (read as 0) but not both.
 *   grad_logits: device [T, grad_row_stride] of grad_dtype, 16-byte aligned,
 *     grad_row_stride >= 152576 with rows a multiple of 16 bytes apart; all
 *     152576 columns of each row are written.  It may not overlap the logits.
 *   out_full / out_restr / out_support: optional forward outputs (NULL to
 *     skip).  top_p / top_k are used (and validated) when grad_restr,
 *     out_restr or out_support is given; otherwise the pass is full-only.
 * One launch on `stream`; reads the logits once and writes the gradient
 * once. */
typedef enum { RLK_GRAD_BF16 = 0, RLK_GRAD_F32 = 1 } rlk_grad_dtype;

rlk_status rlk_logp_backward(const rlk_logp_args* args, const float* grad_full,
                             const float* grad_restr, void* grad_logits, int64_t grad_row_stride,
                             int32_t grad_dtype, float* out_full, float* out_restr,
                             int32_t* out_support, void* stream);

/* rlk_logp_pair plus the per-row record a later backward needs (the usual
 * training order: the forward runs first, the backward later).  out_stats:
 * device rlk_row_stats[T], 16-byte aligned, required; the other outputs as in
 * rlk_logp_pair (at least one of out_full/out_restr). */
rlk_status rlk_logp_pair_save(const rlk_logp_args* args, float* out_full, float* out_restr,
                              int32_t* out_support, rlk_row_stats* out_stats, void* stream);

/* The same gradient as rlk_logp_backward, bit for bit, from a saved record:
 * a streaming pass that reads the logits once and writes the gradient once.
 * args carries the logits, targets and temperatures of the saved forward
 * (top_p/top_k are not read: the support is in the record).  stats: device
 * rlk_row_stats[T] from rlk_logp_pair_save on the same logits and
 * parameters, 16-byte aligned.  grad_full, grad_restr, grad_logits,
 * grad_row_stride and grad_dtype as in rlk_logp_backward.  A row whose record
 * is NaN (a rejected or non-finite row) gets NaN on every real column. */
rlk_status rlk_logp_backward_saved(const rlk_logp_args* args, const rlk_row_stats* stats,
                                   const float* grad_full, const float* grad_restr,
                                   void* grad_logits, int64_t grad_row_stride, int32_t grad_dtype,
                                   void* stream);

/* Sampler: draw one token per row from the same restricted distribution the
 * logprobs use (the rollout side; "Configurable H100 consistency runs",
 * sampling flags: temperature 0 is greedy, top-k then top-p over the real
 * vocabulary), so that the sampled token's restricted logprob is the one the
 * training side later recomputes.  The draw is inverse-CDF sampling with the
 * support in ascending column order: with U = u / 2^32 for a 32-bit random
 * word u, the token is the smallest column a in S whose cumulative
 * renormalised mass exceeds U.  Rows with top-k or top-p use the exact
 * fixed-point integers of the support selection as masses; rows without
 * either (S = every real token) use float masses exp((x - M) / tau) summed in
 * a fixed order (per 16-byte chunk, per 32-chunk word relative to the shard
 * maximum, then a scan over the words) with U = (u >> 8) / 2^24.  Either way
 * the draw is a function of the row and u alone.  Greedy rows give the argmax
 * (lowest column on ties).
 *   args: logits and per-row temperature / top_p / top_k as for
 *     rlk_logp_pair; args->target is not read (may be NULL).
 *   u per row: uniform[i] if uniform is not NULL, else word 0 of
 *     Philox4x32-10 (Salmon et al., SC 2011) with key (seed low, seed high)
 *     and counter (counter[i] low, counter[i] high, 0, 0).  Give each
 *     (request, position) its own counter and the draw does not depend on
 *     the batch.  counter: device uint64[T], 8-byte aligned; uniform: device
 *     uint32[T]; at least one of them.
 *   out_token: device int32[T], required: the sampled column; -1 for a row
 *     whose outputs are NaN (rejected parameters, non-finite logits).
 *   out_restr / out_full: optional float[T]: the sampled token's restricted
 *     and full logprobs, bit-identical to rlk_logp_pair with target = token.
 *   out_support: optional int32[T], as in rlk_logp_pair.
 *   workspace: device scratch of RLK_SAMPLE_WORKSPACE_BYTES(T) bytes,
 *     16-byte aligned, owned by the caller: the pair pass leaves a 16-byte
 *     record per row there for the draw, then (from byte 16 T on, 2432 bytes
 *     per row) for a filtered row one bit per 16-byte chunk marking the
 *     chunks that reach the row's candidate window, for an unfiltered row
 *     the float mass of every 32-chunk word and the shard maxima.  Its
 *     contents on entry do not matter; calls that share a workspace must not
 *     overlap on the GPU.
 * A row whose support reaches below the 1024-key window is resolved exactly
 * (slower path), as in rlk_logp_pair.  Two launches on `stream`: the pair
 * pass that resolves every row (greedy and NaN rows finish there), then one
 * block per drawing row, which reads the marked chunks when a filtered
 * row's support lies inside its candidate window, every real chunk for a
 * wider support, and for an unfiltered row the word masses and then the one
 * word the draw lands in; each case computes the same masses in the same
 * order as a read of every chunk would, so the result does not depend on
 * which chunks are read. */
#define RLK_SAMPLE_WORKSPACE_BYTES(T) ((size_t)(T) * (16u + 2432u))

rlk_status rlk_sample(const rlk_logp_args* args, unsigned long long seed,
                      const unsigned long long* counter, const uint32_t* uniform,
                      int32_t* out_token, float* out_restr, float* out_full,
                      int32_t* out_support, void* workspace, void* stream);

/* rlk_sample without a workspace argument, for callers that cannot allocate
 * device memory when they call (their memory belongs to a framework
 * allocator or a fixed plan, e.g. an inference-engine plugin at enqueue
 * time, where a cudaMalloc would bypass the plan and may synchronise the
 * device).  The pages have no counterpart: this is a packaging of
 * rlk_sample, with the same arguments (minus workspace) and results.
 *   Scratch: a fixed array inside the library, RLK_SAMPLE_NOALLOC_MAX_ROWS x
 *     16 bytes (1 MiB) of device memory on every GPU that loads the library,
 *     held until the process exits.  T above RLK_SAMPLE_NOALLOC_MAX_ROWS is
 *     rejected with RLK_EINVAL (split the batch, or use rlk_sample).
 *   Set-up: every call looks up the array's device address on the current
 *     device (cudaGetSymbolAddress, no stream work).  The first call on a
 *     device also loads the library's device code there: make that first
 *     call before any stream capture.  Nothing is allocated by any call.
 *   Sharing: every call on a device uses the same array.  Each call writes
 *     every record it reads, so leftovers from an earlier call never matter,
 *     but calls that overlap on the GPU (different streams, or host threads
 *     sharing a device) race on the array: order them. */
#define RLK_SAMPLE_NOALLOC_MAX_ROWS 65536

rlk_status rlk_sample_noalloc(const rlk_logp_args* args, unsigned long long seed,
                              const unsigned long long* counter, const uint32_t* uniform,
                              int32_t* out_token, float* out_restr, float* out_full,
                              int32_t* out_support, void* stream);

/* Full-vocabulary logprob straight from the LM head, without storing the
 * logits (the KL-reference side, "Configurable H100 consistency runs",
 * KL-reference paragraph: the reference is scaled over the whole real
 * vocabulary).  x = h . W^T is formed on the tensor cores (bf16 products,
 * fp32 accumulation in a fixed K order), each 128-row x 256-column tile of x
 * is reduced to one (max, sum-exp) pair per row, and the 596 tiles of a row
 * are folded in a fixed order:  full[i] = (x_it - M_i) / tau_i - ln Z_i.
 * The logits keep fp32 precision (they are not rounded to bf16), so results
 * differ from rlk_logp_full on bf16 logits by that rounding.
 *   hidden: bf16 [T, hidden_stride], H columns used; weight: bf16
 *     [152576, weight_stride] (the padded LM head; rows >= 151936 ignored).
 *     Both 16-byte aligned, strides multiples of 8 elements; H a multiple of
 *     64.
 *   target: int32 [T]; temperature: per-row float [T] or the scalar (> 0).
 *   out_full: float [T].
 *   workspace: RLK_LINEAR_WORKSPACE_BYTES(T) bytes of device scratch,
 *     16-byte aligned (per-row tile summaries and the target's logit).
 *   Rows with a rejected temperature or target get NaN and count in
 *     err_count (optional).
 * Two launches on `stream`. */
#define RLK_LINEAR_WORKSPACE_BYTES(T) ((size_t)(T) * (596u * 8u + 4u))

rlk_status rlk_linear_logp(const void* hidden, int64_t T, int64_t H, int64_t hidden_stride,
                           const void* weight, int64_t weight_stride, const int32_t* target,
                           const float* temperature, float temperature_scalar, float* out_full,
                           void* workspace, int32_t* err_count, void* stream);

/* Full and restricted logprob straight from the LM head, without storing the
 * logits: the policy side keeps its top-k-then-top-p support while the
 * reference side is scaled over the whole vocabulary ("Configurable H100
 * consistency runs", KL-reference and sampling-flags paragraphs).  The
 * logits are the fp32 x = h . W^T of rlk_linear_logp, s = x / tau, and
 * full, restr and support follow the definitions at the top of this file on
 * those fp32 values (order keys of fp32; -0 ties with +0); the nucleus uses
 * the fixed-point masses of rlk_logp_pair (exp(s_j - s_max) in units of
 * 2^-44, Z_k their exact sum; without top-k, Z_k is the float normaliser of
 * the full side scaled to those units).  out_full is bit-identical to
 * rlk_linear_logp.
 *   hidden, weight, H, strides, target, temperature: as rlk_linear_logp
 *     (tau > 0: no greedy rows).
 *   top_p / top_k: per-row device arrays [T] or NULL for the scalars, domains
 *     as in rlk_logp_args.
 *   out_restr: float [T], required; out_full: float [T] or NULL; out_support:
 *     int32 [T] or NULL.
 *   workspace: RLK_LINEAR_PAIR_WORKSPACE_BYTES(T) bytes of device scratch,
 *     256-byte aligned (tile summaries, the 8 largest logits of every
 *     256-column tile, per-row search state, bucket counts and listed keys).
 * The support is found by exact selection over the fp32 order keys.  The
 * first GEMM pass keeps each tile's 8 largest logits; a row whose first
 * window (top-k: at or above the k-th largest tile maximum, else the k-th
 * largest kept logit; top-p alone: the a-priori mass bound) they provably
 * contain is resolved from them.  Other rows go through rounds that
 * recompute the GEMM for the row tiles holding them, histogramming and
 * listing the keys of each row's current window (at most five rounds per
 * stage).  One memset and 3 + 2 x 12 launches on `stream`; rounds with no
 * unresolved row do no GEMM work.  A rejected row gets NaN outputs, support
 * -1 and counts in err_count; a row with a NaN or infinite logit gets NaN
 * restr and support -1; a wait that gives up leaves NaN and counts in
 * err_count; a row still unresolved after the last round (not expected) gets
 * NaN and support -2. */
#define RLK_LINEAR_PAIR_WORKSPACE_BYTES(T) ((size_t)(T) * 52640u + 4096u)

rlk_status rlk_linear_logp_pair(const void* hidden, int64_t T, int64_t H, int64_t hidden_stride,
                                const void* weight, int64_t weight_stride, const int32_t* target,
                                const float* temperature, float temperature_scalar, const float* top_p,
                                float top_p_scalar, const int32_t* top_k, int32_t top_k_scalar,
                                float* out_full, float* out_restr, int32_t* out_support, void* workspace,
                                int32_t* err_count, void* stream);

/* ---------------------------------------------------------------------
 * Vocabulary-sharded form: the fixed virtual TP8 partition with each shard
 * in its own buffer, as a tensor-parallel rank would hold it ("Reproduce and
 * profile the Qwen3-8B TP4/CP2 experiment", section "How non-default CUDA
 * topology reuses TP4/CP2": every shard yields a summary and the summaries
 * combine in one fixed vocabulary order).
 *
 * Phase 1: rlk_logp_shard_summary on each shard (on whichever device holds
 * it); gather the [T] outputs of the 8 shards into shard-major [8][T] arrays
 * (the summary exchange of the tensor-parallel setting); rlk_logp_merge then
 * gives the full logprob, bit-identical to rlk_logp_full/pair on the whole
 * row.  Phase 2 (restricted side): rlk_logp_shard_counts on each shard with
 * the gathered summaries, then rlk_logp_merge with the counts of all shards
 * gives the restricted logprob and support, bit-identical to rlk_logp_pair
 * for every row whose support lies within 1024 order keys of the row maximum
 * (8 binades of bf16); other rows get NaN and support -2 (the fused entry
 * points resolve them by re-reading the row).
 *
 * Rows are validated as in rlk_logp_pair.  A rejected row gets NaN summaries
 * and NaN outputs with support -1; only shard 0 increments err_count, so one
 * pass over the 8 shards counts each rejected row once.
 * ------------------------------------------------------------------- */

typedef struct rlk_shard_args {
  /* bf16 [T, row_stride]: the shard's columns; column 0 is vocabulary column
   * 19072*shard.  Shards 0..6 read 19072 columns, shard 7 its 18432 real
   * ones.  Base 16-byte aligned. */
  const void* logits;
  int64_t T;                 /* rows, < 2^31 */
  int64_t row_stride;        /* elements; >= 19072, % 8 == 0 */
  int32_t shard;             /* 0..7 */
  const int32_t* target;     /* [T] target column in the whole vocabulary */
  const float* temperature;  float temperature_scalar;
  const float* top_p;        float top_p_scalar;
  const int32_t* top_k;      int32_t top_k_scalar;
  int32_t* err_count;        /* optional; counted by shard 0 only */
} rlk_shard_args;

/* Per-row summary of one shard, each output a device [T] array:
 *   out_max     the shard maximum of the logits (a bf16 value; -inf if all
 *               -inf; NaN for a rejected row);
 *   out_sumexp  sum over the shard of exp((x_j - out_max) / tau) in the fixed
 *               tree of the fused kernel (NaN if the shard holds a NaN or for
 *               a rejected row, 0 for greedy rows);
 *   out_aux     greedy rows: first vocabulary column holding the shard
 *               maximum; rows with 1 <= k <= 1024: the shard's top-k witness
 *               (an order key); otherwise 0;
 *   out_target_logit  the target's logit, written only for rows whose target
 *               lies in this shard (other entries are left untouched);
 *   out_chunk_max  optional (NULL: not written), device uint16 [T][2384],
 *               16-byte aligned: the maximum (bf16 bits) of each 16-byte chunk
 *               (8 columns) of the shard, for rlk_logp_shard_counts; shard 7
 *               writes its 2304 real chunks. */
#define RLK_SHARD_CHUNKS 2384

rlk_status rlk_logp_shard_summary(const rlk_shard_args* args, float* out_max, float* out_sumexp,
                                  int32_t* out_aux, float* out_target_logit, uint16_t* out_chunk_max,
                                  void* stream);

/* Per-row exact counts of this shard's tokens on the row's candidate window
 * (at most 1024 order keys below the row maximum, derived from the 8
 * summaries exactly as the fused kernel derives it).  maxes, sumexps, aux
 * are the gathered shard-major [8][T] phase-1 outputs.  chunk_max: optional,
 * this shard's out_chunk_max from phase 1; given, only the chunks whose
 * maximum reaches the window are read (a few percent of the shard on typical
 * rows) instead of the whole shard, with the same counts.  out_counts: device
 * uint32 [T][1024], 16-byte aligned; entry i counts the tokens whose bf16
 * order key is the row maximum's key minus i (zero beyond the window and for
 * rows without a top-k or top-p filter). */
rlk_status rlk_logp_shard_counts(const rlk_shard_args* args, const float* maxes,
                                 const float* sumexps, const int32_t* aux,
                                 const uint16_t* chunk_max, uint32_t* out_counts, void* stream);

/* Merge of the 8 summaries of every row in fixed shard order.
 *   maxes, sumexps, aux: shard-major [8][T]; target_logit: [T] (from the
 *   shard holding each target); target, temperature/top_p/top_k as in
 *   rlk_shard_args (per-row array or scalar).
 *   out_full: [T] full logprob (required).
 *   counts == NULL: full logprob only (top_p/top_k ignored).  Otherwise
 *   count_shards (1 or 8) count arrays of [T][1024] each, summed here (pass
 *   1 if they were already summed across shards), and out_restr /
 *   out_support (at least one given) receive the restricted logprob and the
 *   support size. */
rlk_status rlk_logp_merge(const float* maxes, const float* sumexps, const int32_t* aux,
                          const float* target_logit, int64_t T, const int32_t* target,
                          const float* temperature, float temperature_scalar,
                          const float* top_p, float top_p_scalar,
                          const int32_t* top_k, int32_t top_k_scalar,
                          const uint32_t* counts, int32_t count_shards,
                          float* out_full, float* out_restr, int32_t* out_support,
                          void* stream);

/* Rows whose support reaches below the first window.  rlk_logp_merge cannot
 * resolve a row whose top-k or top-p threshold lies more than 1024 order keys
 * below the row maximum (support -2): the fused kernel re-reads such a row,
 * a shard holder cannot.  The resumable pair below continues such rows over
 * successive lower windows of 1024 keys, the caller counting each window on
 * every shard in between, exactly as the fused kernel's fallback walks them
 * (top-k first, from the top; then the nucleus, from the top again), so the
 * results are bit-identical to rlk_logp_pair.  Same sources as the merge:
 * each shard yields a summary and the summaries combine in a fixed order of
 * vocabulary position ("Reproduce and profile the Qwen3-8B TP4/CP2
 * experiment", "How non-default CUDA topology reuses TP4/CP2").
 *
 * Per-row state, device [T], caller-owned, zeroed by the caller before the
 * first merge call (stage 0 = the first window). */
typedef struct rlk_merge_state {
  int32_t stage;      /* 0 first window; 1 toward the k-th largest value; 2 toward the nucleus
                         threshold; 3 resolved (the row's outputs are final) */
  int32_t hi, lo;     /* stages 1, 2: the window (order keys, inclusive) the next counts cover */
  int32_t vk_key;     /* stage 2: lowest order key of the top-k set (-1: top-k off) */
  uint32_t carry_c;   /* tokens above the window, in the current stage */
  uint32_t pad;
  uint64_t carry_m;   /* their mass, exp((x - M) / tau) in 2^-44 fixed point */
  uint64_t zk;        /* stage 2: mass of the top-k set in the same units */
} rlk_merge_state;

/* rlk_logp_merge for restricted rows with a resolution state.  counts must
 * hold, per row, the counts of the window its state names: for stage-0 rows
 * rlk_logp_shard_counts' first window, for stage-1/2 rows
 * rlk_logp_shard_counts_window's.  Rows in stage 3 are skipped (outputs and
 * state untouched).  A row resolved by this call gets its outputs and stage
 * 3; a row that needs a lower window gets restricted NaN, support -2 and the
 * window in its state, and counts one in out_pending (optional device
 * int32, added to: zero it before the call).  Repeat counts + merge until no
 * row is pending (at most 2 * 64 rounds; one or two in practice).  Other
 * arguments and errors as rlk_logp_merge (counts required). */
rlk_status rlk_logp_merge_resumable(const float* maxes, const float* sumexps, const int32_t* aux,
                                    const float* target_logit, int64_t T, const int32_t* target,
                                    const float* temperature, float temperature_scalar,
                                    const float* top_p, float top_p_scalar,
                                    const int32_t* top_k, int32_t top_k_scalar,
                                    const uint32_t* counts, int32_t count_shards,
                                    rlk_merge_state* state, float* out_full, float* out_restr,
                                    int32_t* out_support, int32_t* out_pending, void* stream);

/* Per-row exact counts of this shard's real tokens on the window that each
 * row's state names (stages 1 and 2: order keys state.lo .. state.hi, entry i
 * counting key state.hi - i); rows in stages 0 and 3 get zeros.  chunk_max as
 * in rlk_logp_shard_counts (optional; given, only chunks whose maximum
 * reaches state.lo are read).  out_counts: device uint32 [T][1024], 16-byte
 * aligned. */
rlk_status rlk_logp_shard_counts_window(const rlk_shard_args* args, const rlk_merge_state* state,
                                        const uint16_t* chunk_max, uint32_t* out_counts, void* stream);

/* Static message for a status code. */
const char* rlk_status_string(rlk_status status);

/* Message for the last non-OK status returned on the calling host thread. */
const char* rlk_last_error(void);

/* RLK_ABI_VERSION of the built library. */
int rlk_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* RLK_LOGP_H */
