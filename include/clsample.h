/* clsample.h: C ABI of the GB300 (sm_103a) batched constrained logits sampler.
 *
 * One call turns a [B, V] next-token logits matrix into one token id per row, plus the
 * drawn token's logprob.  For every row it applies, in order:
 *
 *   1. sanitising of non-finite logits
 *        (SGLang source teardown (10): Sampling, Grammar and structured output,
 *         section "_preprocess_logits");
 *   2. frequency / presence penalties (additive), then the repetition penalty (scaling),
 *      then sparse logit_bias (a repeated id keeps its last value)
 *        (same page, sections "Order semantics of the penalties" and "Why logit_bias is
 *         built from triples");
 *   3. the int32 grammar bitmask: bit (i & 31) of word i >> 5 equal to 0 sets logit i to
 *      -inf, before any truncation
 *        (same page, section "Bitmask: one int32 covers 32 tokens");
 *   4. the greedy rule: temperature < 1e-5 (GLM-5.3 inference (7): output side, section
 *      "Sampling") or top_k in {0, 1} (SGLang page, section "Field groups");
 *   5. temperature, then top-k -> top-p -> min-p truncation on the tempered distribution
 *        (SGLang page, section "The maths of the three cuts": S_k, S_p, S_m);
 *   6. an exponential race keyed by (seed, position): token = argmax_i p_i / E_i over the
 *      kept set, E_i = -ln U_i with U_i from Philox4x32-10 (Salmon et al., SC'11) at
 *      counter (i / 4, position, 0) and key seed, so a request's draw does not depend on
 *      the batch it is in (SGLang page, section "Call site"; GLM-5.3 page: one random
 *      stream per request);
 *   7. the logprob of the drawn token under the full tempered distribution, computed as
 *      log-softmax (SGLang page, section "Numerical consistency of logprobs").
 *
 * Threading and ownership.  A handle is bound to the CUDA device that was current at
 * clsample_create and owns device scratch sized for max_batch rows (row order and
 * counters, per-slice records, per-row lists of penalised and biased tokens, compacted
 * candidates, and a spill area of one row per batch row; about 1.5 MB per row for
 * V = 151936).  Every array in clsample_args_t is a DEVICE pointer owned by the caller;
 * it must stay valid until the work enqueued on the stream has finished.  The logits are
 * read-only (never written in place).  Calls on one handle must be ordered (one stream,
 * or streams joined by events): they share the handle's scratch.  Separate handles are
 * independent.
 *
 * Errors.  Every entry point validates its arguments on the host, without any device
 * synchronisation, and returns a negative CLSAMPLE_ERR_* code on a bad argument;
 * nothing is enqueued then.  Data errors found on the device (ids outside [0, V),
 * decreasing CSR offsets, NaN parameters, a row with no allowed token) never trap:
 * they go to the per-row status (OK < OVERFLOW < INVALID, ordered by severity so that
 * a MAX reduction over rows gives one verdict; SGLang page, section
 * "LogitsProcessorOutput"), and such a row gets token -1 and logprob -inf.
 */
#ifndef CLSAMPLE_H
#define CLSAMPLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* clsample_stream_t;
typedef struct clsample_handle clsample_t;

enum {
  CLSAMPLE_LOGITS_F32 = 0,  /* float32 logits */
  CLSAMPLE_LOGITS_BF16 = 1  /* bfloat16 logits, widened exactly to float32 */
};

/* Per-row status codes written to row_status. */
enum { CLSAMPLE_ROW_OK = 0, CLSAMPLE_ROW_OVERFLOW = 1, CLSAMPLE_ROW_INVALID = 2 };

/* Return codes. */
enum {
  CLSAMPLE_SUCCESS = 0,
  CLSAMPLE_ERR_NULL = -1,       /* a required pointer is NULL */
  CLSAMPLE_ERR_BATCH = -2,      /* B < 0 or B > max_batch */
  CLSAMPLE_ERR_VOCAB = -3,      /* V <= 0, V != the handle's vocab, or V > 262144 */
  CLSAMPLE_ERR_STRIDE = -4,     /* logits_row_stride < V or bitmask_row_stride < ceil(V/32) */
  CLSAMPLE_ERR_DTYPE = -5,      /* logits_dtype is not a CLSAMPLE_LOGITS_* value */
  CLSAMPLE_ERR_CUDA = -6,       /* a CUDA runtime call failed (launch, attribute, device) */
  CLSAMPLE_ERR_DEVICE = -7,     /* the current device is not the handle's or not sm_103 */
  CLSAMPLE_ERR_MODE = -8        /* mode has a bit that is not a CLSAMPLE_MODE_* flag */
};

/* Bits of clsample_args_t.mode (0: sequential truncation, one draw per row). */
enum {
  /* Top-p over the whole distribution, intersected with the top-k set (SGLang page,
   * the sampler's "joint" filter order), instead of top-p over the renormalised top-k
   * set.  Rows with a top-k cut and top_p < 1 then take the co-resident row-group route. */
  CLSAMPLE_MODE_JOINT_TOPK_TOPP = 1,
  /* Scoring only (SGLang page, logprobs-only computation): the same transforms, no draw.
   * Every row takes the greedy route whatever its parameters -- token = argmax of z',
   * logprobs at T_eff -- and the requested ids (tid_*) get their logprobs. */
  CLSAMPLE_MODE_SCORE_ONLY = 2,
  /* Batch fast path (SGLang page, "Field groups": the host-side batch booleans
   * is_all_greedy and need_top_k/top_p/min_p_sampling, and the sampler's simple-sampling
   * branch; GLM page, "Sampling").  The caller asserts that every row is greedy (T < 1e-5,
   * top_k 0 or 1, or SCORE_ONLY) or untruncated (top_p 1, min_p 0, top_k -1 or at least
   * the row's allowed tokens).  The call is then one sweep over the logits -- no
   * preparation launch -- with the same results as without the flag.  A row that breaks
   * the assertion, or has 2^20 or more history ids or 4095 or more bias entries, gets
   * status INVALID.  Requested-id and top-N logprobs are not available (ERR_MODE).
   * An untruncated row draws from candidates within 2e-3 of each slice's best fast race
   * score; a slice with more than 64 of them (not seen in practice) makes the row
   * OVERFLOW. */
  CLSAMPLE_MODE_FAST_SWEEP = 4
};

/* Arguments of one sampler call.  B rows, V vocabulary entries.
 *
 * mode              CLSAMPLE_MODE_* bits, 0 for plain sampling; other bits: ERR_MODE.
 * logits            [B, logits_row_stride] elements of logits_dtype, row-major.
 * temperatures      f32[B]; NULL = 1.0.  T < 1e-5 (including 0 and negatives) is greedy;
 *                   NaN or +inf is INVALID.
 * top_ks            i32[B]; NULL = -1.  -1 (or >= the number of allowed tokens) keeps the
 *                   whole vocabulary; 0 and 1 are greedy; < -1 is INVALID.  Every token
 *                   tied with the k-th largest probability is kept.
 * top_ps            f32[B]; NULL = 1.0.  Must lie in (0, 1], else INVALID.
 * min_ps            f32[B]; NULL = 0.0.  Must lie in [0, 1], else INVALID.
 * rep, freq, pres   f32[B] each, NULL = 1.0 / 0.0 / 0.0.  For a token seen c > 0 times in
 *                   the row's history: z -= freq*c; z -= pres; then z = z > 0 ? z/rep :
 *                   z*rep.  rep must be finite and > 0, freq and pres finite.
 * hist_offs/ids     CSR of the rows' token histories: ids hist_ids[hist_offs[r] ..
 *                   hist_offs[r+1]), duplicates counted.  NULL offs = no penalties.
 * bias_offs/ids/vals CSR of logit_bias entries; z += val; for a repeated id the LAST
 *                   entry of the row wins.  NULL offs = no bias.  NaN values are INVALID.
 * bitmask           i32[B, bitmask_row_stride] words, bit i & 31 of word i >> 5 allows
 *                   token i; NULL = unconstrained.  A row of all -1 words is unconstrained.
 * seeds             u64[B]; NULL = 0 for every row.  The request's random key.
 * positions         i64[B]; NULL = `step` for every row.  The request's token position;
 *                   rows of one request at different positions draw independently.
 * tokens            i32[B] output (required).
 * logprobs          f32[B] output or NULL: ln p(token) under softmax(z'/T_eff) over all
 *                   allowed tokens (T_eff = 1 for rows with T < 1e-5).
 * row_status        i32[B] output or NULL.
 * dbg_transformed   f32[B, V] output or NULL: the transformed logits z' (after penalties,
 *                   bias and mask), row-major with row stride V.
 * dbg_kept_count    i32[B] output or NULL: size of the kept set K (1 for greedy rows).
 * dbg_cut           f32[B] output or NULL: min over K of y = (z' - max z') * (1/T).
 * logprobs_orig     f32[B] output or NULL: ln p(token) under softmax(z') at T = 1, the
 *                   distribution before temperature (SGLang page, "Numerical consistency
 *                   of logprobs": the original logprobs).  Costs one more exponential
 *                   per logit when requested.
 * logprobs_kept     f32[B] output or NULL: ln of the token's probability renormalised
 *                   over the kept set K, the distribution it was drawn from (GLM page,
 *                   "Sampling": the top-k/top-p sampler's processed logprobs); 0 for
 *                   greedy rows (K is the token alone).
 * tid_offs/ids      CSR of requested token ids (SGLang page, the output container's
 *                   token-ids logprobs): ids tid_ids[tid_offs[r] .. tid_offs[r+1]), in
 *                   any order, repeats allowed.  NULL offs = none.  An id outside [0, V)
 *                   or a decreasing offset makes the row INVALID.
 * tid_logprobs      f32[tid_offs[B]] output (required with tid_offs): ln p(id) under the
 *                   same distribution as `logprobs` (softmax(z'/T_eff), pre-truncation);
 *                   -inf for a masked id and for every id of an INVALID row.
 * top_ns            i32[B] or NULL: N, the number of most probable tokens to report for
 *                   row r (SGLang page, the output container's top logprobs); 0 <= N <=
 *                   min(32, top_n_stride), else the row is INVALID.  Order: probability
 *                   descending; y is monotone in z', so equal probabilities are ranked
 *                   by z' descending, then by id ascending.
 * top_n_stride      row stride (elements) of top_ids / top_logprobs, >= 1 with top_ns.
 * top_ids           i32[B, top_n_stride] output (required with top_ns): places 0..N-1 of
 *                   row r; -1 past the row's allowed tokens and for an INVALID row; places
 *                   N.. untouched.
 * top_logprobs      f32[B, top_n_stride] output (required with top_ns): ln p of those
 *                   tokens under softmax(z'/T_eff) (pre-truncation); -inf where the id is -1.
 *
 * Limits: V <= 262144 (at most 18 slices of at most 15360 tokens per row).  Any number
 * of penalised, biased or allowed tokens is handled exactly.  A row whose candidate set
 * must spill (a slice with more than 2048 candidates: flat or heavily tied rows) takes a
 * spill row for the call.  A handle has one spill row per batch row, so no valid row of
 * clsample_apply runs out; clsample_apply_static has 4, and a fifth row that must spill
 * in one of its calls gets status OVERFLOW.  A row whose bounded waits for other CTAs
 * gave up (a GPU that stopped scheduling them) is OVERFLOW too.
 */
typedef struct {
  int32_t B, V;
  int32_t logits_dtype;
  int32_t mode;
  const void* logits;
  int64_t logits_row_stride;
  const float* temperatures;
  const int32_t* top_ks;
  const float* top_ps;
  const float* min_ps;
  const float* rep;
  const float* freq;
  const float* pres;
  const int32_t* hist_offs;
  const int32_t* hist_ids;
  const int32_t* bias_offs;
  const int32_t* bias_ids;
  const float* bias_vals;
  const int32_t* bitmask;
  int64_t bitmask_row_stride;
  const uint64_t* seeds;
  const int64_t* positions;
  int64_t step;
  int32_t* tokens;
  float* logprobs;
  int32_t* row_status;
  float* dbg_transformed;
  int32_t* dbg_kept_count;
  float* dbg_cut;
  float* logprobs_orig;
  float* logprobs_kept;
  const int32_t* tid_offs;
  const int32_t* tid_ids;
  float* tid_logprobs;
  const int32_t* top_ns;
  int32_t top_n_stride;
  int32_t reserved1;
  int32_t* top_ids;
  float* top_logprobs;
} clsample_args_t;

/* Creates a handle for batches of up to max_batch rows over a vocabulary of `vocab`
 * tokens on the current CUDA device.  Sets the kernels' shared-memory attributes and
 * allocates the handle's device scratch (cudaMalloc; freed by clsample_destroy).
 * Returns CLSAMPLE_SUCCESS and *out, or a negative code (*out = NULL; nothing kept). */
int clsample_create(int32_t max_batch, int32_t vocab, clsample_t** out);

/* Releases a handle and its scratch (NULL is ignored).  cudaFree synchronises the
 * device, so no call on the handle may still be running. */
void clsample_destroy(clsample_t* handle);

/* Enqueues one sampler call on `stream`: the preparation launch (one CTA orders the
 * rows, heavy rows first, and resets the call's counters; when the call has penalties,
 * logit_bias or a bitmask, one more CTA per row lists the row's distinct penalised and
 * biased tokens by vocabulary slice and counts its allowed tokens), then the sampler
 * kernel (one CTA per (row, slice), launched with programmatic stream serialisation; its
 * CTAs wait, bounded, only for the flags the preparation launch sets); nothing when
 * B == 0.  Returns after enqueueing; results are valid once the stream reaches this
 * point. */
int clsample_apply(clsample_t* handle, const clsample_args_t* args, clsample_stream_t stream);

/* The two halves of clsample_apply, for callers that schedule or time them apart:
 * clsample_prepare enqueues the preparation launch, clsample_sample the sampler kernel,
 * which consumes what the last clsample_prepare on this handle wrote (each
 * clsample_sample needs its own clsample_prepare before it: the sampler clears the
 * preparation's flags when it ends; a sample without one waits a few seconds at most
 * and reports every row OVERFLOW, touching no row past B; a preparation that no sample consumes is harmless, the
 * next one clears its flags first).  The pair, with the same arguments on one stream,
 * equals clsample_apply.  Same validation and return codes. */
int clsample_prepare(clsample_t* handle, const clsample_args_t* args, clsample_stream_t stream);
int clsample_sample(clsample_t* handle, const clsample_args_t* args, clsample_stream_t stream);

/* One sampler call without a handle that allocates nothing.  The pages have no
 * counterpart: this is a deployment convenience of this library, and it samples
 * exactly like clsample_apply.  Its scratch is one fixed device array compiled into
 * the library (about 37 MB, zero when the library loads); no cudaMalloc or cudaFree
 * ever happens.  The first call on a device looks up the array's address on that
 * device (cudaGetSymbolAddress) and sets the kernels' shared-memory limit, once per
 * device, under a host lock.  Limits: B <= 64 (else CLSAMPLE_ERR_BATCH) and
 * V <= 262144 (else CLSAMPLE_ERR_VOCAB); nothing is enqueued on an error.  The array
 * holds 4 spill rows (see the limits of clsample_args_t): at most 4 rows of a call may
 * spill; a further row that must spill reports OVERFLOW.
 * Races: every call on a device, from any host thread or stream, uses the same array,
 * so calls of this entry point on one device must be ordered (one stream, or streams
 * joined by events); two overlapping calls corrupt each other's row order and records.
 * Calls through handles are unaffected, and each process has its own array. */
int clsample_apply_static(const clsample_args_t* args, clsample_stream_t stream);

/* Static description of a return code. */
const char* clsample_strerror(int code);

/* Launch geometry chosen for a vocabulary size: slices per row, tokens per slice and
 * dynamic shared memory per CTA.  Host-only; needs no GPU.  Returns CLSAMPLE_SUCCESS or
 * CLSAMPLE_ERR_VOCAB. */
int clsample_geometry(int32_t vocab, int32_t* slices, int32_t* chunk, int32_t* smem_bytes);

/* How many sampler-kernel CTAs of this handle can be resident on the device at once
 * (cudaOccupancyMaxActiveBlocksPerMultiprocessor times the SM count), computed at
 * clsample_create; the kernel launches one CTA per (row, slice). */
int clsample_occupancy(clsample_t* handle, int32_t logits_dtype, int32_t* resident_ctas);

/* Builds grammar-bitmask rows from allowed-token lists (vLLM page, "allowed token ids",
 * a hard-coded constraint of the sampler, expressed here as the bitmask the sampler
 * takes).  offs i32[B+1] and ids (DEVICE) give row r's allowed ids ids[offs[r] ..
 * offs[r+1]); bitmask i32[B, bitmask_row_stride] (DEVICE, written; words past
 * ceil(V/32) untouched) gets bit id & 31 of word id >> 5 set for each listed id and every
 * other bit cleared.  A row with an id outside [0, V), a decreasing offset or an empty
 * list ends all-zero, which clsample_apply reports as INVALID.  Enqueue only on `stream`;
 * returns a negative code for bad sizes or NULL pointers (nothing launched). */
int clsample_allowed_to_bitmask(const int32_t* offs, const int32_t* ids, int32_t B, int32_t V, int32_t* bitmask,
                                int64_t bitmask_row_stride, clsample_stream_t stream);

/* Diagnostics of the building blocks, on device arrays of length n (enqueued on
 * `stream`): the fixed-point top-p weight floor(exp32(y) * 2^40) of each y (y <= 0),
 * and the race uniform U of (seed, position, token).  They run the same device code
 * as clsample_apply, so tests can compare them with an independent implementation. */
int clsample_debug_weights(const float* y, uint64_t* weights, int32_t n, clsample_stream_t stream);
int clsample_debug_uniforms(const uint64_t* seeds, const int64_t* positions, const int64_t* tokens,
                            float* u, int32_t n, clsample_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* CLSAMPLE_H */
