/*
 * spec_verify.h -- C ABI of a GB300 (sm_103a) library for the batched
 * draft-verification step of speculative decoding.
 *
 * The operation (sources are web pages, cited by title and section):
 *  [P1] reactapp.top, "Speculative decoding and early exit: speeding up
 *       autoregressive decode", section "Speculative decoding: draft first,
 *       then verify": the target scores the K drafted positions plus one more
 *       in a single pass; each target row becomes p = softmax(logits / T);
 *       positions are tested in order and the first rejection ends the pass;
 *       a rejection is replaced by a token drawn from relu(p - q) normalised;
 *       when all K drafts pass, one bonus token is drawn from the last row.
 *  [P2] trefon.com, "Decode is memory-bound: a ~59 tok/s ceiling on an RTX
 *       4090 and how speculative decoding breaks it", section "Speculative
 *       decoding": draft token x is kept with probability min(1, p(x)/q(x)),
 *       which makes the output follow the target distribution exactly.
 *  [P3] agentnet.co.il, "New technical post reveals how speculative decoding
 *       speeds up LLM inference without hurting accuracy", section "How it
 *       works in practice": with D drafts the accepted length AL is in
 *       [1, 1 + D].
 *
 * Conventions shared by every entry point:
 *  - Arrays are row-major and dense with the vocabulary (V) innermost.
 *  - logits [B, K+1, V]: row i < K scores draft position i, row K is the bonus
 *    row.  dtype SV_F32 (float) or SV_BF16 (bfloat16 bit patterns).
 *  - q [B, K, V] float: the draft's probabilities, already at the draft's
 *    temperature; used as given (not renormalised).
 *  - draft_tokens [B, K] int32.
 *  - uniforms [B, K+1] float in [0, 1): u[b, i] drives the test at position i
 *    (accept iff u * q(x) < p(x), i.e. u < min(1, p/q)); u[b, K] drives the
 *    one corrected-or-bonus draw, an inverse-CDF draw over token ids in
 *    ascending order (the first token whose running weight exceeds u * S).
 *    Uniforms are inputs so that results are reproducible and testable.
 *  - Outputs: accept_len [B] int32 = accepted drafts + 1 in [1, K+1] (0 marks
 *    a sequence error); out_tokens [B, K+1] int32 = accepted drafts, then the
 *    drawn token, then -1; accept_mask [B, K] uint8 = 1 on accepted positions.
 *  - Optional outputs (pass NULL to skip): row_stats [B, K+1, 2] float =
 *    (max_v logits/T, sum_v exp(logits/T - max)) for every row the pass
 *    reached, NaN for rows it never needed; p_draft [B, K] float = p_i(x_i)
 *    for the tests that ran, NaN otherwise; status [B] int32 = SV_* code of
 *    each sequence.
 *  - Rows after the first rejection are never read: the test loop of [P1]
 *    stops there, and so does the kernel.
 *  - Shapes: 1 <= B, 0 <= K <= 32 (K = 0 draws one token from row 0),
 *    1 <= V, B*(K+1)*V < 2^40.  Every pointer must be aligned to its element
 *    size.  16-byte aligned logits with V*sizeof(element) a multiple of 16 take
 *    the bulk-copy path; other layouts take a slower element-wise path.
 *
 * Ownership and threading: the caller owns every array.  A context owns only
 * its own small device state (an error word) and, after the first host-buffer
 * call, staging buffers sized to the largest host-buffer call so far.  spec_verify_run
 * allocates nothing and never synchronises.  One context serves one stream at
 * a time; calls on one context from several host threads must be serialised
 * by the caller.
 *
 * Errors: host-detectable problems return at once and launch nothing.  Errors
 * found on the device (a draft token outside [0, V), a uniform outside [0, 1),
 * a NaN / +inf / all -inf target row that the pass reaches, a NaN, infinite or
 * negative q value that the pass reads) mark only that sequence (accept_len 0,
 * out_tokens -1, mask 0, stats NaN, status code) and set a bit in the
 * context's sticky error word, read with spec_verify_get_error.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

typedef enum {
    SV_OK = 0,
    SV_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad shape, T <= 0 or not finite   */
    SV_ERR_UNSUPPORTED = 2,   /* shape beyond what one launch plan can hold                  */
    SV_ERR_CUDA = 3,          /* a CUDA runtime call failed                                   */
    SV_ERR_TOKEN_RANGE = 4,   /* device: a draft token outside [0, V)                         */
    SV_ERR_NONFINITE = 5,     /* device: NaN/+inf/all -inf logits row, or NaN/inf/negative q  */
    SV_ERR_TIMEOUT = 6,       /* device: a bounded wait for a bulk copy ran out               */
    SV_ERR_UNIFORM_RANGE = 7, /* device: a uniform outside [0, 1)                             */
    SV_ERR_BAD_OFFSETS = 8    /* device: ragged-batch row offsets that describe no packing    */
} sv_status;

/* Opaque context: device id, limits, launch-plan cache, error word. */
typedef struct sv_ctx sv_ctx;

/* Launch plan the library picks for a shape (reported for tests and tuning). */
typedef struct {
    int cluster;       /* CTAs per sequence, one thread-block cluster (1..16)          */
    int group;         /* target rows a cluster loads before deciding (1..K+1)         */
    int threads;       /* threads per CTA                                              */
    int smem_bytes;    /* dynamic shared memory per CTA                                */
    int64_t slice;     /* vocabulary entries per CTA (a multiple of 8)                 */
    int64_t grid;      /* CTAs in the launch = B * cluster                             */
    int bulk_copy;     /* 1: row slices move with cp.async.bulk; 0: element-wise loads */
    int prefetch_next; /* 1: the next row slice is prefetched into L2 while one is reduced */
    int stages;        /* 2 KB ring stages per warp (3, or 6 for batches that leave SMs
                          room; 0 for the kernels without a ring)                     */
} sv_plan;

/* Create a context on `device` for calls with B <= max_B, K <= max_K (<= 32)
 * and V <= max_V.  Queries the device, sets kernel attributes, allocates the
 * 4-byte device error word.  *out is set only on success.
 * Returns SV_OK, SV_ERR_INVALID_ARG or SV_ERR_CUDA (no usable device). */
int spec_verify_init(sv_ctx** out, int device, int max_B, int max_K, int64_t max_V);

/* One batched verify on `stream` (a cudaStream_t; NULL = legacy default
 * stream), device pointers throughout, asynchronous.  Layouts, meaning and
 * error behaviour as described at the top of this file.  `stream` must belong
 * to the context's device.  Safe to capture in a CUDA graph. */
int spec_verify_run(sv_ctx* ctx,
                    const void* target_logits, int logits_dtype,
                    const float* q, const int32_t* draft_tokens, const float* uniforms,
                    int B, int K, int64_t V, float temperature,
                    int32_t* accept_len, int32_t* out_tokens, uint8_t* accept_mask,
                    float* row_stats, float* p_draft, int32_t* status,
                    void* stream);

/* The same verify with HOST buffers for every array (pinned memory gives the
 * fastest copies).  Copies the inputs to context-owned device staging buffers
 * (allocated by the first call, re-allocated only when a later call needs
 * more, kept until destroy), runs, copies the outputs back and synchronises
 * `stream` before returning.  Returns the launch status, or the lowest device
 * error code seen by this call (the sticky error word is cleared). */
int spec_verify_run_host(sv_ctx* ctx,
                         const void* target_logits, int logits_dtype,
                         const float* q, const int32_t* draft_tokens, const float* uniforms,
                         int B, int K, int64_t V, float temperature,
                         int32_t* accept_len, int32_t* out_tokens, uint8_t* accept_mask,
                         float* row_stats, float* p_draft, int32_t* status,
                         void* stream);

/* Synchronise `stream`, read and clear the context's sticky device error
 * word.  *mask (if not NULL) receives a bit (1 << code) per error kind seen
 * since the last read.  Returns SV_OK or the lowest code present. */
int spec_verify_get_error(sv_ctx* ctx, void* stream, uint32_t* mask);

/* Launch plan for a shape on the context's device (no launch). */
int spec_verify_get_plan(sv_ctx* ctx, int B, int K, int64_t V, int logits_dtype, sv_plan* out);

/* Force parts of the plan (0 = automatic): cluster size 1..16, rows per group
 * 1..K+1 (clamped), threads per CTA 128/256/512.  Used by tests to cover every
 * plan and by tuning sweeps.  The greedy, truncated and draft-logit calls take
 * only the cluster size (the truncated kernel, also under a draft-logit call
 * with a filter on, caps it at 8).  Returns
 * SV_ERR_INVALID_ARG on values outside those sets. */
int spec_verify_set_plan_override(sv_ctx* ctx, int cluster, int group, int threads);

/* The planner as a pure host function of the device limits, for tests:
 * num_sms, max dynamic shared memory per CTA, largest cluster the device
 * allows, and the same overrides.  No CUDA call is made. */
int spec_verify_plan_for(int num_sms, int smem_per_cta, int max_cluster,
                         int B, int K, int64_t V, int logits_dtype,
                         int ovr_cluster, int ovr_group, int ovr_threads, sv_plan* out);

/* Ragged batch ([P1] "Scheduling interaction": continuous batching mixes
 * sequences at different points): every sequence b has its own draft depth
 * K_b <= K_max and its rows are packed.  `row_offsets` [B+1] (int32, device)
 * gives sequence b the target rows row_offsets[b] .. row_offsets[b+1]-1, so
 * K_b = row_offsets[b+1] - row_offsets[b] - 1, with row_offsets[0] = 0 and
 * row_offsets[B] = total_rows.  Packed layouts (device, V innermost):
 *   target_logits [total_rows, V]   rows of b from row_offsets[b]
 *   q             [total_rows-B, V] draft rows of b from row_offsets[b] - b
 *   draft_tokens  [total_rows-B]    from row_offsets[b] - b
 *   uniforms      [total_rows]      from row_offsets[b]: K_b tests, then the draw
 *   accept_len    [B]               in [1, K_b+1]; 0 = sequence error
 *   out_tokens    [total_rows]      from row_offsets[b], -1 padded
 *   accept_mask   [total_rows-B]    from row_offsets[b] - b
 *   row_stats     [total_rows, 2]   optional, from row_offsets[b]
 *   p_draft       [total_rows-B]    optional, from row_offsets[b] - b
 *   status        [B]               optional
 * Each sequence is verified exactly as spec_verify_run verifies it alone.
 * Offsets are read on the device: a sequence whose pair describes no packing
 * (row_offsets[b] < b, K_b < 0 or > K_max, or fewer than B-1-b rows left after
 * it within total_rows) gets SV_ERR_BAD_OFFSETS (status, error word,
 * accept_len 0) and nothing else of it is read or written.
 * Returns SV_OK, SV_ERR_INVALID_ARG (as spec_verify_run, with B <= total_rows
 * <= B*(K_max+1)), SV_ERR_UNSUPPORTED or SV_ERR_CUDA. */
int spec_verify_run_ragged(sv_ctx* ctx,
                           const void* target_logits, int logits_dtype,
                           const float* q, const int32_t* draft_tokens, const float* uniforms,
                           const int32_t* row_offsets, int64_t total_rows,
                           int B, int K_max, int64_t V, float temperature,
                           int32_t* accept_len, int32_t* out_tokens, uint8_t* accept_mask,
                           float* row_stats, float* p_draft, int32_t* status, void* stream);

/* Verification against a truncated target ([P2] "Two things that follow from
 * the math" names the production settings temperature 0.6, top-p 0.95, min-p
 * 0.05).  The target distribution of every row becomes p~: token v is kept
 * when p_v >= min_p * max p (min-p) and when the mass of the tokens strictly
 * more probable than v is below top_p (top-p; every token tied at the
 * boundary is kept); both filters look at the untruncated p = softmax(l/T),
 * and p~ is p on the kept tokens divided by their sum.  p~ replaces p in the
 * test (u*q(x) < p~(x)), the residual max(0, p~_j - q_j) and the bonus draw.
 * top_p >= 1 turns top-p off, min_p <= 0 turns min-p off (both off: the same
 * outputs as spec_verify_run up to rounding).
 *
 * Arguments, layouts and errors as spec_verify_run, except that with a filter
 * on the rejected draft row q_j is read -- and checked for values that are
 * not probabilities (SV_ERR_NONFINITE) -- only at the kept tokens, since
 * max(0, p~_j - q_j) is zero wherever p~_j is; row_stats are those of the
 * untruncated softmax of the rows read, p_draft = p~(x_i).  Requires
 * 0 < top_p and min_p < 1 (SV_ERR_INVALID_ARG otherwise).  With min-p on, the
 * kernel reads each row it reaches once in full and then only the stretches
 * that can hold min-p survivors, and takes the top-p cut and the draw over
 * the survivors; without min-p (or with more survivors than its lists hold)
 * it takes the cut by histogram passes over the row, two (bf16) to four (f32)
 * more reads from L2.  Clusters have at most 8 CTAs. */
int spec_verify_run_truncated(sv_ctx* ctx,
                              const void* target_logits, int logits_dtype,
                              const float* q, const int32_t* draft_tokens, const float* uniforms,
                              int B, int K, int64_t V, float temperature,
                              double top_p, double min_p,
                              int32_t* accept_len, int32_t* out_tokens, uint8_t* accept_mask,
                              float* row_stats, float* p_draft, int32_t* status, void* stream);

/* The truncated-target kernel's launch plan on the context's device. */
int spec_verify_get_plan_truncated(sv_ctx* ctx, int B, int K, int64_t V, int logits_dtype,
                                   sv_plan* out);

/* Its planner as a pure host function (no CUDA call), for tests. */
int spec_verify_plan_truncated_for(int num_sms, int max_cluster, int B, int K, int64_t V,
                                   int logits_dtype, int ovr_cluster, sv_plan* out);

/* Verification with draft LOGITS instead of draft probabilities ([P1]
 * "Speculative decoding: draft first, then verify": the drafter's distribution
 * is q = softmax(draft_logits / T), formed from its logits at its temperature).
 * Position i uses q_i = softmax(draft_logits[b, i] / draft_temperature): the
 * test u*q(x) < p(x), and after a rejection at j the residual max(0, p_j - q_j).
 * The kernel forms q from the draft row's own maximum and normaliser, taken in
 * the same pass as the target row's, so no q array exists anywhere.  top_p < 1
 * or min_p > 0 verify against the truncated target exactly as
 * spec_verify_run_truncated does (q itself is never truncated); top_p >= 1
 * with min_p <= 0 is the plain verify, run by spec_verify_run's kernel in its
 * draft-logit form: each test row's draft row streams through the same
 * shared-memory ring right after it.
 *
 *   draft_logits [B, K, V]  the target's dtype (logits_dtype), device; row i is
 *                           the drafter's scores at position i (may be NULL
 *                           when K == 0)
 *   draft_temperature       > 0 and finite
 * Every other argument, layout and output as spec_verify_run_truncated
 * (row_stats: the target rows' untruncated statistics; p_draft: p~(x_i)).
 *
 * Bytes: each row the pass reaches is read with its draft row (rows after the
 * first rejection are never read; without filters the row after it is read
 * only as far as it got before the decision), plus the rejected pair again
 * for the draw (with min-p on, only the kept tokens of the pair).
 * Device-detected errors as spec_verify_run, plus: a draft row the pass
 * reaches holding a NaN or +inf, or only -inf, is SV_ERR_NONFINITE for that
 * sequence.  16-byte aligned target and draft rows (V * element size a
 * multiple of 16) take the vector path; other layouts the element path.
 * Asynchronous, no allocation, one launch on `stream`.  Returns SV_OK,
 * SV_ERR_INVALID_ARG (as spec_verify_run_truncated, plus a null or misaligned
 * draft_logits with K > 0, or a draft temperature that is not positive and
 * finite) or SV_ERR_CUDA. */
int spec_verify_run_draft_logits(sv_ctx* ctx,
                                 const void* target_logits, int logits_dtype,
                                 const void* draft_logits, const int32_t* draft_tokens,
                                 const float* uniforms, int B, int K, int64_t V,
                                 float temperature, float draft_temperature,
                                 double top_p, double min_p,
                                 int32_t* accept_len, int32_t* out_tokens, uint8_t* accept_mask,
                                 float* row_stats, float* p_draft, int32_t* status, void* stream);

/* The draft-logit kernel's launch plan on the context's device (filters: 1
 * when top-p or min-p is on). */
int spec_verify_get_plan_draft_logits(sv_ctx* ctx, int B, int K, int64_t V, int logits_dtype,
                                      int filters, sv_plan* out);

/* Its planner as a pure host function (no CUDA call), for tests: the
 * truncated planner when filters is 1; without filters spec_verify_plan_for's
 * mapping for 128-thread CTAs with the 227 KB of shared memory a GB300 CTA
 * may opt into, and room for two rows of partials (target and draft) per
 * group row. */
int spec_verify_plan_draft_logits_for(int num_sms, int max_cluster, int B, int K, int64_t V,
                                      int logits_dtype, int filters, int ovr_cluster,
                                      sv_plan* out);

/* Greedy verification: the verify of spec_verify_run in the limit T -> 0
 * ([P1] "Speculative decoding: draft first, then verify": as T falls, the
 * softmax of logits/T puts all its mass on the largest logit).  Row i becomes
 * one-hot at a_i = argmax_v target_logits[b, i, v], the LOWEST token id among
 * equal maxima; draft x_i is accepted iff x_i == a_i (the test u*q(x) < p(x)
 * with a one-hot p); the first rejected position j emits a_j (the only token
 * with max(0, p_j - q_j) > 0), and a fully accepted sequence emits the bonus
 * a_K.  So neither draft probabilities nor uniforms are taken.
 *
 *   target_logits [B, K+1, V]  float32 or bfloat16 (SV_F32 / SV_BF16), device
 *   draft_tokens  [B, K]       int32, device (may be NULL when K == 0)
 *   accept_len    [B]          out, accepted drafts + 1 in [1, K+1]; 0 = sequence error
 *   out_tokens    [B, K+1]     out, accepted drafts, then a_j, then -1
 *   accept_mask   [B, K]       out, 1 for accepted positions (may be NULL when K == 0)
 *   row_argmax    [B, K+1]     optional out: a_i for the rows read, -1 for the others
 *                              (and for every row of an erroneous sequence)
 *   status        [B]          optional out: per-sequence status
 *
 * Rows are read in order and not past the first rejection.  Device-detected
 * errors (a draft token outside [0, V); a row the loop reaches holding a NaN
 * or +inf, or only -inf) mark the sequence as for spec_verify_run, set the
 * context's error word, and count in bin 0 of the telemetry histogram if one
 * is set.  Asynchronous, no allocation, one launch on `stream`.
 * Returns SV_OK, SV_ERR_INVALID_ARG (null or misaligned pointers, shapes outside
 * the context's limits, telemetry bins < K + 2) or SV_ERR_CUDA (launch failed). */
int spec_verify_run_greedy(sv_ctx* ctx,
                           const void* target_logits, int logits_dtype,
                           const int32_t* draft_tokens, int B, int K, int64_t V,
                           int32_t* accept_len, int32_t* out_tokens, uint8_t* accept_mask,
                           int32_t* row_argmax, int32_t* status, void* stream);

/* The greedy kernel's launch plan for a shape on the context's device. */
int spec_verify_get_plan_greedy(sv_ctx* ctx, int B, int K, int64_t V, int logits_dtype,
                                sv_plan* out);

/* The greedy planner as a pure host function (no CUDA call), for tests:
 * one cluster per sequence, the largest that keeps the batch resident (eight
 * 128-thread CTAs per SM) and gives every warp enough work; ovr_cluster > 0
 * forces the cluster size. */
int spec_verify_plan_greedy_for(int num_sms, int max_cluster, int B, int K, int64_t V,
                                int logits_dtype, int ovr_cluster, sv_plan* out);

/* Acceptance telemetry ([P1] "Production perspective": ship the acceptance
 * rate and the mean accepted length; its operational checklist: record
 * acceptance histograms).  With `accept_hist` set, every later verify on this
 * context adds 1, per sequence, to accept_hist[AL] (AL = accepted length,
 * 1..K+1; bin 0 counts sequences that reported an error).  `accept_hist` is a
 * DEVICE array of `bins` uint32 counters owned by the caller, who zeroes it and
 * keeps it alive while set; counts accumulate across calls (atomic adds on the
 * launch stream).  A run whose K + 2 exceeds `bins` returns SV_ERR_INVALID_ARG.
 * NULL (bins ignored) turns the counting off.  Keep one histogram per draft
 * depth K: spec_adapt reads it for one K.
 * Returns SV_OK or SV_ERR_INVALID_ARG (no context, bins < 2, misaligned). */
int spec_verify_set_telemetry(sv_ctx* ctx, uint32_t* accept_hist, int bins);

/* What a histogram of accepted lengths for one draft depth K says. */
typedef struct {
    uint64_t sequences;          /* sequences counted (bins 1..K+1)                       */
    uint64_t errors;             /* bin 0                                                  */
    uint64_t tested;             /* draft tokens tested: sum of min(AL, K)                 */
    uint64_t accepted;           /* draft tokens accepted: sum of AL - 1                   */
    double acceptance;           /* accepted / tested (NaN if nothing was tested)          */
    double mean_accept_len;      /* tokens emitted per pass (NaN if no sequence)           */
    uint64_t pos_tested[32];     /* position i tested by sequences with AL >= i + 1        */
    double pos_acceptance[32];   /* accepted at i / tested at i (NaN if untested or i >= K) */
    int next_K;                  /* the draft depth for the next passes                    */
} sv_adapt;

/* Adaptive draft depth ([P2] "Two things that follow from the math": cap the
 * depth when the measured acceptance falls below 35 %; "Rules I follow": pick
 * the depth from measured acceptance and keep measuring).  Host function, no
 * CUDA call.  `hist` is a HOST copy of a telemetry histogram collected at
 * depth K (bins >= K + 2).  next_K = K (bounded by K_max) while fewer than
 * `min_tested` drafts were tested; K_floor when acceptance < threshold (the
 * pages use 0.35); K_max otherwise.
 * Returns SV_OK or SV_ERR_INVALID_ARG (null pointers, K or K_max outside
 * [0, 32], K_floor outside [0, K_max], bins < K + 2, threshold outside [0, 1]). */
int spec_adapt(const uint32_t* hist, int bins, int K, int K_max, int K_floor,
               double threshold, uint64_t min_tested, sv_adapt* out);

/* The verify of spec_verify_run with no context and no allocation of any
 * kind (no cudaMalloc/cudaFree, no host heap, no allocating library call).
 * The pages have no counterpart: this is a deployment convenience, not part of
 * the method.
 *
 * For callers that cannot allocate where they verify: an engine that handed
 * nearly all device memory to its own pool at start-up, a decode loop that
 * must not take the device-wide synchronisation cudaFree implies (so it cannot
 * own a context it later destroys), a plugin behind a fixed function table
 * with nowhere to create or release a context.
 *
 * Arguments, layouts, outputs and per-sequence errors are those of
 * spec_verify_run, with `device` (the CUDA device the pointers and `stream`
 * belong to) in place of the context.  Limits: 0 <= device < 64,
 * 1 <= B <= 2^20, 0 <= K <= 32, 1 <= V <= 2^31 (and B*(K+1)*V < 2^40); larger
 * sizes return SV_ERR_INVALID_ARG before anything is launched.  The launch plan
 * is the planner's automatic choice.
 *
 * Setup: the first call for a device queries it, sets the kernels' attributes
 * and looks up the device address of the library's static scratch, with that
 * device current.  Make that first call before any stream capture begins.  A
 * failed setup returns SV_ERR_CUDA / SV_ERR_UNSUPPORTED and is retried by the
 * next call.
 *
 * Scratch: a 256-byte array in the library's device code, one per device, of
 * which a call uses 4 bytes (the word the kernel ORs error bits into).
 * Nothing in it has to start at zero: the kernel never reads it.  This entry
 * offers no way to read it either, so errors are seen through `status` (pass
 * it) and accept_len == 0.  Every call on a device shares that scratch: calls
 * that can overlap on the GPU (streams not ordered with each other) race on
 * it, so order them on one stream or with events.  Host threads may call
 * concurrently once a device is set up. */
int spec_verify_run_noalloc(int device,
                            const void* target_logits, int logits_dtype,
                            const float* q, const int32_t* draft_tokens, const float* uniforms,
                            int B, int K, int64_t V, float temperature,
                            int32_t* accept_len, int32_t* out_tokens, uint8_t* accept_mask,
                            float* row_stats, float* p_draft, int32_t* status,
                            void* stream);

/* Self-test of the bounded wait the kernels use for every mbarrier wait (the
 * pages have no counterpart: a diagnostic of this library).  One thread on
 * `device` waits on a barrier of its own through the same routine as the
 * greedy kernel's waits; with arrive = 1 the barrier's phase is completed
 * first and the wait succeeds at once, with arrive = 0 nothing ever completes
 * it and the wait gives up after limit_ns.  Outputs: *completed (1 = the wait
 * succeeded, 0 = it ran out) and *elapsed_ns (device global timer).
 * Synchronises the device's legacy default stream.  Returns SV_OK,
 * SV_ERR_INVALID_ARG (null outputs, limit_ns > 2e9) or SV_ERR_CUDA. */
int spec_verify_selftest_wait(int device, unsigned long long limit_ns, int arrive,
                              int* completed, unsigned long long* elapsed_ns);

/* Release the context and everything it owns. */
int spec_verify_destroy(sv_ctx* ctx);

/* Static text for a status code. */
const char* spec_verify_strerror(int code);

/* Library version as major*10000 + minor*100 + patch. */
int spec_verify_version(void);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_VERIFY_H */
