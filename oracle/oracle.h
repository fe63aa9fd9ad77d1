/*
 * oracle.h -- fp64 CPU reference for batched speculative-decoding verification.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the package smoke check and the
 * benchmark's CPU-baseline leg call it; the product library never links it and
 * shares no code, header or constant with it.
 *
 * Citations (page title, then section):
 *  [P1] reactapp.top, "Speculative decoding and early exit: speeding up
 *       autoregressive decode" -- section "Speculative decoding: draft first,
 *       then verify" (the conceptual PyTorch loop: softmax of each target row at
 *       temperature T, acceptance min(1, p(x)/q(x)), stop at the first
 *       rejection, corrected token from relu(p - q) normalised, bonus token from
 *       the last row when every draft token is accepted).
 *  [P2] trefon.com, "Decode is memory-bound: a ~59 tok/s ceiling on an RTX 4090
 *       and how speculative decoding breaks it" -- section "Speculative
 *       decoding" (accept x with probability min(1, p(x)/q(x)); the output law
 *       equals the target's; expected tokens per pass (1 - a^(k+1))/(1 - a) and
 *       its table) and section "Two things that follow from the math"
 *       (expected acceptance = sum_x min(p(x), q(x))).
 *  [P3] agentnet.co.il, "New technical post reveals how speculative decoding
 *       speeds up LLM inference without hurting accuracy" -- section "How it
 *       works in practice" (draft length D; acceptance length AL in [1, 1 + D]).
 */
#ifndef SV_ORACLE_H
#define SV_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Per-sequence status codes (the numbers the product library also reports). */
#define ORACLE_OK 0
#define ORACLE_TOKEN_RANGE 4   /* a draft token outside [0, V)                       */
#define ORACLE_NONFINITE 5     /* NaN / +inf / all -inf target row, or bad q value    */
#define ORACLE_UNIFORM_RANGE 7 /* a uniform outside [0, 1) or NaN                     */
#define ORACLE_BAD_OFFSETS 8   /* ragged batch: offsets that describe no packing      */

/* Softmax of one target row at temperature T, in double precision.
 *   row: V stored logits (dtype 0 = float32, 1 = bfloat16 bit patterns).
 *   p: out, V probabilities.  m_out = max_v row[v]/T, s_out = sum_v exp(row[v]/T - m).
 * Returns ORACLE_OK, or ORACLE_NONFINITE when a value is NaN, a value is +inf,
 * or every value is -inf (p is then left unspecified). */
int oracle_softmax_row(const void* row, int dtype, int64_t V, double T,
                       double* p, double* m_out, double* s_out);

/* Batched verification, sequence by sequence, in the order the pages give.
 *
 * Inputs (host, row-major, V innermost):
 *   logits   [B, K+1, V]  float32 or bf16 bits (dtype 0 / 1); row i is the
 *                         target's distribution at draft position i, row K the
 *                         bonus row
 *   q        [B, K, V]    float32 draft probabilities, used as given
 *   tokens   [B, K]       int32 draft tokens
 *   uniforms [B, K+1]     float32; u[b,i] drives the test at position i and
 *                         u[b,K] the single corrected-or-bonus sample
 * Outputs (any of the optional ones may be NULL):
 *   accept_len [B]        accepted drafts + 1, in [1, K+1]; 0 on a sequence error
 *   out_tokens [B, K+1]   accepted prefix, then the sampled token, then -1
 *   accept_mask [B, K]    1 for accepted positions, else 0
 *   status [B]            ORACLE_* code of the sequence
 *   row_m, row_s [B, K+1] softmax max and normaliser of the rows the loop
 *                         reached; NaN for rows it never reached (optional)
 *   p_draft [B, K]        p_i(x_i) for the tests that ran; NaN otherwise (optional)
 *   accept_margin [B]     min over the tests that ran of |u_i - p/q| (inf when
 *                         none ran or q(x) = 0) (optional)
 *   sample_margin [B]     distance of u[b,K] to the nearer normalised CDF
 *                         boundary around the sampled token, counting only
 *                         boundaries that have a positive-weight token on the
 *                         far side (inf when neither does) (optional)
 *   sample_alt [B]        the positive-weight token across that nearer
 *                         boundary, or -1 (optional)
 */
/* Host threads oracle_verify and its variants use for a batch: 1 in the plain
 * build, OpenMP's thread count in a build with -fopenmp. */
int oracle_threads(void);
/* Sets that count (OpenMP build, n >= 1); returns the count now in force. */
int oracle_set_threads(int n);

int oracle_verify(const void* logits, int dtype, const float* q, const int32_t* tokens,
                  const float* uniforms, int64_t B, int K, int64_t V, float temperature,
                  int32_t* accept_len, int32_t* out_tokens, uint8_t* accept_mask,
                  int32_t* status, double* row_m, double* row_s, double* p_draft,
                  double* accept_margin, double* sample_margin, int32_t* sample_alt);

/* Verification against the truncated target ([P2] "Two things that follow
 * from the math": production settings temperature 0.6, top-p 0.95, min-p
 * 0.05).  p~ keeps token v when p_v >= min_p * max p (min-p) and the mass of
 * the tokens strictly more probable than v is below top_p (top-p, ties at the
 * boundary kept), both on the untruncated p; p~ is p on the kept tokens over
 * their sum and replaces p in the test, the residual and the bonus draw.
 * top_p >= 1 / min_p <= 0 switch a filter off; top_p must be > 0, min_p < 1.
 * Outputs as oracle_verify (p_draft = p~(x)); trunc_margin [B] (optional) is
 * the smallest distance of a reached row from a filter boundary:
 * |log(p_v/p_max) - log(min_p)| and |mass above v - top_p| over its tokens. */
int oracle_verify_truncated(const void* logits, int dtype, const float* q, const int32_t* tokens,
                            const float* uniforms, int64_t B, int K, int64_t V,
                            float temperature, double top_p, double min_p, int32_t* accept_len,
                            int32_t* out_tokens, uint8_t* accept_mask, int32_t* status,
                            double* row_m, double* row_s, double* p_draft,
                            double* accept_margin, double* sample_margin, int32_t* sample_alt,
                            double* trunc_margin);

/* The verify (optionally against the truncated target) with draft LOGITS
 * dlogits [B, K, V] (the target's dtype) instead of draft probabilities: q_i =
 * softmax(d_i / T_d), in double precision, computed when the loop reaches row
 * i.  A reached draft row with a NaN or +inf, or only -inf, is a sequence error.
 * top_p >= 1 and min_p <= 0 leave the target untruncated.  Outputs as
 * oracle_verify_truncated. */
int oracle_verify_draft_logits(const void* logits, int dtype, const void* dlogits,
                               const int32_t* tokens, const float* uniforms, int64_t B, int K,
                               int64_t V, float temperature, float draft_temperature,
                               double top_p, double min_p, int32_t* accept_len,
                               int32_t* out_tokens, uint8_t* accept_mask, int32_t* status,
                               double* row_m, double* row_s, double* p_draft,
                               double* accept_margin, double* sample_margin,
                               int32_t* sample_alt, double* trunc_margin);

/* Ragged batch: sequence b owns packed target rows [off[b], off[b+1]) of R,
 * K_b = off[b+1] - off[b] - 1 <= K_max; its draft rows, tokens, mask and
 * p_draft start at off[b] - b, its uniforms, out_tokens and row stats at
 * off[b].  Each sequence is verified by oracle_verify with its own K_b;
 * offsets that describe no packing give ORACLE_BAD_OFFSETS for that sequence. */
int oracle_verify_ragged(const void* logits, int dtype, const float* q, const int32_t* tokens,
                         const float* uniforms, const int32_t* off, int64_t B, int K_max,
                         int64_t R, int64_t V, float temperature, int32_t* accept_len,
                         int32_t* out_tokens, uint8_t* accept_mask, int32_t* status,
                         double* row_m, double* row_s, double* p_draft, double* accept_margin,
                         double* sample_margin, int32_t* sample_alt);

/* Greedy verification, the limit T -> 0 of oracle_verify: a_i = the first
 * token holding the largest logit of row i; draft x_i is accepted iff
 * x_i = a_i; the first rejected position j emits a_j, and a fully accepted
 * sequence emits the bonus a_K.  No q and no uniforms.  Outputs as
 * oracle_verify (accept_len 0 and tokens -1 on a sequence error); row_argmax
 * [B, K+1] (optional) holds a_i for the rows reached, -1 for the others and for
 * every row of an erroneous sequence. */
int oracle_verify_greedy(const void* logits, int dtype, const int32_t* tokens, int64_t B, int K,
                         int64_t V, int32_t* accept_len, int32_t* out_tokens,
                         uint8_t* accept_mask, int32_t* status, int32_t* row_argmax);

/* Histogram of accepted lengths: hist[n] = sequences with accept_len n,
 * n = 0..K+1 (0 = sequence error).  Returns 1 if a length is outside that range. */
int oracle_accept_hist(const int32_t* accept_len, int64_t B, int K, uint64_t* hist);

/* Acceptance rate (accepted / tested drafts), mean accepted length, per-position
 * acceptance (K values) of a histogram taken at depth K, and the next depth:
 * K (bounded by K_max) while fewer than min_tested drafts were tested, K_floor
 * when the acceptance is below `threshold`, K_max otherwise. */
int oracle_adapt(const uint64_t* hist, int K, int K_max, int K_floor, double threshold,
                 uint64_t min_tested, double* acceptance, double* mean_len,
                 double* pos_acceptance, int* next_K);

#ifdef __cplusplus
}
#endif
#endif
