/*
 * oracle.c -- fp64 CPU reference for batched speculative-decoding verification.
 *
 * TEST INFRASTRUCTURE ONLY (see oracle.h for the citations [P1]-[P3]).  It is
 * slow and plain on purpose: one sequence at a time, one row at a time, every
 * sum a left-to-right loop in double precision.  It follows the method step by
 * step as the pages state it; where the pages leave a step open, the reading
 * taken is stated next to the step.
 *
 * Build: gcc -O2 -ffp-contract=off -shared -fPIC oracle.c -lm
 * The same source built with -fopenmp verifies the sequences of a batch on
 * several host threads (each sequence on one thread, with its own scratch
 * rows); every sequence's arithmetic is the same either way.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Host threads the batch loops use: 1 unless built with OpenMP. */
int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Sets the thread count of later batch loops (OpenMP build; n >= 1) and
 * returns the count now in force. */
int oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n >= 1)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
    return oracle_threads();
}

/* One stored logit as an exact double.  bf16 widens to fp32 by placing its 16
 * bits in the high half of the word; both widen exactly to double. */
static double logit_at(const void* base, int dtype, int64_t idx)
{
    if (dtype == 0)
        return (double)((const float*)base)[idx];
    uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* [P1] "Speculative decoding: draft first, then verify": each target row is
 * turned into a distribution by a softmax of logits / T.  Written out: z = l/T,
 * m = max z, s = sum exp(z - m), p = exp(z - m) / s.  A NaN, a +inf, or a row
 * with no finite-or-smaller value (all -inf) has no distribution; the pages are
 * silent, and the reading taken is that such a sequence is an error. */
int oracle_softmax_row(const void* row, int dtype, int64_t V, double T,
                       double* p, double* m_out, double* s_out)
{
    double m = -INFINITY;
    for (int64_t v = 0; v < V; ++v) {
        double z = logit_at(row, dtype, v) / T;
        if (isnan(z))
            return ORACLE_NONFINITE;
        if (z > m)
            m = z;
    }
    if (!isfinite(m))
        return ORACLE_NONFINITE;
    double s = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        double e = exp(logit_at(row, dtype, v) / T - m);
        p[v] = e;
        s += e;
    }
    for (int64_t v = 0; v < V; ++v)
        p[v] /= s;
    *m_out = m;
    *s_out = s;
    return ORACLE_OK;
}

static int q_value_ok(float x)
{
    return x >= 0.0f && isfinite(x);
}

/* Inverse-CDF draw from weights w[0..V) with the single uniform u: the first
 * token whose running sum exceeds u * S, tokens taken in ascending id order.
 * The pages call torch.multinomial and do not fix which exact sampler it is;
 * any exact sampler has the right law, and this one is the plain definition.
 * A weight of zero can never be drawn.  If rounding leaves u * S at or past the
 * last running sum, the last positive-weight token is taken.
 * Also reports the tie margin: the distance from u to the normalised running
 * sums just below and at the drawn token, each counted only when a
 * positive-weight token lies on the far side of that boundary. */
static int64_t draw_inverse_cdf(const double* w, int64_t V, double S, double u,
                                double* margin, int32_t* alt)
{
    const double t = u * S;
    double run = 0.0, before = 0.0;
    int64_t tok = -1;
    for (int64_t v = 0; v < V; ++v) {
        before = run;
        run += w[v];
        if (run > t) {
            tok = v;
            break;
        }
    }
    if (tok < 0) {
        for (int64_t v = V - 1; v >= 0; --v)
            if (w[v] > 0.0) {
                tok = v;
                break;
            }
        before = 0.0;
        for (int64_t v = 0; v < tok; ++v)
            before += w[v];
        run = before + w[tok];
    }
    int64_t prev = -1, next = -1;
    for (int64_t v = tok - 1; v >= 0; --v)
        if (w[v] > 0.0) {
            prev = v;
            break;
        }
    for (int64_t v = tok + 1; v < V; ++v)
        if (w[v] > 0.0) {
            next = v;
            break;
        }
    double m_lo = prev >= 0 ? fabs(u - before / S) : INFINITY;
    double m_hi = next >= 0 ? fabs(u - run / S) : INFINITY;
    if (m_lo <= m_hi) {
        *margin = m_lo;
        *alt = (int32_t)prev;
    } else {
        *margin = m_hi;
        *alt = (int32_t)next;
    }
    return tok;
}

/* Truncation of a target row (the production sampler settings of [P2] "Two
 * things that follow from the math": temperature 0.6, top-p 0.95, min-p 0.05).
 * The pages name the settings, not the definitions or their order; the
 * readings taken, both on the untruncated p and therefore order-free:
 *   min-p keeps v when p_v >= min_p * max_u p_u;
 *   top-p keeps v when the mass of the tokens strictly more probable than v
 *         is below top_p (the smallest set of most probable tokens whose mass
 *         reaches top_p, with every token tied at its boundary kept);
 * a token is kept when both keep it, and p~ = p on the kept tokens, divided by
 * their sum.  top_p >= 1 and min_p <= 0 switch a filter off. */
typedef struct {
    double top_p, min_p;
} trunc_opts;

/* the row qsort orders: one per thread in the OpenMP build */
#ifdef _OPENMP
static __thread const double* g_sort_p;
#else
static const double* g_sort_p;
#endif

static int by_p_desc(const void* a, const void* b)
{
    const int64_t i = *(const int64_t*)a, j = *(const int64_t*)b;
    if (g_sort_p[i] != g_sort_p[j])
        return g_sort_p[i] > g_sort_p[j] ? -1 : 1;
    return i < j ? -1 : (i > j);
}

/* p (a softmax row) becomes p~ in place.  *margin is lowered to the distance
 * of the row from a filter boundary: |log(p_v / p_max) - log(min_p)| over
 * tokens, and |mass above v - top_p| over tokens, for the filters in use. */
static int truncate_row(double* p, int64_t V, const trunc_opts* tr, double* margin)
{
    double pmax = 0.0;
    for (int64_t v = 0; v < V; ++v)
        if (p[v] > pmax)
            pmax = p[v];
    unsigned char* keep = (unsigned char*)malloc((size_t)V);
    int64_t* order = (int64_t*)malloc((size_t)V * sizeof(int64_t));
    if (!keep || !order) {
        free(keep);
        free(order);
        return -2;
    }
    for (int64_t v = 0; v < V; ++v) {
        keep[v] = 1;
        if (tr->min_p > 0.0) {
            if (!(p[v] >= tr->min_p * pmax))
                keep[v] = 0;
            const double d = fabs(log(p[v] / pmax) - log(tr->min_p));
            if (d < *margin)
                *margin = d;
        }
    }
    if (tr->top_p < 1.0) {
        for (int64_t v = 0; v < V; ++v)
            order[v] = v;
        g_sort_p = p;
        qsort(order, (size_t)V, sizeof(int64_t), by_p_desc);
        double above = 0.0; /* mass of the tokens strictly more probable */
        int64_t g0 = 0;
        while (g0 < V) {
            int64_t g1 = g0;
            double gm = 0.0;
            while (g1 < V && p[order[g1]] == p[order[g0]]) {
                gm += p[order[g1]];
                ++g1;
            }
            const double d = fabs(above - tr->top_p);
            if (d < *margin)
                *margin = d;
            if (!(above < tr->top_p))
                for (int64_t k = g0; k < g1; ++k)
                    keep[order[k]] = 0;
            above += gm;
            g0 = g1;
        }
    }
    /* nothing dropped: p~ is p itself (no second normalisation) */
    int64_t dropped = 0;
    for (int64_t v = 0; v < V; ++v)
        dropped += !keep[v];
    double kept = 0.0;
    for (int64_t v = 0; v < V; ++v)
        if (keep[v])
            kept += p[v];
    for (int64_t v = 0; v < V && dropped; ++v)
        p[v] = keep[v] ? p[v] / kept : 0.0;
    free(keep);
    free(order);
    return ORACLE_OK;
}

/* One sequence.  p and w are scratch rows of V doubles.  With `tr`, every
 * target row is truncated (truncate_row) before it is used. */
static int verify_one(const void* logits, int dtype, const float* q, const int32_t* x,
                      const float* u, int K, int64_t V, double T, double* p, double* w,
                      int32_t* out_tok, uint8_t* mask, double* rm, double* rs, double* pd,
                      double* a_margin, double* s_margin, int32_t* s_alt, int32_t* len,
                      const trunc_opts* tr, double* t_margin, const void* dlog, double Td,
                      double* qrow)
{
    const size_t esz = dtype == 0 ? 4 : 2;
    const char* lbase = (const char*)logits;

    /* Every draft token must name a vocabulary entry and every uniform must lie
     * in [0, 1) (the pages draw them with torch.rand, which has that range). */
    for (int i = 0; i < K; ++i)
        if (x[i] < 0 || (int64_t)x[i] >= V)
            return ORACLE_TOKEN_RANGE;
    for (int i = 0; i <= K; ++i)
        if (!(u[i] >= 0.0f && u[i] < 1.0f))
            return ORACLE_UNIFORM_RANGE;

    /* [P1] verify loop: positions in order, stop at the first rejection.
     * Acceptance probability is min(1, p(x)/q(x)) ([P1]; [P2] "Speculative
     * decoding").  The test "u < min(1, p/q)" with u in [0, 1) is written as
     * u * q(x) < p(x): identical for q(x) > 0, and for q(x) = 0 it accepts
     * exactly when p(x) > 0.  The pages' prior-art code adds 1e-9 to q(x) as a
     * guard; the method itself has no such term and it is left out. */
    int j = K;
    double m = 0.0, s = 0.0;
    for (int i = 0; i < K; ++i) {
        int st = oracle_softmax_row(lbase + (size_t)i * (size_t)V * esz, dtype, V, T, p, &m, &s);
        if (st != ORACLE_OK)
            return st;
        if (tr && (st = truncate_row(p, V, tr, t_margin)) != ORACLE_OK)
            return st;
        rm[i] = m;
        rs[i] = s;
        const double px = p[x[i]];
        double qx;
        if (dlog) {
            /* draft logits given: q_i = softmax(d_i / T_d), the row the drafter
             * sampled x_i from, computed when its test runs */
            double dm, ds;
            st = oracle_softmax_row((const char*)dlog + (size_t)i * (size_t)V * esz, dtype, V, Td,
                                    qrow, &dm, &ds);
            if (st != ORACLE_OK)
                return st;
            qx = qrow[x[i]];
        } else {
            const float qf = q[(size_t)i * (size_t)V + (size_t)x[i]];
            if (!q_value_ok(qf))
                return ORACLE_NONFINITE;
            qx = (double)qf;
        }
        pd[i] = px;
        if (qx > 0.0) {
            double mg = fabs((double)u[i] - px / qx);
            if (mg < *a_margin)
                *a_margin = mg;
        }
        if ((double)u[i] * qx < px)
            continue; /* accepted */
        j = i;
        break;
    }

    double S = 0.0;
    if (j < K) {
        /* [P1] rejection at position j: the corrected token comes from
         * relu(p_j - q_j) normalised by its sum. */
        const float* qj = dlog ? 0 : q + (size_t)j * (size_t)V;
        for (int64_t v = 0; v < V; ++v) {
            double qv;
            if (tr && (tr->top_p < 1.0 || tr->min_p > 0.0) && p[v] == 0.0) {
                /* Against a truncated target the residual max(0, p~ - q) is
                 * zero wherever p~ is: q_j enters only at the kept tokens,
                 * and is read (and checked) there alone, as q(x_i) is in the
                 * test. */
                w[v] = 0.0;
                continue;
            }
            if (dlog) {
                qv = qrow[v]; /* row j: the last row tested */
            } else {
                if (!q_value_ok(qj[v]))
                    return ORACLE_NONFINITE;
                qv = (double)qj[v];
            }
            const double d = p[v] - qv;
            w[v] = d > 0.0 ? d : 0.0;
            S += w[v];
        }
        /* Exact arithmetic cannot reject with S = 0 when both rows sum to one;
         * rounding or an unnormalised q can.  The pages are silent; the reading
         * taken is to draw from p_j itself with the same uniform. */
        if (S == 0.0) {
            for (int64_t v = 0; v < V; ++v) {
                w[v] = p[v];
                S += w[v];
            }
        }
    } else {
        /* [P1] every draft accepted: the bonus token comes from the softmax of
         * the last target row. */
        int st = oracle_softmax_row(lbase + (size_t)K * (size_t)V * esz, dtype, V, T, p, &m, &s);
        if (st != ORACLE_OK)
            return st;
        if (tr && (st = truncate_row(p, V, tr, t_margin)) != ORACLE_OK)
            return st;
        rm[K] = m;
        rs[K] = s;
        for (int64_t v = 0; v < V; ++v) {
            w[v] = p[v];
            S += w[v];
        }
    }

    /* One uniform for the one sample of the pass: u[K]. */
    const int64_t tok = draw_inverse_cdf(w, V, S, (double)u[K], s_margin, s_alt);

    /* [P3] the accepted length counts the accepted drafts plus the one token
     * the target always adds: AL in [1, 1 + D]. */
    *len = j + 1;
    for (int i = 0; i < j; ++i) {
        out_tok[i] = x[i];
        mask[i] = 1;
    }
    out_tok[j] = (int32_t)tok;
    return ORACLE_OK;
}

static int verify_batch(const void* logits, int dtype, const float* q, const int32_t* tokens,
                        const float* uniforms, int64_t B, int K, int64_t V, float temperature,
                        int32_t* accept_len, int32_t* out_tokens, uint8_t* accept_mask,
                        int32_t* status, double* row_m, double* row_s, double* p_draft,
                        double* accept_margin, double* sample_margin, int32_t* sample_alt,
                        const trunc_opts* tr, double* trunc_margin, const void* dlogits,
                        double Td)
{
    if (!logits || !uniforms || !accept_len || !out_tokens || B < 0 || K < 0 || V < 1 ||
        (K > 0 && ((!q && !dlogits) || !tokens || !accept_mask)) || (dtype != 0 && dtype != 1) ||
        !(temperature > 0.0f) || !isfinite(temperature))
        return -1;
    /* scratch per thread: two rows of V doubles (three with draft logits),
     * plus the per-row results of one sequence */
    const int nth = oracle_threads();
    const size_t nr = (size_t)(K + 1);
    double* p_all = (double*)malloc((size_t)nth * (size_t)V * sizeof(double));
    double* w_all = (double*)malloc((size_t)nth * (size_t)V * sizeof(double));
    double* rm_all = (double*)malloc((size_t)nth * nr * sizeof(double));
    double* rs_all = (double*)malloc((size_t)nth * nr * sizeof(double));
    double* pd_all = (double*)malloc((size_t)nth * nr * sizeof(double));
    double* q_all = dlogits ? (double*)malloc((size_t)nth * (size_t)V * sizeof(double)) : 0;
    if (!p_all || !w_all || !rm_all || !rs_all || !pd_all || (dlogits && !q_all)) {
        free(p_all); free(w_all); free(rm_all); free(rs_all); free(pd_all); free(q_all);
        return -2;
    }
    const size_t esz = dtype == 0 ? 4 : 2;
    const double T = (double)temperature;

#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nth)
#endif
    for (int64_t b = 0; b < B; ++b) {
#ifdef _OPENMP
        const size_t th = (size_t)omp_get_thread_num();
#else
        const size_t th = 0;
#endif
        double* p = p_all + th * (size_t)V;
        double* w = w_all + th * (size_t)V;
        double* rm = rm_all + th * nr;
        double* rs = rs_all + th * nr;
        double* pd = pd_all + th * nr;
        double* qrow = q_all ? q_all + th * (size_t)V : 0;
        int32_t* ot = out_tokens + (size_t)b * (size_t)(K + 1);
        uint8_t* mk = K > 0 ? accept_mask + (size_t)b * (size_t)K : 0;
        uint8_t mk_dummy[1];
        for (int i = 0; i <= K; ++i) {
            ot[i] = -1;
            rm[i] = NAN;
            rs[i] = NAN;
            if (i < K) {
                mk[i] = 0;
                pd[i] = NAN;
            }
        }
        double a_mg = INFINITY, s_mg = INFINITY, t_mg = INFINITY;
        int32_t s_alt = -1, len = 0;
        int st = verify_one((const char*)logits + (size_t)b * (size_t)(K + 1) * (size_t)V * esz,
                            dtype, K > 0 && q ? q + (size_t)b * (size_t)K * (size_t)V : 0,
                            K > 0 ? tokens + (size_t)b * (size_t)K : 0,
                            uniforms + (size_t)b * (size_t)(K + 1), K, V, T, p, w, ot,
                            mk ? mk : mk_dummy, rm, rs, pd, &a_mg, &s_mg, &s_alt, &len, tr,
                            &t_mg,
                            dlogits ? (const char*)dlogits +
                                          (size_t)b * (size_t)K * (size_t)V * esz : 0,
                            Td, qrow);
        if (st != ORACLE_OK) {
            /* an erroneous sequence reports nothing but its status */
            len = 0;
            for (int i = 0; i <= K; ++i) {
                ot[i] = -1;
                rm[i] = NAN;
                rs[i] = NAN;
                if (i < K) {
                    mk[i] = 0;
                    pd[i] = NAN;
                }
            }
            a_mg = INFINITY;
            s_mg = INFINITY;
            s_alt = -1;
        }
        accept_len[b] = len;
        if (status)
            status[b] = st;
        if (trunc_margin)
            trunc_margin[b] = st == ORACLE_OK ? t_mg : INFINITY;
        if (row_m)
            for (int i = 0; i <= K; ++i)
                row_m[(size_t)b * (size_t)(K + 1) + (size_t)i] = rm[i];
        if (row_s)
            for (int i = 0; i <= K; ++i)
                row_s[(size_t)b * (size_t)(K + 1) + (size_t)i] = rs[i];
        if (p_draft)
            for (int i = 0; i < K; ++i)
                p_draft[(size_t)b * (size_t)K + (size_t)i] = pd[i];
        if (accept_margin)
            accept_margin[b] = a_mg;
        if (sample_margin)
            sample_margin[b] = s_mg;
        if (sample_alt)
            sample_alt[b] = s_alt;
    }
    free(p_all); free(w_all); free(rm_all); free(rs_all); free(pd_all); free(q_all);
    return 0;
}

int oracle_verify(const void* logits, int dtype, const float* q, const int32_t* tokens,
                  const float* uniforms, int64_t B, int K, int64_t V, float temperature,
                  int32_t* accept_len, int32_t* out_tokens, uint8_t* accept_mask,
                  int32_t* status, double* row_m, double* row_s, double* p_draft,
                  double* accept_margin, double* sample_margin, int32_t* sample_alt)
{
    return verify_batch(logits, dtype, q, tokens, uniforms, B, K, V, temperature, accept_len,
                        out_tokens, accept_mask, status, row_m, row_s, p_draft, accept_margin,
                        sample_margin, sample_alt, 0, 0, 0, 1.0);
}

/* The verify with the truncated target p~ (truncate_row) in place of p in
 * every step: the test u*q(x) < p~(x), the residual max(0, p~_j - q_j), the
 * bonus row p~_K.  Row statistics stay those of the untruncated softmax;
 * p_draft reports p~(x).  trunc_margin [B] (optional): the smallest distance of
 * a reached row from a filter boundary (see truncate_row). */
int oracle_verify_truncated(const void* logits, int dtype, const float* q, const int32_t* tokens,
                            const float* uniforms, int64_t B, int K, int64_t V,
                            float temperature, double top_p, double min_p, int32_t* accept_len,
                            int32_t* out_tokens, uint8_t* accept_mask, int32_t* status,
                            double* row_m, double* row_s, double* p_draft,
                            double* accept_margin, double* sample_margin, int32_t* sample_alt,
                            double* trunc_margin)
{
    if (!(top_p > 0.0) || !(min_p < 1.0) || isnan(top_p) || isnan(min_p))
        return -1;
    trunc_opts tr = {top_p, min_p};
    return verify_batch(logits, dtype, q, tokens, uniforms, B, K, V, temperature, accept_len,
                        out_tokens, accept_mask, status, row_m, row_s, p_draft, accept_margin,
                        sample_margin, sample_alt, &tr, trunc_margin, 0, 1.0);
}

/* The verify with draft LOGITS in place of draft probabilities: the drafter's
 * distribution at position i is q_i = softmax(d_i / T_d) ([P1]'s loop forms it
 * the same way from the draft model's logits), computed in double precision
 * when the loop needs it (the test at i; the residual at the rejected row).
 * A draft row that holds a NaN or +inf, or only -inf, is a sequence error when
 * the loop reaches it.  dlogits [B, K, V] has the target's dtype.  top_p >= 1
 * and min_p <= 0 leave the target untruncated. */
int oracle_verify_draft_logits(const void* logits, int dtype, const void* dlogits,
                               const int32_t* tokens, const float* uniforms, int64_t B, int K,
                               int64_t V, float temperature, float draft_temperature,
                               double top_p, double min_p, int32_t* accept_len,
                               int32_t* out_tokens, uint8_t* accept_mask, int32_t* status,
                               double* row_m, double* row_s, double* p_draft,
                               double* accept_margin, double* sample_margin,
                               int32_t* sample_alt, double* trunc_margin)
{
    if (!dlogits || !(top_p > 0.0) || !(min_p < 1.0) || isnan(top_p) || isnan(min_p) ||
        !(draft_temperature > 0.0f) || !isfinite(draft_temperature))
        return -1;
    trunc_opts tr = {top_p, min_p};
    const int off = top_p >= 1.0 && min_p <= 0.0;
    return verify_batch(logits, dtype, 0, tokens, uniforms, B, K, V, temperature, accept_len,
                        out_tokens, accept_mask, status, row_m, row_s, p_draft, accept_margin,
                        sample_margin, sample_alt, off ? 0 : &tr, trunc_margin, dlogits,
                        (double)draft_temperature);
}

/* Acceptance telemetry ([P1] "Production perspective" and its operational
 * checklist: acceptance rate, mean accepted length, acceptance histograms),
 * from the definitions, one sequence at a time. */
int oracle_accept_hist(const int32_t* accept_len, int64_t B, int K, uint64_t* hist) {
    if (K < 0 || B < 0)
        return 1;
    for (int n = 0; n <= K + 1; ++n)
        hist[n] = 0;
    for (int64_t b = 0; b < B; ++b) {
        const int32_t n = accept_len[b];
        if (n < 0 || n > K + 1)
            return 1;
        hist[n] += 1;
    }
    return 0;
}

/* What a histogram at depth K says, and the depth rule of [P2] ("Two things
 * that follow from the math": cap the depth when the measured acceptance is
 * below the threshold, 35 % on the page).  A sequence with accepted length n
 * (1 <= n <= K+1) tested min(n, K) drafts and accepted n - 1 of them; it
 * tested position i when n >= i + 1 and accepted it when n >= i + 2. */
int oracle_adapt(const uint64_t* hist, int K, int K_max, int K_floor, double threshold,
                 uint64_t min_tested, double* acceptance, double* mean_len,
                 double* pos_acceptance, int* next_K) {
    if (K < 0 || K_floor < 0 || K_floor > K_max)
        return 1;
    uint64_t seqs = 0, tested = 0, accepted = 0, len_sum = 0;
    for (int n = 1; n <= K + 1; ++n) {
        seqs += hist[n];
        tested += hist[n] * (uint64_t)(n < K ? n : K);
        accepted += hist[n] * (uint64_t)(n - 1);
        len_sum += hist[n] * (uint64_t)n;
    }
    for (int i = 0; i < K; ++i) {
        uint64_t t = 0, a = 0;
        for (int n = i + 1; n <= K + 1; ++n)
            t += hist[n];
        for (int n = i + 2; n <= K + 1; ++n)
            a += hist[n];
        pos_acceptance[i] = t ? (double)a / (double)t : NAN;
    }
    *acceptance = tested ? (double)accepted / (double)tested : NAN;
    *mean_len = seqs ? (double)len_sum / (double)seqs : NAN;
    if (tested == 0 || tested < min_tested)
        *next_K = K < K_max ? K : K_max;
    else if (*acceptance < threshold)
        *next_K = K_floor;
    else
        *next_K = K_max;
    return 0;
}

/* Greedy verification: the verify step in the limit T -> 0.  As T falls, the
 * softmax of l/T ([P1] "Speculative decoding: draft first, then verify")
 * puts all of its mass on the largest logit, so p_i becomes one-hot at
 * a_i = argmax_v l[b,i,v].  Then [P1]'s test u*q(x) < p(x) accepts exactly
 * when x_i = a_i (p(x) = 1 > u*q(x) for u < 1, q <= 1; p(x) = 0 otherwise),
 * the residual max(0, p_j - q_j) is positive only at a_j, and the bonus row
 * draws a_K, so neither q nor u is needed.  Readings where the limit is not
 * unique: among equal largest logits the lowest token id is a_i (the
 * first-occurrence rule of argmax); a row the loop reaches that holds a NaN or
 * +inf, or only -inf, is a sequence error, as for the sampled verify.
 *
 * Outputs as oracle_verify; row_argmax [B, K+1] (optional) holds a_i for the
 * rows the loop reached and -1 for the others. */
int oracle_verify_greedy(const void* logits, int dtype, const int32_t* tokens, int64_t B, int K,
                         int64_t V, int32_t* accept_len, int32_t* out_tokens,
                         uint8_t* accept_mask, int32_t* status, int32_t* row_argmax)
{
    if (B < 0 || K < 0 || V < 1)
        return 1;
    const size_t es = dtype == 0 ? 4 : 2;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t b = 0; b < B; ++b) {
        int st = ORACLE_OK, len = 0;
        int32_t* ot = out_tokens + (size_t)b * (size_t)(K + 1);
        for (int i = 0; i <= K; ++i)
            ot[i] = -1;
        for (int i = 0; i < K; ++i)
            accept_mask[(size_t)b * (size_t)K + (size_t)i] = 0;
        if (row_argmax)
            for (int i = 0; i <= K; ++i)
                row_argmax[(size_t)b * (size_t)(K + 1) + (size_t)i] = -1;
        for (int i = 0; i < K; ++i) {
            const int32_t x = tokens[(size_t)b * (size_t)K + (size_t)i];
            if (x < 0 || (int64_t)x >= V)
                st = ORACLE_TOKEN_RANGE;
        }
        for (int i = 0; st == ORACLE_OK && i <= K; ++i) {
            const char* row = (const char*)logits + ((size_t)b * (size_t)(K + 1) + (size_t)i) *
                                                        (size_t)V * es;
            /* a_i: the first token holding the largest logit */
            double best = -INFINITY;
            int64_t a = -1;
            for (int64_t v = 0; v < V; ++v) {
                const double l = logit_at(row, dtype, v);
                if (isnan(l) || l == INFINITY) {
                    st = ORACLE_NONFINITE;
                    break;
                }
                if (l > best) {
                    best = l;
                    a = v;
                }
            }
            if (st == ORACLE_OK && a < 0)
                st = ORACLE_NONFINITE; /* every logit is -inf */
            if (st != ORACLE_OK)
                break;
            if (row_argmax)
                row_argmax[(size_t)b * (size_t)(K + 1) + (size_t)i] = (int32_t)a;
            if (i < K && tokens[(size_t)b * (size_t)K + (size_t)i] == (int32_t)a) {
                ot[i] = (int32_t)a; /* accepted: the draft token stays */
                accept_mask[(size_t)b * (size_t)K + (size_t)i] = 1;
                continue;
            }
            ot[i] = (int32_t)a; /* the corrected token (i < K) or the bonus token (i = K) */
            len = i + 1;
            break;
        }
        if (st != ORACLE_OK) { /* an erroneous sequence reports no per-row outputs */
            len = 0;
            for (int i = 0; i <= K; ++i)
                ot[i] = -1;
            for (int i = 0; i < K; ++i)
                accept_mask[(size_t)b * (size_t)K + (size_t)i] = 0;
            if (row_argmax)
                for (int i = 0; i <= K; ++i)
                    row_argmax[(size_t)b * (size_t)(K + 1) + (size_t)i] = -1;
        }
        accept_len[b] = len;
        if (status)
            status[b] = st;
    }
    return 0;
}

/* Ragged batches: sequence b owns target rows [off[b], off[b+1]) of a packed
 * [R, V] logits array, so its draft depth is K_b = off[b+1] - off[b] - 1.  The
 * pages verify one sequence at a time ([P1]'s loop); batching is a scheduling
 * matter ([P1] "Scheduling interaction"), so each sequence is verified on its
 * own by oracle_verify with its own K_b.  Its draft rows, tokens, mask and
 * draft probabilities start at off[b] - b (K_b of them); uniforms, output
 * tokens and row statistics at off[b] (K_b + 1).  Offsets that do not describe
 * such a packing (off[b] < b, off[b+1] <= off[b], K_b > K_max, or too few rows
 * left for the sequences after b) make that sequence an error
 * (ORACLE_BAD_OFFSETS, accept_len 0) and nothing of it is read or written
 * except accept_len and status. */
int oracle_verify_ragged(const void* logits, int dtype, const float* q, const int32_t* tokens,
                         const float* uniforms, const int32_t* off, int64_t B, int K_max,
                         int64_t R, int64_t V, float temperature, int32_t* accept_len,
                         int32_t* out_tokens, uint8_t* accept_mask, int32_t* status,
                         double* row_m, double* row_s, double* p_draft, double* accept_margin,
                         double* sample_margin, int32_t* sample_alt)
{
    if (!off || B < 0 || K_max < 0 || R < B)
        return -1;
    const size_t esz = dtype == 0 ? 4 : 2;
    int rc_any = 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t b = 0; b < B; ++b) {
        const int64_t o0 = off[b], o1 = off[b + 1];
        const int64_t Kb = o1 - o0 - 1;
        if (o0 < b || Kb < 0 || Kb > K_max || o1 + (B - b - 1) > R) {
            accept_len[b] = 0;
            if (status)
                status[b] = ORACLE_BAD_OFFSETS;
            if (accept_margin)
                accept_margin[b] = INFINITY;
            if (sample_margin)
                sample_margin[b] = INFINITY;
            if (sample_alt)
                sample_alt[b] = -1;
            continue;
        }
        const int64_t d0 = o0 - b; /* first draft row of sequence b */
        const int rc = oracle_verify(
            (const char*)logits + (size_t)o0 * (size_t)V * esz, dtype,
            Kb ? q + (size_t)d0 * (size_t)V : 0, Kb ? tokens + d0 : 0, uniforms + o0, 1, (int)Kb, V,
            temperature, accept_len + b, out_tokens + o0, Kb ? accept_mask + d0 : 0,
            status ? status + b : 0, row_m ? row_m + o0 : 0, row_s ? row_s + o0 : 0,
            p_draft && Kb ? p_draft + d0 : 0, accept_margin ? accept_margin + b : 0,
            sample_margin ? sample_margin + b : 0, sample_alt ? sample_alt + b : 0);
        if (rc != 0) {
#ifdef _OPENMP
#pragma omp critical
#endif
            rc_any = rc;
        }
    }
    return rc_any;
}
