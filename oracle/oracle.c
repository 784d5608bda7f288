/*
 * oracle.c -- plain, slow fp64 CPU oracle for the speculative-decoding
 * verification step (the vectorised rejection sampler).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA implementation.
 *
 * Source of every step ("P3"): the speculative-decoding tutorial page at
 * http://www.dpshk.com/news/5598276/ (its HTML title, "企业官网建设流程全解析",
 * is unrelated to its content).  Sections cited below are that page's:
 *   §3.1  problem statement, steps 1-4 (draft, verify, accept with
 *         min(1, p/q), resample from (p - q)_+ at the first rejection)
 *   §3.2  why the output is exactly distributed as p (residual r(x))
 *   §3.3  expected emitted tokens (1 - a^(g+1)) / (1 - a)
 *   §4    flow diagram: worked example with ratios 0.92 / 0.75 / 0.31
 *   §5.2  RejectionSampler walk-through, steps (1)-(5): softmax of the target
 *         logits, accept_prob = min(1, p / clamp(q, 1e-10)), uniform < accept
 *         _prob, cumprod prefix mask, residual resample (_recover_rejected)
 *   §5.3  bonus token from the (g+1)-th target row when every draft is kept
 *   §8    pitfall 2: temperature 0 is greedy decoding
 *
 * Readings where the page is silent (each is listed with its reason in the
 * design notes of this repository):
 *   - temperature T divides the target logits before the softmax; T = 0 means
 *     the target distribution is one-hot at the lowest-index argmax;
 *   - the page's torch.multinomial draw is replaced by an inverse-CDF draw on
 *     a caller-supplied uniform: token = min{ j : C_j > u * S }, C the
 *     inclusive prefix sum of the residual, S its total;
 *   - if the residual total S is 0 at a rejection, sample from p instead;
 *   - draft_probs == NULL means every draft is deterministic: q is one-hot at
 *     the drafted token (prompt-lookup drafting, P3 §7);
 *   - unused output slots are -1; a request with invalid inputs gets
 *     num_accepted = -1 and an all -1 token row.
 *
 * Everything is computed in fp64; bf16 and fp32 inputs convert to fp64 exactly.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Bits of the per-request "bad input" word.  Same meaning as the CUDA
 * library's documented flags, but defined here on their own. */
enum {
    ORC_BAD_DRAFT_LEN = 1,   /* draft length outside [0, gamma_max]          */
    ORC_BAD_TEMP = 2,        /* temperature NaN, inf, negative or subnormal  */
    ORC_BAD_TOKEN = 4,       /* a draft token id outside [0, V)              */
    ORC_BAD_U_ACCEPT = 8,    /* an acceptance uniform outside [0, 1)         */
    ORC_BAD_U_SAMPLE = 16,   /* the sampling uniform outside [0, 1)          */
    ORC_BAD_NORMALISER = 32  /* non-finite softmax normaliser (T > 0 rows)   */
};

/* P3 §5.2 step (2): the divisor of the acceptance ratio is clamped at 1e-10. */
static const double ORC_Q_FLOOR = 1e-10;

/* log2(e) and the largest finite binary32 value (the range check of the
 * temperature-scaled row maximum). */
static const float ORC_LOG2E_F = 1.4426950408889634f;
static const float ORC_EXP_LIMIT = 16777216.0f; /* 2^24 */

/* |fl32(m * fl32(log2(e) / T))| < 2^24, in binary32 arithmetic. */
static int exponent_range_ok(double m, double T) {
    volatile float cs = ORC_LOG2E_F / (float)T;
    volatile float o = (float)m * cs;
    return fabsf(o) < ORC_EXP_LIMIT;
}

/* Optional outputs.  Any pointer may be NULL except tokens / num_accepted.
 * Shapes: [B] per request, [B, gmax] per draft position, [B, gmax+1] per row.
 */
typedef struct {
    int32_t *tokens;          /* [B, gmax+1] emitted tokens, -1 padded        */
    int32_t *num_accepted;    /* [B] accepted drafts, -1 for bad input        */
    int32_t *bad;             /* [B] ORC_BAD_* bits                           */
    double *resid_mass;       /* [B] S = sum (p_k - q_k)_+ (NaN if no draw)   */
    double *sample_margin;    /* [B] min(uS - C_{j-1}, C_j - uS); inf if exact*/
    int32_t *sample_fallback; /* [B] 1 if S == 0 forced a draw from p_k       */
    double *p_tok;            /* [B, gmax] p_i(x_i)                           */
    double *q_tok;            /* [B, gmax] q_i(x_i) before the clamp          */
    double *accept_prob;      /* [B, gmax] a_i = min(1, p / max(q, 1e-10))    */
    uint8_t *flags;           /* [B, gmax] 1 accept, 0 reject, 2 not evaluated*/
    double *accept_margin;    /* [B, gmax] |u_i - a_i|; inf if exact          */
    double *row_max;          /* [B, gmax+1] max_j logit                      */
    double *row_sum;          /* [B, gmax+1] sum_j exp((l_j - max)/T), T > 0  */
    int32_t *row_argmax;      /* [B, gmax+1] lowest index of the max          */
} orc_outputs;

/* ---- input element access ------------------------------------------------ */

/* A bf16 value is the upper half of an IEEE binary32; widening is exact. */
static double bf16_bits_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double logit_at(const void *logits, int is_bf16, size_t idx)
{
    if (is_bf16)
        return bf16_bits_to_double(((const uint16_t *)logits)[idx]);
    return (double)((const float *)logits)[idx];
}

/* ---- P3 §5.2 step (1): softmax of one target row ------------------------- */

/* Row statistics of the softmax of l / T: the maximum logit, the lowest index
 * attaining it, and the normaliser s = sum_j exp((l_j - max) / T).  For T = 0
 * the distribution is one-hot at the argmax and s is reported as 1. */
void orc_row_stats(const void *logits, int is_bf16, size_t row_offset, int V,
                   double T, double *out_max, double *out_sum, int *out_argmax)
{
    double mx = logit_at(logits, is_bf16, row_offset);
    int arg = 0;
    for (int j = 1; j < V; ++j) {
        double l = logit_at(logits, is_bf16, row_offset + (size_t)j);
        if (l > mx) {
            mx = l;
            arg = j;
        }
    }
    double s = 1.0;
    if (T > 0.0) {
        s = 0.0;
        for (int j = 0; j < V; ++j)
            s += exp((logit_at(logits, is_bf16, row_offset + (size_t)j) - mx) / T);
    }
    *out_max = mx;
    *out_sum = s;
    *out_argmax = arg;
}

/* p(j) of the temperature-scaled target softmax, given the row statistics. */
static double target_prob(double l_j, int j, double mx, double s, int argmax,
                          double T)
{
    if (T == 0.0)
        return j == argmax ? 1.0 : 0.0;
    return exp((l_j - mx) / T) / s;
}

/* ---- P3 §3.1 step 4 / §5.2 step (5): inverse-CDF draw --------------------- */

/* Draw from the unnormalised non-negative weights r[0..n-1] with the uniform
 * u in [0, 1): the smallest j whose inclusive prefix sum exceeds u * S, S the
 * total.  Zero-weight entries can never be chosen.  If rounding leaves no such
 * j, the last j with r_j > 0 is returned and the margin is 0.  *margin is the
 * distance of u * S to the nearer edge of the chosen token's CDF interval. */
int orc_inverse_cdf(const double *r, int n, double u, double *margin)
{
    double S = 0.0;
    for (int j = 0; j < n; ++j)
        S += r[j];
    double target = u * S;
    double c = 0.0;
    for (int j = 0; j < n; ++j) {
        double prev = c;
        c += r[j];
        if (c > target) {
            if (margin)
                *margin = fmin(target - prev, c - target);
            return j;
        }
    }
    if (margin)
        *margin = 0.0;
    for (int j = n - 1; j >= 0; --j)
        if (r[j] > 0.0)
            return j;
    return -1;
}

/* ---- input validation ----------------------------------------------------- */

static int valid_uniform(double u) { return u >= 0.0 && u < 1.0; }

static int request_bad_bits(const int32_t *draft_ids, const float *u_acc,
                            const float *u_samp, const float *temperature,
                            const int32_t *draft_lens, int b, int gmax, int V,
                            int *gamma_out)
{
    int bad = 0;
    int g = draft_lens ? draft_lens[b] : gmax;
    if (g < 0 || g > gmax) {
        bad |= ORC_BAD_DRAFT_LEN;
        g = 0;
    }
    double T = (double)temperature[b];
    /* 0 is greedy; otherwise a normal positive finite binary32 value. */
    if (!(T == 0.0 || (isfinite(T) && T >= 1.1754943508222875e-38)))
        bad |= ORC_BAD_TEMP;
    if (!valid_uniform((double)u_samp[b]))
        bad |= ORC_BAD_U_SAMPLE;
    for (int i = 0; i < g; ++i) {
        int32_t x = draft_ids[(size_t)b * gmax + i];
        if (x < 0 || x >= V)
            bad |= ORC_BAD_TOKEN;
        if (!valid_uniform((double)u_acc[(size_t)b * gmax + i]))
            bad |= ORC_BAD_U_ACCEPT;
    }
    *gamma_out = g;
    return bad;
}

/* ---- the verification step, one request at a time ------------------------ */

/*
 * Inputs (host memory, row-major):
 *   logits       [B, gmax+1, V]  bf16 bits (is_bf16 = 1) or fp32
 *   draft_ids    [B, gmax]       int32
 *   draft_probs  [B, gmax, V]    fp32, or NULL (deterministic drafts)
 *   u_acc        [B, gmax]       fp32 uniforms for the accept test
 *   u_samp       [B]             fp32 uniform for the resample / bonus draw
 *   temperature  [B]             fp32, 0 = greedy
 *   draft_lens   [B]             int32 in [0, gmax], or NULL (all gmax)
 * Returns 0, or -1 if the scratch allocation fails.
 */
/* The weights of the draw at position k of request b (P3 §3.1 step 4, §3.2,
 * §5.2 (5)): r_j = (p_k(j) - q_k(j))_+ at a rejection (k < g), p_g(j) for the
 * bonus draw (§5.3), written to r[0..V-1].  Returns S = sum_j (p_k - q_k)_+
 * (the residual mass before the fallback) and sets *fallback when S = 0 made
 * the draw use p_k itself. */
static double draw_weights(const void *logits, int is_bf16, const int32_t *draft_ids,
                           const float *draft_probs, int b, int k, int g, int gmax, int V,
                           size_t off, double mx, double s, int argmax, double T,
                           double *r, int *fallback)
{
    double S = 0.0;
    for (int j = 0; j < V; ++j) {
        double p = target_prob(logit_at(logits, is_bf16, off + (size_t)j), j, mx, s, argmax, T);
        double q = 0.0; /* bonus row: nothing to subtract */
        if (k < g) {
            if (draft_probs)
                q = (double)draft_probs[((size_t)b * gmax + k) * (size_t)V + j];
            else
                q = (j == draft_ids[(size_t)b * gmax + k]) ? 1.0 : 0.0;
        }
        r[j] = fmax(p - q, 0.0);
        S += r[j];
    }
    *fallback = 0;
    if (!(S > 0.0)) {
        /* Reading: an empty residual means p_k <= q_k everywhere; draw from
         * p_k itself. */
        for (int j = 0; j < V; ++j)
            r[j] = target_prob(logit_at(logits, is_bf16, off + (size_t)j), j, mx, s, argmax, T);
        *fallback = 1;
    }
    return S;
}

/* Requests b0 .. b1-1 of the batch (each request is independent of the
 * others; every output slot of a request is written by its own iteration). */
static int verify_range(const void *logits, int is_bf16, const int32_t *draft_ids,
                        const float *draft_probs, const float *u_acc,
                        const float *u_samp, const float *temperature,
                        const int32_t *draft_lens, int b0, int b1, int gmax, int V,
                        orc_outputs *out)
{
    const size_t rows_per_req = (size_t)gmax + 1;
    double *row_m = malloc(rows_per_req * sizeof(double));
    double *row_s = malloc(rows_per_req * sizeof(double));
    int *row_a = malloc(rows_per_req * sizeof(int));
    double *resid = malloc((size_t)(V > 0 ? V : 1) * sizeof(double));
    if (!row_m || !row_s || !row_a || !resid) {
        free(row_m); free(row_s); free(row_a); free(resid);
        return -1;
    }

    for (int b = b0; b < b1; ++b) {
        int32_t *tok = out->tokens + (size_t)b * rows_per_req;
        for (size_t i = 0; i < rows_per_req; ++i)
            tok[i] = -1;
        if (out->resid_mass) out->resid_mass[b] = NAN;
        if (out->sample_margin) out->sample_margin[b] = INFINITY;
        if (out->sample_fallback) out->sample_fallback[b] = 0;
        for (int i = 0; i < gmax; ++i) {
            size_t pi = (size_t)b * gmax + i;
            if (out->p_tok) out->p_tok[pi] = NAN;
            if (out->q_tok) out->q_tok[pi] = NAN;
            if (out->accept_prob) out->accept_prob[pi] = NAN;
            if (out->flags) out->flags[pi] = 2;
            if (out->accept_margin) out->accept_margin[pi] = INFINITY;
        }
        for (size_t i = 0; i < rows_per_req; ++i) {
            size_t ri = (size_t)b * rows_per_req + i;
            if (out->row_max) out->row_max[ri] = NAN;
            if (out->row_sum) out->row_sum[ri] = NAN;
            if (out->row_argmax) out->row_argmax[ri] = -1;
        }

        int g;
        int bad = request_bad_bits(draft_ids, u_acc, u_samp, temperature,
                                   draft_lens, b, gmax, V, &g);
        const double T = (double)temperature[b];

        /* P3 §3.1 step 2 / §5.2 (1): the target distribution of each of the
         * g+1 rows; row g is the bonus row (§5.3). */
        if (!bad) {
            for (int i = 0; i <= g; ++i) {
                size_t off = ((size_t)b * rows_per_req + i) * (size_t)V;
                orc_row_stats(logits, is_bf16, off, V, T, &row_m[i], &row_s[i],
                              &row_a[i]);
                if (T > 0.0 && !(isfinite(row_m[i]) && isfinite(row_s[i])))
                    bad |= ORC_BAD_NORMALISER;
                /* Reading: the step works on binary32 logits (the pages' fp32
                 * tensors) and so in binary32 arithmetic, where p is formed
                 * from exponents (l - m) * log2(e) / T.  A temperature so
                 * small that the row maximum in log2 units, m * cs with
                 * cs = log2(e) / T (both rounded to binary32), reaches 2^24
                 * in magnitude leaves no binary32 room to form those
                 * exponents (the rounding error of m * cs alone exceeds 1):
                 * invalid data, like a non-finite normaliser.  The product is
                 * taken in binary32, as the step takes it. */
                if (T > 0.0 && isfinite(row_m[i]) && !exponent_range_ok(row_m[i], T))
                    bad |= ORC_BAD_NORMALISER;
            }
        }
        if (out->bad) out->bad[b] = bad;
        if (bad) {
            out->num_accepted[b] = -1;
            continue;
        }
        for (int i = 0; i <= g; ++i) {
            size_t ri = (size_t)b * rows_per_req + i;
            if (out->row_max) out->row_max[ri] = row_m[i];
            if (out->row_sum) out->row_sum[ri] = row_s[i];
            if (out->row_argmax) out->row_argmax[ri] = row_a[i];
        }

        /* P3 §3.1 step 3 / §5.2 (2)-(3): a_i = min(1, p_i(x_i) / max(q_i(x_i),
         * 1e-10)), accepted iff u_i < a_i.  Every position is evaluated (the
         * flags after the first rejection are diagnostics only). */
        int k = g; /* P3 §5.2 (4): cumprod of the flags = first rejection */
        for (int i = 0; i < g; ++i) {
            size_t pi = (size_t)b * gmax + i;
            size_t off = ((size_t)b * rows_per_req + i) * (size_t)V;
            int x = draft_ids[pi];
            double P = target_prob(logit_at(logits, is_bf16, off + (size_t)x),
                                   x, row_m[i], row_s[i], row_a[i], T);
            double q = draft_probs
                           ? (double)draft_probs[((size_t)b * gmax + i) * (size_t)V + x]
                           : 1.0;
            double a = fmin(1.0, P / fmax(q, ORC_Q_FLOOR));
            double u = (double)u_acc[pi];
            int f = u < a;
            if (f == 0 && k == g)
                k = i;
            if (out->p_tok) out->p_tok[pi] = P;
            if (out->q_tok) out->q_tok[pi] = q;
            if (out->accept_prob) out->accept_prob[pi] = a;
            if (out->flags) out->flags[pi] = (uint8_t)f;
            /* Greedy targets give a of exactly 0 or 1: the decision is exact. */
            if (out->accept_margin)
                out->accept_margin[pi] =
                    (T == 0.0 && (a == 0.0 || a == 1.0)) ? INFINITY : fabs(u - a);
        }
        out->num_accepted[b] = k;

        /* P3 §4 / §5.4: the k accepted drafts are emitted, later ones dropped. */
        for (int i = 0; i < k; ++i)
            tok[i] = draft_ids[(size_t)b * gmax + i];

        /* Token at position k: the residual resample at a rejection (P3 §3.1
         * step 4, §3.2, §5.2 (5)) or the bonus draw from row g (§5.3). */
        size_t off = ((size_t)b * rows_per_req + k) * (size_t)V;
        if (T == 0.0) {
            tok[k] = row_a[k]; /* p_k is one-hot at its argmax */
            continue;
        }
        int fallback = 0;
        double S = draw_weights(logits, is_bf16, draft_ids, draft_probs, b, k, g, gmax, V,
                                off, row_m[k], row_s[k], row_a[k], T, resid, &fallback);
        if (out->resid_mass) out->resid_mass[b] = S;
        if (out->sample_fallback) out->sample_fallback[b] = fallback;
        double margin = 0.0;
        tok[k] = orc_inverse_cdf(resid, V, (double)u_samp[b], &margin);
        if (out->sample_margin) out->sample_margin[b] = margin;
    }

    free(row_m);
    free(row_s);
    free(row_a);
    free(resid);
    return 0;
}

int orc_verify(const void *logits, int is_bf16, const int32_t *draft_ids,
               const float *draft_probs, const float *u_acc,
               const float *u_samp, const float *temperature,
               const int32_t *draft_lens, int B, int gmax, int V,
               orc_outputs *out)
{
    return verify_range(logits, is_bf16, draft_ids, draft_probs, u_acc, u_samp,
                        temperature, draft_lens, 0, B, gmax, V, out);
}

/* ---- the same step on several host threads (for timing on many cores) -- */

typedef struct {
    const void *logits;
    int is_bf16;
    const int32_t *draft_ids;
    const float *draft_probs, *u_acc, *u_samp, *temperature;
    const int32_t *draft_lens;
    int b0, b1, gmax, V;
    orc_outputs *out;
    int rc;
} orc_range_job;

static void *run_range(void *arg)
{
    orc_range_job *j = (orc_range_job *)arg;
    j->rc = verify_range(j->logits, j->is_bf16, j->draft_ids, j->draft_probs,
                         j->u_acc, j->u_samp, j->temperature, j->draft_lens,
                         j->b0, j->b1, j->gmax, j->V, j->out);
    return NULL;
}

/* orc_verify with the requests split into contiguous ranges over nthreads
 * POSIX threads.  The per-request arithmetic is verify_range's, unchanged;
 * results are identical to orc_verify's.  Returns 0, or -1 if a scratch
 * allocation or a thread creation fails. */
int orc_verify_mt(const void *logits, int is_bf16, const int32_t *draft_ids,
                  const float *draft_probs, const float *u_acc,
                  const float *u_samp, const float *temperature,
                  const int32_t *draft_lens, int B, int gmax, int V,
                  orc_outputs *out, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > B) nthreads = B > 0 ? B : 1;
    if (nthreads == 1)
        return orc_verify(logits, is_bf16, draft_ids, draft_probs, u_acc, u_samp,
                          temperature, draft_lens, B, gmax, V, out);
    orc_range_job *jobs = calloc((size_t)nthreads, sizeof *jobs);
    pthread_t *tid = calloc((size_t)nthreads, sizeof *tid);
    int rc = 0;
    if (!jobs || !tid) {
        free(jobs); free(tid);
        return -1;
    }
    int started = 0;
    for (int k = 0; k < nthreads; ++k) {
        orc_range_job *j = &jobs[k];
        j->logits = logits; j->is_bf16 = is_bf16; j->draft_ids = draft_ids;
        j->draft_probs = draft_probs; j->u_acc = u_acc; j->u_samp = u_samp;
        j->temperature = temperature; j->draft_lens = draft_lens;
        j->b0 = (int)((long long)B * k / nthreads);
        j->b1 = (int)((long long)B * (k + 1) / nthreads);
        j->gmax = gmax; j->V = V; j->out = out;
        if (pthread_create(&tid[k], NULL, run_range, j) != 0) {
            rc = -1;
            break;
        }
        ++started;
    }
    for (int k = 0; k < started; ++k) {
        pthread_join(tid[k], NULL);
        if (jobs[k].rc != 0) rc = -1;
    }
    free(jobs);
    free(tid);
    return rc;
}

/* Test support: the weights w_0 .. w_{V-1} that the draw at position k of
 * request b walks (draw_weights, with the request's row statistics
 * recomputed), so that a drawn token's own mass can be checked even where it
 * lies below the resolution of the prefix sums.  Returns 0, or -1 for T <= 0
 * (no draw). */
int orc_draw_weights(const void *logits, int is_bf16, const int32_t *draft_ids,
                     const float *draft_probs, const float *temperature, int b, int k,
                     int g, int gmax, int V, double *w)
{
    const double T = (double)temperature[b];
    if (!(T > 0.0)) return -1;
    const size_t off = ((size_t)b * ((size_t)gmax + 1) + (size_t)k) * (size_t)V;
    double mx, s;
    int argmax, fallback;
    orc_row_stats(logits, is_bf16, off, V, T, &mx, &s, &argmax);
    draw_weights(logits, is_bf16, draft_ids, draft_probs, b, k, g, gmax, V, off, mx, s,
                 argmax, T, w, &fallback);
    return 0;
}

/* Test support: the inclusive prefix sums C_0 .. C_{V-1} of those weights,
 * so that a drawn token j can be checked against its interval
 * [C_{j-1}, C_j) when u * C_{V-1} falls near an edge.  Returns 0, or -1 for
 * T <= 0 (no draw). */
int orc_draw_cdf(const void *logits, int is_bf16, const int32_t *draft_ids,
                 const float *draft_probs, const float *temperature, int b, int k, int g,
                 int gmax, int V, double *cdf)
{
    if (orc_draw_weights(logits, is_bf16, draft_ids, draft_probs, temperature, b, k, g, gmax,
                         V, cdf) != 0)
        return -1;
    double c = 0.0;
    for (int j = 0; j < V; ++j) {
        c += cdf[j];
        cdf[j] = c;
    }
    return 0;
}
