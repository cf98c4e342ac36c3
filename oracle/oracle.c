/*
 * oracle.c -- TEST INFRASTRUCTURE, NOT PRODUCT CODE.
 *
 * A plain, slow, fp64 CPU oracle for causal linear attention and its chunkwise,
 * normalised, feature-mapped and log-linear variants.  Only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg load it.  It includes nothing from
 * the CUDA library and the CUDA library never links, loads or calls it.
 *
 * Every routine is single-threaded, loops in the order its source describes, and
 * accumulates in double.  Callers pass float64 arrays holding the stored input
 * values exactly (bf16 and fp32 values are doubles), row-major, one (b,h) head:
 *   q, k : [L, d_in]   v : [L, dv]   feature-mapped rows : [L, D]
 *
 * Sources (page title, then section / equation / listing):
 *   [chunked]   "attention と線形の間" (sharin-2a1.pages.dev, parts/chunked.html):
 *               section 1 (ScoresFirst / StateFirst, the state-size table),
 *               section 2 (Chunked, CausalScoresFirst, CausalStateFirst, tril),
 *               section 3 (the Shape cost model and its two tables).
 *   [perf]      "Linear Attention / Performerの理論と実装" (disassemble-channel.com):
 *               ELU feature map, FAVOR+ positive random features, the normalised
 *               output equation, "再帰的な状態更新" (S_t, z_t recurrence).
 *   [loglinear] "論文紹介：Log Linear Attention" (docswell slides): Fenwick tree
 *               partition (slides 15-16, 20-21), level weights (slide 17), decoding
 *               update rule (slide 22).
 *   [perf] also gives the Retention form of the update, S_t = gamma S_{t-1} + phi(k_t)
 *               v_t^T with 0 < gamma < 1 (the section on the RNN without forgetting).
 *
 * Parity status: every routine here is pinned by CPU tests against printed values,
 * closed forms, library routines or brute force (tests/test_oracle_*.py).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* feature maps phi                                                           */
/* ------------------------------------------------------------------------- */

/* Identity: phi(x) = x (plain linear attention, [chunked] section 1). */
void orc_phi_identity(const double *x, long n, double *out)
{
    for (long i = 0; i < n; ++i) out[i] = x[i];
}

/* [perf] ELU feature map: phi(x) = elu(x) + 1, i.e. x + 1 where x >= 0, e^x below. */
void orc_phi_elu1(const double *x, long n, double *out)
{
    for (long i = 0; i < n; ++i) out[i] = (x[i] >= 0.0) ? x[i] + 1.0 : exp(x[i]);
}

/* [perf] FAVOR+ positive random features.  The inputs are first scaled by d^{-1/4}
 * (the Performer implementation scales both q and k), then
 *     phi(x) = exp(omega x - |x|^2 / 2) / sqrt(m),  omega: [m, d] (rows omega_l).
 * rows x: [rows, d] -> out: [rows, m]. */
void orc_phi_favor(const double *x, long rows, int d, const double *omega, int m, double *out)
{
    const double s = pow((double)d, -0.25);
    double *xs = (double *)malloc(sizeof(double) * (size_t)d);
    for (long r = 0; r < rows; ++r) {
        double nrm2 = 0.0;
        for (int j = 0; j < d; ++j) {
            xs[j] = x[r * d + j] * s;
            nrm2 += xs[j] * xs[j];
        }
        for (int l = 0; l < m; ++l) {
            double p = 0.0;
            for (int j = 0; j < d; ++j) p += omega[(long)l * d + j] * xs[j];
            out[r * m + l] = exp(p - 0.5 * nrm2) / sqrt((double)m);
        }
    }
    free(xs);
}

/* ------------------------------------------------------------------------- */
/* Fenwick level of a (query t, key s) pair                                   */
/* ------------------------------------------------------------------------- */

/* [loglinear] slides 16 and 20-21: for query t the past splits into buckets of sizes
 * 1, 1, 2, 4, ...; level 0 is t itself and level l >= 1 holds the keys s < t whose
 * highest bit differing from t is bit l-1.  So level = 0 if s == t, else
 * 1 + floor(log2(t XOR s)).  Worked case t = 7: {7}, {6}, {4,5}, {0,1,2,3}. */
int orc_fenwick_level(long t, long s)
{
    if (s == t) return 0;
    uint64_t x = (uint64_t)(t ^ s);
    int lg = 0;
    while (x >>= 1) ++lg;
    return 1 + lg;
}

static double dot(const double *a, const double *b, int n)
{
    double acc = 0.0;
    for (int i = 0; i < n; ++i) acc += a[i] * b[i];
    return acc;
}

/* ------------------------------------------------------------------------- */
/* Definition, scores first                                                    */
/* ------------------------------------------------------------------------- */

/* The plain definition, one output row at a time:
 *   num_t = sum_{s<=t} M[t,s] (phi(q_t) . phi(k_s)) v_s
 *   den_t = sum_{s<=t} M[t,s] (phi(q_t) . phi(k_s))
 *   out_t = normalize ? num_t / den_t : num_t
 * with M[t,s] = 1, or lam[t, level(t,s)] when lam is given (log-linear mask).
 * [chunked] CausalScoresFirst and tril (the diagonal is kept: s <= t);
 * [perf] normalised output equation y_t (sums over j = 1..t);
 * [loglinear] slide 17 (M built from per-level weights lambda_t^(l)).
 * causal = 0 gives the non-causal ScoresFirst order ([chunked] section 1), s over all L.
 * rows: the output rows to compute (NULL = all L, in order); out: [nrows, dv].
 * Returns 0, or -1 when a needed level is >= nl. */
int orc_scores_first(const double *fq, const double *fk, const double *v, long L, int D, int dv,
                     int causal, int normalize, const double *lam, int nl,
                     const long *rows, long nrows, double *out)
{
    double *num = (double *)malloc(sizeof(double) * (size_t)dv);
    long n = rows ? nrows : L;
    for (long r = 0; r < n; ++r) {
        long t = rows ? rows[r] : r;
        long smax = causal ? t : L - 1;
        double den = 0.0;
        for (int j = 0; j < dv; ++j) num[j] = 0.0;
        for (long s = 0; s <= smax; ++s) {
            double a = dot(fq + t * D, fk + s * D, D);
            if (lam) {
                int l = orc_fenwick_level(t, s);
                if (l >= nl) { free(num); return -1; }
                a *= lam[t * nl + l];
            }
            for (int j = 0; j < dv; ++j) num[j] += a * v[s * dv + j];
            den += a;
        }
        for (int j = 0; j < dv; ++j) out[r * dv + j] = normalize ? num[j] / den : num[j];
    }
    free(num);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Non-causal state first                                                      */
/* ------------------------------------------------------------------------- */

/* [chunked] section 1, StateFirst: out = phi(Q) (phi(K)^T V); the state phi(K)^T V is
 * D x dv whatever L is.  With normalize, [perf]'s non-causal normalised form
 * out_i = phi(q_i)^T S / phi(q_i)^T z with z = sum_j phi(k_j).
 * S_out (D x dv) and z_out (D) receive the state if non-NULL. */
void orc_state_first(const double *fq, const double *fk, const double *v, long L, int D, int dv,
                     int normalize, double *out, double *S_out, double *z_out)
{
    double *S = (double *)calloc((size_t)D * dv, sizeof(double));
    double *z = (double *)calloc((size_t)D, sizeof(double));
    for (long s = 0; s < L; ++s)
        for (int i = 0; i < D; ++i) {
            z[i] += fk[s * D + i];
            for (int j = 0; j < dv; ++j) S[i * dv + j] += fk[s * D + i] * v[s * dv + j];
        }
    for (long t = 0; t < L; ++t) {
        double den = dot(fq + t * D, z, D);
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < D; ++i) acc += fq[t * D + i] * S[i * dv + j];
            out[t * dv + j] = normalize ? acc / den : acc;
        }
    }
    if (S_out) memcpy(S_out, S, sizeof(double) * (size_t)D * dv);
    if (z_out) memcpy(z_out, z, sizeof(double) * (size_t)D);
    free(S);
    free(z);
}

/* ------------------------------------------------------------------------- */
/* Causal state recurrence (chunk size 1)                                      */
/* ------------------------------------------------------------------------- */

/* [chunked] CausalStateFirst and [perf] "再帰的な状態更新":
 *   S_t = S_{t-1} + phi(k_t) v_t^T,  z_t = z_{t-1} + phi(k_t),
 *   out_t = phi(q_t)^T S_t  (/ phi(q_t)^T z_t when normalize).
 * S0 (D x dv) / z0 (D): optional starting state (NULL = zero); S_out / z_out: optional
 * final state S_L, z_L. */
void orc_state_recurrence(const double *fq, const double *fk, const double *v, long L, int D,
                          int dv, int normalize, const double *S0, const double *z0,
                          double *out, double *S_out, double *z_out)
{
    double *S = (double *)calloc((size_t)D * dv, sizeof(double));
    double *z = (double *)calloc((size_t)D, sizeof(double));
    if (S0) memcpy(S, S0, sizeof(double) * (size_t)D * dv);
    if (z0) memcpy(z, z0, sizeof(double) * (size_t)D);
    for (long t = 0; t < L; ++t) {
        const double *kt = fk + t * D, *vt = v + t * dv, *qt = fq + t * D;
        for (int i = 0; i < D; ++i) {
            z[i] += kt[i];
            for (int j = 0; j < dv; ++j) S[i * dv + j] += kt[i] * vt[j];
        }
        double den = dot(qt, z, D);
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < D; ++i) acc += qt[i] * S[i * dv + j];
            out[t * dv + j] = normalize ? acc / den : acc;
        }
    }
    if (S_out) memcpy(S_out, S, sizeof(double) * (size_t)D * dv);
    if (z_out) memcpy(z_out, z, sizeof(double) * (size_t)D);
    free(S);
    free(z);
}

/* ------------------------------------------------------------------------- */
/* Chunked form (self-check of the chunk-size invariant only)                  */
/* ------------------------------------------------------------------------- */

/* [chunked] section 2, Chunked(q, k, v, c): chunk size c <= 0 becomes 1; the sequence
 * is cut into chunks of c rows (the last may be shorter).  Per chunk, the part of the
 * past before the chunk is read from the carried state (inter = q_c . state), the part
 * inside the chunk from the causally masked scores (tril(q_c k_c^T) v_c), the two are
 * added, and then the state takes the chunk's k_c^T v_c.  The normaliser rides along
 * the same way (z carried, masked score row sums inside the chunk).
 * unmasked_intra = 1 plants the mistake the page reports making first (no mask inside
 * the chunk); it exists only so a test can show that the checks catch it. */
void orc_chunked(const double *fq, const double *fk, const double *v, long L, int D, int dv,
                 long C, int normalize, int unmasked_intra, double *out)
{
    if (C <= 0) C = 1;
    double *S = (double *)calloc((size_t)D * dv, sizeof(double));
    double *z = (double *)calloc((size_t)D, sizeof(double));
    double *num = (double *)malloc(sizeof(double) * (size_t)dv);
    for (long start = 0; start < L; start += C) {
        long end = start + C < L ? start + C : L;
        for (long t = start; t < end; ++t) {
            const double *qt = fq + t * D;
            /* inter: from the carried state */
            double den = dot(qt, z, D);
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < D; ++i) acc += qt[i] * S[i * dv + j];
                num[j] = acc;
            }
            /* intra: masked scores inside the chunk */
            for (long s = start; s < end; ++s) {
                if (s > t && !unmasked_intra) continue;
                double a = dot(qt, fk + s * D, D);
                for (int j = 0; j < dv; ++j) num[j] += a * v[s * dv + j];
                den += a;
            }
            for (int j = 0; j < dv; ++j) out[t * dv + j] = normalize ? num[j] / den : num[j];
        }
        /* carry the chunk into the state */
        for (long s = start; s < end; ++s)
            for (int i = 0; i < D; ++i) {
                z[i] += fk[s * D + i];
                for (int j = 0; j < dv; ++j) S[i * dv + j] += fk[s * D + i] * v[s * dv + j];
            }
    }
    free(S);
    free(z);
    free(num);
}

/* ------------------------------------------------------------------------- */
/* Log-linear Fenwick recurrence (chunk size 1)                                 */
/* ------------------------------------------------------------------------- */

/* [loglinear] slides 18-22, read so that it produces the mask of orc_fenwick_level.
 * Level states S^(l), l = 1..nl-1, each hold sum phi(k_s) v_s^T over the keys of
 * bucket l of the current query (z^(l) likewise for the normaliser).  At step t:
 *   out_t = lam[t,0] (phi(q_t).phi(k_t)) v_t + sum_{l>=1} lam[t,l] phi(q_t)^T S^(l)
 * then, with r = number of trailing zero bits of t+1 (slide 22's lssb):
 *   level 0 takes the current token, levels 1..r are emptied into level r+1,
 *   S^(r+1) = phi(k_t) v_t^T + sum_{l=1..r} S^(l),  S^(1..r) = 0,
 *   higher levels are kept as they are.
 * Returns 0, or -1 if a level >= nl would be needed before the end of the sequence. */
int orc_loglinear_recurrence(const double *fq, const double *fk, const double *v, long L, int D,
                             int dv, const double *lam, int nl, int normalize, double *out)
{
    size_t sz = (size_t)D * dv;
    double *S = (double *)calloc(sz * (size_t)nl, sizeof(double));
    double *z = (double *)calloc((size_t)D * nl, sizeof(double));
    double *num = (double *)malloc(sizeof(double) * (size_t)dv);
    int rc = 0;
    for (long t = 0; t < L; ++t) {
        const double *qt = fq + t * D, *kt = fk + t * D, *vt = v + t * dv;
        const double *lt = lam + t * nl;
        double a0 = lt[0] * dot(qt, kt, D);
        double den = a0;
        for (int j = 0; j < dv; ++j) num[j] = a0 * vt[j];
        for (int l = 1; l < nl; ++l) {
            const double *Sl = S + sz * l;
            den += lt[l] * dot(qt, z + (size_t)D * l, D);
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < D; ++i) acc += qt[i] * Sl[i * dv + j];
                num[j] += lt[l] * acc;
            }
        }
        for (int j = 0; j < dv; ++j) out[t * dv + j] = normalize ? num[j] / den : num[j];
        if (t + 1 == L) break;
        int r = 0;
        while ((((uint64_t)(t + 1)) >> r & 1u) == 0) ++r;
        if (r + 1 >= nl) { rc = -1; break; }
        double *Sn = S + sz * (r + 1), *zn = z + (size_t)D * (r + 1);
        for (int i = 0; i < D; ++i) {
            zn[i] = kt[i];
            for (int j = 0; j < dv; ++j) Sn[i * dv + j] = kt[i] * vt[j];
        }
        for (int l = 1; l <= r; ++l) {
            double *Sl = S + sz * l, *zl = z + (size_t)D * l;
            for (size_t e = 0; e < sz; ++e) { Sn[e] += Sl[e]; Sl[e] = 0.0; }
            for (int i = 0; i < D; ++i) { zn[i] += zl[i]; zl[i] = 0.0; }
        }
    }
    free(S);
    free(z);
    free(num);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* Decay (Retention)                                                           */
/* ------------------------------------------------------------------------- */

/* [perf], the section on the RNN without forgetting: the Retention update
 *   S_t = gamma S_{t-1} + phi(k_t) v_t^T,   S_{-1} = 0,
 * read by y_t = phi(q_t)^T S_t.  The page gives the update of S only; the normaliser is
 * read the plainest way that keeps y_t a weighted mean of the values: z decays with the
 * same gamma, z_t = gamma z_{t-1} + phi(k_t), and y_t = phi(q_t)^T S_t / phi(q_t)^T z_t.
 * gamma = 1 is the plain recurrence. */
void orc_decay_recurrence(const double *fq, const double *fk, const double *v, long L, int D,
                          int dv, double gamma, int normalize, double *out)
{
    double *S = (double *)calloc((size_t)D * dv, sizeof(double));
    double *z = (double *)calloc((size_t)D, sizeof(double));
    for (long t = 0; t < L; ++t) {
        const double *kt = fk + t * D, *vt = v + t * dv, *qt = fq + t * D;
        for (int i = 0; i < D; ++i) {
            z[i] = gamma * z[i] + kt[i];
            for (int j = 0; j < dv; ++j) S[i * dv + j] = gamma * S[i * dv + j] + kt[i] * vt[j];
        }
        double den = dot(qt, z, D);
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int i = 0; i < D; ++i) acc += qt[i] * S[i * dv + j];
            out[t * dv + j] = normalize ? acc / den : acc;
        }
    }
    free(S);
    free(z);
}

/* The same output written out as a weighted sum over the past (unrolling the update):
 *   num_t = sum_{s<=t} gamma^(t-s) (phi(q_t) . phi(k_s)) v_s,
 *   den_t = sum_{s<=t} gamma^(t-s) (phi(q_t) . phi(k_s)),
 * i.e. the causal mask of [chunked] section 2 with entries gamma^(t-s) instead of 1.
 * rows: the output rows to compute (NULL = all L, in order); out: [nrows, dv]. */
void orc_decay_scores_first(const double *fq, const double *fk, const double *v, long L, int D,
                            int dv, double gamma, int normalize, const long *rows, long nrows,
                            double *out)
{
    double *num = (double *)malloc(sizeof(double) * (size_t)dv);
    long n = rows ? nrows : L;
    for (long r = 0; r < n; ++r) {
        long t = rows ? rows[r] : r;
        double den = 0.0;
        for (int j = 0; j < dv; ++j) num[j] = 0.0;
        for (long s = 0; s <= t; ++s) {
            double a = pow(gamma, (double)(t - s)) * dot(fq + t * D, fk + s * D, D);
            for (int j = 0; j < dv; ++j) num[j] += a * v[s * dv + j];
            den += a;
        }
        for (int j = 0; j < dv; ++j) out[r * dv + j] = normalize ? num[j] / den : num[j];
    }
    free(num);
}

/* ------------------------------------------------------------------------- */
/* Backward pass (gradients of the causal output)                             */
/* ------------------------------------------------------------------------- */

/* The pages give no formulas for the backward pass; this is the chain rule applied to the
 * plain definition used by orc_scores_first / orc_decay_scores_first, with M[t,s] = 1 or
 * gamma^(t-s) for s <= t and a_ts = phi(q_t) . phi(k_s):
 *   num_t = sum_{s<=t} M a_ts v_s,  den_t = sum_{s<=t} M a_ts,
 *   out_t = num_t (unnormalised) or num_t / den_t.
 * Given dout (the gradient of a scalar loss with respect to out), the loss depends on a_ts
 * through num_t (and den_t), so
 *   unnormalised: g_ts = M (dout_t . v_s)
 *   normalised:   g_ts = M (dout_t . v_s - dout_t . out_t) / den_t
 *   dv_s     = sum_{t>=s} M a_ts dout_t   (divided by den_t when normalised)
 *   dphiq_t  = sum_{s<=t} g_ts phi(k_s),   dphik_s = sum_{t>=s} g_ts phi(q_t).
 * gamma <= 0 means no decay (M = 1).  Inputs are feature-mapped rows; out: [L, D], [L, D],
 * [L, dv]. */
void orc_backward_features(const double *fq, const double *fk, const double *v, const double *dout,
                           long L, int D, int dv, int normalize, double gamma, double *dfq,
                           double *dfk, double *dvo)
{
    double *o = (double *)malloc(sizeof(double) * (size_t)dv);
    memset(dfq, 0, sizeof(double) * (size_t)L * D);
    memset(dfk, 0, sizeof(double) * (size_t)L * D);
    memset(dvo, 0, sizeof(double) * (size_t)L * dv);
    for (long t = 0; t < L; ++t) {
        const double *qt = fq + t * D, *dt = dout + t * dv;
        /* the forward row: num_t, den_t, out_t */
        double den = 0.0;
        for (int j = 0; j < dv; ++j) o[j] = 0.0;
        for (long s = 0; s <= t; ++s) {
            double m = gamma > 0.0 ? pow(gamma, (double)(t - s)) : 1.0;
            double a = m * dot(qt, fk + s * D, D);
            for (int j = 0; j < dv; ++j) o[j] += a * v[s * dv + j];
            den += a;
        }
        double scale = 1.0, dto = 0.0;
        if (normalize) {
            for (int j = 0; j < dv; ++j) o[j] /= den;
            scale = 1.0 / den;
            dto = dot(dt, o, dv);
        }
        for (long s = 0; s <= t; ++s) {
            double m = gamma > 0.0 ? pow(gamma, (double)(t - s)) : 1.0;
            double a = m * dot(qt, fk + s * D, D);
            double g = m * (dot(dt, v + s * dv, dv) - dto) * scale;
            for (int i = 0; i < D; ++i) {
                dfq[t * D + i] += g * fk[s * D + i];
                dfk[s * D + i] += g * qt[i];
            }
            for (int j = 0; j < dv; ++j) dvo[s * dv + j] += a * scale * dt[j];
        }
    }
    free(o);
}

/* The same chain rule under the log-linear mask of [loglinear] slide 17:
 * M_ts = lambda_t^(l(t,s)), l from orc_fenwick_level, lam [L, nl] per query row t.
 * With a_ts = phi(q_t).phi(k_s) and the forward out_t = sum_{s<=t} M_ts a_ts v_s (/ den_t,
 * den_t = sum_{s<=t} M_ts a_ts):
 *   G_ts = M_ts (dout_t . v_s - dout_t . out_t) / den_t      (normalised; else M_ts dout_t . v_s)
 *   dphi(q)_t = sum_{s<=t} G_ts phi(k_s),  dphi(k)_s = sum_{t>=s} G_ts phi(q_t),
 *   dv_s = sum_{t>=s} M_ts a_ts dout_t (/ den_t).
 * The level weights are data here (their own gradient is not formed).  Returns -1 when nl
 * does not cover the levels of L rows, else 0. */
int orc_backward_features_ll(const double *fq, const double *fk, const double *v,
                             const double *dout, const double *lam, int nl, long L, int D,
                             int dv, int normalize, double *dfq, double *dfk, double *dvo)
{
    if (L > 1 && orc_fenwick_level(L - 1, 0) >= nl) return -1;
    double *o = (double *)malloc(sizeof(double) * (size_t)dv);
    memset(dfq, 0, sizeof(double) * (size_t)L * D);
    memset(dfk, 0, sizeof(double) * (size_t)L * D);
    memset(dvo, 0, sizeof(double) * (size_t)L * dv);
    for (long t = 0; t < L; ++t) {
        const double *qt = fq + t * D, *dt = dout + t * dv, *lt = lam + t * nl;
        double den = 0.0;
        for (int j = 0; j < dv; ++j) o[j] = 0.0;
        for (long s = 0; s <= t; ++s) {
            double a = lt[orc_fenwick_level(t, s)] * dot(qt, fk + s * D, D);
            for (int j = 0; j < dv; ++j) o[j] += a * v[s * dv + j];
            den += a;
        }
        double scale = 1.0, dto = 0.0;
        if (normalize) {
            for (int j = 0; j < dv; ++j) o[j] /= den;
            scale = 1.0 / den;
            dto = dot(dt, o, dv);
        }
        for (long s = 0; s <= t; ++s) {
            double m = lt[orc_fenwick_level(t, s)];
            double a = m * dot(qt, fk + s * D, D);
            double g = m * (dot(dt, v + s * dv, dv) - dto) * scale;
            for (int i = 0; i < D; ++i) {
                dfq[t * D + i] += g * fk[s * D + i];
                dfk[s * D + i] += g * qt[i];
            }
            for (int j = 0; j < dv; ++j) dvo[s * dv + j] += a * scale * dt[j];
        }
    }
    free(o);
    return 0;
}

/* Chain rule through the feature map: dx from dphi for rows x [rows, d].
 *   identity: dx = dphi;
 *   elu+1:    dx = dphi * (x >= 0 ? 1 : e^x)   ([perf] ELU feature map);
 *   FAVOR+:   with s = d^{-1/4}, xs = s x and phi_l = exp(omega_l . xs - |xs|^2 / 2) / sqrt(m),
 *             d phi_l / d x_i = s phi_l (omega_li - xs_i), so
 *             dx_i = s sum_l dphi_l phi_l (omega_li - xs_i).
 * kind: 0 identity, 1 elu+1, 2 FAVOR+ (omega [m, d], dphi [rows, m]). */
void orc_phi_grad(const double *x, long rows, int d, int kind, const double *omega, int m,
                  const double *dphi, double *dx)
{
    if (kind == 0) {
        for (long e = 0; e < rows * d; ++e) dx[e] = dphi[e];
        return;
    }
    if (kind == 1) {
        for (long e = 0; e < rows * d; ++e) dx[e] = dphi[e] * (x[e] >= 0.0 ? 1.0 : exp(x[e]));
        return;
    }
    const double s = pow((double)d, -0.25);
    double *xs = (double *)malloc(sizeof(double) * (size_t)d);
    double *ph = (double *)malloc(sizeof(double) * (size_t)m);
    for (long r = 0; r < rows; ++r) {
        double nrm2 = 0.0;
        for (int j = 0; j < d; ++j) {
            xs[j] = x[r * d + j] * s;
            nrm2 += xs[j] * xs[j];
        }
        for (int l = 0; l < m; ++l) {
            double p = 0.0;
            for (int j = 0; j < d; ++j) p += omega[(long)l * d + j] * xs[j];
            ph[l] = exp(p - 0.5 * nrm2) / sqrt((double)m);
        }
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int l = 0; l < m; ++l) acc += dphi[r * m + l] * ph[l] * (omega[(long)l * d + i] - xs[i]);
            dx[r * d + i] = s * acc;
        }
    }
    free(xs);
    free(ph);
}

/* ------------------------------------------------------------------------- */
/* Cost model                                                                  */
/* ------------------------------------------------------------------------- */

/* [chunked] section 3, Shape{L, D, C}: multiply-add counts.
 *   state: writing and reading the d x d state, C d^2 each per chunk, L/C chunks
 *          -> 2 L d^2, independent of C;
 *   score: making the scores and mixing the values, C^2 d each per chunk
 *          -> 2 L C d, proportional to C;
 *   intra memory: the C x C score block. */
long long orc_state_flops(long long L, long long D, long long C) { (void)C; return 2 * L * D * D; }
long long orc_score_flops(long long L, long long D, long long C) { return 2 * L * C * D; }
long long orc_total_flops(long long L, long long D, long long C)
{
    return orc_state_flops(L, D, C) + orc_score_flops(L, D, C);
}
long long orc_intra_memory(long long C) { return C * C; }
int orc_is_full_attention(long long L, long long C) { return C >= L; }
int orc_is_linear(long long C) { return C == 1; }

/* [chunked] section 1 table: the d x d state against a KV cache holding k and v rows. */
long long orc_state_elems(long long L, long long d) { (void)L; return d * d; }
long long orc_kv_cache_elems(long long L, long long d) { return 2 * L * d; }
