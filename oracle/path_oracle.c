/*
 * PaTH attention oracle: plain, slow, fp64 CPU code.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load or call this file's library.  The
 * product path (libpath_attn) shares no code with it and never calls it.
 *
 * What it computes (PaTH Attention summary, gist.science/ko/paper/2505.16381,
 * section "2. 방법론 / 핵심 메커니즘", attention-logit equation):
 *
 *     logit(i, j) = scale * k_j^T (H_{j+1} H_{j+2} ... H_i) q_i      (j <= i)
 *     H_s         = I - beta_s w_s w_s^T
 *
 * followed by a causal softmax over j <= i and out_i = sum_j p_ij v_j.
 * The product order H_{j+1} ... H_i (so H_i acts on q_i first) and the empty
 * product for j == i (the identity) are the readings this build takes where
 * the equation writes an order-free product.
 *
 * PaTH-FoX (same page, section "확장: PaTH-FoX"): the forgetting-transformer
 * gate adds a data-dependent additive bias sum_{s=j+1}^{i} log f_s to the
 * logit.  The bias is not multiplied by `scale`.
 *
 * Inference (same page, section "3. 효율적인 학습 및 추론", bullet "추론"):
 * at step t every cached key is updated in place with the current
 * transition, k_j <- H_t k_j (j < t), and the new key k_t is appended
 * untransformed; attention then reads the cache like ordinary attention.
 *
 * Backward (path_oracle_prefill_bwd): reverse-mode differentiation of the
 * same equation, one transition at a time (see row_backward); the pages give
 * no gradient formulas of their own.
 *
 * Everything below applies one reflection at a time to a vector.  It never
 * forms the UT / compact-WY representation and never blocks, fuses or
 * reorders the steps of the definition.  lse is the natural log of the sum of
 * exp(logit) over the causal row (logits include scale and the FoX bias).
 *
 * Layouts: q, k, v, w are [BH][L][d] row-major doubles; beta and log_f are
 * [BH][L].  All entry points return 0 on success and a negative value on a
 * bad argument.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double dot(const double *a, const double *b, int64_t d)
{
    double s = 0.0;
    for (int64_t m = 0; m < d; ++m)
        s += a[m] * b[m];
    return s;
}

/* u <- H u with H = I - beta w w^T (one Householder-like transition). */
static void apply_transition(double *u, const double *w, double beta, int64_t d)
{
    double c = beta * dot(w, u, d);
    for (int64_t m = 0; m < d; ++m)
        u[m] -= c * w[m];
}

/*
 * Logits of query row i of one head, for keys j = 0..i.
 * Walk j from i down to 0.  At key j the running vector equals
 * (H_{j+1} ... H_i) q_i, so the logit is scale * k_j . u; then u moves past
 * position j (u <- H_j u) and the FoX bias picks up log f_j.  If B is not
 * NULL, row j of B receives the running vector seen by key j.
 */
static void row_logits(int64_t i, int64_t d, double scale, const double *q_i,
                       const double *k, const double *w, const double *beta,
                       const double *log_f, double *u, double *logit, double *B)
{
    memcpy(u, q_i, (size_t)d * sizeof(double));
    double bias = 0.0;
    for (int64_t j = i; j >= 0; --j) {
        if (B)
            memcpy(B + j * d, u, (size_t)d * sizeof(double));
        logit[j] = scale * dot(k + j * d, u, d) + bias;
        apply_transition(u, w + j * d, beta[j], d);
        if (log_f)
            bias += log_f[j];
    }
}

/* Explicit softmax of logit[0..n-1] applied to the value rows v[0..n-1]. */
static void softmax_rows(int64_t n, int64_t d, const double *logit,
                         const double *v, double *out, double *lse)
{
    double mx = -INFINITY;
    for (int64_t j = 0; j < n; ++j)
        if (logit[j] > mx)
            mx = logit[j];
    double sum = 0.0;
    for (int64_t m = 0; m < d; ++m)
        out[m] = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double p = exp(logit[j] - mx);
        sum += p;
        for (int64_t m = 0; m < d; ++m)
            out[m] += p * v[j * d + m];
    }
    for (int64_t m = 0; m < d; ++m)
        out[m] /= sum;
    if (lse)
        *lse = mx + log(sum);
}

/*
 * Prefill forward.  rows == NULL computes every query row (nrows must be L);
 * otherwise only the listed query positions.  out is [BH][nrows][d], lse is
 * [BH][nrows] (lse may be NULL).  log_f == NULL is plain PaTH.
 */
int path_oracle_prefill(int64_t BH, int64_t L, int64_t d, double scale,
                        const double *q, const double *k, const double *v,
                        const double *w, const double *beta, const double *log_f,
                        int64_t nrows, const int64_t *rows, double *out,
                        double *lse, int nthreads)
{
    if (BH < 0 || L < 0 || d <= 0 || nrows < 0 || (!rows && nrows != L))
        return -1;
    if (rows)
        for (int64_t r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= L)
                return -2;
    int64_t total = BH * nrows;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int err = 0;
#pragma omp parallel
    {
        double *u = (double *)malloc((size_t)d * sizeof(double));
        double *logit = (double *)malloc((size_t)(L > 0 ? L : 1) * sizeof(double));
        if (!u || !logit) {
#pragma omp atomic write
            err = -3;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t t = 0; t < total; ++t) {
                int64_t bh = t / nrows, r = t % nrows;
                int64_t i = rows ? rows[r] : r;
                const double *qh = q + bh * L * d, *kh = k + bh * L * d;
                const double *vh = v + bh * L * d, *wh = w + bh * L * d;
                const double *bh_beta = beta + bh * L;
                const double *bh_f = log_f ? log_f + bh * L : NULL;
                row_logits(i, d, scale, qh + i * d, kh, wh, bh_beta, bh_f, u, logit, NULL);
                softmax_rows(i + 1, d, logit, vh, out + t * d, lse ? lse + t : NULL);
            }
        }
        free(u);
        free(logit);
    }
    return err;
}

/*
 * Full logit matrix of one head (tiny inputs only): logits is [L][L] with
 * logits[i][j] for j <= i and -inf above the diagonal.
 */
int path_oracle_logits(int64_t L, int64_t d, double scale, const double *q,
                       const double *k, const double *w, const double *beta,
                       const double *log_f, double *logits)
{
    if (L < 0 || d <= 0)
        return -1;
    double *u = (double *)malloc((size_t)d * sizeof(double));
    if (!u)
        return -3;
    for (int64_t i = 0; i < L; ++i) {
        double *row = logits + i * L;
        row_logits(i, d, scale, q + i * d, k, w, beta, log_f, u, row, NULL);
        for (int64_t j = i + 1; j < L; ++j)
            row[j] = -INFINITY;
    }
    free(u);
    return 0;
}

/*
 * One head of a decode step (inference bullet of section 3): cached keys
 * j < t take the new token's transition in place, k_j <- H_t k_j; (k_t, v_t)
 * are written at slot t; then softmax attention of q_t over slots 0..t.  With
 * a forget-gate history lf (PaTH-FoX, section 2), log f_t is stored at slot t
 * and the logit of key j gains sum_{s=j+1}^{t} log f_s, accumulated from the
 * right one term per key; the new token's own logit gains nothing.
 */
static int decode_head(int64_t cap, int64_t t, int64_t d, double scale, double *kc,
                       double *vc, double *lf, const double *q_t, const double *k_t,
                       const double *v_t, const double *w_t, double beta_t, double log_f_t,
                       double *out)
{
    (void)cap;
    for (int64_t j = 0; j < t; ++j)
        apply_transition(kc + j * d, w_t, beta_t, d);
    memcpy(kc + t * d, k_t, (size_t)d * sizeof(double));
    memcpy(vc + t * d, v_t, (size_t)d * sizeof(double));
    if (lf)
        lf[t] = log_f_t;
    double *logit = (double *)malloc((size_t)(t + 1) * sizeof(double));
    if (!logit)
        return -3;
    double bias = 0.0;  /* sum_{s=j+1}^{t} log f_s */
    for (int64_t j = t; j >= 0; --j) {
        logit[j] = scale * dot(kc + j * d, q_t, d) + bias;
        if (lf)
            bias += lf[j];
    }
    softmax_rows(t + 1, d, logit, vc, out, NULL);
    free(logit);
    return 0;
}

/*
 * One PaTH decode step for BH independent heads (see decode_head).
 * k_cache, v_cache: [BH][cap][d], modified in place.
 */
int path_oracle_decode_step(int64_t BH, int64_t cap, int64_t t, int64_t d,
                            double scale, double *k_cache, double *v_cache,
                            const double *q_t, const double *k_t,
                            const double *v_t, const double *w_t,
                            const double *beta_t, double *out, int nthreads)
{
    if (BH < 0 || d <= 0 || t < 0 || t >= cap)
        return -1;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < BH; ++bh) {
        int e = decode_head(cap, t, d, scale, k_cache + bh * cap * d, v_cache + bh * cap * d,
                            NULL, q_t + bh * d, k_t + bh * d, v_t + bh * d, w_t + bh * d,
                            beta_t[bh], 0.0, out + bh * d);
        if (e) {
#pragma omp atomic write
            err = e;
        }
    }
    return err;
}

/*
 * One PaTH-FoX decode step (see decode_head).  lf_hist: [BH][cap], log f of
 * tokens 0..t-1 on entry; log_f_t is stored at slot t.
 */
int path_oracle_decode_step_fox(int64_t BH, int64_t cap, int64_t t, int64_t d,
                                double scale, double *k_cache, double *v_cache,
                                double *lf_hist, const double *q_t, const double *k_t,
                                const double *v_t, const double *w_t,
                                const double *beta_t, const double *log_f_t, double *out,
                                int nthreads)
{
    if (BH < 0 || d <= 0 || t < 0 || t >= cap || !lf_hist || !log_f_t)
        return -1;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < BH; ++bh) {
        int e = decode_head(cap, t, d, scale, k_cache + bh * cap * d, v_cache + bh * cap * d,
                            lf_hist + bh * cap, q_t + bh * d, k_t + bh * d, v_t + bh * d,
                            w_t + bh * d, beta_t[bh], log_f_t[bh], out + bh * d);
        if (e) {
#pragma omp atomic write
            err = e;
        }
    }
    return err;
}

/*
 * Key cache as left by L0 decode steps over tokens 0..L0-1:
 *     kc_j = H_{L0-1} H_{L0-2} ... H_{j+1} k_j.
 * Built with an explicit d x d matrix M swept from the right: M starts as I,
 * kc_j = M k_j, then M <- M H_j.  k, w are [BH][L0][d], beta [BH][L0];
 * k_cache is [BH][cap][d] (rows 0..L0-1 written).
 */
int path_oracle_build_kcache(int64_t BH, int64_t L0, int64_t cap, int64_t d,
                             const double *k, const double *w,
                             const double *beta, double *k_cache, int nthreads)
{
    if (BH < 0 || L0 < 0 || L0 > cap || d <= 0)
        return -1;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < BH; ++bh) {
        double *M = (double *)calloc((size_t)(d * d), sizeof(double));
        double *Mw = (double *)malloc((size_t)d * sizeof(double));
        if (!M || !Mw) {
#pragma omp atomic write
            err = -3;
            free(M);
            free(Mw);
            continue;
        }
        for (int64_t m = 0; m < d; ++m)
            M[m * d + m] = 1.0;
        const double *kh = k + bh * L0 * d, *wh = w + bh * L0 * d;
        const double *bb = beta + bh * L0;
        double *kc = k_cache + bh * cap * d;
        for (int64_t j = L0 - 1; j >= 0; --j) {
            for (int64_t r = 0; r < d; ++r)
                kc[j * d + r] = dot(M + r * d, kh + j * d, d);
            /* M <- M - beta_j (M w_j) w_j^T */
            for (int64_t r = 0; r < d; ++r)
                Mw[r] = dot(M + r * d, wh + j * d, d);
            for (int64_t r = 0; r < d; ++r)
                for (int64_t c = 0; c < d; ++c)
                    M[r * d + c] -= bb[j] * Mw[r] * wh[j * d + c];
        }
        free(M);
        free(Mw);
    }
    return err;
}

/*
 * Boundary-adjusted rows of one head for a chunk length C (section 3,
 * FlashAttention-style algorithm, first bullet: per block, precompute
 * boundary-adjusted query and key rows).  Chunk c covers positions
 * [cC, min(cC+C, L)).  For i in chunk c with first position s0 and last
 * position e:
 *     qb_i = H_{s0} ... H_i q_i          (apply H_i first, H_{s0} last)
 *     kb_j = H_e ... H_{j+1} k_j          (apply H_{j+1} first, H_e last)
 * so that for j in an earlier chunk than i, logit(i, j) equals
 * scale * kb_j^T (whole-chunk products in between) qb_i.
 */
int path_oracle_boundary_rows(int64_t L, int64_t d, int64_t C, const double *q,
                              const double *k, const double *w,
                              const double *beta, double *qb, double *kb)
{
    if (L < 0 || d <= 0 || C <= 0)
        return -1;
    for (int64_t i = 0; i < L; ++i) {
        int64_t s0 = (i / C) * C;
        int64_t e = s0 + C - 1 < L - 1 ? s0 + C - 1 : L - 1;
        double *u = qb + i * d;
        memcpy(u, q + i * d, (size_t)d * sizeof(double));
        for (int64_t s = i; s >= s0; --s)
            apply_transition(u, w + s * d, beta[s], d);
        double *x = kb + i * d;
        memcpy(x, k + i * d, (size_t)d * sizeof(double));
        for (int64_t s = i + 1; s <= e; ++s)
            apply_transition(x, w + s * d, beta[s], d);
    }
    return 0;
}

/*
 * Gradients of one query row i of one head, added into the head's
 * accumulators (dk, dv, dw, dbeta, dlog_f) and written to dq_i.
 *
 * The backward pass is not spelled out on the pages (the PaTH lecture notes,
 * open questions, only remark that it costs more than the forward); this is
 * reverse-mode differentiation of the attention-logit equation, one
 * transition at a time.  With b_s = H_{s+1} ... H_i q_i (the running vector of
 * row_logits at key s) and, for j < s, a_{j,s} = H_{s-1} ... H_{j+1} k_j, the
 * logit is scale * a_{j,s}^T H_s b_s, so
 *     dL/dH_s = scale * g_s b_s^T,  g_s = sum_{j<s} dlogit_j a_{j,s},
 * and g obeys g_{s+1} = H_s g_s + dlogit_s k_s (g_0 = 0).  For
 * H_s = I - beta_s w_s w_s^T that gives
 *     dbeta_s = -w_s^T (dL/dH_s) w_s,
 *     dw_s    = -beta_s (dL/dH_s + dL/dH_s^T) w_s,
 * and dq_i = scale * g_{i+1}, dk_j = scale * dlogit_j b_j.  The softmax part
 * is the usual one: dlogit_j = p_j (dout_i . v_j - dout_i . out_i + dlse_i).
 * The FoX bias of logit j is sum_{s=j+1}^{i} log f_s, so
 * dlog_f_s = sum_{j<s} dlogit_j.
 */
static void row_backward(int64_t i, int64_t d, double scale, const double *q_i,
                         const double *k, const double *v, const double *w,
                         const double *beta, const double *log_f, const double *dout_i,
                         double dlse_i, double *B, double *logit, double *dl, double *g,
                         double *dq_i, double *dk, double *dv, double *dw, double *dbeta,
                         double *dlog_f)
{
    /* the logits, and b_j for j = i..0 */
    row_logits(i, d, scale, q_i, k, w, beta, log_f, g, logit, B);
    /* softmax and its gradient */
    double mx = -INFINITY;
    for (int64_t j = 0; j <= i; ++j)
        if (logit[j] > mx)
            mx = logit[j];
    double sum = 0.0;
    for (int64_t j = 0; j <= i; ++j)
        sum += exp(logit[j] - mx);
    const double lse = mx + log(sum);
    double D = 0.0;
    for (int64_t j = 0; j <= i; ++j) {
        double p = exp(logit[j] - lse);
        double dp = dot(dout_i, v + j * d, d);
        dl[j] = p * dp;   /* p_j (dout . v_j), finished below */
        D += p * dp;
        for (int64_t m = 0; m < d; ++m)
            dv[j * d + m] += p * dout_i[m];
    }
    for (int64_t j = 0; j <= i; ++j) {
        double p = exp(logit[j] - lse);
        dl[j] -= p * (D - dlse_i);
        for (int64_t m = 0; m < d; ++m)
            dk[j * d + m] += scale * dl[j] * B[j * d + m];
    }
    /* left-to-right sweep over the transitions */
    for (int64_t m = 0; m < d; ++m)
        g[m] = 0.0;
    double cum = 0.0;  /* sum_{j<s} dlogit_j */
    for (int64_t s = 0; s <= i; ++s) {
        if (s > 0) {
            const double *ws = w + s * d, *bs = B + s * d;
            double alpha = dot(ws, g, d), gamma = dot(ws, bs, d);
            dbeta[s] -= scale * alpha * gamma;
            for (int64_t m = 0; m < d; ++m)
                dw[s * d + m] -= beta[s] * scale * (gamma * g[m] + alpha * bs[m]);
        }
        if (log_f)
            dlog_f[s] += cum;
        cum += dl[s];
        apply_transition(g, w + s * d, beta[s], d);
        for (int64_t m = 0; m < d; ++m)
            g[m] += dl[s] * k[s * d + m];
    }
    for (int64_t m = 0; m < d; ++m)
        dq_i[m] = scale * g[m];
}

/*
 * Prefill backward: gradients of sum(dout * out) + sum(dlse * lse) with
 * respect to q, k, v, w, beta and (PaTH-FoX) log_f.  Same layouts as
 * path_oracle_prefill; dlse may be NULL (zero); dlog_f is written only when
 * log_f is given.  Rows of one head run in parallel, each thread with its own
 * accumulators, summed at the end of the head.
 */
int path_oracle_prefill_bwd(int64_t BH, int64_t L, int64_t d, double scale,
                            const double *q, const double *k, const double *v,
                            const double *w, const double *beta, const double *log_f,
                            const double *dout, const double *dlse, double *dq,
                            double *dk, double *dv, double *dw, double *dbeta,
                            double *dlog_f, int nthreads)
{
    if (BH < 0 || L < 0 || d <= 0)
        return -1;
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    const size_t Ld = (size_t)L * d;
    memset(dk, 0, BH * Ld * sizeof(double));
    memset(dv, 0, BH * Ld * sizeof(double));
    memset(dw, 0, BH * Ld * sizeof(double));
    memset(dbeta, 0, (size_t)(BH * L) * sizeof(double));
    if (log_f)
        memset(dlog_f, 0, (size_t)(BH * L) * sizeof(double));
    int err = 0;
    for (int64_t bh = 0; bh < BH; ++bh) {
        const double *qh = q + bh * Ld, *kh = k + bh * Ld, *vh = v + bh * Ld;
        const double *wh = w + bh * Ld, *bb = beta + bh * L, *oh = dout + bh * Ld;
        const double *fh = log_f ? log_f + bh * L : NULL;
#pragma omp parallel
        {
            size_t n1 = L > 0 ? (size_t)L : 1;
            double *B = (double *)malloc(n1 * d * sizeof(double));
            double *logit = (double *)malloc(n1 * sizeof(double));
            double *dl = (double *)malloc(n1 * sizeof(double));
            double *g = (double *)malloc((size_t)d * sizeof(double));
            double *acc = (double *)calloc(3 * n1 * d + 2 * n1, sizeof(double));
            if (!B || !logit || !dl || !g || !acc) {
#pragma omp atomic write
                err = -3;
            } else {
                double *adk = acc, *adv = acc + n1 * d, *adw = acc + 2 * n1 * d;
                double *adb = acc + 3 * n1 * d, *adf = adb + n1;
#pragma omp for schedule(dynamic, 4)
                for (int64_t i = 0; i < L; ++i)
                    row_backward(i, d, scale, qh + i * d, kh, vh, wh, bb, fh, oh + i * d,
                                 dlse ? dlse[bh * L + i] : 0.0, B, logit, dl, g,
                                 dq + bh * Ld + i * d, adk, adv, adw, adb, adf);
#pragma omp critical
                {
                    for (size_t e = 0; e < Ld; ++e) {
                        dk[bh * Ld + e] += adk[e];
                        dv[bh * Ld + e] += adv[e];
                        dw[bh * Ld + e] += adw[e];
                    }
                    for (int64_t s = 0; s < L; ++s) {
                        dbeta[bh * L + s] += adb[s];
                        if (log_f)
                            dlog_f[bh * L + s] += adf[s];
                    }
                }
            }
            free(B);
            free(logit);
            free(dl);
            free(g);
            free(acc);
        }
    }
    return err;
}
