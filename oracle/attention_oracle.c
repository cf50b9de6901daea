/*
 * attention_oracle.c -- plain fp64 CPU oracle for the attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the tests, the smoke check and the bench's CPU-baseline leg
 * do.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (for every head (b,h) and query row i, keys j):
 *
 *   s_j   = scale * <q_i, k_j>                       for the allowed keys j
 *   m     = max_j s_j
 *   l     = sum_j exp(s_j - m)
 *   o_i   = (sum_j exp(s_j - m) * v_j) / l
 *   lse_i = m + ln(l)
 *
 * The allowed keys are all j (non-causal) or j <= i (causal).
 *
 * Sources (page title, section):
 *  - "FlashAttention-2를 CuTe로 밑바닥부터 구현하며 겪은 GPU 커널 지옥기",
 *    section "커널 구조는 단순한데, 디테일이 지옥임": the attention formula
 *    (scores = QK^T / sqrt(d_h), row softmax, times V).
 *  - "3.6 어텐션 I — 메모리 문제·FlashAttention 원리", section 3.6.4: the
 *    max-shifted (stable) softmax and the online recurrence in the state
 *    (m, l, O) with alpha = exp(m_old - m_new), normalised once at the end.
 *  - same page, section 3.6.6: causal masking skips keys j > i.
 *  - same page, section 3.6.7: the saved row statistic L = m + log(l),
 *    read here as the natural logarithm over the scaled scores.
 *
 * Two entry families:
 *  - oracle_attention_rows / oracle_attention_fwd: the plain definition,
 *    computed two-pass per row (max first, then the sums).  Because the
 *    tiled online method reaches this same result exactly (section 3.6.4
 *    states that it is exact, not an approximation), this plain definition
 *    is what the GPU path is compared against.
 *  - oracle_online_row: the online recurrence of section 3.6.4, applied to
 *    one row of scores split into caller-chosen blocks processed in a
 *    caller-chosen order.  It records the state after every block so the
 *    tests can check the page's hand-worked intermediate values
 *    (section 3.6.5) and the block-order independence the page claims.
 *
 *  - oracle_attention_decode: the plain definition for Nq queries against
 *    Nk >= Nq keys (decoding; causal aligns the queries with the end).
 *  - oracle_attention_bwd: the gradients of the plain definition (softmax
 *    Jacobian), for the backward pass; oracle_attention_bwd_rows: dq of
 *    listed query rows only (O(N d) each, for full-size samples).
 *
 * Every function here is pinned by tests under tests/ (worked example,
 * exercise, closed forms, invariants, finite differences, source mutations).
 *
 * Arithmetic: IEEE fp64, evaluated in source order (built without
 * fast-math, so the compiler does not reassociate the sums).
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_ENOMEM 2

/* Scores of query row i against the first n_keys keys of one head.
 * q, k point at the head's [N, d] blocks (row-major). */
static void scores_row(const double *q, const double *k, long i, long n_keys,
                       long d, double scale, double *s)
{
    for (long j = 0; j < n_keys; ++j) {
        double dot = 0.0;
        for (long c = 0; c < d; ++c)
            dot += q[i * d + c] * k[j * d + c];
        s[j] = scale * dot;
    }
}

/* Number of keys query row i may attend to (causal: keys 0..i). */
static long allowed_keys(long i, long n, int causal)
{
    if (causal)
        return i + 1;
    return n;
}

/* Plain definition for one query row against its first n_keys keys:
 * stable softmax of the scores, times V. */
static void attention_row_keys(const double *q, const double *k, const double *v,
                               long i, long n_keys, long d, double scale,
                               double *s, double *o_i, double *lse_i)
{
    scores_row(q, k, i, n_keys, d, scale, s);

    double m = -INFINITY;
    for (long j = 0; j < n_keys; ++j)
        if (s[j] > m)
            m = s[j];

    double l = 0.0;
    for (long j = 0; j < n_keys; ++j)
        l += exp(s[j] - m);

    for (long c = 0; c < d; ++c)
        o_i[c] = 0.0;
    for (long j = 0; j < n_keys; ++j) {
        double p = exp(s[j] - m);
        for (long c = 0; c < d; ++c)
            o_i[c] += p * v[j * d + c];
    }
    for (long c = 0; c < d; ++c)
        o_i[c] = o_i[c] / l;

    *lse_i = m + log(l);
}

/* Plain definition for row i of a square (queries = keys = n) problem. */
static void attention_row(const double *q, const double *k, const double *v,
                          long i, long n, long d, double scale, int causal,
                          double *s, double *o_i, double *lse_i)
{
    attention_row_keys(q, k, v, i, allowed_keys(i, n, causal), d, scale, s, o_i, lse_i);
}

/* ------------------------------------------------------------------ */
/* Threaded driver over a list of (head, row) pairs.                    */

typedef struct {
    const double *q, *k, *v;
    const long *rows; /* pairs: head index bh, query index i */
    long nrows, n, d;
    double scale;
    int causal;
    double *o, *lse;
    long begin, end;
    int status;
} row_job;

static void *row_worker(void *arg)
{
    row_job *job = (row_job *)arg;
    double *s = (double *)malloc((size_t)(job->n > 0 ? job->n : 1) * sizeof(double));
    if (!s) {
        job->status = ORACLE_ENOMEM;
        return NULL;
    }
    long head_elems = job->n * job->d;
    for (long r = job->begin; r < job->end; ++r) {
        long bh = job->rows[2 * r];
        long i = job->rows[2 * r + 1];
        const double *qh = job->q + bh * head_elems;
        const double *kh = job->k + bh * head_elems;
        const double *vh = job->v + bh * head_elems;
        attention_row(qh, kh, vh, i, job->n, job->d, job->scale, job->causal, s,
                      job->o + r * job->d, job->lse + r);
    }
    free(s);
    job->status = ORACLE_OK;
    return NULL;
}

/*
 * oracle_attention_rows: the plain definition for selected rows.
 *   q, k, v : [BH, N, d] fp64, contiguous (BH = batch * heads)
 *   rows    : nrows pairs (bh, i), 0 <= bh < BH, 0 <= i < N
 *   o       : [nrows, d] fp64 output, lse : [nrows] fp64 output
 *   nthreads: worker threads (<= 0 means 1)
 * Returns 0 on success, 1 on an invalid argument, 2 when out of memory.
 */
int oracle_attention_rows(const double *q, const double *k, const double *v,
                          long BH, long N, long d, double scale, int causal,
                          const long *rows, long nrows, double *o, double *lse,
                          int nthreads)
{
    if (BH < 0 || N < 0 || d < 1 || nrows < 0 || (causal != 0 && causal != 1))
        return ORACLE_EINVAL;
    if (nrows == 0)
        return ORACLE_OK;
    if (!q || !k || !v || !rows || !o || !lse || N == 0 || BH == 0)
        return ORACLE_EINVAL;
    for (long r = 0; r < nrows; ++r) {
        if (rows[2 * r] < 0 || rows[2 * r] >= BH || rows[2 * r + 1] < 0 ||
            rows[2 * r + 1] >= N)
            return ORACLE_EINVAL;
    }
    if (nthreads <= 0)
        nthreads = 1;
    if (nthreads > nrows)
        nthreads = (int)nrows;

    row_job *jobs = (row_job *)calloc((size_t)nthreads, sizeof(row_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    unsigned char *spawned = (unsigned char *)calloc((size_t)nthreads, 1);
    if (!jobs || !tids || !spawned) {
        free(jobs);
        free(tids);
        free(spawned);
        return ORACLE_ENOMEM;
    }
    long per = (nrows + nthreads - 1) / nthreads;
    int status = ORACLE_OK;
    for (int t = 0; t < nthreads; ++t) {
        row_job *jb = &jobs[t];
        jb->q = q; jb->k = k; jb->v = v; jb->rows = rows; jb->nrows = nrows;
        jb->n = N; jb->d = d; jb->scale = scale; jb->causal = causal;
        jb->o = o; jb->lse = lse;
        jb->begin = t * per;
        jb->end = (t + 1) * per < nrows ? (t + 1) * per : nrows;
        jb->status = ORACLE_OK;
        if (jb->begin >= jb->end)
            continue;
        /* the last slice, or one whose thread failed to start, runs here */
        if (t < nthreads - 1 && pthread_create(&tids[t], NULL, row_worker, jb) == 0)
            spawned[t] = 1;
        else
            row_worker(jb);
    }
    for (int t = 0; t < nthreads; ++t) {
        if (spawned[t])
            pthread_join(tids[t], NULL);
        if (jobs[t].status != ORACLE_OK)
            status = jobs[t].status;
    }
    free(spawned);
    free(jobs);
    free(tids);
    return status;
}

/*
 * oracle_attention_fwd: the plain definition for every row of every head.
 *   q, k, v, o : [BH, N, d] fp64 contiguous; lse : [BH, N] fp64.
 */
int oracle_attention_fwd(const double *q, const double *k, const double *v,
                         long BH, long N, long d, double scale, int causal,
                         double *o, double *lse, int nthreads)
{
    if (BH < 0 || N < 0 || d < 1)
        return ORACLE_EINVAL;
    long nrows = BH * N;
    if (nrows == 0)
        return ORACLE_OK;
    long *rows = (long *)malloc((size_t)nrows * 2 * sizeof(long));
    if (!rows)
        return ORACLE_ENOMEM;
    for (long bh = 0; bh < BH; ++bh)
        for (long i = 0; i < N; ++i) {
            rows[2 * (bh * N + i)] = bh;
            rows[2 * (bh * N + i) + 1] = i;
        }
    int st = oracle_attention_rows(q, k, v, BH, N, d, scale, causal, rows, nrows,
                                   o, lse, nthreads);
    free(rows);
    return st;
}

/*
 * oracle_scores_row: the scaled scores of query row i of one head against
 * its allowed keys (all N, or 0..i when causal).  q, k: [N, d] fp64.
 * s must hold N doubles; returns the number of scores written via *n_out.
 */
int oracle_scores_row(const double *q, const double *k, long N, long d, long i,
                      double scale, int causal, double *s, long *n_out)
{
    if (!q || !k || !s || !n_out || N < 1 || d < 1 || i < 0 || i >= N)
        return ORACLE_EINVAL;
    long n_keys = allowed_keys(i, N, causal);
    scores_row(q, k, i, n_keys, d, scale, s);
    *n_out = n_keys;
    return ORACLE_OK;
}

/*
 * oracle_online_row: the online-softmax recurrence ("3.6 어텐션 I",
 * section 3.6.4) over one row of scores s[0..n) with values v [n, d].
 *
 * The row is cut into nblocks blocks; block t covers scores
 * [block_start[t], block_start[t] + block_len[t]) and blocks are processed
 * in the order given (any order; the blocks need not be sorted).  State
 * starts at m = -inf, l = 0, O = 0.  For every block:
 *     m_tilde = max of the block's scores
 *     m_new   = max(m, m_tilde)
 *     alpha   = exp(m - m_new)          (0 on the first block: exp(-inf))
 *     p_j     = exp(s_j - m_new)        for the block's scores
 *     l       = alpha * l + sum_j p_j
 *     O       = alpha * O + sum_j p_j * v_j
 *     m       = m_new
 * and at the end o = O / l.
 *
 * Outputs: o_out [d] (normalised), *l_out, *m_out.  If trace is not NULL it
 * receives, per processed block, (m_tilde, m_new, alpha, l, O[0..d)) with O
 * unnormalised: nblocks * (4 + d) doubles.
 * The blocks must cover every score exactly once; otherwise returns 1.
 */
int oracle_online_row(const double *s, const double *v, long n, long d,
                      const long *block_start, const long *block_len,
                      long nblocks, double *o_out, double *l_out, double *m_out,
                      double *trace)
{
    if (!s || !v || !block_start || !block_len || !o_out || !l_out || !m_out ||
        n < 1 || d < 1 || nblocks < 1)
        return ORACLE_EINVAL;
    unsigned char *seen = (unsigned char *)calloc((size_t)n, 1);
    double *acc = (double *)calloc((size_t)d, sizeof(double));
    if (!seen || !acc) {
        free(seen);
        free(acc);
        return ORACLE_ENOMEM;
    }
    int status = ORACLE_OK;
    for (long t = 0; t < nblocks && status == ORACLE_OK; ++t) {
        if (block_len[t] < 1 || block_start[t] < 0 || block_start[t] + block_len[t] > n) {
            status = ORACLE_EINVAL;
            break;
        }
        for (long j = block_start[t]; j < block_start[t] + block_len[t]; ++j) {
            if (seen[j])
                status = ORACLE_EINVAL;
            seen[j] = 1;
        }
    }
    for (long j = 0; j < n && status == ORACLE_OK; ++j)
        if (!seen[j])
            status = ORACLE_EINVAL;
    if (status != ORACLE_OK) {
        free(seen);
        free(acc);
        return status;
    }

    double m = -INFINITY;
    double l = 0.0;
    for (long t = 0; t < nblocks; ++t) {
        long j0 = block_start[t], j1 = block_start[t] + block_len[t];
        double m_tilde = -INFINITY;
        for (long j = j0; j < j1; ++j)
            if (s[j] > m_tilde)
                m_tilde = s[j];
        double m_new = m > m_tilde ? m : m_tilde;
        double alpha = exp(m - m_new);
        double block_sum = 0.0;
        for (long j = j0; j < j1; ++j)
            block_sum += exp(s[j] - m_new);
        l = alpha * l + block_sum;
        for (long c = 0; c < d; ++c) {
            double pv = 0.0;
            for (long j = j0; j < j1; ++j)
                pv += exp(s[j] - m_new) * v[j * d + c];
            acc[c] = alpha * acc[c] + pv;
        }
        m = m_new;
        if (trace) {
            double *tr = trace + t * (4 + d);
            tr[0] = m_tilde;
            tr[1] = m_new;
            tr[2] = alpha;
            tr[3] = l;
            for (long c = 0; c < d; ++c)
                tr[4 + c] = acc[c];
        }
    }
    for (long c = 0; c < d; ++c)
        o_out[c] = acc[c] / l;
    *l_out = l;
    *m_out = m;
    free(seen);
    free(acc);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* Backward pass: gradients of the plain definition.                    */
/*
 * For one head with scores s_ij = scale * <q_i, k_j> over the allowed keys,
 * p_ij = softmax_j(s_ij) and o_i = sum_j p_ij v_j, and an upstream gradient
 * g_i = dL/do_i, the chain rule through the row softmax gives
 *     dv_j  = sum_i p_ij g_i
 *     dp_ij = <g_i, v_j>
 *     ds_ij = p_ij * (dp_ij - sum_k p_ik dp_ik)          (softmax Jacobian)
 *     dq_i  = scale * sum_j ds_ij k_j
 *     dk_j  = scale * sum_i ds_ij q_i
 * "3.6 어텐션 I", section 3.6.7, describes the backward as recomputing S and P
 * from Q, K and the saved row statistics; this is the quantity it computes.
 * Rows are processed one at a time (two passes over the keys, like the
 * forward), so memory is O(N d) per head.
 */
/* One query row i of one head over its n_keys allowed keys: leaves
 * s[j] = p_ij and dp[j] = <g_i, v_j>, writes dq_i, and returns
 * sum_j p_ij dp_ij (the row's D term of the softmax Jacobian). */
static double backward_row(const double *q, const double *k, const double *v, const double *g,
                           long i, long n_keys, long d, double scale, double *s, double *dp,
                           double *dq_i)
{
    scores_row(q, k, i, n_keys, d, scale, s);
    double m = -INFINITY;
    for (long j = 0; j < n_keys; ++j)
        if (s[j] > m)
            m = s[j];
    double row_sum = 0.0;
    for (long j = 0; j < n_keys; ++j)
        row_sum += exp(s[j] - m);
    /* s <- p_ij, dp <- <g_i, v_j> */
    double pdp = 0.0;
    for (long j = 0; j < n_keys; ++j) {
        s[j] = exp(s[j] - m) / row_sum;
        double dot = 0.0;
        for (long c = 0; c < d; ++c)
            dot += g[i * d + c] * v[j * d + c];
        dp[j] = dot;
        pdp += s[j] * dot;
    }
    for (long c = 0; c < d; ++c)
        dq_i[c] = 0.0;
    for (long j = 0; j < n_keys; ++j) {
        const double ds_ij = s[j] * (dp[j] - pdp);
        for (long c = 0; c < d; ++c)
            dq_i[c] += scale * ds_ij * k[j * d + c];
    }
    return pdp;
}

/* Query rows [i0, i1) of one head: their dq rows are written, and their
 * contributions are added into dk and dv. */
static void backward_rows(const double *q, const double *k, const double *v, const double *g,
                          long n, long d, double scale, int causal, long i0, long i1, double *s,
                          double *dp, double *dq, double *dk, double *dv)
{
    for (long i = i0; i < i1; ++i) {
        long n_keys = allowed_keys(i, n, causal);
        double pdp = backward_row(q, k, v, g, i, n_keys, d, scale, s, dp, dq + i * d);
        for (long j = 0; j < n_keys; ++j) {
            double ds = s[j] * (dp[j] - pdp);
            for (long c = 0; c < d; ++c) {
                dv[j * d + c] += s[j] * g[i * d + c];
                dk[j * d + c] += scale * ds * q[i * d + c];
            }
        }
    }
}

/* A share of the work: query rows [i0, i1) of head `head`.  dk and dv point
 * at the head's outputs when one job covers the whole head, else at private
 * accumulators that are summed afterwards in job order. */
typedef struct {
    const double *q, *k, *v, *g;
    long n, d;
    double scale;
    int causal;
    long head, i0, i1;
    double *dq, *dk, *dv;
    int status;
} rows_job;

static void run_rows_job(rows_job *jb)
{
    double *s = (double *)malloc((size_t)(jb->n > 0 ? jb->n : 1) * sizeof(double));
    double *dp = (double *)malloc((size_t)(jb->n > 0 ? jb->n : 1) * sizeof(double));
    if (!s || !dp) {
        free(s);
        free(dp);
        jb->status = ORACLE_ENOMEM;
        return;
    }
    long he = jb->n * jb->d;
    for (long x = 0; x < he; ++x) {
        jb->dk[x] = 0.0;
        jb->dv[x] = 0.0;
    }
    backward_rows(jb->q + jb->head * he, jb->k + jb->head * he, jb->v + jb->head * he,
                  jb->g + jb->head * he, jb->n, jb->d, jb->scale, jb->causal, jb->i0, jb->i1, s, dp,
                  jb->dq + jb->head * he, jb->dk, jb->dv);
    free(s);
    free(dp);
    jb->status = ORACLE_OK;
}

typedef struct {
    rows_job *jobs;
    long begin, end;
} job_range;

static void *jobs_worker(void *arg)
{
    job_range *r = (job_range *)arg;
    for (long t = r->begin; t < r->end; ++t)
        run_rows_job(&r->jobs[t]);
    return NULL;
}

/*
 * oracle_attention_bwd: gradients dq, dk, dv ([BH, N, d] fp64) of
 * L = sum(o * g) for the plain definition, given q, k, v and g = dL/do
 * ([BH, N, d] fp64).  The work is split into (head, query-row range) jobs:
 * one job per head when there are at least as many heads as threads, else
 * each head's rows are split so that every thread has work; split heads sum
 * their jobs' dk, dv in job order.
 */
int oracle_attention_bwd(const double *q, const double *k, const double *v, const double *g,
                         long BH, long N, long d, double scale, int causal, double *dq,
                         double *dk, double *dv, int nthreads)
{
    if (BH < 0 || N < 0 || d < 1 || (causal != 0 && causal != 1))
        return ORACLE_EINVAL;
    if (BH == 0 || N == 0)
        return ORACLE_OK;
    if (!q || !k || !v || !g || !dq || !dk || !dv)
        return ORACLE_EINVAL;
    if (nthreads <= 0)
        nthreads = 1;
    long splits = nthreads > BH ? nthreads / BH : 1;
    if (splits > N)
        splits = N;
    const long njobs = BH * splits;
    const long he = N * d;
    rows_job *jobs = (rows_job *)calloc((size_t)njobs, sizeof(rows_job));
    double *priv = splits > 1 ? (double *)malloc((size_t)njobs * 2 * (size_t)he * sizeof(double)) : NULL;
    if (!jobs || (splits > 1 && !priv)) {
        free(jobs);
        free(priv);
        return ORACLE_ENOMEM;
    }
    const long rows_per = (N + splits - 1) / splits;
    for (long h = 0; h < BH; ++h) {
        for (long sp = 0; sp < splits; ++sp) {
            rows_job *jb = &jobs[h * splits + sp];
            jb->q = q; jb->k = k; jb->v = v; jb->g = g; jb->n = N; jb->d = d;
            jb->scale = scale; jb->causal = causal; jb->head = h; jb->dq = dq;
            jb->i0 = sp * rows_per < N ? sp * rows_per : N;
            jb->i1 = (sp + 1) * rows_per < N ? (sp + 1) * rows_per : N;
            if (splits > 1) {
                jb->dk = priv + (size_t)(h * splits + sp) * 2 * (size_t)he;
                jb->dv = jb->dk + he;
            } else {
                jb->dk = dk + h * he;
                jb->dv = dv + h * he;
            }
            jb->status = ORACLE_OK;
        }
    }
    int nt = nthreads < njobs ? nthreads : (int)njobs;
    job_range *ranges = (job_range *)calloc((size_t)nt, sizeof(job_range));
    pthread_t *tids = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
    unsigned char *spawned = (unsigned char *)calloc((size_t)nt, 1);
    if (!ranges || !tids || !spawned) {
        free(ranges); free(tids); free(spawned); free(jobs); free(priv);
        return ORACLE_ENOMEM;
    }
    const long per = (njobs + nt - 1) / nt;
    for (int t = 0; t < nt; ++t) {
        ranges[t].jobs = jobs;
        ranges[t].begin = t * per < njobs ? t * per : njobs;
        ranges[t].end = (t + 1) * per < njobs ? (t + 1) * per : njobs;
        if (t < nt - 1 && pthread_create(&tids[t], NULL, jobs_worker, &ranges[t]) == 0)
            spawned[t] = 1;
        else
            jobs_worker(&ranges[t]);
    }
    int status = ORACLE_OK;
    for (int t = 0; t < nt; ++t)
        if (spawned[t])
            pthread_join(tids[t], NULL);
    for (long x = 0; x < njobs; ++x)
        if (jobs[x].status != ORACLE_OK)
            status = jobs[x].status;
    if (status == ORACLE_OK && splits > 1) {
        for (long h = 0; h < BH; ++h) {
            double *dkh = dk + h * he, *dvh = dv + h * he;
            for (long x = 0; x < he; ++x) {
                dkh[x] = 0.0;
                dvh[x] = 0.0;
            }
            for (long sp = 0; sp < splits; ++sp) {
                const rows_job *jb = &jobs[h * splits + sp];
                for (long x = 0; x < he; ++x) {
                    dkh[x] += jb->dk[x];
                    dvh[x] += jb->dv[x];
                }
            }
        }
    }
    free(ranges); free(tids); free(spawned); free(jobs); free(priv);
    return status;
}

/*
 * oracle_attention_bwd_rows: dq for the listed query rows only (rows[2r] =
 * flattened head, rows[2r+1] = query index), into dq_out [nrows, d].  One
 * row needs only its own softmax, so each costs O(N d).  Threads split the
 * rows.
 */
typedef struct {
    const double *q, *k, *v, *g;
    long N, d;
    double scale;
    int causal;
    const long *rows;
    double *out;
    long begin, end;
    int status;
} dq_rows_job;

static void *dq_rows_worker(void *arg)
{
    dq_rows_job *jb = (dq_rows_job *)arg;
    double *s = (double *)malloc((size_t)jb->N * sizeof(double));
    double *dp = (double *)malloc((size_t)jb->N * sizeof(double));
    if (!s || !dp) {
        free(s);
        free(dp);
        jb->status = ORACLE_ENOMEM;
        return NULL;
    }
    const long he = jb->N * jb->d;
    for (long r = jb->begin; r < jb->end; ++r) {
        const long bh = jb->rows[2 * r], i = jb->rows[2 * r + 1];
        backward_row(jb->q + bh * he, jb->k + bh * he, jb->v + bh * he, jb->g + bh * he, i,
                     allowed_keys(i, jb->N, jb->causal), jb->d, jb->scale, s, dp, jb->out + r * jb->d);
    }
    free(s);
    free(dp);
    jb->status = ORACLE_OK;
    return NULL;
}

int oracle_attention_bwd_rows(const double *q, const double *k, const double *v, const double *g,
                              long BH, long N, long d, double scale, int causal, const long *rows,
                              long nrows, double *dq_out, int nthreads)
{
    if (BH < 0 || N < 0 || d < 1 || nrows < 0 || (causal != 0 && causal != 1))
        return ORACLE_EINVAL;
    if (nrows == 0)
        return ORACLE_OK;
    if (!q || !k || !v || !g || !rows || !dq_out || N == 0)
        return ORACLE_EINVAL;
    for (long r = 0; r < nrows; ++r)
        if (rows[2 * r] < 0 || rows[2 * r] >= BH || rows[2 * r + 1] < 0 || rows[2 * r + 1] >= N)
            return ORACLE_EINVAL;
    if (nthreads <= 0)
        nthreads = 1;
    if (nthreads > nrows)
        nthreads = (int)nrows;
    dq_rows_job *jobs = (dq_rows_job *)calloc((size_t)nthreads, sizeof(dq_rows_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    unsigned char *spawned = (unsigned char *)calloc((size_t)nthreads, 1);
    if (!jobs || !tids || !spawned) {
        free(jobs); free(tids); free(spawned);
        return ORACLE_ENOMEM;
    }
    const long per = (nrows + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        dq_rows_job *jb = &jobs[t];
        jb->q = q; jb->k = k; jb->v = v; jb->g = g; jb->N = N; jb->d = d; jb->scale = scale;
        jb->causal = causal; jb->rows = rows; jb->out = dq_out;
        jb->begin = t * per < nrows ? t * per : nrows;
        jb->end = (t + 1) * per < nrows ? (t + 1) * per : nrows;
        jb->status = ORACLE_OK;
        if (t < nthreads - 1 && pthread_create(&tids[t], NULL, dq_rows_worker, jb) == 0)
            spawned[t] = 1;
        else
            dq_rows_worker(jb);
    }
    int status = ORACLE_OK;
    for (int t = 0; t < nthreads; ++t) {
        if (spawned[t])
            pthread_join(tids[t], NULL);
        if (jobs[t].status != ORACLE_OK)
            status = jobs[t].status;
    }
    free(jobs); free(tids); free(spawned);
    return status;
}

/* ------------------------------------------------------------------ */
/* Decoding: few queries against a long key sequence.                   */
/*
 * The plain definition for Nq queries against Nk keys (Nq <= Nk).  Causal
 * aligns the queries with the end of the key sequence: query i sits at
 * position Nk - Nq + i and attends to keys 0 .. Nk - Nq + i (for Nq = 1,
 * every key).  "3.6 어텐션 I", section 3.6.9: decoding (one query) is the
 * case that needs a different parallelisation; the quantity is unchanged.
 */
static long decode_keys(long i, long nq, long nk, int causal)
{
    return causal ? nk - nq + i + 1 : nk;
}

typedef struct {
    const double *q, *k, *v;
    long nq, nk, d;
    double scale;
    int causal;
    double *o, *lse;
    long begin, end; /* flattened (head, query) rows */
    int status;
} decode_job;

static void *decode_worker(void *arg)
{
    decode_job *jb = (decode_job *)arg;
    double *s = (double *)malloc((size_t)jb->nk * sizeof(double));
    if (!s) {
        jb->status = ORACLE_ENOMEM;
        return NULL;
    }
    for (long r = jb->begin; r < jb->end; ++r) {
        const long bh = r / jb->nq, i = r % jb->nq;
        attention_row_keys(jb->q + bh * jb->nq * jb->d, jb->k + bh * jb->nk * jb->d,
                           jb->v + bh * jb->nk * jb->d, i, decode_keys(i, jb->nq, jb->nk, jb->causal),
                           jb->d, jb->scale, s, jb->o + r * jb->d, jb->lse + r);
    }
    free(s);
    jb->status = ORACLE_OK;
    return NULL;
}

/*
 * oracle_attention_decode: q [BH, Nq, d], k and v [BH, Nk, d] fp64
 * contiguous; o [BH, Nq, d], lse [BH, Nq].  Requires 1 <= Nq <= Nk.
 */
int oracle_attention_decode(const double *q, const double *k, const double *v, long BH, long Nq,
                            long Nk, long d, double scale, int causal, double *o, double *lse,
                            int nthreads)
{
    if (BH < 0 || Nq < 1 || Nk < Nq || d < 1 || (causal != 0 && causal != 1))
        return ORACLE_EINVAL;
    if (BH == 0)
        return ORACLE_OK;
    if (!q || !k || !v || !o || !lse)
        return ORACLE_EINVAL;
    const long nrows = BH * Nq;
    if (nthreads <= 0)
        nthreads = 1;
    if (nthreads > nrows)
        nthreads = (int)nrows;
    decode_job *jobs = (decode_job *)calloc((size_t)nthreads, sizeof(decode_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    unsigned char *spawned = (unsigned char *)calloc((size_t)nthreads, 1);
    if (!jobs || !tids || !spawned) {
        free(jobs); free(tids); free(spawned);
        return ORACLE_ENOMEM;
    }
    const long per = (nrows + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        decode_job *jb = &jobs[t];
        jb->q = q; jb->k = k; jb->v = v; jb->nq = Nq; jb->nk = Nk; jb->d = d;
        jb->scale = scale; jb->causal = causal; jb->o = o; jb->lse = lse;
        jb->begin = t * per < nrows ? t * per : nrows;
        jb->end = (t + 1) * per < nrows ? (t + 1) * per : nrows;
        jb->status = ORACLE_OK;
        if (t < nthreads - 1 && pthread_create(&tids[t], NULL, decode_worker, jb) == 0)
            spawned[t] = 1;
        else
            decode_worker(jb);
    }
    int status = ORACLE_OK;
    for (int t = 0; t < nthreads; ++t) {
        if (spawned[t])
            pthread_join(tids[t], NULL);
        if (jobs[t].status != ORACLE_OK)
            status = jobs[t].status;
    }
    free(jobs); free(tids); free(spawned);
    return status;
}

int oracle_abi_version(void) { return 1; }
