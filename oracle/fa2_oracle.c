/*
 * CPU oracle for the FlashAttention-2 forward pass — TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this code. The product library never links, loads or calls it.
 *
 * What it computes is the plain definition, in fp64, with no tiling, no
 * online rescaling and no reordering beyond one pass for the scores and one
 * pass for the weighted sum:
 *
 *   for every head (b, h) and query row i:
 *     J(i) = { j : 0 <= j < N, and j <= i when the causal mask is on }
 *     s_j  = scale * sum_d Q[i,d] * K[j,d]                        (j in J(i))
 *     m    = max_j s_j,   l = sum_j exp(s_j - m)
 *     O[i] = sum_j exp(s_j - m) * V[j] / l,   LSE[i] = m + ln(l)
 *     J(i) empty  =>  O[i] = 0, LSE[i] = +inf
 *
 * Sources: "FlashAttention-2 MMA 代码学习" step 0 (standard attention
 * O = softmax(QK^T/sqrt(d)) V) and step 1 (the (m, l) statistics); the
 * yangyitao.com CUDA book ch. 15, section 15.1 (change 4: LSE = m + log l),
 * section 15.3 (softmax_scale applied to the dot product before the max,
 * causal rule "col > row is masked", columns >= N masked, an all-masked row
 * gives O = 0 and LSE = +inf, and LSE uses the natural log).
 *
 * Inputs are the exact values of the 16-bit tensors, widened to double by
 * the caller. Work is split over POSIX threads by rows; each row is computed
 * by exactly one thread with the same loop order, so results do not depend
 * on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *q, *k, *v;   /* one head: [N, D] each, row-major        */
    long n, d;
    double scale;
    int causal;
    const long *rows;          /* query rows to compute (NULL: all rows)  */
    long nrows;
    double *o;                 /* [nrows, D]                              */
    double *lse;               /* [nrows]                                 */
    long begin, end;           /* this worker's slice of [0, nrows)       */
    double *scores;            /* scratch, length N                       */
} oracle_job;

static void oracle_row(const oracle_job *jb, long i, double *o_row, double *lse_out)
{
    const long n = jb->n, d = jb->d;
    long nvis = n;                              /* |J(i)| for a prefix set */
    if (jb->causal) nvis = (i + 1 < n) ? i + 1 : n;
    if (nvis <= 0) {
        for (long c = 0; c < d; ++c) o_row[c] = 0.0;
        *lse_out = INFINITY;
        return;
    }
    const double *qi = jb->q + i * d;
    double m = -INFINITY;
    for (long j = 0; j < nvis; ++j) {
        const double *kj = jb->k + j * d;
        double dot = 0.0;
        for (long c = 0; c < d; ++c) dot += qi[c] * kj[c];
        const double s = jb->scale * dot;
        jb->scores[j] = s;
        if (s > m) m = s;
    }
    double l = 0.0;
    for (long c = 0; c < d; ++c) o_row[c] = 0.0;
    for (long j = 0; j < nvis; ++j) {
        const double w = exp(jb->scores[j] - m);
        const double *vj = jb->v + j * d;
        l += w;
        for (long c = 0; c < d; ++c) o_row[c] += w * vj[c];
    }
    for (long c = 0; c < d; ++c) o_row[c] /= l;
    *lse_out = m + log(l);
}

static void *oracle_worker(void *arg)
{
    oracle_job *jb = (oracle_job *)arg;
    for (long r = jb->begin; r < jb->end; ++r) {
        const long i = jb->rows ? jb->rows[r] : r;
        oracle_row(jb, i, jb->o + r * jb->d, jb->lse + r);
    }
    return NULL;
}

/*
 * One head. q, k, v: [n, d] row-major doubles. rows: query indices (or NULL
 * for all n rows, in which case nrows must equal n). o: [nrows, d]. lse:
 * [nrows]. Returns 0, or -1 on a bad argument / allocation failure.
 */
int fa2_oracle_head(const double *q, const double *k, const double *v,
                    long n, long d, double scale, int causal,
                    const long *rows, long nrows,
                    double *o, double *lse, int nthreads)
{
    if (!q || !k || !v || !o || !lse || n < 1 || d < 1 || nrows < 0) return -1;
    if (!rows && nrows != n) return -1;
    for (long r = 0; rows && r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= n) return -1;
    if (nrows == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > nrows) nthreads = (int)nrows;

    oracle_job *jobs = (oracle_job *)calloc((size_t)nthreads, sizeof(oracle_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    double *scratch = (double *)malloc((size_t)nthreads * (size_t)n * sizeof(double));
    if (!jobs || !tids || !scratch) {
        free(jobs); free(tids); free(scratch);
        return -1;
    }
    const long per = (nrows + nthreads - 1) / nthreads;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        oracle_job *jb = &jobs[t];
        jb->q = q; jb->k = k; jb->v = v;
        jb->n = n; jb->d = d; jb->scale = scale; jb->causal = causal;
        jb->rows = rows; jb->nrows = nrows; jb->o = o; jb->lse = lse;
        jb->begin = (long)t * per;
        jb->end = jb->begin + per < nrows ? jb->begin + per : nrows;
        jb->scores = scratch + (size_t)t * (size_t)n;
        if (jb->begin >= jb->end) continue;
        if (t == 0) continue;                    /* run slice 0 on this thread */
        if (pthread_create(&tids[t], NULL, oracle_worker, jb) != 0) {
            oracle_worker(jb);                   /* fall back to inline */
            tids[t] = 0;
        } else {
            ++started;
        }
    }
    oracle_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (tids[t]) pthread_join(tids[t], NULL);
    (void)started;
    free(jobs); free(tids); free(scratch);
    return 0;
}
