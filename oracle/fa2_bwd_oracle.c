/*
 * CPU oracle for the gradient of the attention forward pass (the backward
 * pass of FlashAttention-2) — TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite and the benchmark's CPU-baseline leg may load this
 * code. The product library never links, loads or calls it.
 *
 * It is the gradient of the forward definition, written out by the chain
 * rule, in fp64, with no tiling and no reordering. For one head, with the
 * forward quantities
 *
 *   J(i)  = { j : 0 <= j < N, and j <= i when the causal mask is on }
 *   s_ij  = scale * <Q_i, K_j>,   P_ij = exp(s_ij) / sum_{j' in J(i)} exp(s_ij')
 *   O_i   = sum_{j in J(i)} P_ij V_j
 *
 * and an upstream gradient dO (the gradient of a scalar loss w.r.t. O):
 *
 *   dV_j   = sum_{i : j in J(i)} P_ij dO_i
 *   dP_ij  = <dO_i, V_j>
 *   Delta_i = <dO_i, O_i>                     (= sum_j P_ij dP_ij)
 *   dS_ij  = P_ij (dP_ij - Delta_i)           (softmax Jacobian)
 *   dQ_i   = scale * sum_{j in J(i)} dS_ij K_j
 *   dK_j   = scale * sum_{i : j in J(i)} dS_ij Q_i
 *
 * Sources: the yangyitao.com CUDA book, ch. 15, section 15.1 (change 4: the
 * backward pass keeps only LSE = m + log l per row and recomputes S and P
 * from it) and the closing paragraph of the chapter (the backward recomputes
 * S and P, accumulates dQ across key tiles, and runs the outer loop over
 * K/V); the forward definition itself is the one in fa2_oracle.c.
 *
 * Two passes: over query rows (row statistics m_i, l_i, O_i, Delta_i, then
 * dQ_i), and over key rows (dK_j, dV_j, recomputing P_ij from the stored
 * m_i, l_i). Each output row is computed by one thread with a fixed loop
 * order, so results do not depend on the thread count.
 *
 * Optional outputs *_mag are per-element condition sums for error bounds:
 *   dV_mag = sum_i |P_ij dO_id|
 *   dQ_mag = scale * sum_j P_ij (|dP_ij - Delta_i| + A_i) |K_jd|
 *   dK_mag = scale * sum_i P_ij (|dP_ij - Delta_i| + A_i) |Q_id|
 * with A_i = sum_d |dO_id O_id|. A relative perturbation of size u of each
 * P_ij, of each dS_ij and of each O_id (16-bit rounding of those operands)
 * moves an element by at most about u times its condition sum. Each is at
 * least the sum of the absolute values of the element's terms.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *q, *k, *v, *dout;    /* one head: [N, D] row-major          */
    long n, d;
    double scale;
    int causal;
    double *m, *l, *delta;             /* [N] row statistics (pass 1 output)  */
    double *amag;                      /* [N] sum_d |dO_id O_id| (pass 1)     */
    double *dq, *dk, *dv;              /* [N, D]                              */
    double *dq_mag, *dk_mag, *dv_mag;  /* [N, D] or NULL                      */
} bwd_ctx;

typedef struct {
    const bwd_ctx *c;
    long begin, end;
    double *scratch;                   /* length N                            */
    int pass;
} bwd_job;

static double dot(const double *a, const double *b, long d)
{
    double s = 0.0;
    for (long c = 0; c < d; ++c) s += a[c] * b[c];
    return s;
}

/* Number of keys query row i may attend to (the keys are 0 .. nvis-1). */
static long visible_keys(const bwd_ctx *c, long i)
{
    if (!c->causal) return c->n;
    return (i + 1 < c->n) ? i + 1 : c->n;
}

/* First query row that may attend to key j (the rows are first .. N-1). */
static long first_query(const bwd_ctx *c, long j)
{
    return c->causal ? j : 0;
}

/* Pass 1, query row i: softmax statistics, O_i, Delta_i, then dQ_i. */
static void bwd_query_row(const bwd_ctx *c, long i, double *s)
{
    const long d = c->d, nvis = visible_keys(c, i);
    const double *qi = c->q + i * d, *doi = c->dout + i * d;
    double *dqi = c->dq + i * d;
    double *dqm = c->dq_mag ? c->dq_mag + i * d : NULL;
    double m = -INFINITY;
    for (long j = 0; j < nvis; ++j) {
        s[j] = c->scale * dot(qi, c->k + j * d, d);
        if (s[j] > m) m = s[j];
    }
    /* s[j] <- exp(s_ij - m), the unnormalised softmax weights */
    double l = 0.0;
    for (long j = 0; j < nvis; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    /* O_i, then Delta_i = <dO_i, O_i> */
    double delta = 0.0, amag = 0.0;
    for (long col = 0; col < d; ++col) {
        double o = 0.0;
        for (long j = 0; j < nvis; ++j) o += s[j] * c->v[j * d + col];
        delta += doi[col] * (o / l);
        amag += fabs(doi[col] * (o / l));
    }
    c->m[i] = m;
    c->l[i] = l;
    c->delta[i] = delta;
    c->amag[i] = amag;
    for (long col = 0; col < d; ++col) {
        dqi[col] = 0.0;
        if (dqm) dqm[col] = 0.0;
    }
    for (long j = 0; j < nvis; ++j) {
        const double *kj = c->k + j * d;
        const double p = s[j] / l;
        const double dp = dot(doi, c->v + j * d, d);
        const double ds = p * (dp - delta);
        const double cond = c->scale * p * (fabs(dp - delta) + amag);
        for (long col = 0; col < d; ++col) {
            const double t = c->scale * ds * kj[col];
            dqi[col] += t;
            if (dqm) dqm[col] += cond * fabs(kj[col]);
        }
    }
}

/* Pass 2, key row j: dV_j and dK_j from the stored row statistics. */
static void bwd_key_row(const bwd_ctx *c, long j)
{
    const long d = c->d, n = c->n;
    const double *kj = c->k + j * d, *vj = c->v + j * d;
    double *dkj = c->dk + j * d, *dvj = c->dv + j * d;
    double *dkm = c->dk_mag ? c->dk_mag + j * d : NULL;
    double *dvm = c->dv_mag ? c->dv_mag + j * d : NULL;
    for (long col = 0; col < d; ++col) {
        dkj[col] = 0.0;
        dvj[col] = 0.0;
        if (dkm) dkm[col] = 0.0;
        if (dvm) dvm[col] = 0.0;
    }
    for (long i = first_query(c, j); i < n; ++i) {
        const double *qi = c->q + i * d, *doi = c->dout + i * d;
        const double sij = c->scale * dot(qi, kj, d);
        const double p = exp(sij - c->m[i]) / c->l[i];
        const double dp = dot(doi, vj, d);
        const double ds = p * (dp - c->delta[i]);
        const double cond = c->scale * p * (fabs(dp - c->delta[i]) + c->amag[i]);
        for (long col = 0; col < d; ++col) {
            const double tv = p * doi[col];
            const double tk = c->scale * ds * qi[col];
            dvj[col] += tv;
            dkj[col] += tk;
            if (dvm) dvm[col] += fabs(tv);
            if (dkm) dkm[col] += cond * fabs(qi[col]);
        }
    }
}

static void *bwd_worker(void *arg)
{
    bwd_job *jb = (bwd_job *)arg;
    for (long r = jb->begin; r < jb->end; ++r) {
        if (jb->pass == 1)
            bwd_query_row(jb->c, r, jb->scratch);
        else
            bwd_key_row(jb->c, r);
    }
    return NULL;
}

/* Runs one pass over rows [0, n) on up to nthreads threads. */
static int run_pass(const bwd_ctx *c, int pass, int nthreads)
{
    const long n = c->n;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n) nthreads = (int)n;
    bwd_job *jobs = (bwd_job *)calloc((size_t)nthreads, sizeof(bwd_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    double *scratch = (double *)malloc((size_t)nthreads * (size_t)n * sizeof(double));
    if (!jobs || !tids || !scratch) {
        free(jobs); free(tids); free(scratch);
        return -1;
    }
    const long per = (n + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        bwd_job *jb = &jobs[t];
        jb->c = c;
        jb->pass = pass;
        jb->begin = (long)t * per;
        jb->end = jb->begin + per < n ? jb->begin + per : n;
        jb->scratch = scratch + (size_t)t * (size_t)n;
        if (t == 0 || jb->begin >= jb->end) continue;
        if (pthread_create(&tids[t], NULL, bwd_worker, jb) != 0) {
            bwd_worker(jb);
            tids[t] = 0;
        }
    }
    bwd_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t)
        if (tids[t]) pthread_join(tids[t], NULL);
    free(jobs); free(tids); free(scratch);
    return 0;
}

/*
 * One head. q, k, v, dout: [n, d] row-major doubles. dq, dk, dv: [n, d]
 * outputs. delta (optional, [n]): receives Delta_i. *_mag (optional, [n, d]):
 * per-element condition sums (see above). Returns 0, or -1 on
 * a bad argument or an allocation failure.
 */
int fa2_oracle_bwd_head(const double *q, const double *k, const double *v, const double *dout,
                        long n, long d, double scale, int causal,
                        double *dq, double *dk, double *dv, double *delta,
                        double *dq_mag, double *dk_mag, double *dv_mag, int nthreads)
{
    if (!q || !k || !v || !dout || !dq || !dk || !dv || n < 1 || d < 1) return -1;
    double *stats = (double *)malloc((size_t)4 * (size_t)n * sizeof(double));
    if (!stats) return -1;
    bwd_ctx c;
    memset(&c, 0, sizeof(c));
    c.q = q; c.k = k; c.v = v; c.dout = dout;
    c.n = n; c.d = d; c.scale = scale; c.causal = causal;
    c.m = stats; c.l = stats + n; c.delta = stats + 2 * n; c.amag = stats + 3 * n;
    c.dq = dq; c.dk = dk; c.dv = dv;
    c.dq_mag = dq_mag; c.dk_mag = dk_mag; c.dv_mag = dv_mag;
    int rc = run_pass(&c, 1, nthreads);
    if (rc == 0) rc = run_pass(&c, 2, nthreads);
    if (rc == 0 && delta) memcpy(delta, c.delta, (size_t)n * sizeof(double));
    free(stats);
    return rc;
}
