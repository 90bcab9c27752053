/*
 * attn_oracle.c -- plain, slow CPU reference ("oracle") for the fused
 * attention forward, in fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file: it exists so that tests, the smoke check and the CPU
 * baseline leg of the benchmark can compare the CUDA kernels against an
 * independent definition.  It shares no code, header, table or constant with
 * the CUDA library (attention_fa2_fwd_gb300/csrc) and includes none of it.
 *
 * What it computes (one query row at a time, no tiling, no online softmax):
 *
 *   For every batch b, query head h < H_q and query row i < N_q
 *     1. kv head        hk = floor(h / (H_q / H_kv))
 *          ("Skill: Write a Triton Attention Kernel", Required reasoning
 *           process, step 1: the KV head is the Q head divided by the
 *           group size; the GQA/MQA note on "Triton-FlashAttention" uses
 *           the same index_head // group_size mapping.)
 *     2. score row      s_j = scale * sum_d Q[b,h,i,d] * K[b,hk,j,d]
 *                       for every j < N_kv  (step 5b: S = Q K^T * scale)
 *     3. mask           s_j = -inf where j > i when causal
 *                       (step 5c: keep q_pos >= kv_pos, top-left aligned:
 *                        the pages compare absolute positions with no
 *                        offset between the query and key sequences)
 *     4. softmax        m = max_j s_j, e_j = exp(s_j - m), l = sum_j e_j
 *     5. output         O[b,h,i,:] = sum_j (e_j / l) * V[b,hk,j,:]
 *                       (Correctness requirements: after the loop O / l
 *                        is the softmax-weighted average of the V rows)
 *     6. log-sum-exp    LSE[b,h,i] = m + ln(l)
 *                       (step 8: natural log, and not m alone)
 *
 * This is exactly the value that the tiled online-softmax algorithm of the
 * pages reaches in exact arithmetic; the oracle writes the explicit full
 * score row instead.  exp/log are the C library's, in double precision.
 *
 * Decode (one new query token over a cache of cache_len valid positions,
 * "Triton-FlashAttention", Phase 2: all cache_len cached positions take part) is the
 * same definition with N_q = 1, N_kv = cache_len and no causal mask.
 *
 * Layout: every tensor is a dense, contiguous fp64 array in (b, h, n, d)
 * order: Q (B,H_q,N_q,D), K and V (B,H_kv,N_kv,D), O (B,H_q,N_q,D),
 * LSE (B,H_q,N_q).  Callers convert/permute before calling.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL 1
#define ORACLE_ENOMEM 2

typedef struct {
    const double *q, *k, *v;
    double *o, *lse;
    int64_t B, Hq, Hkv, Nq, Nkv, D;
    int causal;
    double scale;
    /* either a dense range of flattened (b,h,i) rows, or a list of triples */
    const int64_t *sel; /* NULL for dense */
    int64_t first, last; /* [first, last) of flattened rows or of sel entries */
    int failed;
} job_t;

/* Steps 1-6 above for one (b, h, i).  s is scratch of N_kv doubles. */
static void attention_row(const job_t *J, int64_t b, int64_t h, int64_t i,
                          double *s, double *o_row, double *lse_out)
{
    const int64_t D = J->D, Nkv = J->Nkv;
    const int64_t group = J->Hq / J->Hkv;
    const int64_t hk = h / group;                                   /* step 1 */
    const double *qrow = J->q + ((b * J->Hq + h) * J->Nq + i) * D;
    const double *kh = J->k + (b * J->Hkv + hk) * Nkv * D;
    const double *vh = J->v + (b * J->Hkv + hk) * Nkv * D;

    double m = -INFINITY;
    for (int64_t j = 0; j < Nkv; ++j) {
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d) dot += qrow[d] * kh[j * D + d];
        double sj = J->scale * dot;                                 /* step 2 */
        if (J->causal && j > i) sj = -INFINITY;                     /* step 3 */
        s[j] = sj;
        if (sj > m) m = sj;
    }
    double l = 0.0;
    for (int64_t j = 0; j < Nkv; ++j) {                             /* step 4 */
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    for (int64_t d = 0; d < D; ++d) o_row[d] = 0.0;
    for (int64_t j = 0; j < Nkv; ++j) {                             /* step 5 */
        const double w = s[j] / l;
        if (w == 0.0) continue;
        for (int64_t d = 0; d < D; ++d) o_row[d] += w * vh[j * D + d];
    }
    *lse_out = m + log(l);                                          /* step 6 */
}

static void *run_job(void *arg)
{
    job_t *J = (job_t *)arg;
    double *s = (double *)malloc((size_t)(J->Nkv > 0 ? J->Nkv : 1) * sizeof(double));
    if (!s) {
        J->failed = 1;
        return NULL;
    }
    for (int64_t r = J->first; r < J->last; ++r) {
        int64_t b, h, i;
        double *o_row, *lse_out;
        if (J->sel) {
            b = J->sel[3 * r + 0];
            h = J->sel[3 * r + 1];
            i = J->sel[3 * r + 2];
            o_row = J->o + r * J->D;
            lse_out = J->lse + r;
        } else {
            i = r % J->Nq;
            h = (r / J->Nq) % J->Hq;
            b = r / (J->Nq * J->Hq);
            o_row = J->o + r * J->D;
            lse_out = J->lse + r;
        }
        attention_row(J, b, h, i, s, o_row, lse_out);
    }
    free(s);
    return NULL;
}

static int run_threads(job_t *proto, int64_t nrows, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    if ((int64_t)nthreads > nrows) nthreads = (int)(nrows > 0 ? nrows : 1);
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !tids) {
        free(jobs);
        free(tids);
        return ORACLE_ENOMEM;
    }
    int rc = ORACLE_OK;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *proto;
        jobs[t].first = nrows * t / nthreads;
        jobs[t].last = nrows * (t + 1) / nthreads;
    }
    int started = 0;
    for (int t = 1; t < nthreads; ++t) {
        if (pthread_create(&tids[t], NULL, run_job, &jobs[t]) != 0) break;
        started = t;
    }
    run_job(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
    for (int t = started + 1; t < nthreads; ++t) run_job(&jobs[t]); /* threads that failed to start */
    for (int t = 0; t < nthreads; ++t)
        if (jobs[t].failed) rc = ORACLE_ENOMEM;
    free(jobs);
    free(tids);
    return rc;
}

static int check_shape(int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nkv, int64_t D)
{
    if (B < 1 || Hq < 1 || Hkv < 1 || Nq < 1 || Nkv < 1 || D < 1) return ORACLE_EINVAL;
    if (Hq % Hkv != 0) return ORACLE_EINVAL;
    return ORACLE_OK;
}

/* All rows.  o: (B,H_q,N_q,D), lse: (B,H_q,N_q). */
int oracle_attention_fwd(const double *q, const double *k, const double *v, double *o, double *lse,
                         int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nkv, int64_t D,
                         int causal, double scale, int nthreads)
{
    int rc = check_shape(B, Hq, Hkv, Nq, Nkv, D);
    if (rc) return rc;
    if (!q || !k || !v || !o || !lse) return ORACLE_EINVAL;
    job_t J = {q, k, v, o, lse, B, Hq, Hkv, Nq, Nkv, D, causal ? 1 : 0, scale, NULL, 0, 0, 0};
    return run_threads(&J, B * Hq * Nq, nthreads);
}

/* Selected rows only: sel holds nsel triples (b, h, i); o_rows is (nsel, D)
 * and lse_rows is (nsel).  Used to check sampled rows of workloads whose full
 * output would take the oracle too long. */
int oracle_attention_rows(const double *q, const double *k, const double *v,
                          int64_t B, int64_t Hq, int64_t Hkv, int64_t Nq, int64_t Nkv, int64_t D,
                          int causal, double scale, const int64_t *sel, int64_t nsel,
                          double *o_rows, double *lse_rows, int nthreads)
{
    int rc = check_shape(B, Hq, Hkv, Nq, Nkv, D);
    if (rc) return rc;
    if (!q || !k || !v || !sel || !o_rows || !lse_rows || nsel < 0) return ORACLE_EINVAL;
    for (int64_t r = 0; r < nsel; ++r) {
        if (sel[3 * r] < 0 || sel[3 * r] >= B || sel[3 * r + 1] < 0 || sel[3 * r + 1] >= Hq ||
            sel[3 * r + 2] < 0 || sel[3 * r + 2] >= Nq)
            return ORACLE_EINVAL;
    }
    job_t J = {q, k, v, o_rows, lse_rows, B, Hq, Hkv, Nq, Nkv, D, causal ? 1 : 0, scale, sel, 0, 0, 0};
    return run_threads(&J, nsel, nthreads);
}
