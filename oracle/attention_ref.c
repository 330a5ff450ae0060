/*
 * Plain fp64 CPU attention forward -- TEST INFRASTRUCTURE, not product code.
 *
 * Only the tests, the package's smoke check and the benchmark's CPU-baseline
 * leg may load this library.  It shares no code with the CUDA path.
 *
 * What it computes is the definition of scaled dot-product attention, one
 * query row at a time, with the score row S and the probability row P
 * materialised in full (FlashAttention from Scratch, sec. 2 "Begin with one
 * attention row" and sec. 5 "Run the math before writing a GPU kernel";
 * FlashAttention Cheat Sheet, sec. 1 "The whole operation"):
 *
 *   s_j   = scale * sum_d q[d] * k_j[d]
 *   s_j   = -inf  if causal and key position j > i + (Lk - Lq)
 *           (bottom-right alignment: the queries are the last Lq positions
 *            of the Lk-long key sequence; sec. 5 "Rectangular causal masking")
 *   m     = max_j s_j
 *   p_j   = exp(s_j - m),  l = sum_j p_j,  P_j = p_j / l     (safe softmax)
 *   o     = sum_j P_j v_j
 *   lse   = m + ln(l)                                         (natural log)
 *
 * A row whose keys are all masked returns o = 0 and lse = -inf
 * (sec. 4.4 "Handle the empty state deliberately").
 *
 * GQA: query head h reads KV head h / (Hq / Hkv)
 * (sec. 9.2 "GQA and MQA change decode traffic").
 *
 * Queries and keys have D elements per row, values and outputs Dv; the two
 * differ in the (192, 128) case of the FlashAttention-4 benchmarks
 * (FlashAttention-4: Blackwell Attention Kernel Co-Design, "How we know").
 *
 * Inputs are fp32 arrays holding exact bf16 values; every product and sum is
 * done in double.  Element (b, h, i, d) of a tensor X lives at
 * X + b*xs[0] + h*xs[1] + i*xs[2] + d, so the same routine reads the dense
 * [B,H,L,D] layout and one sequence of a packed [T,H,D] batch.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    const float *q, *k, *v;
    int64_t qs[3], ks[3], vs[3];
    int B, Hq, Hkv, Lq, Lk, D, Dv;
    int causal;
    double scale;
    const int64_t *rows; /* flat row ids (b*Hq + h)*Lq + i, or NULL = all */
    int64_t nrows;
    double *o;   /* nrows x Dv */
    double *lse; /* nrows */
    int64_t begin, end;
    int status;
} job_t;

static void one_row(const job_t *J, int64_t flat, double *S, double *P, double *o, double *lse)
{
    const int64_t i = flat % J->Lq;
    const int64_t bh = flat / J->Lq;
    const int h = (int)(bh % J->Hq);
    const int b = (int)(bh / J->Hq);
    const int group = J->Hq / J->Hkv;
    const int hk = h / group;
    const float *qrow = J->q + b * J->qs[0] + h * J->qs[1] + i * J->qs[2];
    const float *kb = J->k + b * J->ks[0] + hk * J->ks[1];
    const float *vb = J->v + b * J->vs[0] + hk * J->vs[1];
    const int64_t last_allowed = i + (int64_t)J->Lk - (int64_t)J->Lq;

    /* score row S (materialised) */
    for (int64_t j = 0; j < J->Lk; ++j) {
        if (J->causal && j > last_allowed) {
            S[j] = -INFINITY;
            continue;
        }
        const float *krow = kb + j * J->ks[2];
        double acc = 0.0;
        for (int d = 0; d < J->D; ++d) acc += (double)qrow[d] * (double)krow[d];
        S[j] = J->scale * acc;
    }
    double m = -INFINITY;
    for (int64_t j = 0; j < J->Lk; ++j)
        if (S[j] > m) m = S[j];
    if (m == -INFINITY) { /* every key masked */
        for (int d = 0; d < J->Dv; ++d) o[d] = 0.0;
        *lse = -INFINITY;
        return;
    }
    /* probability row P (materialised) */
    double l = 0.0;
    for (int64_t j = 0; j < J->Lk; ++j) {
        P[j] = exp(S[j] - m);
        l += P[j];
    }
    for (int64_t j = 0; j < J->Lk; ++j) P[j] /= l;
    /* o = P V */
    for (int d = 0; d < J->Dv; ++d) o[d] = 0.0;
    for (int64_t j = 0; j < J->Lk; ++j) {
        if (P[j] == 0.0) continue; /* masked key: its term is exactly zero */
        const float *vrow = vb + j * J->vs[2];
        for (int d = 0; d < J->Dv; ++d) o[d] += P[j] * (double)vrow[d];
    }
    *lse = m + log(l);
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    double *S = (double *)malloc(sizeof(double) * (size_t)J->Lk);
    double *P = (double *)malloc(sizeof(double) * (size_t)J->Lk);
    if (!S || !P) {
        J->status = 1;
        free(S);
        free(P);
        return NULL;
    }
    for (int64_t r = J->begin; r < J->end; ++r) {
        const int64_t flat = J->rows ? J->rows[r] : r;
        one_row(J, flat, S, P, J->o + r * J->Dv, J->lse + r);
    }
    free(S);
    free(P);
    return NULL;
}

int oracle_num_cpus(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * Computes nrows output rows (all B*Hq*Lq rows when rows == NULL) into
 * o[nrows][Dv] and lse[nrows].  Returns 0 on success, nonzero on bad
 * arguments or allocation failure.  nthreads <= 0 uses every online CPU.
 */
int oracle_attention_rows(const float *q, const float *k, const float *v,
                          const int64_t *q_strides, const int64_t *k_strides,
                          const int64_t *v_strides, int B, int Hq, int Hkv, int Lq,
                          int Lk, int D, int Dv, int causal, double scale, const int64_t *rows,
                          int64_t nrows, double *o, double *lse, int nthreads)
{
    if (!q || !k || !v || !o || !lse || B <= 0 || Hq <= 0 || Hkv <= 0 || Lq <= 0 ||
        Lk <= 0 || D <= 0 || Dv <= 0 || Hq % Hkv != 0)
        return 2;
    if (!rows) nrows = (int64_t)B * Hq * Lq;
    if (nrows <= 0) return 0;
    if (nthreads <= 0) nthreads = oracle_num_cpus();
    if (nthreads > nrows) nthreads = (int)nrows;

    job_t base;
    memset(&base, 0, sizeof(base));
    base.q = q;
    base.k = k;
    base.v = v;
    memcpy(base.qs, q_strides, sizeof(base.qs));
    memcpy(base.ks, k_strides, sizeof(base.ks));
    memcpy(base.vs, v_strides, sizeof(base.vs));
    base.B = B;
    base.Hq = Hq;
    base.Hkv = Hkv;
    base.Lq = Lq;
    base.Lk = Lk;
    base.D = D;
    base.Dv = Dv;
    base.causal = causal;
    base.scale = scale;
    base.rows = rows;
    base.nrows = nrows;
    base.o = o;
    base.lse = lse;

    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *tids = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    char *started = (char *)calloc((size_t)nthreads, 1);
    if (!jobs || !tids || !started) {
        free(jobs);
        free(tids);
        free(started);
        return 1;
    }
    int status = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].begin = nrows * t / nthreads;
        jobs[t].end = nrows * (t + 1) / nthreads;
        if (pthread_create(&tids[t], NULL, worker, &jobs[t]) == 0)
            started[t] = 1;
        else
            worker(&jobs[t]); /* run inline if a thread cannot start */
    }
    for (int t = 0; t < nthreads; ++t) {
        if (started[t]) pthread_join(tids[t], NULL);
        status |= jobs[t].status;
    }
    free(jobs);
    free(tids);
    free(started);
    return status;
}
