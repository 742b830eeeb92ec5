/*
 * oracle.c -- float64 CPU reference for exact scaled-dot-product softmax
 * attention (decode and causal prefill), for split-KV partials, and for
 * the log-sum-exp merge of partials.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this library.  The CUDA library shares no code,
 * header, table or helper with it, and neither includes the other.
 *
 * What it computes
 * ----------------
 * Attention glossary (jisaku.com/glossary/attention), section "basic
 * concepts and operating principle": a query takes the inner product with
 * every key to give a score, softmax turns the scores into weights, and
 * the output is the weight-averaged value vector.  The Tree Attention
 * explainer (aibr.jp/archives/143699), section 2, stresses that the
 * tree-parallel method is exact -- it changes the parallel strategy, not
 * the result -- so this oracle is that definition written out, with no
 * tiling, blocking or reordering:
 *
 *   s_j   = scale * sum_d q[d] * k[j][d]            for the attended keys j
 *   m     = max_j s_j
 *   lse   = m + ln( sum_j exp(s_j - m) )            (natural log, scaled logits)
 *   out_d = sum_j exp(s_j - lse) * v[j][d]
 *
 * The log-sum-exp is the "energy" whose gradient gives attention in the
 * Tree Attention explainer, sections 1 and 3; the same explainer reduces
 * it along the sequence axis as an associative tree.  The partial of a
 * chunk C of keys and the merge of partials are
 *
 *   partial(C) = (m_C, l_C, o_C),  m_C = max_{j in C} s_j,
 *                l_C = sum_{j in C} exp(s_j - m_C),
 *                o_C = sum_{j in C} exp(s_j - m_C) v_j       (unnormalised)
 *   merge:      m* = max_i m_i,  l* = sum_i l_i exp(m_i - m*),
 *               o* = sum_i o_i exp(m_i - m*),
 *               out = o* / l*,   lse = m* + ln l*.
 *   An empty chunk is (m = -inf, l = 0, o = 0) and carries weight 0.
 *
 * Readings where the pages are silent: query head h reads KV head
 * floor(h / (Hq/Hkv)); an empty attended set gives out = 0, lse = -inf;
 * causal prefill is top-left aligned with the diagonal included (query i
 * attends keys 0..i).
 *
 * Inputs arrive as the exact bf16 or fp32 values the GPU sees and are
 * widened to double element by element (exact), so input rounding is not
 * counted as error.  Parity: pinned (see the tests that check this file
 * against closed forms, brute force and library routines).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F64 = 2 };
enum { ORACLE_OK = 0, ORACLE_BAD_ARG = 1, ORACLE_NO_MEMORY = 2 };

/* Widen element i of a bf16 (raw bits), fp32 or fp64 array to double
 * (fp64 carries already-widened values, e.g. a dequantised cache). */
static double widen(const void *base, int dtype, size_t i)
{
    if (dtype == ORACLE_F64)
        return ((const double *)base)[i];
    if (dtype == ORACLE_F32)
        return (double)((const float *)base)[i];
    uint32_t bits = (uint32_t)((const uint16_t *)base)[i] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

/* Scores s_j = scale * <q, k_j> for keys j in [j0, j1) of one KV head. */
static void scores(const double *q, const void *k, int kv_dtype, size_t kv_base,
                   long j0, long j1, int D, double scale, double *s)
{
    for (long j = j0; j < j1; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += q[d] * widen(k, kv_dtype, kv_base + (size_t)j * D + d);
        s[j - j0] = scale * dot;
    }
}

/* Full attention of one query over keys [0, L) of one KV head. */
static void attend(const double *q, const void *k, const void *v, int kv_dtype,
                   size_t kv_base, long L, int D, double scale, double *s,
                   double *out, double *lse)
{
    if (L <= 0) {
        for (int d = 0; d < D; ++d)
            out[d] = 0.0;
        *lse = -INFINITY;
        return;
    }
    scores(q, k, kv_dtype, kv_base, 0, L, D, scale, s);
    double m = -INFINITY;
    for (long j = 0; j < L; ++j)
        if (s[j] > m)
            m = s[j];
    double sum = 0.0;
    for (long j = 0; j < L; ++j)
        sum += exp(s[j] - m);
    double lse_v = m + log(sum);
    for (int d = 0; d < D; ++d)
        out[d] = 0.0;
    for (long j = 0; j < L; ++j) {
        double w = exp(s[j] - lse_v);
        for (int d = 0; d < D; ++d)
            out[d] += w * widen(v, kv_dtype, kv_base + (size_t)j * D + d);
    }
    *lse = lse_v;
}

/* ---------------------------------------------------------------- threads */

typedef struct {
    int kind; /* 0 = decode rows, 1 = causal prefill rows */
    const void *q, *k, *v;
    int q_dtype, kv_dtype;
    long B, Hq, Hkv, S, D;
    double scale;
    const int32_t *seqlens;
    const int64_t *rows;
    long n_rows;
    double *out, *lse;
    long next; /* shared work counter */
    int status;
    pthread_mutex_t lock;
} job_t;

static long take_row(job_t *job)
{
    pthread_mutex_lock(&job->lock);
    long r = job->next++;
    pthread_mutex_unlock(&job->lock);
    return r;
}

static void *worker(void *arg)
{
    job_t *job = (job_t *)arg;
    long D = job->D, S = job->S;
    double *qd = (double *)malloc(sizeof(double) * D);
    double *s = (double *)malloc(sizeof(double) * (S > 0 ? S : 1));
    if (!qd || !s) {
        free(qd);
        free(s);
        pthread_mutex_lock(&job->lock);
        job->status = ORACLE_NO_MEMORY;
        pthread_mutex_unlock(&job->lock);
        return NULL;
    }
    long G = job->Hq / job->Hkv;
    for (;;) {
        long r = take_row(job);
        if (r >= job->n_rows)
            break;
        long id = job->rows ? (long)job->rows[r] : r;
        long b, h, L;
        size_t q_base;
        if (job->kind == 0) { /* decode: id = b*Hq + h */
            b = id / job->Hq;
            h = id % job->Hq;
            L = job->seqlens ? job->seqlens[b] : S;
            q_base = (size_t)id * D;
        } else { /* prefill: id = (b*Hq + h)*S + i, keys 0..i */
            long bh = id / S;
            long i = id % S;
            b = bh / job->Hq;
            h = bh % job->Hq;
            L = i + 1;
            q_base = (size_t)id * D;
        }
        for (long d = 0; d < D; ++d)
            qd[d] = widen(job->q, job->q_dtype, q_base + d);
        size_t kv_base = ((size_t)b * job->Hkv + (size_t)(h / G)) * (size_t)S * D;
        attend(qd, job->k, job->v, job->kv_dtype, kv_base, L, (int)D, job->scale, s,
               job->out + (size_t)r * D, job->lse + r);
    }
    free(qd);
    free(s);
    return NULL;
}

static int run_job(job_t *job, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 1024)
        nthreads = 1024;
    pthread_mutex_init(&job->lock, NULL);
    job->next = 0;
    job->status = ORACLE_OK;
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
    if (!tid)
        return ORACLE_NO_MEMORY;
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&tid[t], NULL, worker, job) != 0)
            break;
        ++started;
    }
    if (started == 0)
        worker(job);
    for (int t = 0; t < started; ++t)
        pthread_join(tid[t], NULL);
    free(tid);
    pthread_mutex_destroy(&job->lock);
    return job->status;
}

/* ---------------------------------------------------------------- exports */

/*
 * Decode: one query per (b, h) attends keys [0, L_b) of its KV head,
 * L_b = seqlens[b] (host array, may be NULL meaning S).
 * q [B,Hq,D]; k, v [B,Hkv,S,D].  rows: optional list of b*Hq + h to
 * compute (NULL = all B*Hq in order).  out [n_rows, D], lse [n_rows].
 */
int oracle_decode(const void *q, int q_dtype, const void *k, const void *v, int kv_dtype,
                  long B, long Hq, long Hkv, long S, long D, double scale,
                  const int32_t *seqlens, const int64_t *rows, long n_rows,
                  double *out, double *lse, int nthreads)
{
    if (B < 1 || Hq < 1 || Hkv < 1 || Hq % Hkv || S < 0 || D < 1 || !q || !k || !v || !out || !lse)
        return ORACLE_BAD_ARG;
    if (seqlens)
        for (long b = 0; b < B; ++b)
            if (seqlens[b] < 0 || seqlens[b] > S)
                return ORACLE_BAD_ARG;
    if (!rows)
        n_rows = B * Hq;
    for (long r = 0; rows && r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= B * Hq)
            return ORACLE_BAD_ARG;
    job_t job = {0};
    job.kind = 0;
    job.q = q; job.k = k; job.v = v;
    job.q_dtype = q_dtype; job.kv_dtype = kv_dtype;
    job.B = B; job.Hq = Hq; job.Hkv = Hkv; job.S = S; job.D = D;
    job.scale = scale; job.seqlens = seqlens; job.rows = rows; job.n_rows = n_rows;
    job.out = out; job.lse = lse;
    return run_job(&job, nthreads);
}

/*
 * Causal prefill: query row i of head h attends keys 0..i of KV head
 * floor(h/G).  q [B,H,S,D]; k, v [B,Hkv,S,D].  rows: optional list of
 * (b*H + h)*S + i (NULL = all).  out [n_rows, D], lse [n_rows].
 */
int oracle_prefill_causal(const void *q, const void *k, const void *v, int dtype,
                          long B, long H, long Hkv, long S, long D, double scale,
                          const int64_t *rows, long n_rows, double *out, double *lse,
                          int nthreads)
{
    if (B < 1 || H < 1 || Hkv < 1 || H % Hkv || S < 1 || D < 1 || !q || !k || !v || !out || !lse)
        return ORACLE_BAD_ARG;
    if (!rows)
        n_rows = B * H * S;
    for (long r = 0; rows && r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= B * H * S)
            return ORACLE_BAD_ARG;
    job_t job = {0};
    job.kind = 1;
    job.q = q; job.k = k; job.v = v;
    job.q_dtype = dtype; job.kv_dtype = dtype;
    job.B = B; job.Hq = H; job.Hkv = Hkv; job.S = S; job.D = D;
    job.scale = scale; job.seqlens = NULL; job.rows = rows; job.n_rows = n_rows;
    job.out = out; job.lse = lse;
    return run_job(&job, nthreads);
}

/*
 * Split-KV partials of one decode row (b, h): chunk c covers keys
 * [bounds[c], bounds[c+1]) intersected with [0, L_b).  Writes m[c], l[c]
 * and o[c][D] as defined in the header comment; an empty chunk gives
 * (-inf, 0, 0).  bounds has N+1 entries, non-decreasing, within [0, S].
 */
int oracle_decode_partials(const void *q, int q_dtype, const void *k, const void *v,
                           int kv_dtype, long B, long Hq, long Hkv, long S, long D,
                           double scale, const int32_t *seqlens, long b, long h,
                           const int64_t *bounds, long N, double *m, double *l, double *o)
{
    if (b < 0 || b >= B || h < 0 || h >= Hq || Hq % Hkv || N < 1 || !bounds)
        return ORACLE_BAD_ARG;
    for (long c = 0; c < N; ++c)
        if (bounds[c] < 0 || bounds[c] > bounds[c + 1] || bounds[c + 1] > S)
            return ORACLE_BAD_ARG;
    long L = seqlens ? seqlens[b] : S;
    if (L < 0 || L > S)
        return ORACLE_BAD_ARG;
    double *qd = (double *)malloc(sizeof(double) * D);
    double *s = (double *)malloc(sizeof(double) * (S > 0 ? S : 1));
    if (!qd || !s) {
        free(qd);
        free(s);
        return ORACLE_NO_MEMORY;
    }
    for (long d = 0; d < D; ++d)
        qd[d] = widen(q, q_dtype, (size_t)(b * Hq + h) * D + d);
    size_t kv_base = ((size_t)b * Hkv + (size_t)(h / (Hq / Hkv))) * (size_t)S * D;
    for (long c = 0; c < N; ++c) {
        long j0 = bounds[c], j1 = bounds[c + 1] < L ? bounds[c + 1] : L;
        double *oc = o + (size_t)c * D;
        for (long d = 0; d < D; ++d)
            oc[d] = 0.0;
        if (j1 <= j0) {
            m[c] = -INFINITY;
            l[c] = 0.0;
            continue;
        }
        scores(qd, k, kv_dtype, kv_base, j0, j1, (int)D, scale, s);
        double mc = -INFINITY;
        for (long j = 0; j < j1 - j0; ++j)
            if (s[j] > mc)
                mc = s[j];
        double lc = 0.0;
        for (long j = 0; j < j1 - j0; ++j) {
            double w = exp(s[j] - mc);
            lc += w;
            for (long d = 0; d < D; ++d)
                oc[d] += w * widen(v, kv_dtype, kv_base + (size_t)(j0 + j) * D + d);
        }
        m[c] = mc;
        l[c] = lc;
    }
    free(qd);
    free(s);
    return ORACLE_OK;
}

/*
 * Log-sum-exp merge of N partials for each of R rows (Tree Attention
 * explainer, sections 1 and 3: the sequence-axis reduction is associative).
 * m, l [R,N]; o [R,N,D]; out [R,D]; lse [R].  Partials with m = -inf have
 * weight 0; a row whose partials are all empty gives out = 0, lse = -inf.
 */
int oracle_combine(const double *m, const double *l, const double *o, long R, long N, long D,
                   double *out, double *lse)
{
    if (R < 0 || N < 1 || D < 1 || !m || !l || !o || !out || !lse)
        return ORACLE_BAD_ARG;
    for (long r = 0; r < R; ++r) {
        const double *mr = m + (size_t)r * N, *lr = l + (size_t)r * N;
        const double *orow = o + (size_t)r * N * D;
        double *out_r = out + (size_t)r * D;
        double ms = -INFINITY;
        for (long i = 0; i < N; ++i)
            if (mr[i] > ms)
                ms = mr[i];
        for (long d = 0; d < D; ++d)
            out_r[d] = 0.0;
        if (ms == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double ls = 0.0;
        for (long i = 0; i < N; ++i) {
            if (mr[i] == -INFINITY)
                continue;
            double w = exp(mr[i] - ms);
            ls += lr[i] * w;
            for (long d = 0; d < D; ++d)
                out_r[d] += orow[(size_t)i * D + d] * w;
        }
        for (long d = 0; d < D; ++d)
            out_r[d] /= ls;
        lse[r] = ms + log(ls);
    }
    return ORACLE_OK;
}
