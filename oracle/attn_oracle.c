/*
 * attn_oracle.c — plain CPU float64 reference for exact multi-head attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it.  It shares no code with the CUDA library.
 *
 * What it computes (the definition, written out):
 *   For every batch b, head h and query row i < Nq, with K(i) the set of
 *   allowed keys
 *       K(i) = { j < Nk : !causal  or  j <= i }              (top-left causal)
 *       s_j    = scale * sum_x q[i,x] * k[j,x]                 for j in K(i)
 *       m      = max_{j in K(i)} s_j
 *       l      = sum_{j in K(i)} exp(s_j - m)
 *       O[i,:] = sum_{j in K(i)} exp(s_j - m) * v[j,:] / l
 *       LSE[i] = m + log(l)                                    (natural log)
 *
 * Sources, by page:
 *   - "flash_attention_2.cu" (leloykun/flash-hyperbolic-attention-minimal),
 *     forward kernel: S = softmax_scale * Q K^T with the scale applied to the
 *     dot product before the row max; P = exp(S - m); l = row sum of P;
 *     O = P V / l; L = m + log(l); the causal rule keeps key j for query i only
 *     while i >= j; keys and rows past N are excluded.
 *   - "Add Fused Multi-Head Attention example" (JuliaGPU/cuTile.jl PR #16),
 *     masking snippet: masked positions get an additive -Inf, i.e. they drop
 *     out of both the max and the sum.
 *
 * Layout: q [B,H,Nq,d], k and v [B,H,Nk,d], o [B,H,Nq,d], lse [B,H,Nq], all
 * contiguous row-major.  Inputs are float (the exact values the GPU reads:
 * bf16 inputs are widened to float without rounding); every operation here is
 * in double.  exp and log come from the host C library.
 *
 * Functions:
 *   oracle_attn_fwd         the definition above, two passes per row.
 *   oracle_attn_rows        the same definition for a list of rows only.
 *   oracle_attn_probs       the probability matrix P (tiny problems).
 *   oracle_attn_fwd_online  the online-softmax recurrence over key tiles, in
 *                           double; it exists only so the tests can show the
 *                           tiled algorithm equals the definition.
 *   oracle_attn_bwd         the gradients dQ, dK, dV of the forward for an
 *                           upstream gradient dO (see its comment).
 * Every function returns 0 on success and -1 on a bad argument.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* Number of keys query row i may attend to (the set K(i) is 0 .. n-1). */
static long allowed_keys(long i, long Nk, int causal)
{
    if (!causal) return Nk;
    return (i + 1 < Nk) ? (i + 1) : Nk;
}

/* One query row of the definition.  s is scratch of length >= Nk. */
static void attn_row(const float *qrow, const float *kh, const float *vh,
                     long nk, long d, double scale,
                     double *orow, double *lse, double *s)
{
    /* scores, scaled before the max is taken */
    double m = -INFINITY;
    for (long j = 0; j < nk; ++j) {
        double dot = 0.0;
        for (long x = 0; x < d; ++x)
            dot += (double)qrow[x] * (double)kh[j * d + x];
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
    }
    /* second pass: unnormalised probabilities, their sum and P V */
    double l = 0.0;
    for (long x = 0; x < d; ++x) orow[x] = 0.0;
    for (long j = 0; j < nk; ++j) {
        double p = exp(s[j] - m);
        l += p;
        for (long x = 0; x < d; ++x)
            orow[x] += p * (double)vh[j * d + x];
    }
    for (long x = 0; x < d; ++x) orow[x] /= l;
    *lse = m + log(l);
}

/* ---- thread pool over work items ------------------------------------- */

typedef struct {
    const float *q, *k, *v;
    double *o, *lse;
    long B, H, Nq, Nk, d;
    double scale;
    int causal;
    const long *rows; /* NULL: whole heads; else flat row ids bh*Nq+i */
    long nitems;
    long next;        /* next work item (guarded by mu) */
    pthread_mutex_t mu;
} job_t;

static long take_item(job_t *J)
{
    pthread_mutex_lock(&J->mu);
    long it = J->next++;
    pthread_mutex_unlock(&J->mu);
    return it;
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)(J->Nk > 0 ? J->Nk : 1));
    if (!s) return (void *)1;
    for (;;) {
        long it = take_item(J);
        if (it >= J->nitems) break;
        if (J->rows == NULL) {
            /* one (b, h) head per item */
            long bh = it;
            const float *qh = J->q + bh * J->Nq * J->d;
            const float *kh = J->k + bh * J->Nk * J->d;
            const float *vh = J->v + bh * J->Nk * J->d;
            for (long i = 0; i < J->Nq; ++i)
                attn_row(qh + i * J->d, kh, vh, allowed_keys(i, J->Nk, J->causal),
                         J->d, J->scale, J->o + (bh * J->Nq + i) * J->d,
                         J->lse + bh * J->Nq + i, s);
        } else {
            /* one listed row per item; outputs packed in list order */
            long r = J->rows[it];
            long bh = r / J->Nq, i = r % J->Nq;
            attn_row(J->q + r * J->d, J->k + bh * J->Nk * J->d,
                     J->v + bh * J->Nk * J->d, allowed_keys(i, J->Nk, J->causal),
                     J->d, J->scale, J->o + it * J->d, J->lse + it, s);
        }
    }
    free(s);
    return NULL;
}

static int run_job(job_t *J, int nthreads)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 1024) nthreads = 1024;
    if ((long)nthreads > J->nitems) nthreads = (int)(J->nitems > 0 ? J->nitems : 1);
    J->next = 0;
    pthread_mutex_init(&J->mu, NULL);
    pthread_t th[1024];
    int started = 0, rc = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, worker, J) != 0) break;
        ++started;
    }
    if (started == 0) rc = (worker(J) == NULL) ? 0 : -1;
    for (int t = 0; t < started; ++t) {
        void *ret = NULL;
        pthread_join(th[t], &ret);
        if (ret != NULL) rc = -1;
    }
    pthread_mutex_destroy(&J->mu);
    return rc;
}

static int bad_sizes(long B, long H, long Nq, long Nk, long d)
{
    return B < 1 || H < 1 || Nq < 1 || Nk < 1 || d < 1;
}

int oracle_attn_fwd(const float *q, const float *k, const float *v,
                    double *o, double *lse,
                    long B, long H, long Nq, long Nk, long d,
                    double scale, int causal, int nthreads)
{
    if (!q || !k || !v || !o || !lse || bad_sizes(B, H, Nq, Nk, d)) return -1;
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v; J.o = o; J.lse = lse;
    J.B = B; J.H = H; J.Nq = Nq; J.Nk = Nk; J.d = d;
    J.scale = scale; J.causal = causal ? 1 : 0;
    J.rows = NULL; J.nitems = B * H;
    return run_job(&J, nthreads);
}

int oracle_attn_rows(const float *q, const float *k, const float *v,
                     const long *rows, long nrows, double *o, double *lse,
                     long B, long H, long Nq, long Nk, long d,
                     double scale, int causal, int nthreads)
{
    if (!q || !k || !v || !rows || !o || !lse || nrows < 0 ||
        bad_sizes(B, H, Nq, Nk, d)) return -1;
    for (long r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= B * H * Nq) return -1;
    job_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v; J.o = o; J.lse = lse;
    J.B = B; J.H = H; J.Nq = Nq; J.Nk = Nk; J.d = d;
    J.scale = scale; J.causal = causal ? 1 : 0;
    J.rows = rows; J.nitems = nrows;
    return run_job(&J, nthreads);
}

/* P[b,h,i,j] = exp(s_j - m) / l for allowed keys, 0 for excluded ones. */
int oracle_attn_probs(const float *q, const float *k, double *p,
                      long B, long H, long Nq, long Nk, long d,
                      double scale, int causal)
{
    if (!q || !k || !p || bad_sizes(B, H, Nq, Nk, d)) return -1;
    for (long bh = 0; bh < B * H; ++bh) {
        for (long i = 0; i < Nq; ++i) {
            const float *qrow = q + (bh * Nq + i) * d;
            const float *kh = k + bh * Nk * d;
            double *prow = p + (bh * Nq + i) * Nk;
            long nk = allowed_keys(i, Nk, causal);
            double m = -INFINITY;
            for (long j = 0; j < nk; ++j) {
                double dot = 0.0;
                for (long x = 0; x < d; ++x)
                    dot += (double)qrow[x] * (double)kh[j * d + x];
                prow[j] = scale * dot;
                if (prow[j] > m) m = prow[j];
            }
            double l = 0.0;
            for (long j = 0; j < nk; ++j) {
                prow[j] = exp(prow[j] - m);
                l += prow[j];
            }
            for (long j = 0; j < nk; ++j) prow[j] /= l;
            for (long j = nk; j < Nk; ++j) prow[j] = 0.0;
        }
    }
    return 0;
}

/*
 * The online-softmax recurrence, in double, over key tiles of bc keys
 * ("flash_attention_2.cu", forward kernel; the swapped loop order of
 * "parallel execution of read/write operations (paper vs implementation)":
 * each query row starts from m = -inf, l = 0, O = 0 and visits key tiles in
 * order).  For tile t with scores s_j:
 *     m_new = max(m, max_j s_j)
 *     l     = exp(m - m_new) * l + sum_j exp(s_j - m_new)
 *     O     = exp(m - m_new) * O + sum_j exp(s_j - m_new) * v_j
 *     m     = m_new
 * and at the end O /= l, LSE = m + log(l).
 */
int oracle_attn_fwd_online(const float *q, const float *k, const float *v,
                           double *o, double *lse,
                           long B, long H, long Nq, long Nk, long d,
                           double scale, int causal, long bc)
{
    if (!q || !k || !v || !o || !lse || bc < 1 || bad_sizes(B, H, Nq, Nk, d))
        return -1;
    double *s = (double *)malloc(sizeof(double) * (size_t)bc);
    if (!s) return -1;
    for (long bh = 0; bh < B * H; ++bh) {
        const float *kh = k + bh * Nk * d;
        const float *vh = v + bh * Nk * d;
        for (long i = 0; i < Nq; ++i) {
            const float *qrow = q + (bh * Nq + i) * d;
            double *orow = o + (bh * Nq + i) * d;
            long nk = allowed_keys(i, Nk, causal);
            double m = -INFINITY, l = 0.0;
            for (long x = 0; x < d; ++x) orow[x] = 0.0;
            for (long j0 = 0; j0 < nk; j0 += bc) {
                long n = (nk - j0 < bc) ? (nk - j0) : bc;
                double mt = -INFINITY;
                for (long c = 0; c < n; ++c) {
                    double dot = 0.0;
                    for (long x = 0; x < d; ++x)
                        dot += (double)qrow[x] * (double)kh[(j0 + c) * d + x];
                    s[c] = scale * dot;
                    if (s[c] > mt) mt = s[c];
                }
                double m_new = (mt > m) ? mt : m;
                double alpha = exp(m - m_new); /* exp(-inf) = 0 on the first tile */
                double lt = 0.0;
                for (long x = 0; x < d; ++x) orow[x] *= alpha;
                for (long c = 0; c < n; ++c) {
                    double p = exp(s[c] - m_new);
                    lt += p;
                    for (long x = 0; x < d; ++x)
                        orow[x] += p * (double)vh[(j0 + c) * d + x];
                }
                l = alpha * l + lt;
                m = m_new;
            }
            for (long x = 0; x < d; ++x) orow[x] /= l;
            lse[bh * Nq + i] = m + log(l);
        }
    }
    free(s);
    return 0;
}

/*
 * Gradients of the forward above for an upstream gradient dO (the quantities
 * of the backward kernel of "flash_attention_2.cu"), from the definition:
 *   P_ij  = softmax over allowed keys j of s_ij = scale * q_i . k_j
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = dO_i . v_j
 *   D_i   = sum_j P_ij dP_ij
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale * sum_j dS_ij k_j
 *   dK_j  = scale * sum_i dS_ij q_i
 * The page forms D_i as rowsum(dO_i * O_i); D_i = sum_j P_ij dP_ij is the same
 * number because O_i = sum_j P_ij v_j, and needs no forward output.
 * Excluded keys have P_ij = 0 and take no part.  Outputs are float64 with the
 * layouts of q (dq) and k (dk, dv).
 */
typedef struct {
    const float *q, *k, *v, *dout;
    double *dq, *dk, *dv;
    long B, H, Nq, Nk, d;
    double scale;
    int causal;
    long next;
    pthread_mutex_t mu;
} bjob_t;

static void bwd_head(bjob_t *J, long bh, double *p, double *dp)
{
    const long Nq = J->Nq, Nk = J->Nk, d = J->d;
    const float *qh = J->q + bh * Nq * d, *kh = J->k + bh * Nk * d;
    const float *vh = J->v + bh * Nk * d, *doh = J->dout + bh * Nq * d;
    double *dqh = J->dq + bh * Nq * d, *dkh = J->dk + bh * Nk * d, *dvh = J->dv + bh * Nk * d;
    for (long x = 0; x < Nk * d; ++x) { dkh[x] = 0.0; dvh[x] = 0.0; }
    for (long i = 0; i < Nq; ++i) {
        const float *qi = qh + i * d, *doi = doh + i * d;
        const long nk = allowed_keys(i, Nk, J->causal);
        /* probabilities of row i (two passes, as the forward) */
        double m = -INFINITY;
        for (long j = 0; j < nk; ++j) {
            double dot = 0.0;
            for (long x = 0; x < d; ++x) dot += (double)qi[x] * (double)kh[j * d + x];
            p[j] = J->scale * dot;
            if (p[j] > m) m = p[j];
        }
        double l = 0.0;
        for (long j = 0; j < nk; ++j) { p[j] = exp(p[j] - m); l += p[j]; }
        for (long j = 0; j < nk; ++j) p[j] /= l;
        /* dP, D */
        double D = 0.0;
        for (long j = 0; j < nk; ++j) {
            double dot = 0.0;
            for (long x = 0; x < d; ++x) dot += (double)doi[x] * (double)vh[j * d + x];
            dp[j] = dot;
            D += p[j] * dot;
        }
        /* dS and the three gradients */
        for (long x = 0; x < d; ++x) dqh[i * d + x] = 0.0;
        for (long j = 0; j < nk; ++j) {
            const double ds = p[j] * (dp[j] - D);
            for (long x = 0; x < d; ++x) {
                dqh[i * d + x] += J->scale * ds * (double)kh[j * d + x];
                dkh[j * d + x] += J->scale * ds * (double)qi[x];
                dvh[j * d + x] += p[j] * (double)doi[x];
            }
        }
    }
}

static void *bwd_worker(void *arg)
{
    bjob_t *J = (bjob_t *)arg;
    double *p = (double *)malloc(sizeof(double) * (size_t)J->Nk);
    double *dp = (double *)malloc(sizeof(double) * (size_t)J->Nk);
    if (!p || !dp) { free(p); free(dp); return (void *)1; }
    for (;;) {
        pthread_mutex_lock(&J->mu);
        long bh = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (bh >= J->B * J->H) break;
        bwd_head(J, bh, p, dp);
    }
    free(p);
    free(dp);
    return NULL;
}

int oracle_attn_bwd(const float *q, const float *k, const float *v, const float *dout,
                    double *dq, double *dk, double *dv,
                    long B, long H, long Nq, long Nk, long d,
                    double scale, int causal, int nthreads)
{
    if (!q || !k || !v || !dout || !dq || !dk || !dv || bad_sizes(B, H, Nq, Nk, d)) return -1;
    bjob_t J;
    memset(&J, 0, sizeof J);
    J.q = q; J.k = k; J.v = v; J.dout = dout; J.dq = dq; J.dk = dk; J.dv = dv;
    J.B = B; J.H = H; J.Nq = Nq; J.Nk = Nk; J.d = d; J.scale = scale;
    J.causal = causal ? 1 : 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 1024) nthreads = 1024;
    if ((long)nthreads > B * H) nthreads = (int)(B * H);
    pthread_mutex_init(&J.mu, NULL);
    pthread_t th[1024];
    int started = 0, rc = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (pthread_create(&th[t], NULL, bwd_worker, &J) != 0) break;
        ++started;
    }
    if (started == 0) rc = (bwd_worker(&J) == NULL) ? 0 : -1;
    for (int t = 0; t < started; ++t) {
        void *ret = NULL;
        pthread_join(th[t], &ret);
        if (ret != NULL) rc = -1;
    }
    pthread_mutex_destroy(&J.mu);
    return rc;
}
