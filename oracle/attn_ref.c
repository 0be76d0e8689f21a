/*
 * CPU fp64 oracle for the attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or
 * load this file; only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it. It shares no code, header, table or helper with the
 * CUDA library.
 *
 * Sources (the three web pages on FlashAttention):
 *  - MUSA SDK programming guide, "FlashAttention 优化", section
 *    "标准 Self-Attention 的问题 / 计算流程": Attention(Q,K,V) =
 *    softmax(Q K^T / sqrt(d)) V computed as S = Q K^T, P = softmax(S), O = P V.
 *  - same page, "online softmax / 标准 Softmax 回顾": the three-pass safe
 *    softmax m = max(S), Z = sum exp(S - m), P = exp(S - m) / Z, and
 *    "数值稳定性" (subtracting the row maximum).
 *  - same page, "FlashAttention 完整算法", formula steps 1-4 and the flow
 *    chart: the tiled recurrence over key blocks (m, l, O updated per block,
 *    O divided by l at the end).
 *
 * Reading taken where the pages are silent: the scale is an argument applied
 * to the dot product (s = scale * q.k); LSE = m + ln Z in natural log; row
 * statistics are per row.
 *
 * Layouts: Q [BH, Nq, d], K and V [BH, Nk, d], O [BH, Nq, d], LSE [BH, Nq],
 * all row-major fp64. Build: gcc -O2 (no -ffast-math), libm exp/log.
 *
 * oracle_attn_bwd_fp64 is the backward pass (gradients of Q, K, V for a given
 * dO) written out from the chain rule on the same definition, P recomputed
 * from the saved LSE; oracle_attn_bwd_masked_fp64 is the same with the causal
 * and key-length masks.
 *
 * ORACLE_MUTANT (compile-time, default 0) plants one deliberate mistake so
 * the pin tests can show that each such mistake is caught. Mutant builds are
 * made only by the tests, in a temporary directory.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

typedef struct {
    const double *Q, *K, *V;
    double *O, *LSE;
    long BH, Nq, Nk, d;
    double scale;
    long row_begin, row_end; /* flattened (bh, i) rows */
    /* online model */
    long block_n;
    double tau;
    double *trace_m, *trace_l; /* [BH*Nq, nblocks] or NULL */
    int ok;
} job_t;

/* s_j = scale * sum_k q_k * k_jk for one query row against all Nk keys. */
static void scores_row(const double *q, const double *K, long Nk, long d, double scale, double *s)
{
    for (long j = 0; j < Nk; ++j) {
        const double *kj = K + j * d;
        double acc = 0.0;
        for (long c = 0; c < d; ++c) {
#if ORACLE_MUTANT == 1 /* wrong index: q's components shifted against k's */
            acc += q[(c + 1) % d] * kj[c];
#else
            acc += q[c] * kj[c];
#endif
        }
#if ORACLE_MUTANT == 2 /* scale dropped */
        s[j] = acc;
#else
        s[j] = scale * acc;
#endif
    }
}

/* The three-pass definition for one row: max, normaliser, weighted sum. */
static void three_pass_row(const double *s, const double *V, long Nk, long d, double *o, double *lse)
{
    double m = -INFINITY;
    for (long j = 0; j < Nk; ++j)
        if (s[j] > m) m = s[j];
#if ORACLE_MUTANT == 3 /* max subtraction dropped */
    m = 0.0;
#endif
    double Z = 0.0;
    for (long j = 0; j < Nk; ++j) {
#if ORACLE_MUTANT == 4 /* sign error in the exponent */
        Z += exp(m - s[j]);
#else
        Z += exp(s[j] - m);
#endif
    }
    for (long c = 0; c < d; ++c) o[c] = 0.0;
    for (long j = 0; j < Nk; ++j) {
#if ORACLE_MUTANT == 4
        double p = exp(m - s[j]) / Z;
#else
        double p = exp(s[j] - m) / Z;
#endif
#if ORACLE_MUTANT == 5 /* off-by-one value row */
        const double *vj = V + ((j + 1) % Nk) * d;
#else
        const double *vj = V + j * d;
#endif
        for (long c = 0; c < d; ++c) o[c] += p * vj[c];
    }
#if ORACLE_MUTANT == 6 /* max term dropped from the logsumexp */
    *lse = log(Z);
#else
    *lse = m + log(Z);
#endif
}

static void *three_pass_worker(void *arg)
{
    job_t *jb = (job_t *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)(jb->Nk > 0 ? jb->Nk : 1));
    if (!s) { jb->ok = 0; return NULL; }
    for (long r = jb->row_begin; r < jb->row_end; ++r) {
        long bh = r / jb->Nq;
        const double *q = jb->Q + r * jb->d;
        const double *K = jb->K + bh * jb->Nk * jb->d;
        const double *V = jb->V + bh * jb->Nk * jb->d;
#if ORACLE_MUTANT == 7 /* transposed score matrix: s_ij taken as q_j . k_i */
        {
            long i = r % jb->Nq;
            const double *Qh = jb->Q + bh * jb->Nq * jb->d;
            for (long j = 0; j < jb->Nk; ++j) {
                const double *qj = Qh + (j % jb->Nq) * jb->d, *ki = K + (i % jb->Nk) * jb->d;
                double acc = 0.0;
                for (long c = 0; c < jb->d; ++c) acc += qj[c] * ki[c];
                s[j] = jb->scale * acc;
            }
        }
#else
        scores_row(q, K, jb->Nk, jb->d, jb->scale, s);
#endif
        three_pass_row(s, V, jb->Nk, jb->d, jb->O + r * jb->d, jb->LSE + r);
    }
    free(s);
    jb->ok = 1;
    return NULL;
}

/*
 * Online (tiled) model of the same result, one row at a time, in fp64:
 * keys are taken in blocks of block_n. For each block the block row max is
 * found, the running max m is replaced by max(m, block max) and the running
 * denominator l and the unnormalised output o are multiplied by
 * exp(m_old - m_new) before the block's exp(s - m) terms are added; at the
 * end o is divided by l (formula steps 3a-3f and 4).
 *
 * tau >= 0 makes the replacement lazy: the reference max is only moved when
 * the block max exceeds it by more than tau (natural-log units) or on the
 * first block. tau = 0 is the pages' eager update. Because l and o always
 * share one reference max, the final o / l and m + ln l are the same for
 * every tau up to rounding.
 */
static void *online_worker(void *arg)
{
    job_t *jb = (job_t *)arg;
    long nb = (jb->Nk + jb->block_n - 1) / jb->block_n;
    double *s = (double *)malloc(sizeof(double) * (size_t)jb->block_n);
    double *o = (double *)malloc(sizeof(double) * (size_t)jb->d);
    if (!s || !o) { free(s); free(o); jb->ok = 0; return NULL; }
    for (long r = jb->row_begin; r < jb->row_end; ++r) {
        long bh = r / jb->Nq;
        const double *q = jb->Q + r * jb->d;
        const double *K = jb->K + bh * jb->Nk * jb->d;
        const double *V = jb->V + bh * jb->Nk * jb->d;
        double m = -INFINITY, l = 0.0;
        for (long c = 0; c < jb->d; ++c) o[c] = 0.0;
        for (long b = 0; b < nb; ++b) {
            long j0 = b * jb->block_n;
            long nj = jb->Nk - j0 < jb->block_n ? jb->Nk - j0 : jb->block_n;
            scores_row(q, K + j0 * jb->d, nj, jb->d, jb->scale, s);
            double mb = -INFINITY;
            for (long j = 0; j < nj; ++j)
                if (s[j] > mb) mb = s[j];
            double m_new = mb > m ? mb : m;
            if (b == 0 || m_new - m > jb->tau) {
                double alpha = (b == 0) ? 0.0 : exp(m - m_new);
                l *= alpha;
                for (long c = 0; c < jb->d; ++c) o[c] *= alpha;
                m = m_new;
            }
            for (long j = 0; j < nj; ++j) {
                double p = exp(s[j] - m);
                l += p;
                const double *vj = V + (j0 + j) * jb->d;
                for (long c = 0; c < jb->d; ++c) o[c] += p * vj[c];
            }
            if (jb->trace_m) {
                jb->trace_m[r * nb + b] = m;
                jb->trace_l[r * nb + b] = l;
            }
        }
        for (long c = 0; c < jb->d; ++c) jb->O[r * jb->d + c] = o[c] / l;
        jb->LSE[r] = m + log(l);
    }
    free(s);
    free(o);
    jb->ok = 1;
    return NULL;
}

static int run_jobs(job_t *proto, void *(*fn)(void *), int nthreads)
{
    long rows = proto->BH * proto->Nq;
    if (rows <= 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((long)nthreads > rows) nthreads = (int)rows;
    job_t jobs[256];
    pthread_t th[256];
    int started[256];
    long per = (rows + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = *proto;
        jobs[t].row_begin = t * per;
        jobs[t].row_end = (t + 1) * per < rows ? (t + 1) * per : rows;
        jobs[t].ok = 0;
        started[t] = 0;
        if (jobs[t].row_begin >= jobs[t].row_end) { jobs[t].ok = 1; continue; }
        if (t > 0 && pthread_create(&th[t], NULL, fn, &jobs[t]) == 0) started[t] = 1;
    }
    if (jobs[0].row_begin < jobs[0].row_end) fn(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) {
        if (started[t]) pthread_join(th[t], NULL);
        else if (jobs[t].row_begin < jobs[t].row_end) fn(&jobs[t]); /* thread failed: run inline */
    }
    for (int t = 0; t < nthreads; ++t)
        if (!jobs[t].ok) return -2;
    return 0;
}

/* Three-pass definition. Returns 0, or -1 on bad sizes, -2 on allocation failure. */
int oracle_attn_fp64(const double *Q, const double *K, const double *V, double *O, double *LSE,
                     long BH, long Nq, long Nk, long d, double scale, int nthreads)
{
    if (BH < 0 || Nq < 0 || Nk < 1 || d < 1) return -1;
    job_t p;
    memset(&p, 0, sizeof p);
    p.Q = Q; p.K = K; p.V = V; p.O = O; p.LSE = LSE;
    p.BH = BH; p.Nq = Nq; p.Nk = Nk; p.d = d; p.scale = scale;
    return run_jobs(&p, three_pass_worker, nthreads);
}

/* Online recurrence with key blocks of block_n and lazy threshold tau (natural log).
 * trace_m / trace_l, if not NULL, receive m and l after every block:
 * [BH*Nq, ceil(Nk/block_n)]. */
int oracle_attn_online_fp64(const double *Q, const double *K, const double *V, double *O, double *LSE,
                            long BH, long Nq, long Nk, long d, double scale, long block_n, double tau,
                            double *trace_m, double *trace_l, int nthreads)
{
    if (BH < 0 || Nq < 0 || Nk < 1 || d < 1 || block_n < 1 || tau < 0) return -1;
    job_t p;
    memset(&p, 0, sizeof p);
    p.Q = Q; p.K = K; p.V = V; p.O = O; p.LSE = LSE;
    p.BH = BH; p.Nq = Nq; p.Nk = Nk; p.d = d; p.scale = scale;
    p.block_n = block_n; p.tau = tau; p.trace_m = trace_m; p.trace_l = trace_l;
    return run_jobs(&p, online_worker, nthreads);
}

/*
 * Masked definition (causal and/or per-batch key lengths): row i of batch b
 * attends to the keys j with j < klen[b] (all keys when klen is NULL) and,
 * if causal, j <= i (query and key positions counted from the start of the
 * sequence). The three passes run over the allowed keys only. A row with no
 * allowed key has no softmax (the Triton page, section 5.1, warns that
 * exp(-inf - (-inf)) is NaN there); its reading here: O = 0, LSE = -inf.
 * klen: NULL or [B] (B = BH / H).
 */
typedef struct {
    job_t base;
    int causal;
    const long *klen;
    long H;
} mjob_t;

static void *masked_worker(void *arg)
{
    mjob_t *mj = (mjob_t *)arg;
    job_t *jb = &mj->base;
    double *s = (double *)malloc(sizeof(double) * (size_t)(jb->Nk > 0 ? jb->Nk : 1));
    if (!s) { jb->ok = 0; return NULL; }
    for (long r = jb->row_begin; r < jb->row_end; ++r) {
        long bh = r / jb->Nq, i = r % jb->Nq, b = bh / mj->H;
        long nk = mj->klen ? mj->klen[b] : jb->Nk;
        if (nk > jb->Nk) nk = jb->Nk;
        if (mj->causal && i + 1 < nk) nk = i + 1;
        double *o = jb->O + r * jb->d;
        if (nk <= 0) {
            for (long c = 0; c < jb->d; ++c) o[c] = 0.0;
            jb->LSE[r] = -INFINITY;
            continue;
        }
        const double *q = jb->Q + r * jb->d;
        scores_row(q, jb->K + bh * jb->Nk * jb->d, nk, jb->d, jb->scale, s);
        three_pass_row(s, jb->V + bh * jb->Nk * jb->d, nk, jb->d, o, jb->LSE + r);
    }
    free(s);
    jb->ok = 1;
    return NULL;
}

int oracle_attn_masked_fp64(const double *Q, const double *K, const double *V, double *O, double *LSE,
                            long B, long H, long Nq, long Nk, long d, double scale, int causal,
                            const long *klen, int nthreads)
{
    if (B < 0 || H < 1 || Nq < 0 || Nk < 1 || d < 1) return -1;
    long rows = B * H * Nq;
    if (rows <= 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((long)nthreads > rows) nthreads = (int)rows;
    mjob_t jobs[256];
    pthread_t th[256];
    int started[256];
    long per = (rows + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        memset(&jobs[t], 0, sizeof jobs[t]);
        job_t *p = &jobs[t].base;
        p->Q = Q; p->K = K; p->V = V; p->O = O; p->LSE = LSE;
        p->BH = B * H; p->Nq = Nq; p->Nk = Nk; p->d = d; p->scale = scale;
        p->row_begin = t * per;
        p->row_end = (t + 1) * per < rows ? (t + 1) * per : rows;
        jobs[t].causal = causal; jobs[t].klen = klen; jobs[t].H = H;
        started[t] = 0;
        if (p->row_begin >= p->row_end) { p->ok = 1; continue; }
        if (t > 0 && pthread_create(&th[t], NULL, masked_worker, &jobs[t]) == 0) started[t] = 1;
    }
    if (jobs[0].base.row_begin < jobs[0].base.row_end) masked_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) {
        if (started[t]) pthread_join(th[t], NULL);
        else if (jobs[t].base.row_begin < jobs[t].base.row_end) masked_worker(&jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t)
        if (!jobs[t].base.ok) return -2;
    return 0;
}

/*
 * Backward pass by recomputation (the MUSA guide's "重计算" principle and the
 * Triton page, sections 2.4 and 4.4: P is not stored; it is recomputed from
 * Q, K and the saved row statistics, then the chain rule is applied), for one
 * (batch, head) slice at a time, by the definitions, in fp64:
 *     P_ij  = exp(s_ij - LSE_i),  s_ij = scale * q_i . k_j
 *     D_i   = sum_c dO_ic O_ic
 *     dV_j  = sum_i P_ij dO_i
 *     dP_ij = dO_i . v_j
 *     dS_ij = P_ij (dP_ij - D_i)
 *     dQ_i  = scale * sum_j dS_ij k_j
 *     dK_j  = scale * sum_i dS_ij q_i
 * O and LSE are the forward outputs passed in (from the oracle itself).
 * Layouts as oracle_attn_fp64 (Nq = Nk = N); dQ/dK/dV like Q/K/V.
 * The masked variant takes the masks of oracle_attn_masked_fp64: a masked
 * score is -inf, so P_ij = 0 there (set directly, not through exp of the
 * saved LSE, which is -inf on a row with no key); every sum above then runs
 * over the allowed (i, j) only.
 */
typedef struct {
    const double *Q, *K, *V, *O, *dO, *LSE;
    double *dQ, *dK, *dV;
    long N, d;
    double scale;
    long bh_begin, bh_end;
    int ok;
    /* masks of the masked definition: causal (key j <= query i) and per-batch
     * key lengths klen[b] (keys j >= klen[b] masked; NULL = none); H heads per batch */
    int causal;
    const long *klen;
    long H;
} bjob_t;

static void *bwd_worker(void *arg)
{
    bjob_t *jb = (bjob_t *)arg;
    long N = jb->N, d = jb->d;
    double *P = (double *)malloc(sizeof(double) * (size_t)N * (size_t)N);
    double *dS = (double *)malloc(sizeof(double) * (size_t)N * (size_t)N);
    double *D = (double *)malloc(sizeof(double) * (size_t)N);
    if (!P || !dS || !D) { free(P); free(dS); free(D); jb->ok = 0; return NULL; }
    for (long bh = jb->bh_begin; bh < jb->bh_end; ++bh) {
        const double *Q = jb->Q + bh * N * d, *K = jb->K + bh * N * d, *V = jb->V + bh * N * d;
        const double *O = jb->O + bh * N * d, *dO = jb->dO + bh * N * d, *L = jb->LSE + bh * N;
        double *dQ = jb->dQ + bh * N * d, *dK = jb->dK + bh * N * d, *dV = jb->dV + bh * N * d;
        long key_end = N;
        if (jb->klen) {
            key_end = jb->klen[bh / jb->H];
            if (key_end < 0) key_end = 0;
            if (key_end > N) key_end = N;
        }
        for (long i = 0; i < N; ++i) {
            double acc = 0.0;
            for (long c = 0; c < d; ++c) acc += dO[i * d + c] * O[i * d + c];
            D[i] = acc;
            for (long j = 0; j < N; ++j) {
                double s = 0.0, dp = 0.0;
                for (long c = 0; c < d; ++c) {
                    s += Q[i * d + c] * K[j * d + c];
                    dp += dO[i * d + c] * V[j * d + c];
                }
                /* a masked score is -inf: its P is exactly 0 (and a row with no key has no P at all) */
#if ORACLE_MUTANT == 11 /* backward causal mask off by one: the diagonal key dropped */
                const int allowed = j < key_end && (!jb->causal || j < i);
#else
                const int allowed = j < key_end && (!jb->causal || j <= i);
#endif
                P[i * N + j] = allowed ? exp(jb->scale * s - L[i]) : 0.0;
#if ORACLE_MUTANT == 8 /* the D_i term dropped from dS */
                dS[i * N + j] = P[i * N + j] * dp;
#else
                dS[i * N + j] = P[i * N + j] * (dp - D[i]);
#endif
            }
        }
        for (long j = 0; j < N; ++j)
            for (long c = 0; c < d; ++c) {
                double av = 0.0, ak = 0.0;
                for (long i = 0; i < N; ++i) {
#if ORACLE_MUTANT == 10 /* P transposed in dV */
                    av += P[j * N + i] * dO[i * d + c];
#else
                    av += P[i * N + j] * dO[i * d + c];
#endif
                    ak += dS[i * N + j] * Q[i * d + c];
                }
                dV[j * d + c] = av;
#if ORACLE_MUTANT == 9 /* scale dropped from dK */
                dK[j * d + c] = ak;
#else
                dK[j * d + c] = jb->scale * ak;
#endif
            }
        for (long i = 0; i < N; ++i)
            for (long c = 0; c < d; ++c) {
                double aq = 0.0;
                for (long j = 0; j < N; ++j) aq += dS[i * N + j] * K[j * d + c];
                dQ[i * d + c] = jb->scale * aq;
            }
    }
    free(P); free(dS); free(D);
    jb->ok = 1;
    return NULL;
}

int oracle_attn_bwd_masked_fp64(const double *Q, const double *K, const double *V, const double *O,
                                const double *dO, const double *LSE, double *dQ, double *dK, double *dV, long BH,
                                long N, long d, double scale, int causal, const long *klen, long H, int nthreads)
{
    if (BH < 0 || N < 1 || d < 1) return -1;
    if (BH == 0) return 0;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((long)nthreads > BH) nthreads = (int)BH;
    bjob_t jobs[256];
    pthread_t th[256];
    int started[256];
    long per = (BH + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        bjob_t j = {Q, K, V, O, dO, LSE, dQ, dK, dV, N, d, scale, t * per,
                    (t + 1) * per < BH ? (t + 1) * per : BH, 0, causal, klen, H < 1 ? 1 : H};
        jobs[t] = j;
        started[t] = 0;
        if (jobs[t].bh_begin >= jobs[t].bh_end) { jobs[t].ok = 1; continue; }
        if (t > 0 && pthread_create(&th[t], NULL, bwd_worker, &jobs[t]) == 0) started[t] = 1;
    }
    if (jobs[0].bh_begin < jobs[0].bh_end) bwd_worker(&jobs[0]);
    for (int t = 1; t < nthreads; ++t) {
        if (started[t]) pthread_join(th[t], NULL);
        else if (jobs[t].bh_begin < jobs[t].bh_end) bwd_worker(&jobs[t]);
    }
    for (int t = 0; t < nthreads; ++t)
        if (!jobs[t].ok) return -2;
    return 0;
}

int oracle_attn_bwd_fp64(const double *Q, const double *K, const double *V, const double *O, const double *dO,
                         const double *LSE, double *dQ, double *dK, double *dV, long BH, long N, long d,
                         double scale, int nthreads)
{
    return oracle_attn_bwd_masked_fp64(Q, K, V, O, dO, LSE, dQ, dK, dV, BH, N, d, scale, 0, NULL, 1, nthreads);
}

/*
 * Single rows of the backward pass, same definitions and summation orders as
 * oracle_attn_bwd_fp64: dQ rows given as (bh, i) pairs, dK/dV rows as (bh, j)
 * pairs. Each row costs O(N d); O and LSE must cover every row of the heads
 * named. Outputs are [n, d].
 */
int oracle_bwd_rows_masked_fp64(const double *Q, const double *K, const double *V, const double *O,
                                const double *dO, const double *LSE, long BH, long N, long d, double scale,
                                int causal, const long *klen, long H, const long *dq_rows, long n_dq, double *dQ,
                                const long *dkv_rows, long n_dkv, double *dK, double *dV)
{
    if (N < 1 || d < 1) return -1;
    for (long r = 0; r < n_dq; ++r) {
        long bh = dq_rows[2 * r], i = dq_rows[2 * r + 1];
        if (bh < 0 || bh >= BH || i < 0 || i >= N) return -1;
        const double *q = Q + (bh * N + i) * d, *o = O + (bh * N + i) * d, *g = dO + (bh * N + i) * d;
        long key_end = klen ? klen[bh / (H < 1 ? 1 : H)] : N;
        if (key_end < 0) key_end = 0;
        if (key_end > N) key_end = N;
        if (causal && key_end > i + 1) key_end = i + 1;
        double Di = 0.0;
        for (long c = 0; c < d; ++c) Di += g[c] * o[c];
        double *out = dQ + r * d;
        for (long c = 0; c < d; ++c) out[c] = 0.0;
        for (long j = 0; j < key_end; ++j) {
            const double *kj = K + (bh * N + j) * d, *vj = V + (bh * N + j) * d;
            double sc = 0.0, dp = 0.0;
            for (long c = 0; c < d; ++c) {
                sc += q[c] * kj[c];
                dp += g[c] * vj[c];
            }
            double ds = exp(scale * sc - LSE[bh * N + i]) * (dp - Di);
            for (long c = 0; c < d; ++c) out[c] += ds * kj[c];
        }
        for (long c = 0; c < d; ++c) out[c] *= scale;
    }
    for (long r = 0; r < n_dkv; ++r) {
        long bh = dkv_rows[2 * r], j = dkv_rows[2 * r + 1];
        if (bh < 0 || bh >= BH || j < 0 || j >= N) return -1;
        const double *kj = K + (bh * N + j) * d, *vj = V + (bh * N + j) * d;
        double *ok = dK + r * d, *ov = dV + r * d;
        for (long c = 0; c < d; ++c) ok[c] = ov[c] = 0.0;
        long key_end = klen ? klen[bh / (H < 1 ? 1 : H)] : N;
        if (j >= key_end) continue; /* a masked key gets no gradient */
        for (long i = causal ? j : 0; i < N; ++i) {
            const double *q = Q + (bh * N + i) * d, *o = O + (bh * N + i) * d, *g = dO + (bh * N + i) * d;
            double Di = 0.0, sc = 0.0, dp = 0.0;
            for (long c = 0; c < d; ++c) {
                Di += g[c] * o[c];
                sc += q[c] * kj[c];
                dp += g[c] * vj[c];
            }
            double pij = exp(scale * sc - LSE[bh * N + i]);
            double ds = pij * (dp - Di);
            for (long c = 0; c < d; ++c) {
                ov[c] += pij * g[c];
                ok[c] += ds * q[c];
            }
        }
        for (long c = 0; c < d; ++c) ok[c] *= scale;
    }
    return 0;
}

int oracle_bwd_rows_fp64(const double *Q, const double *K, const double *V, const double *O, const double *dO,
                         const double *LSE, long BH, long N, long d, double scale, const long *dq_rows, long n_dq,
                         double *dQ, const long *dkv_rows, long n_dkv, double *dK, double *dV)
{
    return oracle_bwd_rows_masked_fp64(Q, K, V, O, dO, LSE, BH, N, d, scale, 0, NULL, 1, dq_rows, n_dq, dQ,
                                       dkv_rows, n_dkv, dK, dV);
}

/*
 * Merge of attention results computed over disjoint key ranges (the block
 * merge of the Triton page, section 2.3): parts are folded in order with the
 * running triple (m, l, O): for a part with statistics (m_b, l_b) and its
 * normalised output O_b,
 *     m_new = max(m, m_b)
 *     l_new = l e^(m - m_new) + l_b e^(m_b - m_new)
 *     O_new = (O l e^(m - m_new) + O_b l_b e^(m_b - m_new)) / l_new.
 * A part's (m_b, l_b) enter only through LSE_b = m_b + ln l_b, so each part is
 * taken with m_b = LSE_b and l_b = 1. Result: O and LSE = m + ln l.
 * Layouts: O_parts [nparts, rows, d], LSE_parts [nparts, rows]; O [rows, d], LSE [rows].
 */
int oracle_merge_fp64(const double *O_parts, const double *LSE_parts, long nparts, long rows, long d,
                      double *O, double *LSE)
{
    if (nparts < 1 || rows < 0 || d < 1) return -1;
    for (long r = 0; r < rows; ++r) {
        double m = -INFINITY, l = 0.0;
        double *o = O + r * d;
        for (long c = 0; c < d; ++c) o[c] = 0.0;
        for (long b = 0; b < nparts; ++b) {
            const double mb = LSE_parts[b * rows + r], lb = 1.0;
            const double *ob = O_parts + (b * rows + r) * d;
            const double m_new = mb > m ? mb : m;
            const double wa = (m == -INFINITY) ? 0.0 : l * exp(m - m_new);
            const double wb = lb * exp(mb - m_new);
            const double l_new = wa + wb;
            for (long c = 0; c < d; ++c) o[c] = (o[c] * wa + ob[c] * wb) / l_new;
            m = m_new;
            l = l_new;
        }
        LSE[r] = m + log(l);
    }
    return 0;
}

int oracle_mutant_id(void) { return ORACLE_MUTANT; }
