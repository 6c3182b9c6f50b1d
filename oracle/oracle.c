/*
 * CPU oracle for fused softmax attention, forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is used by the tests, by smoke() and by
 * the benchmark's CPU-baseline / reference leg.  The product (the CUDA library
 * and its Python binding) never links, loads or calls it, and it shares no code
 * with the CUDA path.
 *
 * Source of truth: the page "FlashAttention-T: Towards Fully Tensorized
 * Attention by Exploiting Tensor-Vector Parallelism" (papercache.org summary,
 * PPoPP '26):
 *   - section A3 "fused attention algorithm flow" with Fig. 2: every output row
 *     block of O = softmax(S) V, S = Q K^T * scale, is produced from the row
 *     maximum m, the row sum l of the exponentials and the accumulated P V.
 *   - section A2 "Tensorized online softmax": the surrogate maximum equation
 *     (m_hat[i] = max of m[k] over the X-row tile holding row i), the
 *     any-overflow / all-underflow discussion, and Algorithm 1 steps 1-7.
 *   - section A4 results, Fig. 11: accuracy is judged against an FP64 attention.
 *
 * Functions:
 *   oracle_attn_fwd_qk    the plain definition in double precision (the oracle),
 *                         Nq query rows against Nk keys;
 *   oracle_attn_fwd       the same with Nq = Nk;
 *   oracle_attn_naive     brute force in long double with the full S matrix
 *                         materialised and sorted summation (pins the oracle);
 *   oracle_attn_surrogate the blocked online algorithm with the surrogate
 *                         maximum, in the order of Algorithm 1, in double
 *                         (pins that the surrogate maximum does not change the
 *                         result and exposes the all-underflow condition).
 *
 * Layout of every tensor: row-major [B, H, N, d] for Q, K, V, O and [B, H, N]
 * for LSE; values are doubles (bf16 / e4m3 inputs are widened exactly by the
 * caller).  LSE is the natural-log log-sum-exp of the scaled logits.
 * Causal masking keeps key j for query i iff j <= i (equal query and key
 * lengths, aligned at index 0).
 *
 * Portable C99 + pthreads; no ISA-specific code (the host may be x86-64 or
 * aarch64).
 */
#define _GNU_SOURCE
#include <math.h>
#include <pthread.h>
#include <sched.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------ */
/* threads                                                                   */
/* ------------------------------------------------------------------------ */

int oracle_available_cores(void) {
    cpu_set_t set;
    if (sched_getaffinity(0, sizeof(set), &set) == 0) {
        int c = CPU_COUNT(&set);
        if (c > 0) return c;
    }
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/* ------------------------------------------------------------------------ */
/* 1. The plain definition (the oracle)                                      */
/* ------------------------------------------------------------------------ */
/*
 * For every (b, h, i):
 *   s_j   = scale * (q_i . k_j)            for j in J_i
 *   m_i   = max_j s_j
 *   l_i   = sum_j exp(s_j - m_i)
 *   O_i   = (sum_j exp(s_j - m_i) v_j) / l_i
 *   LSE_i = m_i + ln(l_i)
 * with Nq query rows and Nk keys per (b, h); J_i = {0..Nk-1}, or, causal,
 * {0..i + Nk - Nq}: the queries are the last Nq positions of the key
 * sequence (for Nq = Nk this is the ordinary j <= i).  Rows listed by
 * [row_begin, row_end) with stride row_step are computed, in every (b, h);
 * other rows of o / lse are left untouched.  q, o: [B, H, Nq, d]; k, v:
 * [B, H, Nk, d]; lse: [B, H, Nq].
 */
typedef struct {
    const double *q, *k, *v;
    double *o, *lse;
    long B, H, Nq, Nk, d;
    int causal;
    double scale;
    long row_begin, row_end, row_step;
    long n_rows_per_bh;  /* number of selected rows per (b, h) */
    long task_begin, task_end, task_stride; /* tasks = (bh, selected-row index) pairs */
} exact_job;

static void exact_row(const exact_job *jb, long bh, long i, double *s) {
    const long N = jb->Nk, d = jb->d;
    const double *qi = jb->q + (bh * jb->Nq + i) * d;
    const double *kb = jb->k + bh * N * d;
    const double *vb = jb->v + bh * N * d;
    long nkeys = jb->causal ? i + 1 + (jb->Nk - jb->Nq) : N;
    if (nkeys > N) nkeys = N;
    double m = -INFINITY;
    for (long j = 0; j < nkeys; ++j) {
        const double *kj = kb + j * d;
        double dot = 0.0;
        for (long c = 0; c < d; ++c) dot += qi[c] * kj[c];
        s[j] = jb->scale * dot;
        if (s[j] > m) m = s[j];
    }
    double l = 0.0;
    for (long j = 0; j < nkeys; ++j) {
        s[j] = exp(s[j] - m); /* s now holds the unnormalised weights */
        l += s[j];
    }
    double *oi = jb->o + (bh * jb->Nq + i) * d;
    for (long c = 0; c < d; ++c) oi[c] = 0.0;
    for (long j = 0; j < nkeys; ++j) {
        const double *vj = vb + j * d;
        const double w = s[j];
        for (long c = 0; c < d; ++c) oi[c] += w * vj[c];
    }
    for (long c = 0; c < d; ++c) oi[c] /= l;
    jb->lse[bh * jb->Nq + i] = m + log(l);
}

static void *exact_worker(void *arg) {
    const exact_job *jb = (const exact_job *)arg;
    double *s = (double *)malloc(sizeof(double) * (size_t)(jb->Nk > 0 ? jb->Nk : 1));
    if (!s) return (void *)1;
    for (long t = jb->task_begin; t < jb->task_end; t += jb->task_stride) {
        const long bh = t / jb->n_rows_per_bh;
        const long r = t % jb->n_rows_per_bh;
        const long i = jb->row_begin + r * jb->row_step;
        exact_row(jb, bh, i, s);
    }
    free(s);
    return NULL;
}

int oracle_attn_fwd_qk(const double *q, const double *k, const double *v, double *o, double *lse,
                       long B, long H, long Nq, long Nk, long d, int causal, double scale,
                       long row_begin, long row_end, long row_step, int nthreads) {
    if (!q || !k || !v || !o || !lse) return -1;
    if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || d < 1) return -1;
    if (causal && Nk < Nq) return -1; /* the first queries would see no key */
    if (row_step < 1) row_step = 1;
    if (row_begin < 0) row_begin = 0;
    if (row_end > Nq || row_end < 0) row_end = Nq;
    if (row_end <= row_begin || B * H == 0) return 0;
    const long n_rows = (row_end - row_begin + row_step - 1) / row_step;
    const long n_tasks = B * H * n_rows;
    if (nthreads <= 0) nthreads = oracle_available_cores();
    if (nthreads > n_tasks) nthreads = (int)n_tasks;

    exact_job base = {q, k, v, o, lse, B, H, Nq, Nk, d, causal, scale,
                      row_begin, row_end, row_step, n_rows, 0, 0, 1};
    exact_job *jobs = (exact_job *)calloc((size_t)nthreads, sizeof(exact_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return -2; }
    /* Threads take rows round-robin so that causal rows (whose cost grows
     * with the row index) are balanced across threads. */
    int rc = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].task_begin = t;
        jobs[t].task_end = n_tasks;
        jobs[t].task_stride = nthreads;
    }
    char *started = (char *)calloc((size_t)nthreads, 1);
    if (!started) { free(jobs); free(th); return -2; }
    for (int t = 1; t < nthreads; ++t)
        started[t] = (pthread_create(&th[t], NULL, exact_worker, &jobs[t]) == 0);
    if (exact_worker(&jobs[0]) != NULL) rc = -2;
    for (int t = 1; t < nthreads; ++t) {
        void *ret = NULL;
        if (started[t]) pthread_join(th[t], &ret);
        else ret = exact_worker(&jobs[t]); /* could not start a thread: do its share here */
        if (ret) rc = -2;
    }
    free(started);
    free(jobs);
    free(th);
    return rc;
}

/* Equal query and key lengths (the self-attention case). */
int oracle_attn_fwd(const double *q, const double *k, const double *v, double *o, double *lse,
                    long B, long H, long N, long d, int causal, double scale,
                    long row_begin, long row_end, long row_step, int nthreads) {
    return oracle_attn_fwd_qk(q, k, v, o, lse, B, H, N, N, d, causal, scale, row_begin, row_end,
                              row_step, nthreads);
}

/* ------------------------------------------------------------------------ */
/* 2. Brute force in long double                                             */
/* ------------------------------------------------------------------------ */
/*
 * Materialises S = scale * Q K^T for one (b, h) in long double, takes the
 * softmax of every row with the row maximum, sums the weights in ascending
 * order (so that rounding is as small as the format allows) and forms P V by
 * plain triple loops.  Masked entries are excluded from the row.  Intended for
 * tiny inputs only (it holds N*N long doubles).
 */
static int cmp_ld(const void *a, const void *b) {
    long double x = *(const long double *)a, y = *(const long double *)b;
    return (x > y) - (x < y);
}

int oracle_attn_naive(const double *q, const double *k, const double *v, double *o, double *lse,
                      long B, long H, long N, long d, int causal, double scale) {
    if (!q || !k || !v || !o || !lse || N < 0 || d < 1) return -1;
    long double *S = (long double *)malloc(sizeof(long double) * (size_t)(N * N + 1));
    long double *P = (long double *)malloc(sizeof(long double) * (size_t)(N * N + 1));
    long double *tmp = (long double *)malloc(sizeof(long double) * (size_t)(N + 1));
    if (!S || !P || !tmp) { free(S); free(P); free(tmp); return -2; }
    for (long bh = 0; bh < B * H; ++bh) {
        const double *Qb = q + bh * N * d, *Kb = k + bh * N * d, *Vb = v + bh * N * d;
        /* S = scale * Q K^T, masked entries set to -inf */
        for (long i = 0; i < N; ++i)
            for (long j = 0; j < N; ++j) {
                if (causal && j > i) { S[i * N + j] = -INFINITY; continue; }
                long double acc = 0.0L;
                for (long c = 0; c < d; ++c) acc += (long double)Qb[i * d + c] * (long double)Kb[j * d + c];
                S[i * N + j] = (long double)scale * acc;
            }
        /* row softmax */
        for (long i = 0; i < N; ++i) {
            long double m = -INFINITY;
            for (long j = 0; j < N; ++j) if (S[i * N + j] > m) m = S[i * N + j];
            long cnt = 0;
            for (long j = 0; j < N; ++j) {
                long double w = (S[i * N + j] == -INFINITY) ? 0.0L : expl(S[i * N + j] - m);
                P[i * N + j] = w;
                tmp[cnt++] = w;
            }
            qsort(tmp, (size_t)cnt, sizeof(long double), cmp_ld);
            long double l = 0.0L;
            for (long j = 0; j < cnt; ++j) l += tmp[j];
            for (long j = 0; j < N; ++j) P[i * N + j] /= l;
            lse[bh * N + i] = (double)(m + logl(l));
        }
        /* O = P V */
        for (long i = 0; i < N; ++i)
            for (long c = 0; c < d; ++c) {
                long double acc = 0.0L;
                for (long j = 0; j < N; ++j) acc += P[i * N + j] * (long double)Vb[j * d + c];
                o[(bh * N + i) * d + c] = (double)acc;
            }
    }
    free(S); free(P); free(tmp);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* 3. Blocked online algorithm with the surrogate maximum                    */
/* ------------------------------------------------------------------------ */
/*
 * Follows Algorithm 1 of the page ("Tensorized Online Softmax for Fused
 * Attention") in its order, per query block of BM rows (BM a multiple of X)
 * and key block of BN keys, in double precision:
 *   step 1    m_hat <- max(m_hat_old, tilemax(S, X)): the maximum of the row
 *             maxima over the X-row tile holding each row (tiles aligned to
 *             query index 0, last tile cut at N);
 *   steps 2-3 O <- exp(m_hat_old - m_hat) * O, one factor per X-row tile;
 *   steps 4-5 Z <- log2(e) * S - log2(e) * m_hat;
 *   step 6    P~ <- exp2(Z);
 *   step 7    l <- exp(m_hat_old - m_hat) * l + rowsum(P~);  O += P~ V.
 * The first contributing block uses a factor of 0 on the (empty) O and l.
 * Blocks whose tile maximum is -inf (fully masked) leave the state as is.
 * At the end O /= l and LSE = m_hat + ln(l).
 *
 * Alongside, the exact running row maximum m is kept.  For each row the
 * function reports in gap_log2[row] the final c * (m_hat - m) with
 * c = log2(e) (the gap in binary orders of magnitude between the surrogate
 * and the exact maximum) and returns the number of rows whose every
 * exponential underflowed to 0 (l == 0): the all-underflow case of the page's
 * stability discussion.  Such rows get O = NaN and LSE = -inf.
 */
long oracle_attn_surrogate(const double *q, const double *k, const double *v, double *o, double *lse,
                           double *gap_log2, long B, long H, long N, long d, int causal, double scale,
                           long X, long BM, long BN) {
    if (!q || !k || !v || !o || !lse || N < 0 || d < 1) return -1;
    if (X < 1 || BM < X || BM % X != 0 || BN < 1) return -1;
    const double LOG2E = 1.4426950408889634073599246810018921;
    double *S = (double *)malloc(sizeof(double) * (size_t)(BM * BN));
    double *Oacc = (double *)malloc(sizeof(double) * (size_t)(BM * d));
    double *l = (double *)malloc(sizeof(double) * (size_t)BM);
    double *mhat = (double *)malloc(sizeof(double) * (size_t)BM);
    double *mexact = (double *)malloc(sizeof(double) * (size_t)BM);
    double *rowmax = (double *)malloc(sizeof(double) * (size_t)BM);
    if (!S || !Oacc || !l || !mhat || !mexact || !rowmax) {
        free(S); free(Oacc); free(l); free(mhat); free(mexact); free(rowmax);
        return -2;
    }
    long n_underflow = 0;
    for (long bh = 0; bh < B * H; ++bh) {
        const double *Qb = q + bh * N * d, *Kb = k + bh * N * d, *Vb = v + bh * N * d;
        for (long i0 = 0; i0 < N; i0 += BM) {
            const long rows = (N - i0 < BM) ? N - i0 : BM;
            for (long r = 0; r < BM; ++r) { l[r] = 0.0; mhat[r] = -INFINITY; mexact[r] = -INFINITY; }
            for (long x = 0; x < BM * d; ++x) Oacc[x] = 0.0;
            for (long j0 = 0; j0 < N; j0 += BN) {
                const long cols = (N - j0 < BN) ? N - j0 : BN;
                if (causal && j0 > i0 + rows - 1) break;
                /* S block (masked entries -inf) and row maxima */
                for (long r = 0; r < rows; ++r) {
                    rowmax[r] = -INFINITY;
                    for (long c = 0; c < cols; ++c) {
                        double val;
                        if (causal && j0 + c > i0 + r) val = -INFINITY;
                        else {
                            double dot = 0.0;
                            for (long e = 0; e < d; ++e) dot += Qb[(i0 + r) * d + e] * Kb[(j0 + c) * d + e];
                            val = scale * dot;
                        }
                        S[r * BN + c] = val;
                        if (val > rowmax[r]) rowmax[r] = val;
                    }
                    if (rowmax[r] > mexact[r]) mexact[r] = rowmax[r];
                }
                /* step 1: surrogate maximum over X-row tiles */
                for (long t0 = 0; t0 < rows; t0 += X) {
                    const long t1 = (t0 + X < rows) ? t0 + X : rows;
                    double tmax = -INFINITY;
                    for (long r = t0; r < t1; ++r) if (rowmax[r] > tmax) tmax = rowmax[r];
                    const double m_old = mhat[t0];
                    const double m_new = (tmax > m_old) ? tmax : m_old;
                    if (m_new == -INFINITY) continue; /* fully masked tile: nothing to add */
                    /* steps 2-3: one rescale factor for the whole tile */
                    const double alpha = (m_old == -INFINITY) ? 0.0 : exp(m_old - m_new);
                    for (long r = t0; r < t1; ++r) {
                        mhat[r] = m_new;
                        for (long e = 0; e < d; ++e) Oacc[r * d + e] *= alpha;
                        l[r] *= alpha;
                        /* steps 4-6: Z = log2e*S - log2e*m_hat, P~ = exp2(Z); step 7 */
                        double rs = 0.0;
                        for (long c = 0; c < cols; ++c) {
                            const double z = LOG2E * S[r * BN + c] - LOG2E * m_new;
                            const double p = exp2(z);
                            rs += p;
                            for (long e = 0; e < d; ++e) Oacc[r * d + e] += p * Vb[(j0 + c) * d + e];
                        }
                        l[r] += rs;
                    }
                }
            }
            for (long r = 0; r < rows; ++r) {
                const long row = bh * N + i0 + r;
                if (gap_log2) gap_log2[row] = LOG2E * (mhat[r] - mexact[r]);
                if (l[r] == 0.0) {
                    ++n_underflow;
                    for (long e = 0; e < d; ++e) o[row * d + e] = NAN;
                    lse[row] = -INFINITY;
                    continue;
                }
                for (long e = 0; e < d; ++e) o[row * d + e] = Oacc[r * d + e] / l[r];
                lse[row] = mhat[r] + log(l[r]);
            }
        }
    }
    free(S); free(Oacc); free(l); free(mhat); free(mexact); free(rowmax);
    return n_underflow;
}
