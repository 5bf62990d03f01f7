/*
 * kda_oracle.c -- plain fp64 CPU reference for Kimi Delta Attention (KDA).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle that the CUDA library is
 * checked against.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may build, load or call it.  It shares no code, header or
 * constant with the CUDA library, and the CUDA library never calls it.
 *
 * What it computes (token by token, one head at a time, state S of size
 * dk x dv held in fp64):
 *
 *   alpha = exp(g_t)                 per-channel gate, g = log(alpha) <= 0
 *   S     = Diag(alpha) S            decay first ...
 *   w     = S^T k_t                  ... then read the value stored at key k_t
 *   u     = beta_t (v_t - w)         the delta, scaled by the write strength
 *   S     = S + k_t u^T              write the delta only
 *   o_t   = S^T q_t                  read-out with the updated state
 *
 * Sources ("GPT-2부터 Kimi K3까지" = the lineage essay, page 1 of the pages):
 *   - delta rule: read v_old = k S, delta = v_new - v_old, S += k^T delta
 *     (essay, section "DeltaNet: 이제 메모리를 편집할 수 있습니다");
 *   - gating: decay the old state by alpha first, then write precisely
 *     (essay, section "Gated DeltaNet", the alpha x S_old + k^T delta line);
 *   - per-channel alpha: alpha becomes a vector, one forgetting rate per
 *     dimension (essay, section "KDA: Kimi의 비법"; the Kimi Linear explainer,
 *     section "KDA: 지우고 다시 쓰는 메모, 채널마다 다른 망각률");
 *   - beta_t scaling the delta and o_t = S_t^T q_t with the post-write state
 *     are the readings adopted for points the pages leave open.
 *
 * The columns of S never mix (every operation acts on S from the left or
 * column by column), so work is split over (sequence, head, block of 32
 * state columns) and handed to POSIX threads.  Inputs are consumed exactly as
 * given (fp64 copies of the stored values); nothing is re-rounded.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define KDA_ORACLE_COLS 32

typedef struct {
    const double *q, *k, *v, *g, *beta, *S0;
    const int64_t *cu;
    int64_t N;
    int H, dk, dv;
    double *o, *S_T;
    int64_t n_items;
    int64_t next; /* shared work counter */
    int fail;
} oracle_job;

/* One (sequence, head, column block): the recurrence above over the
 * sequence's tokens, for state columns [c0, c1). */
static int run_unit(const oracle_job *a, int64_t n, int h, int c0, int c1)
{
    const int H = a->H, dk = a->dk, dv = a->dv, W = c1 - c0;
    const int64_t bos = a->cu[n], eos = a->cu[n + 1];
    double *S = (double *)malloc(sizeof(double) * (size_t)dk * W);
    double *w = (double *)malloc(sizeof(double) * W);
    double *u = (double *)malloc(sizeof(double) * W);
    double *alpha = (double *)malloc(sizeof(double) * dk);
    if (!S || !w || !u || !alpha) {
        free(S); free(w); free(u); free(alpha);
        return -1;
    }
    const int64_t sbase = ((int64_t)n * H + h) * (int64_t)dk * dv;
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < W; ++j)
            S[i * W + j] = a->S0 ? a->S0[sbase + (int64_t)i * dv + c0 + j] : 0.0;

    for (int64_t t = bos; t < eos; ++t) {
        const int64_t th = t * H + h;
        const double *kt = a->k + th * dk;
        const double *qt = a->q + th * dk;
        const double *gt = a->g + th * dk;
        const double *vt = a->v + th * dv + c0;
        const double bt = a->beta[th];

        for (int i = 0; i < dk; ++i)
            alpha[i] = exp(gt[i]);
        for (int i = 0; i < dk; ++i)               /* S = Diag(alpha) S */
            for (int j = 0; j < W; ++j)
                S[i * W + j] *= alpha[i];
        for (int j = 0; j < W; ++j) {              /* w = S^T k */
            double acc = 0.0;
            for (int i = 0; i < dk; ++i)
                acc += S[i * W + j] * kt[i];
            w[j] = acc;
        }
        for (int j = 0; j < W; ++j)                /* u = beta (v - w) */
            u[j] = bt * (vt[j] - w[j]);
        for (int i = 0; i < dk; ++i)               /* S = S + k u^T */
            for (int j = 0; j < W; ++j)
                S[i * W + j] += kt[i] * u[j];
        double *ot = a->o + th * dv + c0;
        for (int j = 0; j < W; ++j) {              /* o = S^T q */
            double acc = 0.0;
            for (int i = 0; i < dk; ++i)
                acc += S[i * W + j] * qt[i];
            ot[j] = acc;
        }
    }
    for (int i = 0; i < dk; ++i)
        for (int j = 0; j < W; ++j)
            a->S_T[sbase + (int64_t)i * dv + c0 + j] = S[i * W + j];
    free(S); free(w); free(u); free(alpha);
    return 0;
}

static void *worker(void *p)
{
    oracle_job *a = (oracle_job *)p;
    const int nblk = (a->dv + KDA_ORACLE_COLS - 1) / KDA_ORACLE_COLS;
    for (;;) {
        int64_t it = __atomic_fetch_add(&a->next, 1, __ATOMIC_RELAXED);
        if (it >= a->n_items)
            break;
        int64_t n = it / ((int64_t)a->H * nblk);
        int rem = (int)(it % ((int64_t)a->H * nblk));
        int h = rem / nblk, b = rem % nblk;
        int c0 = b * KDA_ORACLE_COLS;
        int c1 = c0 + KDA_ORACLE_COLS < a->dv ? c0 + KDA_ORACLE_COLS : a->dv;
        if (run_unit(a, n, h, c0, c1) != 0)
            __atomic_store_n(&a->fail, 1, __ATOMIC_RELAXED);
    }
    return NULL;
}

/* Number of threads the oracle uses when the caller passes nthreads <= 0. */
int kda_oracle_default_threads(void)
{
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * Prefill over a packed batch.
 *   q, k, g : [T, H, dk]      v : [T, H, dv]      beta : [T, H]
 *   S0      : [N, H, dk, dv] or NULL (zeros)
 *   cu      : [N + 1], cu[0] = 0, non-decreasing, cu[N] = T
 *   o       : [T, H, dv]      S_T : [N, H, dk, dv] (may alias S0)
 * Returns the number of threads used, or a negative value on bad arguments
 * or allocation failure.
 */
int kda_oracle_prefill(const double *q, const double *k, const double *v,
                       const double *g, const double *beta, const double *S0,
                       const int64_t *cu, int64_t N, int64_t T, int H, int dk,
                       int dv, double *o, double *S_T, int nthreads)
{
    if (!cu || N < 0 || T < 0 || H <= 0 || dk <= 0 || dv <= 0 || !S_T)
        return -1;
    if (cu[0] != 0 || cu[N] != T)
        return -1;
    for (int64_t n = 0; n < N; ++n)
        if (cu[n + 1] < cu[n])
            return -1;
    if (T > 0 && (!q || !k || !v || !g || !beta || !o))
        return -1;

    oracle_job job;
    memset(&job, 0, sizeof job);
    job.q = q; job.k = k; job.v = v; job.g = g; job.beta = beta; job.S0 = S0;
    job.cu = cu; job.N = N; job.H = H; job.dk = dk; job.dv = dv;
    job.o = o; job.S_T = S_T;
    job.n_items = N * H * (int64_t)((dv + KDA_ORACLE_COLS - 1) / KDA_ORACLE_COLS);

    if (nthreads <= 0)
        nthreads = kda_oracle_default_threads();
    if (nthreads > job.n_items)
        nthreads = job.n_items > 0 ? (int)job.n_items : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * nthreads);
    if (!th)
        return -2;
    int started = 0;
    for (int i = 1; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, worker, &job) != 0)
            break;
        ++started;
    }
    worker(&job);
    for (int i = 1; i <= started; ++i)
        pthread_join(th[i], NULL);
    free(th);
    return job.fail ? -2 : started + 1;
}

/*
 * One decode step for B independent sequences: each sequence consumes one
 * token and its state is updated in place.  This is the same recurrence with
 * one token per sequence.
 *   q, k, g : [B, H, dk]   v : [B, H, dv]   beta : [B, H]
 *   S       : [B, H, dk, dv], read and overwritten
 *   o       : [B, H, dv]
 */
int kda_oracle_decode_step(const double *q, const double *k, const double *v,
                           const double *g, const double *beta, double *S,
                           int64_t B, int H, int dk, int dv, double *o,
                           int nthreads)
{
    if (B < 0 || !S)
        return -1;
    int64_t *cu = (int64_t *)malloc(sizeof(int64_t) * (size_t)(B + 1));
    if (!cu)
        return -2;
    for (int64_t b = 0; b <= B; ++b)
        cu[b] = b;
    int r = kda_oracle_prefill(q, k, v, g, beta, S, cu, B, B, H, dk, dv, o, S,
                               nthreads);
    free(cu);
    return r;
}
