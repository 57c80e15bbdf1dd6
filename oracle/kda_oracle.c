/*
 * KDA oracle: the Kimi Delta Attention recurrence, token by token, in fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * What it follows:
 *   - "Kimi K3 Architecture Explained" (meta-quantum.today), section 3
 *     "Kimi Delta Attention (KDA)": a fixed-size recurrent state per head; the
 *     update decays stale context first, then erases conflicting memory, then
 *     writes; the eraser recalls a value with the incoming key and writes only
 *     the difference to the new value (DeltaNet lineage).
 *   - Kimi K3 technical-report digest (devpress.csdn.net), section 2.1 (1):
 *     delta rule plus a channel-wise forget gate; the log-decay is a bounded
 *     scaled sigmoid with g_min = -5 (the caller supplies g itself).
 *
 * Readings taken where the pages are silent (each also listed in the design
 * notes): alpha = exp(g) with the natural log; the decay acts on the key
 * (row) side of S in R^{dk x dv}; beta is one scalar per token and head; the
 * output is read after the update, o_t = S_t^T q_t; there is no 1/sqrt(d)
 * scale and no positional term.
 *
 * Per token t of a sequence, for one head, with S of shape dk x dv:
 *     S <- Diag(exp(g_t)) S                  decay
 *     S <- S - beta_t k_t (k_t^T S)           erase
 *     S <- S + beta_t k_t v_t^T               write
 *     o_t = S^T q_t                           read
 *
 * Columns of S never mix (every step acts on S from the left or adds a rank-1
 * term column by column), so splitting the dv columns over threads is exact:
 * each thread runs the same four steps on its own column range.
 *
 * Setting erase = 0 drops the erase step only (the "gated linear attention"
 * reading used by the self-checks); erase = 1 is KDA.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t T_begin, T_end;   /* token range of this sequence               */
    int64_t n, h;             /* sequence index, head index                 */
    int H, dk, dv, j0, j1;    /* column range [j0, j1) of S this job owns    */
    int erase;
    const double *q, *k, *v, *g, *beta, *S0;
    double *out, *S_final;
} kda_job_t;

static void run_job(const kda_job_t *J)
{
    const int dk = J->dk, dv = J->dv, H = J->H, nc = J->j1 - J->j0;
    double *S = (double *)calloc((size_t)dk * (size_t)(nc > 0 ? nc : 1), sizeof(double));
    double *r = (double *)calloc((size_t)(nc > 0 ? nc : 1), sizeof(double));
    if (!S || !r) { free(S); free(r); return; }

    /* S starts from S0 (or zeros). */
    if (J->S0) {
        const double *S0 = J->S0 + ((size_t)J->n * H + J->h) * (size_t)dk * dv;
        for (int i = 0; i < dk; ++i)
            for (int c = 0; c < nc; ++c)
                S[(size_t)i * nc + c] = S0[(size_t)i * dv + J->j0 + c];
    }

    for (int64_t t = J->T_begin; t < J->T_end; ++t) {
        const double *qt = J->q + ((size_t)t * H + J->h) * dk;
        const double *kt = J->k + ((size_t)t * H + J->h) * dk;
        const double *vt = J->v + ((size_t)t * H + J->h) * dv;
        const double *gt = J->g + ((size_t)t * H + J->h) * dk;
        const double bt = J->beta[(size_t)t * H + J->h];

        /* 1. decay: row i of S scaled by alpha_i = exp(g_i). */
        for (int i = 0; i < dk; ++i) {
            const double a = exp(gt[i]);
            for (int c = 0; c < nc; ++c) S[(size_t)i * nc + c] *= a;
        }
        /* 2. erase: S <- S - beta k (k^T S). */
        if (J->erase) {
            for (int c = 0; c < nc; ++c) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += kt[i] * S[(size_t)i * nc + c];
                r[c] = acc;
            }
            for (int i = 0; i < dk; ++i)
                for (int c = 0; c < nc; ++c) S[(size_t)i * nc + c] -= bt * kt[i] * r[c];
        }
        /* 3. write: S <- S + beta k v^T. */
        for (int i = 0; i < dk; ++i)
            for (int c = 0; c < nc; ++c) S[(size_t)i * nc + c] += bt * kt[i] * vt[J->j0 + c];
        /* 4. read: o = S^T q. */
        if (J->out) {
            double *ot = J->out + ((size_t)t * H + J->h) * dv;
            for (int c = 0; c < nc; ++c) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += qt[i] * S[(size_t)i * nc + c];
                ot[J->j0 + c] = acc;
            }
        }
    }

    if (J->S_final) {
        double *SF = J->S_final + ((size_t)J->n * H + J->h) * (size_t)dk * dv;
        for (int i = 0; i < dk; ++i)
            for (int c = 0; c < nc; ++c) SF[(size_t)i * dv + J->j0 + c] = S[(size_t)i * nc + c];
    }
    free(S);
    free(r);
}

typedef struct {
    kda_job_t *jobs;
    int64_t njobs;
    int64_t next;
    pthread_mutex_t lock;
} kda_pool_t;

static void *worker(void *arg)
{
    kda_pool_t *P = (kda_pool_t *)arg;
    for (;;) {
        pthread_mutex_lock(&P->lock);
        int64_t i = P->next++;
        pthread_mutex_unlock(&P->lock);
        if (i >= P->njobs) return NULL;
        run_job(&P->jobs[i]);
    }
}

/*
 * Run the recurrence over N packed sequences.
 *
 *   cu_seqlens : [N+1] token offsets, cu[0] = 0, non-decreasing.
 *   q, k, g    : [T_tot, H, dk];  v, out : [T_tot, H, dv];  beta : [T_tot, H]
 *   S0         : [N, H, dk, dv] or NULL (zeros);  S_final : [N, H, dk, dv] or NULL
 *   out        : may be NULL (states only).
 *   col_block  : columns of S per job (<= 0 means all dv in one job).
 *   nthreads   : worker threads (<= 0 means 1).
 * Returns 0, or -1 on a bad argument.
 */
int kda_oracle_forward(int N, const int64_t *cu_seqlens, int H, int dk, int dv,
                       const double *q, const double *k, const double *v,
                       const double *g, const double *beta, const double *S0,
                       double *out, double *S_final, int erase, int col_block,
                       int nthreads)
{
    if (N < 0 || H <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens || !k || !v || !g || !beta)
        return -1;
    if (out && !q) return -1;
    if (col_block <= 0 || col_block > dv) col_block = dv;
    const int nblk = (dv + col_block - 1) / col_block;
    const int64_t njobs = (int64_t)N * H * nblk;
    kda_job_t *jobs = (kda_job_t *)calloc((size_t)(njobs > 0 ? njobs : 1), sizeof(kda_job_t));
    if (!jobs) return -1;
    int64_t j = 0;
    for (int n = 0; n < N; ++n) {
        if (cu_seqlens[n + 1] < cu_seqlens[n]) { free(jobs); return -1; }
        for (int h = 0; h < H; ++h)
            for (int b = 0; b < nblk; ++b) {
                kda_job_t *J = &jobs[j++];
                J->T_begin = cu_seqlens[n];
                J->T_end = cu_seqlens[n + 1];
                J->n = n; J->h = h; J->H = H; J->dk = dk; J->dv = dv;
                J->j0 = b * col_block;
                J->j1 = (b + 1) * col_block < dv ? (b + 1) * col_block : dv;
                J->erase = erase;
                J->q = q; J->k = k; J->v = v; J->g = g; J->beta = beta; J->S0 = S0;
                J->out = out; J->S_final = S_final;
            }
    }
    if (nthreads <= 1 || njobs <= 1) {
        for (int64_t i = 0; i < njobs; ++i) run_job(&jobs[i]);
    } else {
        kda_pool_t P;
        P.jobs = jobs; P.njobs = njobs; P.next = 0;
        pthread_mutex_init(&P.lock, NULL);
        int nt = nthreads < njobs ? nthreads : (int)njobs;
        pthread_t *th = (pthread_t *)calloc((size_t)nt, sizeof(pthread_t));
        char *ok = (char *)calloc((size_t)nt, 1);
        for (int i = 0; i < nt; ++i) ok[i] = pthread_create(&th[i], NULL, worker, &P) == 0;
        worker(&P); /* the calling thread takes jobs too; covers a failed create */
        for (int i = 0; i < nt; ++i)
            if (ok[i]) pthread_join(th[i], NULL);
        free(ok);
        pthread_mutex_destroy(&P.lock);
        free(th);
    }
    free(jobs);
    return 0;
}
