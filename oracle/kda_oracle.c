/*
 * KDA oracle: a plain, slow, fp64 CPU statement of Kimi Delta Attention.
 *
 * THIS IS TEST INFRASTRUCTURE. Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load it. The CUDA library never links,
 * loads or calls it, and it shares no code, header or table with the CUDA path.
 *
 * What it computes (token by token, the definition itself, no chunking):
 *
 *   gate   ('From Linear Attention to KDA', blog-3d3.pages.dev/posts/150, §5.4):
 *          log a_t[c] = g_min * sigmoid(exp(A_h) * z_t[c]),  g_min = -5
 *          beta_t     = sigmoid(b_t)                       (same page, §5.3)
 *   update (same page §5.2; 'Kimi K3 attention deep dive', forceinjection.github.io,
 *           §2.1-2.2; 'Kimi K3', llm.rainlin.net, section "Kimi Delta Attention"):
 *          S'  = Diag(a_t) S_{t-1}                 decay the rows (d_k index)
 *          p   = S'^T k_t                          what the decayed table predicts for k_t
 *          S_t = S' + beta_t k_t (v_t - p)^T       write only the prediction error
 *          o_t = S_t^T q_t                         read out after the write
 *
 * The rank-1 form above is the same matrix as (I - beta k k^T) Diag(a) S + beta k v^T,
 * written so that no d_k x d_k matrix is formed (the three-step DPLR update of the
 * deep-dive page, §2.2).
 *
 * A 'delta' switch of 0 drops the correction (p := 0). With it the same loop states
 * the relatives listed in the variant table of the blog's §4: linear attention
 * (a = 1, beta = 1), RetNet (scalar a), GLA (per-channel a). Those variants exist only
 * so the worked examples on the pages can pin this code.
 *
 * Layouts (row-major, tokens of all sequences packed one after another):
 *   q, k : [T_total, H, dk]      v : [T_total, H, dv]
 *   la   : [T_total, H, dk]      beta : [T_total, H]
 *   S0   : [N, H, dk, dv] or NULL (zeros)
 *   cu   : [N + 1] token offsets of the sequences
 *   o    : [T_total, H, dv]      S_out : [N, H, dk, dv]
 *
 * Work is split over (sequence, head, block of d_v columns). The columns of S never
 * mix in the update above (p[j] and o[j] read column j only), so the split is exact.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define KDA_ORACLE_G_MIN (-5.0)

static double sigmoid_d(double x) { return 1.0 / (1.0 + exp(-x)); }

/* Gate of the blog's §5.4 in fp64, from the fp32 values the GPU receives. */
void kda_oracle_gate(const float *z, const float *A, const float *b,
                     int64_t T_total, int64_t H, int64_t dk,
                     double *la, double *beta) {
    for (int64_t t = 0; t < T_total; ++t) {
        for (int64_t h = 0; h < H; ++h) {
            const double eA = exp((double)A[h]);
            const float *zz = z + (t * H + h) * dk;
            double *ll = la + (t * H + h) * dk;
            for (int64_t c = 0; c < dk; ++c)
                ll[c] = KDA_ORACLE_G_MIN * sigmoid_d(eA * (double)zz[c]);
            beta[t * H + h] = sigmoid_d((double)b[t * H + h]);
        }
    }
}

typedef struct {
    int delta;
    const double *q, *k, *v, *la, *beta, *S0;
    const int64_t *cu;
    int64_t N, H, dk, dv, bw, nblk;
    double *o, *S_out;
    int64_t n_units;
    int64_t next;   /* shared work counter */
    int failed;     /* set when a worker could not get its scratch memory */
} job_t;

/* One (sequence n, head h, columns [j0, j0 + w)) unit of the recurrence. */
static void run_unit(const job_t *J, int64_t unit, double *S, double *alpha, double *p) {
    const int64_t H = J->H, dk = J->dk, dv = J->dv;
    const int64_t blk = unit % J->nblk;
    const int64_t h = (unit / J->nblk) % H;
    const int64_t n = unit / (J->nblk * H);
    const int64_t j0 = blk * J->bw;
    const int64_t w = (j0 + J->bw <= dv) ? J->bw : dv - j0;

    /* S <- initial state (or zeros), columns j0..j0+w-1 */
    for (int64_t c = 0; c < dk; ++c)
        for (int64_t j = 0; j < w; ++j)
            S[c * w + j] = J->S0 ? J->S0[((n * H + h) * dk + c) * dv + j0 + j] : 0.0;

    for (int64_t t = J->cu[n]; t < J->cu[n + 1]; ++t) {
        const double *qt = J->q + (t * H + h) * dk;
        const double *kt = J->k + (t * H + h) * dk;
        const double *vt = J->v + (t * H + h) * dv + j0;
        const double *lt = J->la + (t * H + h) * dk;
        const double bt = J->beta[t * H + h];

        /* S' = Diag(a_t) S : row c scaled by a_t[c] = exp(log a_t[c]) */
        for (int64_t c = 0; c < dk; ++c) alpha[c] = exp(lt[c]);
        for (int64_t c = 0; c < dk; ++c)
            for (int64_t j = 0; j < w; ++j) S[c * w + j] *= alpha[c];

        /* p = S'^T k_t (zero when the delta correction is switched off) */
        for (int64_t j = 0; j < w; ++j) p[j] = 0.0;
        if (J->delta)
            for (int64_t c = 0; c < dk; ++c)
                for (int64_t j = 0; j < w; ++j) p[j] += kt[c] * S[c * w + j];

        /* S_t = S' + beta_t k_t (v_t - p)^T */
        for (int64_t c = 0; c < dk; ++c)
            for (int64_t j = 0; j < w; ++j) S[c * w + j] += bt * kt[c] * (vt[j] - p[j]);

        /* o_t = S_t^T q_t */
        double *ot = J->o + (t * H + h) * dv + j0;
        for (int64_t j = 0; j < w; ++j) ot[j] = 0.0;
        for (int64_t c = 0; c < dk; ++c)
            for (int64_t j = 0; j < w; ++j) ot[j] += qt[c] * S[c * w + j];
    }

    for (int64_t c = 0; c < dk; ++c)
        for (int64_t j = 0; j < w; ++j)
            J->S_out[((n * H + h) * dk + c) * dv + j0 + j] = S[c * w + j];
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    double *S = (double *)malloc(sizeof(double) * (size_t)(J->dk * J->bw));
    double *alpha = (double *)malloc(sizeof(double) * (size_t)J->dk);
    double *p = (double *)malloc(sizeof(double) * (size_t)J->bw);
    if (S && alpha && p) {
        for (;;) {
            int64_t u = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
            if (u >= J->n_units) break;
            run_unit(J, u, S, alpha, p);
        }
    } else {
        __atomic_store_n(&J->failed, 1, __ATOMIC_RELAXED);
    }
    free(S);
    free(alpha);
    free(p);
    return NULL;
}

int kda_oracle_hardware_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

/*
 * The recurrence over all sequences and heads. Returns 0 on success, -1 on a bad
 * argument, -2 when memory or threads cannot be had. 'threads' <= 0 uses every
 * online core. 'col_block' <= 0 picks 16 columns per work unit.
 */
int kda_oracle_recurrence(int delta, const double *q, const double *k, const double *v,
                          const double *la, const double *beta, const double *S0,
                          const int64_t *cu, int64_t N, int64_t H, int64_t dk, int64_t dv,
                          double *o, double *S_out, int threads, int64_t col_block) {
    if (!q || !k || !v || !la || !beta || !cu || !o || !S_out) return -1;
    if (N < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
    for (int64_t n = 0; n < N; ++n)
        if (cu[n + 1] < cu[n]) return -1;
    job_t J;
    memset(&J, 0, sizeof(J));
    J.delta = delta;
    J.q = q; J.k = k; J.v = v; J.la = la; J.beta = beta; J.S0 = S0; J.cu = cu;
    J.N = N; J.H = H; J.dk = dk; J.dv = dv;
    J.bw = (col_block > 0 && col_block < dv) ? col_block : (dv < 16 ? dv : 16);
    J.nblk = (dv + J.bw - 1) / J.bw;
    J.o = o; J.S_out = S_out;
    J.n_units = N * H * J.nblk;
    J.next = 0;
    if (J.n_units == 0) return 0;

    int nt = threads > 0 ? threads : kda_oracle_hardware_threads();
    if (nt > J.n_units) nt = (int)J.n_units;
    if (nt <= 1) {
        worker(&J);
        return J.failed ? -2 : 0;
    }
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nt);
    if (!tid) return -2;
    int started = 0;
    for (int i = 0; i < nt; ++i) {
        if (pthread_create(&tid[i], NULL, worker, &J) != 0) break;
        ++started;
    }
    if (started == 0) worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(tid[i], NULL);
    free(tid);
    /* a worker that failed took no unit; the others drained the queue, unless all failed */
    return (J.failed && J.next < J.n_units) ? -2 : 0;
}
