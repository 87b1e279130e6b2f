/*
 * kda_oracle.c -- fp64 token-by-token reference for the KDA operator.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  It shares no code with the CUDA
 * path and neither side includes the other.
 *
 * What it computes (Kimi Delta Attention, "Kimi Delta Attention" deep dive,
 * section 03, the recurrence quoted from the Kimi Linear report, and
 * section 02 for the read):
 *
 *     S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t = S_t^T q_t
 *
 * per sequence and per head, with S a d_k x d_v matrix (rows = key channels,
 * d_v contiguous).  Read right to left, as the deep dive does: first every row
 * i of S is scaled by alpha_t[i]; then the decayed state's prediction at k_t,
 * S'^T k_t, is subtracted from v_t; then beta_t k_t (error)^T is added.  The
 * output is read from the updated state.  alpha_t = exp(log_alpha_t).
 *
 * Columns of S never interact (every operation above acts on one column j
 * using only column j of S and element j of v_t), so the work is split over
 * (sequence, head, block of columns) and run on POSIX threads; each column's
 * arithmetic, and its order, is the same whatever the split.
 *
 * Layouts (row-major, all fp64): q, k, log_alpha [T, H, d_k]; v, out
 * [T, H, d_v]; beta [T, H]; states [N, H, d_k, d_v]; cu_seqlens int32 [N+1].
 */
#include <math.h>
#include <pthread.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t num_seqs, H, dk, dv;
    const int32_t *cu;
    const double *q, *k, *v, *la, *beta, *s0;
    double *out, *sfinal;
    int32_t col_begin, col_end, col_block;
    int64_t num_items;
    atomic_llong next;
} job_t;

/* One (sequence, head) over columns [j0, j1): the recurrence, token by token. */
static void run_item(const job_t *J, int32_t n, int32_t h, int32_t j0, int32_t j1,
                     double *S, double *alpha, double *err)
{
    const int32_t H = J->H, dk = J->dk, dv = J->dv;
    const int64_t t0 = J->cu[n], t1 = J->cu[n + 1];
    const size_t sbase = ((size_t)n * H + h) * (size_t)dk * dv;

    /* S <- initial state (zeros when none is given). */
    for (int32_t i = 0; i < dk; ++i)
        for (int32_t j = j0; j < j1; ++j)
            S[(size_t)i * dv + j] = J->s0 ? J->s0[sbase + (size_t)i * dv + j] : 0.0;

    for (int64_t t = t0; t < t1; ++t) {
        const double *qt = J->q + ((size_t)t * H + h) * dk;
        const double *kt = J->k + ((size_t)t * H + h) * dk;
        const double *lat = J->la + ((size_t)t * H + h) * dk;
        const double *vt = J->v + ((size_t)t * H + h) * dv;
        const double bt = J->beta[(size_t)t * H + h];
        double *ot = J->out + ((size_t)t * H + h) * dv;

        /* alpha_t = exp(log alpha_t); decay: S' = Diag(alpha_t) S (rows). */
        for (int32_t i = 0; i < dk; ++i) alpha[i] = exp(lat[i]);
        for (int32_t i = 0; i < dk; ++i)
            for (int32_t j = j0; j < j1; ++j)
                S[(size_t)i * dv + j] *= alpha[i];

        /* error = v_t - S'^T k_t (what the decayed memory predicts at k_t). */
        for (int32_t j = j0; j < j1; ++j) {
            double pred = 0.0;
            for (int32_t i = 0; i < dk; ++i) pred += kt[i] * S[(size_t)i * dv + j];
            err[j] = vt[j] - pred;
        }

        /* correct-and-write: S = S' + beta_t k_t error^T
         * (= (I - beta k k^T) S' + beta k v^T). */
        for (int32_t i = 0; i < dk; ++i) {
            const double bk = bt * kt[i];
            for (int32_t j = j0; j < j1; ++j) S[(size_t)i * dv + j] += bk * err[j];
        }

        /* read after the update: o_t = S_t^T q_t. */
        for (int32_t j = j0; j < j1; ++j) {
            double o = 0.0;
            for (int32_t i = 0; i < dk; ++i) o += qt[i] * S[(size_t)i * dv + j];
            ot[j] = o;
        }
    }

    if (J->sfinal)
        for (int32_t i = 0; i < dk; ++i)
            for (int32_t j = j0; j < j1; ++j)
                J->sfinal[sbase + (size_t)i * dv + j] = S[(size_t)i * dv + j];
}

static void *worker(void *arg)
{
    job_t *J = (job_t *)arg;
    double *S = (double *)malloc(sizeof(double) * (size_t)J->dk * J->dv);
    double *alpha = (double *)malloc(sizeof(double) * (size_t)J->dk);
    double *err = (double *)malloc(sizeof(double) * (size_t)J->dv);
    if (!S || !alpha || !err) { free(S); free(alpha); free(err); return (void *)1; }
    const int32_t ncols = J->col_end - J->col_begin;
    const int32_t nblk = (ncols + J->col_block - 1) / J->col_block;
    for (;;) {
        long long it = atomic_fetch_add(&J->next, 1);
        if (it >= J->num_items) break;
        const int32_t b = (int32_t)(it % nblk);
        const int64_t nh = it / nblk;
        const int32_t h = (int32_t)(nh % J->H), n = (int32_t)(nh / J->H);
        const int32_t j0 = J->col_begin + b * J->col_block;
        const int32_t j1 = j0 + J->col_block < J->col_end ? j0 + J->col_block : J->col_end;
        run_item(J, n, h, j0, j1, S, alpha, err);
    }
    free(S); free(alpha); free(err);
    return NULL;
}

/*
 * Prefill over a packed batch.  Columns [col_begin, col_end) of out and of
 * final_state are written (pass 0, d_v for all of them); the rest is left
 * untouched.  initial_state may be NULL (zero state) and may alias
 * final_state.  final_state may be NULL.  Returns 0 on success, -1 on bad
 * arguments, -2 if a thread could not be started or ran out of memory.
 */
int kda_oracle_prefill(int32_t num_seqs, int32_t H, int32_t dk, int32_t dv,
                       const int32_t *cu_seqlens,
                       const double *q, const double *k, const double *v,
                       const double *log_alpha, const double *beta,
                       const double *initial_state, double *out, double *final_state,
                       int32_t col_begin, int32_t col_end, int32_t num_threads)
{
    if (num_seqs < 0 || H <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens) return -1;
    if (col_begin < 0 || col_end > dv || col_begin > col_end) return -1;
    for (int32_t n = 0; n < num_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
    if (num_seqs == 0 || col_begin == col_end) return 0;

    job_t J;
    memset(&J, 0, sizeof(J));
    J.num_seqs = num_seqs; J.H = H; J.dk = dk; J.dv = dv; J.cu = cu_seqlens;
    J.q = q; J.k = k; J.v = v; J.la = log_alpha; J.beta = beta;
    J.s0 = initial_state; J.out = out; J.sfinal = final_state;
    J.col_begin = col_begin; J.col_end = col_end;
    if (num_threads < 1) num_threads = 1;
    const int32_t ncols = col_end - col_begin;
    /* Enough column blocks to keep every thread busy, at least 8 columns each. */
    int32_t nblk = 1;
    while ((int64_t)num_seqs * H * nblk < 4LL * num_threads && ncols / (nblk * 2) >= 8) nblk *= 2;
    J.col_block = (ncols + nblk - 1) / nblk;
    nblk = (ncols + J.col_block - 1) / J.col_block;
    J.num_items = (int64_t)num_seqs * H * nblk;
    atomic_init(&J.next, 0);

    if (num_threads > J.num_items) num_threads = (int32_t)J.num_items;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)num_threads);
    if (!th) return -2;
    int started = 0, rc = 0;
    for (int32_t i = 0; i < num_threads; ++i) {
        if (pthread_create(&th[i], NULL, worker, &J) != 0) { rc = -2; break; }
        ++started;
    }
    if (started == 0) rc = -2, worker(&J);   /* keep going single-threaded */
    for (int i = 0; i < started; ++i) {
        void *ret = NULL;
        pthread_join(th[i], &ret);
        if (ret) rc = -2;
    }
    free(th);
    return rc;
}

/*
 * One decode step: every sequence advances by exactly one token, its state
 * updated in place (the same recurrence at T = 1).  Inputs are [N, H, *].
 */
int kda_oracle_decode_step(int32_t num_seqs, int32_t H, int32_t dk, int32_t dv,
                           const double *q, const double *k, const double *v,
                           const double *log_alpha, const double *beta,
                           double *state_inout, double *out, int32_t num_threads)
{
    if (num_seqs < 0) return -1;
    int32_t *cu = (int32_t *)malloc(sizeof(int32_t) * ((size_t)num_seqs + 1));
    if (!cu) return -2;
    for (int32_t n = 0; n <= num_seqs; ++n) cu[n] = n;
    int rc = kda_oracle_prefill(num_seqs, H, dk, dv, cu, q, k, v, log_alpha, beta,
                                state_inout, out, state_inout, 0, dv, num_threads);
    free(cu);
    return rc;
}
