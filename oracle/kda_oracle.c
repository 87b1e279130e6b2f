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

/*
 * Reverse mode (gradients) of the prefill.  Given the gradient of a scalar
 * loss with respect to every output, dout [T, H, d_v], and with respect to
 * the final state, dfinal [N, H, d_k, d_v] (NULL: zero), it returns the
 * gradients with respect to q, k, v, log_alpha ([T, H, d_k] / [T, H, d_v]),
 * beta [T, H] and the initial state ds0 [N, H, d_k, d_v] (NULL: not wanted).
 *
 * Per sequence and head the forward recurrence above is re-run to recover
 * the states, then the chain rule is applied to each token's step in reverse
 * order.  With S' = Diag(alpha_t) S_{t-1}, e = v_t - S'^T k_t,
 * S_t = S' + beta_t k_t e^T and o_t = S_t^T q_t, and dS the gradient with
 * respect to S_t (everything after t folded in):
 *
 *   read:   dq_t = S_t do_t;            dS += q_t do_t^T
 *   write:  u = dS^T k_t;  de = beta_t u;  dbeta_t = e . u;  dv_t = de
 *           dk_t = beta_t dS e - S' de
 *           dS' = dS - k_t de^T
 *   decay:  dlog_alpha_t[i] = alpha_t[i] sum_j dS'[i][j] S_{t-1}[i][j]
 *           dS_{t-1} = Diag(alpha_t) dS'
 *
 * and ds0 = dS after the first token.  States are kept at every
 * kCheckpoint-th token and the ones in between recomputed segment by segment
 * (the same arithmetic in the same order, so the same values); this bounds
 * memory at (L / kCheckpoint + kCheckpoint) states per (sequence, head).
 * Threads split the (sequence, head) pairs.  Returns 0, -1 on bad arguments,
 * -2 if memory or a thread could not be had.
 */
enum { kCheckpoint = 32 };

typedef struct {
    int32_t num_seqs, H, dk, dv;
    const int32_t *cu;
    const double *q, *k, *v, *la, *beta, *s0, *dout, *dfinal;
    double *dq, *dk_, *dv_, *dla, *dbeta, *ds0;
    atomic_llong next;
    atomic_int failed;
} bjob_t;

/* One forward step of the recurrence on the full state (all columns). */
static void fwd_step(const bjob_t *B, int64_t t, int32_t h, const double *Sprev, double *Snext,
                     double *alpha, double *err)
{
    const int32_t H = B->H, dk = B->dk, dv = B->dv;
    const double *kt = B->k + ((size_t)t * H + h) * dk;
    const double *lat = B->la + ((size_t)t * H + h) * dk;
    const double *vt = B->v + ((size_t)t * H + h) * dv;
    const double bt = B->beta[(size_t)t * H + h];
    for (int32_t i = 0; i < dk; ++i) alpha[i] = exp(lat[i]);
    for (int32_t i = 0; i < dk; ++i)
        for (int32_t j = 0; j < dv; ++j)
            Snext[(size_t)i * dv + j] = alpha[i] * Sprev[(size_t)i * dv + j];
    for (int32_t j = 0; j < dv; ++j) {
        double pred = 0.0;
        for (int32_t i = 0; i < dk; ++i) pred += kt[i] * Snext[(size_t)i * dv + j];
        err[j] = vt[j] - pred;
    }
    for (int32_t i = 0; i < dk; ++i) {
        const double bk = bt * kt[i];
        for (int32_t j = 0; j < dv; ++j) Snext[(size_t)i * dv + j] += bk * err[j];
    }
}

static int bwd_item(const bjob_t *B, int32_t n, int32_t h)
{
    const int32_t H = B->H, dk = B->dk, dv = B->dv;
    const int64_t t0 = B->cu[n], t1 = B->cu[n + 1], L = t1 - t0;
    const size_t SZ = (size_t)dk * dv;
    const size_t sbase = ((size_t)n * H + h) * SZ;
    const int64_t ncp = L / kCheckpoint + 1;                  /* states at t0 + m * kCheckpoint */
    double *cp = (double *)malloc(sizeof(double) * SZ * (size_t)ncp);
    double *seg = (double *)malloc(sizeof(double) * SZ * (kCheckpoint + 1));
    double *dS = (double *)malloc(sizeof(double) * SZ);
    double *dSp = (double *)malloc(sizeof(double) * SZ);
    double *Sp = (double *)malloc(sizeof(double) * SZ);
    double *alpha = (double *)malloc(sizeof(double) * (size_t)dk);
    double *err = (double *)malloc(sizeof(double) * (size_t)dv);
    double *de = (double *)malloc(sizeof(double) * (size_t)dv);
    int rc = 0;
    if (!cp || !seg || !dS || !dSp || !Sp || !alpha || !err || !de) { rc = -2; goto done; }

    /* forward: checkpoints */
    for (size_t e = 0; e < SZ; ++e) cp[e] = B->s0 ? B->s0[sbase + e] : 0.0;
    {
        double *cur = seg, *nxt = seg + SZ;
        memcpy(cur, cp, sizeof(double) * SZ);
        for (int64_t r = 0; r < L; ++r) {
            fwd_step(B, t0 + r, h, cur, nxt, alpha, err);
            double *tmp = cur; cur = nxt; nxt = tmp;
            if ((r + 1) % kCheckpoint == 0) memcpy(cp + SZ * (size_t)((r + 1) / kCheckpoint), cur, sizeof(double) * SZ);
        }
    }
    /* reverse */
    for (size_t e = 0; e < SZ; ++e) dS[e] = B->dfinal ? B->dfinal[sbase + e] : 0.0;
    for (int64_t m = (L - 1) / kCheckpoint; L > 0 && m >= 0; --m) {
        const int64_t r0 = m * kCheckpoint, r1 = (r0 + kCheckpoint < L) ? r0 + kCheckpoint : L;
        memcpy(seg, cp + SZ * (size_t)m, sizeof(double) * SZ);          /* seg[s] = state after r0 + s tokens */
        for (int64_t r = r0; r < r1; ++r)
            fwd_step(B, t0 + r, h, seg + SZ * (size_t)(r - r0), seg + SZ * (size_t)(r - r0 + 1), alpha, err);
        for (int64_t r = r1 - 1; r >= r0; --r) {
            const int64_t t = t0 + r;
            const double *Sprev = seg + SZ * (size_t)(r - r0);
            const double *St = seg + SZ * (size_t)(r - r0 + 1);
            const double *qt = B->q + ((size_t)t * H + h) * dk;
            const double *kt = B->k + ((size_t)t * H + h) * dk;
            const double *lat = B->la + ((size_t)t * H + h) * dk;
            const double *vt = B->v + ((size_t)t * H + h) * dv;
            const double *dot = B->dout + ((size_t)t * H + h) * dv;
            const double bt = B->beta[(size_t)t * H + h];
            /* recompute S' and e for this token */
            for (int32_t i = 0; i < dk; ++i) alpha[i] = exp(lat[i]);
            for (int32_t i = 0; i < dk; ++i)
                for (int32_t j = 0; j < dv; ++j) Sp[(size_t)i * dv + j] = alpha[i] * Sprev[(size_t)i * dv + j];
            for (int32_t j = 0; j < dv; ++j) {
                double pred = 0.0;
                for (int32_t i = 0; i < dk; ++i) pred += kt[i] * Sp[(size_t)i * dv + j];
                err[j] = vt[j] - pred;
            }
            /* read: o_t = S_t^T q_t */
            for (int32_t i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (int32_t j = 0; j < dv; ++j) acc += St[(size_t)i * dv + j] * dot[j];
                B->dq[((size_t)t * H + h) * dk + i] = acc;
                for (int32_t j = 0; j < dv; ++j) dS[(size_t)i * dv + j] += qt[i] * dot[j];
            }
            /* write: S_t = S' + beta k e^T, e = v - S'^T k */
            double db = 0.0;
            for (int32_t j = 0; j < dv; ++j) {
                double a = 0.0;
                for (int32_t i = 0; i < dk; ++i) a += kt[i] * dS[(size_t)i * dv + j];
                de[j] = bt * a;
                db += err[j] * a;
                B->dv_[((size_t)t * H + h) * dv + j] = de[j];
            }
            B->dbeta[(size_t)t * H + h] = db;
            for (int32_t i = 0; i < dk; ++i) {
                double a = 0.0, b = 0.0;
                for (int32_t j = 0; j < dv; ++j) {
                    a += dS[(size_t)i * dv + j] * err[j];
                    b += Sp[(size_t)i * dv + j] * de[j];
                }
                B->dk_[((size_t)t * H + h) * dk + i] = bt * a - b;
            }
            for (int32_t i = 0; i < dk; ++i)
                for (int32_t j = 0; j < dv; ++j) dSp[(size_t)i * dv + j] = dS[(size_t)i * dv + j] - kt[i] * de[j];
            /* decay: S' = Diag(alpha) S_{t-1} */
            for (int32_t i = 0; i < dk; ++i) {
                double a = 0.0;
                for (int32_t j = 0; j < dv; ++j) a += dSp[(size_t)i * dv + j] * Sprev[(size_t)i * dv + j];
                B->dla[((size_t)t * H + h) * dk + i] = alpha[i] * a;
                for (int32_t j = 0; j < dv; ++j) dS[(size_t)i * dv + j] = alpha[i] * dSp[(size_t)i * dv + j];
            }
        }
    }
    if (B->ds0) memcpy(B->ds0 + sbase, dS, sizeof(double) * SZ);
done:
    free(cp); free(seg); free(dS); free(dSp); free(Sp); free(alpha); free(err); free(de);
    return rc;
}

static void *bworker(void *arg)
{
    bjob_t *B = (bjob_t *)arg;
    const long long items = (long long)B->num_seqs * B->H;
    for (;;) {
        long long it = atomic_fetch_add(&B->next, 1);
        if (it >= items) break;
        if (bwd_item(B, (int32_t)(it / B->H), (int32_t)(it % B->H)) != 0) atomic_store(&B->failed, 1);
    }
    return NULL;
}

int kda_oracle_backward(int32_t num_seqs, int32_t H, int32_t dk, int32_t dv,
                        const int32_t *cu_seqlens,
                        const double *q, const double *k, const double *v,
                        const double *log_alpha, const double *beta, const double *initial_state,
                        const double *dout, const double *dfinal,
                        double *dq, double *dk_out, double *dv_out, double *dlog_alpha, double *dbeta,
                        double *dinitial, int32_t num_threads)
{
    if (num_seqs < 0 || H <= 0 || dk <= 0 || dv <= 0 || !cu_seqlens) return -1;
    for (int32_t n = 0; n < num_seqs; ++n)
        if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
    if (num_seqs == 0) return 0;
    bjob_t B;
    memset(&B, 0, sizeof(B));
    B.num_seqs = num_seqs; B.H = H; B.dk = dk; B.dv = dv; B.cu = cu_seqlens;
    B.q = q; B.k = k; B.v = v; B.la = log_alpha; B.beta = beta; B.s0 = initial_state;
    B.dout = dout; B.dfinal = dfinal;
    B.dq = dq; B.dk_ = dk_out; B.dv_ = dv_out; B.dla = dlog_alpha; B.dbeta = dbeta; B.ds0 = dinitial;
    atomic_init(&B.next, 0);
    atomic_init(&B.failed, 0);
    const long long items = (long long)num_seqs * H;
    if (num_threads < 1) num_threads = 1;
    if (num_threads > items) num_threads = (int32_t)items;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)num_threads);
    if (!th) return -2;
    int started = 0;
    for (int32_t i = 0; i < num_threads; ++i) {
        if (pthread_create(&th[i], NULL, bworker, &B) != 0) break;
        ++started;
    }
    if (started == 0) bworker(&B);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    return atomic_load(&B.failed) ? -2 : 0;
}
