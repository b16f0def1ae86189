/*
 * KDA oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, double-precision CPU statement of what the KDA state path
 * computes.  Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load this file's library; the product path never does.  It shares
 * no code, header, table or helper with the CUDA library.
 *
 * The method (Kimi Delta Attention, gated delta rule) per (sequence, head)
 * unit with a K x V state S (row k = key channel, column v = value channel):
 *
 *     alpha_t = exp(gk_t)                                  (per key channel)
 *     S_t     = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *     o_t     = S_t^T (scale * q_t)                        (post-update state)
 *
 * Sources: "SGLang and Miles Add Day-0 Support for Kimi K3" (lmsys.org),
 * section "ReplaySSM: raw-input replay for the KDA state" names the per-step
 * inputs S_i = (v_i, k_i, gk_i, beta_i) and K = V = 128; the Kimi K3 on B200
 * deployment notes (zdszero.github.io), timeline entry "FlashKDA", give the
 * [128, 128] fp32 state.  The pages never print the formula; the recurrence
 * above is the problem statement this library is built to, and the oracle is
 * that definition written out.
 *
 * Parity status: every function here is pinned by tests in
 * tests/test_oracle_pins.py (closed forms, invariants, brute force on tiny
 * inputs, chunked == sequential).  No function is "parity unpinned".
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* One token of the recurrence, written as the definition.                   */
/* ------------------------------------------------------------------------ */

/*
 * S (K x V, row-major) <- (I - beta k k^T) Diag(exp(gk)) S + beta k v^T
 * o (V)                <- S^T (scale q)                 (skipped if o == NULL)
 * M is a K x V scratch matrix and kM a V-vector scratch.
 */
static void token_step(int K, int V, double *S, const double *q,
                       const double *k, const double *v, const double *gk,
                       double beta, double scale, double *o, double *M,
                       double *kM)
{
    /* M = Diag(exp(gk)) S : row i scaled by exp(gk_i) */
    for (int i = 0; i < K; ++i) {
        double a = exp(gk[i]);
        for (int j = 0; j < V; ++j) M[(size_t)i * V + j] = a * S[(size_t)i * V + j];
    }
    /* kM = k^T M  (a row vector over V) */
    for (int j = 0; j < V; ++j) kM[j] = 0.0;
    for (int i = 0; i < K; ++i)
        for (int j = 0; j < V; ++j) kM[j] += k[i] * M[(size_t)i * V + j];
    /* S = M - beta k (k^T M) + beta k v^T */
    for (int i = 0; i < K; ++i)
        for (int j = 0; j < V; ++j)
            S[(size_t)i * V + j] = M[(size_t)i * V + j] - beta * k[i] * kM[j]
                                   + beta * k[i] * v[j];
    if (o) {
        /* o = S^T (scale q) */
        for (int j = 0; j < V; ++j) o[j] = 0.0;
        for (int i = 0; i < K; ++i) {
            double sq = scale * q[i];
            for (int j = 0; j < V; ++j) o[j] += S[(size_t)i * V + j] * sq;
        }
    }
}

/*
 * Sequential recurrence over T tokens of one unit.  Token t of the unit reads
 * q/k/gk at t*sk, v at t*sv, beta at t*sb and writes o at t*so (o may be NULL).
 * S is the unit's state, read as S_0 and overwritten with S_T.
 */
void kda_oracle_unit(int T, int K, int V, long sk, long sv, long sb, long so,
                     const double *q, const double *k, const double *v,
                     const double *gk, const double *beta, double scale,
                     double *S, double *o)
{
    double *M = (double *)malloc(sizeof(double) * (size_t)K * V);
    double *kM = (double *)malloc(sizeof(double) * (size_t)V);
    for (int t = 0; t < T; ++t)
        token_step(K, V, S, q + t * sk, k + t * sk, v + t * sv, gk + t * sk,
                   beta[t * sb], scale, o ? o + t * so : NULL, M, kM);
    free(M);
    free(kM);
}

/* ------------------------------------------------------------------------ */
/* Chunked (UT / WY) form -- used only to check "chunked == sequential".     */
/* ------------------------------------------------------------------------ */

/*
 * Same result as kda_oracle_unit, computed chunk by chunk (chunk length C).
 * Within a chunk starting from state S0, with G_r = sum_{j<=r} gk_j (per key
 * channel, inclusive) and G_L the chunk's last row:
 *
 *   u_r = beta_r ( v_r - S0^T (exp(G_r) . k_r) )
 *         - sum_{j<r} beta_r <k_r, exp(G_r - G_j) . k_j> u_j     (forward subst.)
 *   o_r = scale [ S0^T (exp(G_r) . q_r)
 *                 + sum_{j<=r} <q_r, exp(G_r - G_j) . k_j> u_j ]
 *   S_L = Diag(exp(G_L)) S0 + sum_j (exp(G_L - G_j) . k_j) u_j^T
 *
 * These follow from unrolling the recurrence inside the chunk: the state
 * after token r equals Diag(exp(G_r)) [S0 + sum_{j<=r} (exp(-G_j) . k_j) u_j^T]
 * with u_j the delta-rule correction beta_j (v_j - S_{j-1}^T Diag(alpha_j) k_j).
 * The pairwise exponentials are formed from exact differences G_r - G_j.
 */
void kda_oracle_unit_chunked(int T, int K, int V, int C, long sk, long sv,
                             long sb, long so, const double *q, const double *k,
                             const double *v, const double *gk,
                             const double *beta, double scale, double *S,
                             double *o)
{
    double *G = (double *)malloc(sizeof(double) * (size_t)C * K);
    double *U = (double *)malloc(sizeof(double) * (size_t)C * V);
    double *Snew = (double *)malloc(sizeof(double) * (size_t)K * V);
    for (int c0 = 0; c0 < T; c0 += C) {
        int L = (T - c0 < C) ? (T - c0) : C;
        /* cumulative log-decay inside the chunk */
        for (int r = 0; r < L; ++r)
            for (int i = 0; i < K; ++i)
                G[(size_t)r * K + i] = gk[(c0 + r) * sk + i] + (r ? G[(size_t)(r - 1) * K + i] : 0.0);
        /* u by forward substitution */
        for (int r = 0; r < L; ++r) {
            const double *kr = k + (c0 + r) * sk;
            double br = beta[(c0 + r) * sb];
            for (int j = 0; j < V; ++j) {
                double acc = 0.0;
                for (int i = 0; i < K; ++i)
                    acc += S[(size_t)i * V + j] * exp(G[(size_t)r * K + i]) * kr[i];
                U[(size_t)r * V + j] = br * (v[(c0 + r) * sv + j] - acc);
            }
            for (int jj = 0; jj < r; ++jj) {
                const double *kj = k + (c0 + jj) * sk;
                double a = 0.0;
                for (int i = 0; i < K; ++i)
                    a += kr[i] * exp(G[(size_t)r * K + i] - G[(size_t)jj * K + i]) * kj[i];
                a *= br;
                for (int j = 0; j < V; ++j) U[(size_t)r * V + j] -= a * U[(size_t)jj * V + j];
            }
        }
        /* outputs */
        if (o) {
            for (int r = 0; r < L; ++r) {
                const double *qr = q + (c0 + r) * sk;
                double *orow = o + (c0 + r) * so;
                for (int j = 0; j < V; ++j) {
                    double acc = 0.0;
                    for (int i = 0; i < K; ++i)
                        acc += S[(size_t)i * V + j] * exp(G[(size_t)r * K + i]) * qr[i];
                    orow[j] = acc;
                }
                for (int jj = 0; jj <= r; ++jj) {
                    const double *kj = k + (c0 + jj) * sk;
                    double a = 0.0;
                    for (int i = 0; i < K; ++i)
                        a += qr[i] * exp(G[(size_t)r * K + i] - G[(size_t)jj * K + i]) * kj[i];
                    for (int j = 0; j < V; ++j) orow[j] += a * U[(size_t)jj * V + j];
                }
                for (int j = 0; j < V; ++j) orow[j] *= scale;
            }
        }
        /* end-of-chunk state */
        for (int i = 0; i < K; ++i) {
            double gl = G[(size_t)(L - 1) * K + i];
            for (int j = 0; j < V; ++j) Snew[(size_t)i * V + j] = exp(gl) * S[(size_t)i * V + j];
            for (int jj = 0; jj < L; ++jj) {
                double f = exp(gl - G[(size_t)jj * K + i]) * k[(c0 + jj) * sk + i];
                for (int j = 0; j < V; ++j) Snew[(size_t)i * V + j] += f * U[(size_t)jj * V + j];
            }
        }
        memcpy(S, Snew, sizeof(double) * (size_t)K * V);
    }
    free(G);
    free(U);
    free(Snew);
}

/* ------------------------------------------------------------------------ */
/* Many independent units on host threads.                                   */
/* ------------------------------------------------------------------------ */

/*
 * A batch of independent (sequence or request, head) units over packed
 * inputs q/k/gk [tokens, H, K], v [tokens, H, V], beta [tokens, H] and
 * o [tokens, H, V].  Unit u runs T[u] tokens starting at token tok0[u] on head
 * head[u] with state S[u] (K x V, in/out).  C <= 0 selects the sequential
 * form, C > 0 the chunked form with chunk length C.  o may be NULL.
 */
typedef struct {
    int n_units, H, K, V, C;
    const long *tok0;
    const int *T, *head;
    const double *q, *k, *v, *gk, *beta;
    double scale;
    double *S, *o;
    int next;
    pthread_mutex_t lock;
} batch_job;

static void *batch_worker(void *arg)
{
    batch_job *J = (batch_job *)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int u = J->next++;
        pthread_mutex_unlock(&J->lock);
        if (u >= J->n_units) break;
        long t0 = J->tok0[u];
        int h = J->head[u];
        long sk = (long)J->H * J->K, sv = (long)J->H * J->V, sb = J->H;
        const double *q = J->q + t0 * sk + (long)h * J->K;
        const double *k = J->k + t0 * sk + (long)h * J->K;
        const double *gk = J->gk + t0 * sk + (long)h * J->K;
        const double *v = J->v + t0 * sv + (long)h * J->V;
        const double *b = J->beta + t0 * sb + h;
        double *o = J->o ? J->o + t0 * sv + (long)h * J->V : NULL;
        double *S = J->S + (size_t)u * J->K * J->V;
        if (J->C > 0)
            kda_oracle_unit_chunked(J->T[u], J->K, J->V, J->C, sk, sv, sb, sv,
                                    q, k, v, gk, b, J->scale, S, o);
        else
            kda_oracle_unit(J->T[u], J->K, J->V, sk, sv, sb, sv, q, k, v, gk, b,
                            J->scale, S, o);
    }
    return NULL;
}

int kda_oracle_batch(int n_units, const long *tok0, const int *T,
                     const int *head, int H, int K, int V, int C,
                     const double *q, const double *k, const double *v,
                     const double *gk, const double *beta, double scale,
                     double *S, double *o, int nthreads)
{
    batch_job J;
    J.n_units = n_units; J.H = H; J.K = K; J.V = V; J.C = C;
    J.tok0 = tok0; J.T = T; J.head = head;
    J.q = q; J.k = k; J.v = v; J.gk = gk; J.beta = beta;
    J.scale = scale; J.S = S; J.o = o; J.next = 0;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n_units) nthreads = n_units > 0 ? n_units : 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int started = 0;
    for (int i = 1; i < nthreads; ++i)
        if (pthread_create(&th[started], NULL, batch_worker, &J) == 0) ++started;
    /* the calling thread works too */
    batch_worker(&J);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.lock);
    return started + 1;
}
