/*
 * Oracle for the gated delta rule forward pass: TEST INFRASTRUCTURE ONLY.
 *
 * Plain fp64 CPU implementation of the sequential recurrence, token by token.
 * It shares no code, header, table or helper with the CUDA path, and the
 * product path never calls it: only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load it.
 *
 * What it computes (north-star recurrence; "从零开始的 GDN 推导", §"Gated Delta
 * Rule Chunk-wise Parallel 前向推导", recurrent form, transposed to the
 * column-vector orientation with S in R^{d_v x d_k}; "RNN的复兴03：现代RNN的并行
 * 计算", §二 eq. for S_t with a separate write strength eta):
 *
 *     S_t = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + eta_t v_t k_t^T
 *     o_t = S_t q_t                     (post-update state, token t included)
 *
 * with eta_t = beta_t unless an explicit eta is passed.  Expanding the product
 * gives the rank-1 form used below, exact in real arithmetic:
 *
 *     r   = S_{t-1} k_t
 *     S_t = alpha_t S_{t-1} + (eta_t v_t - alpha_t beta_t r) k_t^T
 *
 * Layouts (row-major, C order):
 *   q [B,T,H,d_k]  k [B,T,H,d_k]  v [B,T,H,d_v]  o [B,T,H,d_v]
 *   log_alpha, beta, eta [B,T,H]
 *   S0, S_final [N,H,d_v,d_k]   (N = B; with cu_seqlens the token axis is the
 *   packed axis of length T and sequence n spans [cu[n], cu[n+1]) )
 *
 * Parity is pinned by the tests against explicit dense matrix products, the
 * WY identity of the DPLR product, and closed forms (linear attention, the
 * scalar-gated form, retrieval, pure decay).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    const double *q, *k, *v, *log_alpha, *beta, *eta, *S0;
    double *o, *S_final;
    int N, H, T, dk, dv;
    const int32_t *cu;
    int next_unit; /* guarded by mu */
    pthread_mutex_t mu;
} oracle_job;

/* One (sequence, head) unit, token by token. */
static void run_unit(const oracle_job *J, int n, int h, double *S, double *r)
{
    const int H = J->H, dk = J->dk, dv = J->dv;
    long start, len;
    if (J->cu) {
        start = J->cu[n];
        len = (long)J->cu[n + 1] - J->cu[n];
    } else {
        start = (long)n * J->T;
        len = J->T;
    }
    const size_t sN = (size_t)dv * dk;
    if (J->S0)
        memcpy(S, J->S0 + ((size_t)n * H + h) * sN, sN * sizeof(double));
    else
        memset(S, 0, sN * sizeof(double));

    for (long t = 0; t < len; ++t) {
        const size_t tok = (size_t)(start + t) * H + h; /* index into [*,T,H] */
        const double *kt = J->k + tok * dk;
        const double *qt = J->q + tok * dk;
        const double *vt = J->v + tok * dv;
        const double a = exp(J->log_alpha[tok]);
        const double b = J->beta[tok];
        const double e = J->eta ? J->eta[tok] : b;
        /* r = S k */
        for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            const double *Si = S + (size_t)i * dk;
            for (int j = 0; j < dk; ++j) acc += Si[j] * kt[j];
            r[i] = acc;
        }
        /* S = a S + (e v - a b r) k^T */
        for (int i = 0; i < dv; ++i) {
            const double c = e * vt[i] - a * b * r[i];
            double *Si = S + (size_t)i * dk;
            for (int j = 0; j < dk; ++j) Si[j] = a * Si[j] + c * kt[j];
        }
        /* o = S q */
        double *ot = J->o + tok * dv;
        for (int i = 0; i < dv; ++i) {
            double acc = 0.0;
            const double *Si = S + (size_t)i * dk;
            for (int j = 0; j < dk; ++j) acc += Si[j] * qt[j];
            ot[i] = acc;
        }
    }
    if (J->S_final)
        memcpy(J->S_final + ((size_t)n * H + h) * sN, S, sN * sizeof(double));
}

static void *worker(void *arg)
{
    oracle_job *J = (oracle_job *)arg;
    double *S = (double *)malloc(sizeof(double) * (size_t)J->dv * J->dk);
    double *r = (double *)malloc(sizeof(double) * (size_t)J->dv);
    if (!S || !r) {
        free(S);
        free(r);
        return (void *)1;
    }
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int u = J->next_unit++;
        pthread_mutex_unlock(&J->mu);
        if (u >= J->N * J->H) break;
        run_unit(J, u / J->H, u % J->H, S, r);
    }
    free(S);
    free(r);
    return NULL;
}

/*
 * Returns 0 on success, -1 on bad arguments, -2 on allocation/thread failure.
 * n_threads <= 0 means one thread.  Units (sequence, head) are independent, so
 * the result does not depend on the thread count.
 */
int gdn_oracle_f64(const double *q, const double *k, const double *v,
                   const double *log_alpha, const double *beta, const double *eta,
                   const double *S0, double *o, double *S_final,
                   int B, int H, int T, int dk, int dv,
                   const int32_t *cu_seqlens, int n_threads)
{
    if (B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0) return -1;
    if (B == 0 || H == 0) return 0;
    if (!q || !k || !v || !log_alpha || !beta || !o) return -1;
    if (cu_seqlens) {
        if (cu_seqlens[0] != 0 || cu_seqlens[B] != T) return -1;
        for (int n = 0; n < B; ++n)
            if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
    }
    oracle_job J;
    J.q = q; J.k = k; J.v = v; J.log_alpha = log_alpha; J.beta = beta; J.eta = eta;
    J.S0 = S0; J.o = o; J.S_final = S_final;
    J.N = B; J.H = H; J.T = T; J.dk = dk; J.dv = dv; J.cu = cu_seqlens;
    J.next_unit = 0;
    pthread_mutex_init(&J.mu, NULL);
    if (n_threads < 1) n_threads = 1;
    if (n_threads > B * H) n_threads = B * H;
    int rc = 0;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    if (!th) {
        pthread_mutex_destroy(&J.mu);
        return -2;
    }
    int started = 0;
    for (int i = 0; i < n_threads; ++i) {
        if (pthread_create(&th[i], NULL, worker, &J) != 0) break;
        ++started;
    }
    if (started == 0) {
        /* run inline */
        if (worker(&J) != NULL) rc = -2;
    }
    for (int i = 0; i < started; ++i) {
        void *ret = NULL;
        pthread_join(th[i], &ret);
        if (ret != NULL) rc = -2;
    }
    free(th);
    pthread_mutex_destroy(&J.mu);
    return rc;
}
