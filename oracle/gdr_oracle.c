/*
 * gdr_oracle.c -- CPU FP64 oracle for the gated delta rule forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: it is built and used by the tests, by the smoke check and
 * by the CPU-baseline leg of the benchmark.  It shares no code, header,
 * table or helper with the CUDA library.
 *
 * What it computes (the plain definition, token by token, no chunking):
 *
 *   Per-token recurrence of gated delta-rule linear attention, as stated in
 *   the chunked-gated-delta-rule pages (cuLA PR #127 "Summary": the serial
 *   state recurrence; fla state-scan kernel, Kev PR #259 intro) and written
 *   out in full in the project statement:
 *
 *       S_t = alpha_t * S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T
 *       o_t = S_t q_t / sqrt(K)
 *
 *   with alpha_t = exp(g_t), g_t the per-token log gate.  The state is stored
 *   transposed, h = S^T (K x V), so that one update reads
 *
 *       h <- alpha h;   u = beta (v - h^T k);   h <- h + k u^T
 *
 *   which equals alpha (I - beta k k^T) h_prev + beta k v^T.  In the
 *   beta-free (pure gated linear attention) mode the write is h <- h + k v^T.
 *
 *   The readout scale defaults to 1/sqrt(K); the caller passes it.
 *
 * Also provided: the affine map of the recurrence over a token range,
 * h_out = M h_in + c (M: K x K, c: K x V), the segment summary the
 * segment-split mode composes (cuLA PR #127 "Root cause and implementation":
 * local state plus affine transition per segment).
 *
 * Layouts (row-major, contiguous, FP64):
 *   q, k  [B, T, H, K]     v, o  [B, T, H, V]     g, beta  [B, T, H]
 *   h0, ht [N, H, K, V]    cu_seqlens int64 [N + 1] (varlen: B == 1)
 *
 * Parity pins: every function here is checked in tests/test_oracle_pins.py
 * against independent formulations (explicit S-matrix product, chunked WY
 * form with a library inverse, O(T^2) closed forms, exact retrieval with
 * orthonormal keys, per-sequence runs, state carry, linearity).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    const double *q, *k, *v, *g, *beta, *h0;
    double *o, *ht;
    const int64_t *cu;
    const uint8_t *pair_mask;
    int64_t B, T, H, K, V, N;
    double scale;
    int64_t next;
    int failed;
    pthread_mutex_t mu;
} fwd_job;

/* One (sequence n, head h) pair: the token loop. */
static int run_pair(fwd_job *J, int64_t n, int64_t hh)
{
    const int64_t H = J->H, K = J->K, V = J->V;
    int64_t row, t0, t1;
    if (J->cu) {
        row = 0;
        t0 = J->cu[n];
        t1 = J->cu[n + 1];
    } else {
        row = n;
        t0 = 0;
        t1 = J->T;
    }
    double *S = (double *)malloc(sizeof(double) * (size_t)(K * V));
    double *u = (double *)malloc(sizeof(double) * (size_t)V);
    if (!S || !u) {
        free(S);
        free(u);
        return -1;
    }
    const int64_t sidx = (n * H + hh) * K * V;
    if (J->h0)
        memcpy(S, J->h0 + sidx, sizeof(double) * (size_t)(K * V));
    else
        memset(S, 0, sizeof(double) * (size_t)(K * V));

    for (int64_t t = t0; t < t1; ++t) {
        const int64_t tok = (row * J->T + t) * H + hh;
        const double *kt = J->k + tok * K;
        const double *qt = J->q + tok * K;
        const double *vt = J->v + tok * V;
        const double a = exp(J->g[tok]);

        for (int64_t i = 0; i < K * V; ++i)
            S[i] *= a;

        if (J->beta) {
            /* u = beta (v - h^T k) */
            const double b = J->beta[tok];
            for (int64_t j = 0; j < V; ++j)
                u[j] = 0.0;
            for (int64_t i = 0; i < K; ++i) {
                const double ki = kt[i];
                const double *Si = S + i * V;
                for (int64_t j = 0; j < V; ++j)
                    u[j] += Si[j] * ki;
            }
            for (int64_t j = 0; j < V; ++j)
                u[j] = b * (vt[j] - u[j]);
        } else {
            for (int64_t j = 0; j < V; ++j)
                u[j] = vt[j];
        }
        /* h <- h + k u^T */
        for (int64_t i = 0; i < K; ++i) {
            const double ki = kt[i];
            double *Si = S + i * V;
            for (int64_t j = 0; j < V; ++j)
                Si[j] += ki * u[j];
        }
        /* o_t = h^T q / sqrt(K) */
        double *ot = J->o + tok * V;
        for (int64_t j = 0; j < V; ++j)
            ot[j] = 0.0;
        for (int64_t i = 0; i < K; ++i) {
            const double qi = qt[i];
            const double *Si = S + i * V;
            for (int64_t j = 0; j < V; ++j)
                ot[j] += Si[j] * qi;
        }
        for (int64_t j = 0; j < V; ++j)
            ot[j] *= J->scale;
    }
    if (J->ht)
        memcpy(J->ht + sidx, S, sizeof(double) * (size_t)(K * V));
    free(S);
    free(u);
    return 0;
}

static void *fwd_worker(void *arg)
{
    fwd_job *J = (fwd_job *)arg;
    const int64_t total = J->N * J->H;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int64_t idx = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (idx >= total)
            break;
        if (J->pair_mask && !J->pair_mask[idx])
            continue;
        if (run_pair(J, idx / J->H, idx % J->H) != 0) {
            pthread_mutex_lock(&J->mu);
            J->failed = 1;
            pthread_mutex_unlock(&J->mu);
        }
    }
    return NULL;
}

/*
 * gdr_oracle_fwd: the token recurrence over every (sequence, head) pair.
 *   beta == NULL  -> beta-free mode (h <- alpha h + k v^T)
 *   cu == NULL    -> dense: N = B sequences of T tokens
 *   h0 == NULL    -> zero initial state;  ht == NULL -> final state not kept
 *   pair_mask     -> optional [N*H] bytes; pairs with 0 are skipped (their
 *                    o rows and ht slices are left untouched)
 * Returns the number of threads used (>= 1), or -1 on bad arguments / OOM.
 */
int gdr_oracle_fwd(const double *q, const double *k, const double *v,
                   const double *g, const double *beta, const int64_t *cu,
                   const double *h0, double *o, double *ht, int64_t B,
                   int64_t T, int64_t H, int64_t K, int64_t V, int64_t N,
                   double scale, const uint8_t *pair_mask, int n_threads)
{
    if (!q || !k || !v || !g || !o || B < 1 || T < 0 || H < 1 || K < 1 ||
        V < 1)
        return -1;
    if (cu) {
        if (B != 1 || N < 0)
            return -1;
        if (cu[0] != 0 || cu[N] != T)
            return -1;
        for (int64_t n = 0; n < N; ++n)
            if (cu[n + 1] < cu[n])
                return -1;
    } else {
        N = B;
    }
    fwd_job J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.h0 = h0;
    J.o = o; J.ht = ht; J.cu = cu; J.pair_mask = pair_mask;
    J.B = B; J.T = T; J.H = H; J.K = K; J.V = V; J.N = N;
    J.scale = scale;
    pthread_mutex_init(&J.mu, NULL);

    if (n_threads <= 0) {
        long c = sysconf(_SC_NPROCESSORS_ONLN);
        n_threads = c > 0 ? (int)c : 1;
    }
    if ((int64_t)n_threads > N * H)
        n_threads = (int)(N * H > 0 ? N * H : 1);

    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)n_threads);
    if (!th) {
        pthread_mutex_destroy(&J.mu);
        return -1;
    }
    int started = 0;
    for (int i = 0; i < n_threads - 1; ++i)
        if (pthread_create(&th[started], NULL, fwd_worker, &J) == 0)
            ++started;
    /* the calling thread works too */
    fwd_worker(&J);
    for (int i = 0; i < started; ++i)
        pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.mu);
    return J.failed ? -1 : started + 1;
}

/*
 * gdr_oracle_affine: the affine map of the recurrence over one token range of
 * one (sequence, head), h_out = M h_in + c.  Token by token:
 *     P_t = alpha_t (I - beta_t k_t k_t^T)        (beta-free: alpha_t I)
 *     M <- P_t M;   c <- P_t c + beta_t k_t v_t^T (beta-free: + k_t v_t^T)
 * starting from M = I, c = 0.
 *   k [len, K], v [len, V], g [len], beta [len] or NULL; rows contiguous with
 *   row strides ldk, ldv (elements) and gate stride ldg.
 *   M [K, K], c [K, V] row-major outputs.
 * Returns 0, or -1 on bad arguments / OOM.
 */
int gdr_oracle_affine(const double *k, const double *v, const double *g,
                      const double *beta, int64_t len, int64_t K, int64_t V,
                      int64_t ldk, int64_t ldv, int64_t ldg, double *M,
                      double *c)
{
    if (!k || !v || !g || !M || !c || len < 0 || K < 1 || V < 1)
        return -1;
    double *r = (double *)malloc(sizeof(double) * (size_t)(K > V ? K : V));
    if (!r)
        return -1;
    for (int64_t i = 0; i < K; ++i)
        for (int64_t j = 0; j < K; ++j)
            M[i * K + j] = (i == j) ? 1.0 : 0.0;
    memset(c, 0, sizeof(double) * (size_t)(K * V));

    for (int64_t t = 0; t < len; ++t) {
        const double *kt = k + t * ldk;
        const double *vt = v + t * ldv;
        const double a = exp(g[t * ldg]);
        if (beta) {
            const double b = beta[t * ldg];
            /* M <- a (M - b k (k^T M)) */
            for (int64_t j = 0; j < K; ++j)
                r[j] = 0.0;
            for (int64_t i = 0; i < K; ++i)
                for (int64_t j = 0; j < K; ++j)
                    r[j] += kt[i] * M[i * K + j];
            for (int64_t i = 0; i < K; ++i)
                for (int64_t j = 0; j < K; ++j)
                    M[i * K + j] = a * (M[i * K + j] - b * kt[i] * r[j]);
            /* c <- a (c - b k (k^T c)) + b k v^T */
            for (int64_t j = 0; j < V; ++j)
                r[j] = 0.0;
            for (int64_t i = 0; i < K; ++i)
                for (int64_t j = 0; j < V; ++j)
                    r[j] += kt[i] * c[i * V + j];
            for (int64_t i = 0; i < K; ++i)
                for (int64_t j = 0; j < V; ++j)
                    c[i * V + j] = a * (c[i * V + j] - b * kt[i] * r[j]) +
                                   b * kt[i] * vt[j];
        } else {
            for (int64_t i = 0; i < K * K; ++i)
                M[i] *= a;
            for (int64_t i = 0; i < K; ++i)
                for (int64_t j = 0; j < V; ++j)
                    c[i * V + j] = a * c[i * V + j] + kt[i] * vt[j];
        }
    }
    free(r);
    return 0;
}
