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
 * Also provided: the gradient of that forward pass (gdr_oracle_bwd below),
 * and the affine map of the recurrence over a token range,
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


/*
 * Backward pass: the gradient of the forward recurrence above, by reverse-mode
 * differentiation of each token step (the reverse dH recurrence that the
 * flash-linear-attention ABC issue #23 pages run chunk by chunk, "Problem"
 * and "Proposed Dataflow" step 4; its fixture contract asks for dQ, dK, dV
 * and state gradients).  The scalar loss is L = <do, o> + <dht, ht>.
 *
 * One forward step, with h_prev the state before token t:
 *     h' = a h_prev                    a = exp(g_t)
 *     y  = h'^T k,  u = b (v - y)      (beta-free: u = v)
 *     h  = h' + k u^T
 *     o  = scale h^T q
 * Its reverse, with dh = dL/dh entering from the later tokens (dht at the
 * end of the sequence):
 *     dh += scale q do^T;  dq = scale h do
 *     dk  = dh u;          du = dh^T k
 *     dv  = b du;          db = <du, v - y>;  dy = -b du;
 *     dh += k dy^T;        dk += h' dy        (beta-free: dv = du)
 *     dg  = a <dh, h_prev>;  dh <- a dh       (the gradient for h_prev)
 * and dh0 is dh after the first token.  The states h_prev / h of a token are
 * replayed forward from a checkpoint kept every 64 tokens.
 */
enum { BWD_BLOCK = 64 };

typedef struct {
    const double *q, *k, *v, *g, *beta, *h0, *dout, *dht;
    double *dq, *dk, *dv, *dg, *dbeta, *dh0;
    const int64_t *cu;
    const uint8_t *pair_mask;
    int64_t B, T, H, K, V, N;
    double scale;
    int64_t next;
    int failed;
    pthread_mutex_t mu;
} bwd_job;

/* One forward token step on the state hs (K x V) for token index tok, in
 * place (the same step as run_pair's loop body, without the readout). */
static void step_forward(const bwd_job *J, int64_t tok, double *hs, double *u)
{
    const int64_t K = J->K, V = J->V;
    const double *kt = J->k + tok * K;
    const double *vt = J->v + tok * V;
    const double g_t = J->g[tok];
    const double a = exp(g_t);
    for (int64_t i = 0; i < K * V; ++i)
        hs[i] *= a;
    if (J->beta) {
        const double bb = J->beta[tok];
        for (int64_t j = 0; j < V; ++j)
            u[j] = 0.0;
        for (int64_t i = 0; i < K; ++i)
            for (int64_t j = 0; j < V; ++j)
                u[j] += hs[i * V + j] * kt[i];
        for (int64_t j = 0; j < V; ++j)
            u[j] = bb * (vt[j] - u[j]);
    } else {
        for (int64_t j = 0; j < V; ++j)
            u[j] = vt[j];
    }
    for (int64_t i = 0; i < K; ++i)
        for (int64_t j = 0; j < V; ++j)
            hs[i * V + j] += kt[i] * u[j];
}

static int run_pair_bwd(bwd_job *J, int64_t n, int64_t hh)
{
    const int64_t H = J->H, K = J->K, V = J->V, KV = K * V;
    int64_t row, t0, t1;
    if (J->cu) {
        row = 0;
        t0 = J->cu[n];
        t1 = J->cu[1 + n];
    } else {
        row = n;
        t0 = 0;
        t1 = J->T;
    }
    const int64_t len = t1 - t0;
    const int64_t nblk = (len + BWD_BLOCK - 1) / BWD_BLOCK;
    /* ck[b]: state before block b's first token; st[i]: state after token i
     * of the block being reversed (st[0] = the block's checkpoint) */
    double *ck = (double *)malloc(sizeof(double) * (size_t)((nblk > 0 ? nblk : 1) * KV));
    double *st = (double *)malloc(sizeof(double) * (size_t)((BWD_BLOCK + 1) * KV));
    double *dh = (double *)malloc(sizeof(double) * (size_t)KV);
    double *hp = (double *)malloc(sizeof(double) * (size_t)KV);
    double *u = (double *)malloc(sizeof(double) * (size_t)V);
    double *y = (double *)malloc(sizeof(double) * (size_t)V);
    double *du = (double *)malloc(sizeof(double) * (size_t)V);
    if (!ck || !st || !dh || !hp || !u || !y || !du) {
        free(ck); free(st); free(dh); free(hp); free(u); free(y); free(du);
        return -1;
    }
    const int64_t sidx = (n * H + hh) * KV;
    /* forward sweep, keeping each block's starting state */
    if (J->h0)
        memcpy(st, J->h0 + sidx, sizeof(double) * (size_t)KV);
    else
        memset(st, 0, sizeof(double) * (size_t)KV);
    for (int64_t b = 0; b < nblk; ++b) {
        memcpy(ck + b * KV, st, sizeof(double) * (size_t)KV);
        const int64_t e = (b + 1) * BWD_BLOCK < len ? (b + 1) * BWD_BLOCK : len;
        for (int64_t t = t0 + b * BWD_BLOCK; t < t0 + e; ++t)
            step_forward(J, (row * J->T + t) * H + hh, st, u);
    }
    /* reverse sweep */
    if (J->dht)
        memcpy(dh, J->dht + sidx, sizeof(double) * (size_t)KV);
    else
        memset(dh, 0, sizeof(double) * (size_t)KV);
    for (int64_t b = nblk - 1; b >= 0; --b) {
        const int64_t s = t0 + b * BWD_BLOCK;
        const int64_t e = (b + 1) * BWD_BLOCK < len ? t0 + (b + 1) * BWD_BLOCK : t1;
        memcpy(st, ck + b * KV, sizeof(double) * (size_t)KV);
        for (int64_t t = s; t < e; ++t) {
            memcpy(st + (t - s + 1) * KV, st + (t - s) * KV, sizeof(double) * (size_t)KV);
            step_forward(J, (row * J->T + t) * H + hh, st + (t - s + 1) * KV, u);
        }
        for (int64_t t = e - 1; t >= s; --t) {
            const int64_t tok = hh + H * (row * J->T + t);
            const double *kt = J->k + tok * K, *qt = J->q + tok * K;
            const double *vt = J->v + tok * V, *dot = J->dout + tok * V;
            const double *hprev = st + (t - s) * KV, *hcur = st + (t - s + 1) * KV;
            const double g_t = J->g[tok];
            const double a = exp(g_t);
            double *dqt = J->dq + tok * K, *dkt = J->dk + tok * K, *dvt = J->dv + tok * V;
            /* h' = a h_prev, and u (with y = h'^T k) as in the forward step */
            for (int64_t i = 0; i < KV; ++i)
                hp[i] = a * hprev[i];
            if (J->beta) {
                const double bb = J->beta[tok];
                for (int64_t j = 0; j < V; ++j)
                    y[j] = 0.0;
                for (int64_t i = 0; i < K; ++i)
                    for (int64_t j = 0; j < V; ++j)
                        y[j] += hp[i * V + j] * kt[i];
                for (int64_t j = 0; j < V; ++j)
                    u[j] = bb * (vt[j] - y[j]);
            } else {
                for (int64_t j = 0; j < V; ++j)
                    u[j] = vt[j];
            }
            /* readout: dh += scale q do^T;  dq = scale h do */
            for (int64_t i = 0; i < K; ++i)
                for (int64_t j = 0; j < V; ++j)
                    dh[i * V + j] += J->scale * qt[i] * dot[j];
            for (int64_t i = 0; i < K; ++i) {
                double acc = 0.0;
                for (int64_t j = 0; j < V; ++j)
                    acc += hcur[i * V + j] * dot[j];
                dqt[i] = J->scale * acc;
            }
            /* write h = h' + k u^T:  dk = dh u;  du = dh^T k */
            for (int64_t i = 0; i < K; ++i) {
                double acc = 0.0;
                for (int64_t j = 0; j < V; ++j)
                    acc += dh[i * V + j] * u[j];
                dkt[i] = acc;
            }
            for (int64_t j = 0; j < V; ++j)
                du[j] = 0.0;
            for (int64_t i = 0; i < K; ++i)
                for (int64_t j = 0; j < V; ++j)
                    du[j] += dh[i * V + j] * kt[i];
            if (J->beta) {
                /* u = b (v - y):  dv = b du;  db = <du, v - y>;  dy = -b du */
                const double bb = J->beta[tok];
                double db = 0.0;
                for (int64_t j = 0; j < V; ++j) {
                    dvt[j] = bb * du[j];
                    db += du[j] * (vt[j] - y[j]);
                }
                J->dbeta[tok] = db;
                /* y = h'^T k:  dh' += k dy^T;  dk += h' dy */
                for (int64_t i = 0; i < K; ++i) {
                    double acc = 0.0;
                    for (int64_t j = 0; j < V; ++j) {
                        const double dy = -bb * du[j];
                        dh[i * V + j] += kt[i] * dy;
                        acc += hp[i * V + j] * dy;
                    }
                    dkt[i] += acc;
                }
            } else {
                for (int64_t j = 0; j < V; ++j)
                    dvt[j] = du[j];
            }
            /* h' = a h_prev:  dg = a <dh', h_prev>;  dh_prev = a dh' */
            double da = 0.0;
            for (int64_t i = 0; i < KV; ++i)
                da += dh[i] * hprev[i];
            J->dg[tok] = a * da;
            for (int64_t i = 0; i < KV; ++i)
                dh[i] *= a;
        }
    }
    if (J->dh0)
        memcpy(J->dh0 + sidx, dh, sizeof(double) * (size_t)KV);
    free(ck); free(st); free(dh); free(hp); free(u); free(y); free(du);
    return 0;
}

static void *bwd_worker(void *arg)
{
    bwd_job *J = (bwd_job *)arg;
    const int64_t total = J->N * J->H;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        int64_t idx = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (idx >= total)
            break;
        if (J->pair_mask && !J->pair_mask[idx])
            continue;
        if (run_pair_bwd(J, idx / J->H, idx % J->H) != 0) {
            pthread_mutex_lock(&J->mu);
            J->failed = 1;
            pthread_mutex_unlock(&J->mu);
        }
    }
    return NULL;
}

/*
 * gdr_oracle_bwd: gradients of L = <do, o> + <dht, ht> with respect to q, k,
 * v, g, beta and h0, for every (sequence, head) pair.  Layouts as for
 * gdr_oracle_fwd; do has o's layout, dht and dh0 the state layout.
 *   beta == NULL -> beta-free mode (dbeta is not written)
 *   h0 == NULL   -> zero initial state;  dht == NULL -> no final-state term
 *   dh0 == NULL  -> the initial-state gradient is not kept
 *   pair_mask    -> optional [N*H] bytes; pairs with 0 are skipped
 * Returns the number of threads used (>= 1), or -1 on bad arguments / OOM.
 */
int gdr_oracle_bwd(const double *q, const double *k, const double *v,
                   const double *g, const double *beta, const int64_t *cu,
                   const double *h0, const double *dout, const double *dht,
                   double *dq, double *dk, double *dv, double *dg,
                   double *dbeta, double *dh0, int64_t B, int64_t T,
                   int64_t H, int64_t K, int64_t V, int64_t N, double scale,
                   const uint8_t *pair_mask, int n_threads)
{
    if (!q || !k || !v || !g || !dout || !dq || !dk || !dv || !dg ||
        (beta && !dbeta) || B < 1 || T < 0 || H < 1 || K < 1 || V < 1)
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
    bwd_job J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.h0 = h0;
    J.dout = dout; J.dht = dht;
    J.dq = dq; J.dk = dk; J.dv = dv; J.dg = dg; J.dbeta = dbeta; J.dh0 = dh0;
    J.cu = cu; J.pair_mask = pair_mask;
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
        if (pthread_create(&th[started], NULL, bwd_worker, &J) == 0)
            ++started;
    bwd_worker(&J);
    for (int i = 0; i < started; ++i)
        pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&J.mu);
    return J.failed ? -1 : started + 1;
}
