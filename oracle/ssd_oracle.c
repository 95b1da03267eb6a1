/*
 * ssd_oracle.c -- fp64 CPU oracle for the Mamba-2 SSD layer and for the
 * K-token multi-step verification decode.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this file's library.  It shares no code, header,
 * table or helper with the CUDA library; the two meet only in the seeded
 * input arrays.
 *
 * What it computes (per batch row b and head h, state h of shape N x P):
 *
 *   dt_t = softplus(dt_raw_t)            (optional; z > 20 -> z)
 *   a_t  = exp(dt_t * A_h)
 *   h_t  = a_t * h_{t-1} + B_t x_t^T     (B_t in R^N, x_t in R^P)
 *   y_t  = C_t^T h_t + D_h * x_t
 *
 * This is the selective state-space recurrence that Mamba-2 restricts to a
 * scalar-times-identity A per head ("Transformers are SSMs", the SSD layer;
 * summarised on the cloud.tencent page "Mamba 2 ... SSD", section
 * "核心创新——SSD" and section "SSD算法").  The input term carries no dt
 * factor; B and C are shared by contiguous groups of heads, head h using
 * group h / (H / G).
 *
 * Three entry points:
 *   oracle_ssd_seq        -- the plain sequential recurrence (the definition);
 *   oracle_ssd_chunked    -- the four-step chunked block decomposition
 *                            (diagonal blocks, chunk states, state passing,
 *                            output from each chunk's true initial state),
 *                            used only to pin chunk-size invariance;
 *   oracle_ssd_multistep  -- K steps from a cached state, returning y[K],
 *                            the state after the first j tokens and after K
 *                            ("Mamba in the Llama", section 推测解码, the
 *                            MultiStep function).
 *
 * Inputs are float32 arrays (holding the exact generated values, bf16 or
 * fp32); all arithmetic is double.  Outputs are "pair-compact": pair index
 * q enumerates the requested (b, h) pairs and
 *   y[q][t][p], h_final[q][n][p]           (seq / chunked)
 *   y[q][k][p], h_j[q][n][p], h_K[q][n][p] (multistep).
 * Work is spread over (b, h) pairs with POSIX threads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

typedef struct {
    int64_t batch, T, H, P, N, GB, GC;
    const float *x, *dt, *A, *B, *C, *D, *h0;
    const int32_t *j;      /* multistep only */
    int dt_softplus;
    int64_t chunk;         /* chunked only */
    const int64_t *pairs;  /* b*H + h, or NULL = all pairs in order */
    int64_t npairs;
    double *y, *h_out, *h_j;
    int64_t next;          /* work counter */
    int err;
} job_t;

static double softplus(double z) { return z > 20.0 ? z : log1p(exp(z)); }

static double step_dt(const job_t *J, int64_t b, int64_t t, int64_t h) {
    double z = (double)J->dt[(b * J->T + t) * J->H + h];
    return J->dt_softplus ? softplus(z) : z;
}

static int64_t pair_of(const job_t *J, int64_t q) { return J->pairs ? J->pairs[q] : q; }

/* Sequential recurrence for one (b, h) pair. */
static void seq_pair(job_t *J, int64_t q, double *st) {
    const int64_t pr = pair_of(J, q), b = pr / J->H, h = pr % J->H;
    const int64_t T = J->T, H = J->H, P = J->P, N = J->N;
    const int64_t gb = h / (H / J->GB), gc = h / (H / J->GC);
    const double Ah = J->A[h], Dh = J->D ? J->D[h] : 0.0;
    for (int64_t i = 0; i < N * P; i++)
        st[i] = J->h0 ? (double)J->h0[(b * H + h) * N * P + i] : 0.0;
    for (int64_t t = 0; t < T; t++) {
        const double a = exp(step_dt(J, b, t, h) * Ah);
        const float *xt = J->x + ((b * T + t) * H + h) * P;
        const float *Bt = J->B + ((b * T + t) * J->GB + gb) * N;
        const float *Ct = J->C + ((b * T + t) * J->GC + gc) * N;
        for (int64_t n = 0; n < N; n++)
            for (int64_t p = 0; p < P; p++)
                st[n * P + p] = a * st[n * P + p] + (double)Bt[n] * (double)xt[p];
        double *yt = J->y + (q * T + t) * P;
        for (int64_t p = 0; p < P; p++) {
            double acc = 0.0;
            for (int64_t n = 0; n < N; n++) acc += (double)Ct[n] * st[n * P + p];
            yt[p] = acc + Dh * (double)xt[p];
        }
    }
    if (J->h_out) memcpy(J->h_out + q * N * P, st, sizeof(double) * N * P);
}

/*
 * Chunked block decomposition for one (b, h) pair with chunk length Q (any
 * Q >= 1; the last chunk may be short).  With cs the inclusive running sum of
 * dt*A inside a chunk, the four steps are written out one after another over
 * all chunks:
 *   1. diagonal blocks (quadratic, attention-like):
 *        Ydiag_i = sum_{j<=i} exp(cs_i - cs_j) (C_i . B_j) x_j
 *   2. chunk-final states from a zero initial state:
 *        S_c = sum_j exp(cs_last - cs_j) B_j x_j^T
 *   3. state passing across chunks (a scan with the chunk decays):
 *        Hin_0 = h0,  Hin_{c+1} = exp(cs_last(c)) Hin_c + S_c
 *   4. each chunk's output from its true initial state:
 *        Yoff_i = exp(cs_i) C_i^T Hin_c
 *   y = Ydiag + Yoff + D x,  h_final = Hin_nc.
 */
static void chunked_pair(job_t *J, int64_t q, double *work) {
    const int64_t pr = pair_of(J, q), b = pr / J->H, h = pr % J->H;
    const int64_t T = J->T, H = J->H, P = J->P, N = J->N, Q = J->chunk;
    const int64_t gb = h / (H / J->GB), gc = h / (H / J->GC);
    const int64_t nc = (T + Q - 1) / Q;
    const double Ah = J->A[h], Dh = J->D ? J->D[h] : 0.0;
    double *cs = work;                 /* [T]            */
    double *S = cs + T;                /* [nc][N][P]     */
    double *Hin = S + nc * N * P;      /* [nc + 1][N][P] */
    double *y = J->y + q * T * P;
#define XV(t, p) ((double)J->x[(((b) * T + (t)) * H + h) * P + (p)])
#define BV(t, n) ((double)J->B[(((b) * T + (t)) * J->GB + gb) * N + (n)])
#define CV(t, n) ((double)J->C[(((b) * T + (t)) * J->GC + gc) * N + (n)])
    for (int64_t c = 0; c < nc; c++) {
        const int64_t t0 = c * Q, L = (T - t0 < Q) ? T - t0 : Q;
        double run = 0.0;
        for (int64_t i = 0; i < L; i++) { run += step_dt(J, b, t0 + i, h) * Ah; cs[t0 + i] = run; }
    }
    /* step 1: diagonal blocks */
    for (int64_t c = 0; c < nc; c++) {
        const int64_t t0 = c * Q, L = (T - t0 < Q) ? T - t0 : Q;
        for (int64_t i = 0; i < L; i++) {
            for (int64_t p = 0; p < P; p++) y[(t0 + i) * P + p] = 0.0;
            for (int64_t jj = 0; jj <= i; jj++) {
                double cb = 0.0;
                for (int64_t n = 0; n < N; n++) cb += CV(t0 + i, n) * BV(t0 + jj, n);
                const double m = exp(cs[t0 + i] - cs[t0 + jj]) * cb;
                for (int64_t p = 0; p < P; p++) y[(t0 + i) * P + p] += m * XV(t0 + jj, p);
            }
        }
    }
    /* step 2: chunk states */
    for (int64_t c = 0; c < nc; c++) {
        const int64_t t0 = c * Q, L = (T - t0 < Q) ? T - t0 : Q;
        double *Sc = S + c * N * P;
        for (int64_t i = 0; i < N * P; i++) Sc[i] = 0.0;
        for (int64_t jj = 0; jj < L; jj++) {
            const double w = exp(cs[t0 + L - 1] - cs[t0 + jj]);
            for (int64_t n = 0; n < N; n++)
                for (int64_t p = 0; p < P; p++) Sc[n * P + p] += w * BV(t0 + jj, n) * XV(t0 + jj, p);
        }
    }
    /* step 3: state passing */
    for (int64_t i = 0; i < N * P; i++) Hin[i] = J->h0 ? (double)J->h0[(b * H + h) * N * P + i] : 0.0;
    for (int64_t c = 0; c < nc; c++) {
        const int64_t t0 = c * Q, L = (T - t0 < Q) ? T - t0 : Q;
        const double decay = exp(cs[t0 + L - 1]);
        for (int64_t i = 0; i < N * P; i++)
            Hin[(c + 1) * N * P + i] = decay * Hin[c * N * P + i] + S[c * N * P + i];
    }
    /* step 4: outputs from the true initial states, plus the skip term */
    for (int64_t c = 0; c < nc; c++) {
        const int64_t t0 = c * Q, L = (T - t0 < Q) ? T - t0 : Q;
        const double *Hc = Hin + c * N * P;
        for (int64_t i = 0; i < L; i++) {
            const double e = exp(cs[t0 + i]);
            for (int64_t p = 0; p < P; p++) {
                double acc = 0.0;
                for (int64_t n = 0; n < N; n++) acc += CV(t0 + i, n) * Hc[n * P + p];
                y[(t0 + i) * P + p] += e * acc + Dh * XV(t0 + i, p);
            }
        }
    }
    if (J->h_out) memcpy(J->h_out + q * N * P, Hin + nc * N * P, sizeof(double) * N * P);
#undef XV
#undef BV
#undef CV
}

/* K steps from the cached state; records the state after j[b] tokens. */
static void multistep_pair(job_t *J, int64_t q, double *st) {
    const int64_t pr = pair_of(J, q), b = pr / J->H, h = pr % J->H;
    const int64_t K = J->T, H = J->H, P = J->P, N = J->N;
    const int64_t gb = h / (H / J->GB), gc = h / (H / J->GC);
    const double Ah = J->A[h], Dh = J->D ? J->D[h] : 0.0;
    const int64_t jb = J->j[b];
    for (int64_t i = 0; i < N * P; i++) st[i] = (double)J->h0[(b * H + h) * N * P + i];
    if (jb == 0) memcpy(J->h_j + q * N * P, st, sizeof(double) * N * P);
    for (int64_t k = 0; k < K; k++) {
        const double a = exp(step_dt(J, b, k, h) * Ah);
        const float *xk = J->x + ((b * K + k) * H + h) * P;
        const float *Bk = J->B + ((b * K + k) * J->GB + gb) * N;
        const float *Ck = J->C + ((b * K + k) * J->GC + gc) * N;
        for (int64_t n = 0; n < N; n++)
            for (int64_t p = 0; p < P; p++)
                st[n * P + p] = a * st[n * P + p] + (double)Bk[n] * (double)xk[p];
        double *yk = J->y + (q * K + k) * P;
        for (int64_t p = 0; p < P; p++) {
            double acc = 0.0;
            for (int64_t n = 0; n < N; n++) acc += (double)Ck[n] * st[n * P + p];
            yk[p] = acc + Dh * (double)xk[p];
        }
        if (k + 1 == jb) memcpy(J->h_j + q * N * P, st, sizeof(double) * N * P);
    }
    memcpy(J->h_out + q * N * P, st, sizeof(double) * N * P);
}

typedef enum { MODE_SEQ, MODE_CHUNKED, MODE_MULTISTEP } mode_t_;
typedef struct { job_t *J; mode_t_ mode; } worker_arg;

static void *worker(void *argp) {
    worker_arg *w = (worker_arg *)argp;
    job_t *J = w->J;
    size_t words = (size_t)(J->N * J->P);
    if (w->mode == MODE_CHUNKED) {
        const int64_t nc = (J->T + J->chunk - 1) / J->chunk;
        words = (size_t)(J->T + (2 * nc + 1) * J->N * J->P);
    }
    double *buf = (double *)malloc(sizeof(double) * words);
    if (!buf) { __atomic_store_n(&J->err, 1, __ATOMIC_RELAXED); return NULL; }
    for (;;) {
        int64_t q = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
        if (q >= J->npairs) break;
        if (w->mode == MODE_SEQ) seq_pair(J, q, buf);
        else if (w->mode == MODE_CHUNKED) chunked_pair(J, q, buf);
        else multistep_pair(J, q, buf);
    }
    free(buf);
    return NULL;
}

int oracle_default_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int)n : 1;
}

static int run(job_t *J, mode_t_ mode, int nthreads) {
    if (J->batch <= 0 || J->T <= 0 || J->H <= 0 || J->P <= 0 || J->N <= 0 || J->GB <= 0 ||
        J->GC <= 0 || J->H % J->GB || J->H % J->GC)
        return 1;
    if (!J->pairs) J->npairs = J->batch * J->H;
    if (nthreads <= 0) nthreads = oracle_default_threads();
    if (nthreads > J->npairs) nthreads = (int)J->npairs;
    if (nthreads < 1) nthreads = 1;
    J->next = 0;
    J->err = 0;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    worker_arg wa = {J, mode};
    int started = 0;
    for (int i = 1; i < nthreads; i++)
        if (pthread_create(&th[started], NULL, worker, &wa) == 0) started++;
    worker(&wa);
    for (int i = 0; i < started; i++) pthread_join(th[i], NULL);
    free(th);
    return J->err;
}

int oracle_ssd_seq(int64_t batch, int64_t T, int64_t H, int64_t P, int64_t N, int64_t GB,
                   int64_t GC, const float *x, const float *dt, const float *A, const float *B,
                   const float *C, const float *D, const float *h0, int dt_softplus,
                   const int64_t *pairs, int64_t npairs, double *y, double *h_final,
                   int nthreads) {
    job_t J = {batch, T, H, P, N, GB, GC, x, dt, A, B, C, D, h0, NULL, dt_softplus, 0,
               pairs, npairs, y, h_final, NULL, 0, 0};
    return run(&J, MODE_SEQ, nthreads);
}

int oracle_ssd_chunked(int64_t batch, int64_t T, int64_t H, int64_t P, int64_t N, int64_t GB,
                       int64_t GC, const float *x, const float *dt, const float *A,
                       const float *B, const float *C, const float *D, const float *h0,
                       int dt_softplus, int64_t chunk, const int64_t *pairs, int64_t npairs,
                       double *y, double *h_final, int nthreads) {
    if (chunk < 1) return 1;
    job_t J = {batch, T, H, P, N, GB, GC, x, dt, A, B, C, D, h0, NULL, dt_softplus, chunk,
               pairs, npairs, y, h_final, NULL, 0, 0};
    return run(&J, MODE_CHUNKED, nthreads);
}

int oracle_ssd_multistep(int64_t batch, int64_t K, int64_t H, int64_t P, int64_t N, int64_t GB,
                         int64_t GC, const float *x, const float *dt, const float *A,
                         const float *B, const float *C, const float *D, const float *h_cache,
                         const int32_t *j, int dt_softplus, const int64_t *pairs,
                         int64_t npairs, double *y, double *h_j, double *h_K, int nthreads) {
    if (!h_cache || !j) return 1;
    for (int64_t b = 0; b < batch; b++)
        if (j[b] < 0 || j[b] > K) return 1;
    job_t J = {batch, K, H, P, N, GB, GC, x, dt, A, B, C, D, h_cache, j, dt_softplus, 0,
               pairs, npairs, y, h_K, h_j, 0, 0};
    return run(&J, MODE_MULTISTEP, nthreads);
}
