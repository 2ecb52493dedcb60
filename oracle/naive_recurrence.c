/*
 * Oracle: the gated delta rule, one token at a time, in float64.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the CPU reference that the CUDA path
 * is checked against.  Nothing in the library links, includes or calls it; only
 * the tests, the smoke check and the benchmark's CPU-baseline leg do.
 *
 * What it computes (the definition the chunked method reaches exactly, up to
 * rounding order).  Per batch b and head h, with the state S a K x V matrix,
 * S_0 = h0 (or zero), and for t = 1..T:
 *
 *     D_t     = exp(g_t)            (scalar gate, "GDN")
 *             = diag(exp(g_t[:]))   (per-key-dim gate, "KDA")
 *     S~      = D_t S_{t-1}
 *     delta_t = beta_t (v_t - S~^T k_t)
 *     S_t     = S~ + k_t delta_t^T       ( = (I - beta_t k_t k_t^T) D_t S_{t-1} + beta_t k_t v_t^T )
 *     o_t     = scale * S_t^T q_t
 *
 * h_final = S_T, and the checkpoint of chunk c is the state before chunk c,
 * ckpt[c] = S_{c*C}.  This is the gated delta rule in its token form
 * (S_t = exp(g_t)(I - beta k k^T) S_{t-1} + beta k v^T for a scalar gate), the
 * recurrence whose chunked form the two method pages compute: the fused WY
 * prepare of "Reuse P as beta tiles in gated deltanet fused prepare" and the
 * state scan of "kernel_fun/kda/_kernels/bwd_scan.py" (module docstring: h
 * checkpointed before the update, v' = u - w h, h = exp2(gd) h + kg^T v').  For
 * the per-key-dim gate the decay acts before the delta step, the one ordering
 * under which that page's per-dim scan (gd a K-vector broadcast over V) is the
 * chunked form of the recurrence.
 *
 * Column independence: given k, beta and g, each column j of S evolves on its
 * own (every step acts on S from the left), so the work is split over
 * (b, h, block of V columns) across threads.  That split changes no arithmetic.
 *
 * Layouts (all float64, contiguous, head dim last):
 *   q, k [B,T,H,K]; v [B,T,H,V]; g [B,T,H] or [B,T,H,K]; beta [B,T,H];
 *   h0 [B,H,K,V] or NULL; o [B,T,H,V]; h_final [B,H,K,V];
 *   ckpt [B,NT,H,K,V] or NULL (NT = ceil(T / C); a last, partial chunk has its
 *   checkpoint like any other).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t B, T, H, K, V, C;
    int per_k_gate;
    double scale;
    const double *q, *k, *v, *g, *beta, *h0;
    double *o, *h_final, *ckpt;
    int64_t vblock;
    int64_t n_items;
    int64_t next_item;
    pthread_mutex_t lock;
} job_t;

static void run_item(const job_t *J, int64_t item) {
    const int64_t nvb = (J->V + J->vblock - 1) / J->vblock;
    const int64_t bh = item / nvb, vb = item % nvb;
    const int64_t b = bh / J->H, h = bh % J->H;
    const int64_t K = J->K, V = J->V, H = J->H, T = J->T, C = J->C;
    const int64_t j0 = vb * J->vblock;
    const int64_t nj = (j0 + J->vblock <= V) ? J->vblock : V - j0;

    double *S = (double *)calloc((size_t)(K * nj), sizeof(double)); /* S[i*nj + jj] */
    double *r = (double *)malloc((size_t)nj * sizeof(double));
    double *dk = (double *)malloc((size_t)K * sizeof(double));
    if (J->h0) {
        const double *src = J->h0 + ((b * H + h) * K) * V;
        for (int64_t i = 0; i < K; ++i)
            for (int64_t jj = 0; jj < nj; ++jj) S[i * nj + jj] = src[i * V + j0 + jj];
    }
    for (int64_t t = 0; t < T; ++t) {
        if (J->ckpt && (t % C) == 0) {
            double *dst = J->ckpt + (((b * ((T + C - 1) / C) + t / C) * H + h) * K) * V;
            for (int64_t i = 0; i < K; ++i)
                for (int64_t jj = 0; jj < nj; ++jj) dst[i * V + j0 + jj] = S[i * nj + jj];
        }
        const int64_t tok = (b * T + t) * H + h;
        const double *kt = J->k + tok * K;
        const double *qt = J->q + tok * K;
        const double *vt = J->v + tok * V;
        const double bt = J->beta[tok];
        /* decay: S~ = D_t S */
        if (J->per_k_gate) {
            for (int64_t i = 0; i < K; ++i) dk[i] = exp(J->g[tok * K + i]);
        } else {
            const double a = exp(J->g[tok]);
            for (int64_t i = 0; i < K; ++i) dk[i] = a;
        }
        for (int64_t i = 0; i < K; ++i)
            for (int64_t jj = 0; jj < nj; ++jj) S[i * nj + jj] *= dk[i];
        /* r = S~^T k ; delta = beta (v - r) */
        for (int64_t jj = 0; jj < nj; ++jj) r[jj] = 0.0;
        for (int64_t i = 0; i < K; ++i) {
            const double ki = kt[i];
            for (int64_t jj = 0; jj < nj; ++jj) r[jj] += S[i * nj + jj] * ki;
        }
        for (int64_t jj = 0; jj < nj; ++jj) r[jj] = bt * (vt[j0 + jj] - r[jj]);
        /* S = S~ + k delta^T */
        for (int64_t i = 0; i < K; ++i) {
            const double ki = kt[i];
            for (int64_t jj = 0; jj < nj; ++jj) S[i * nj + jj] += ki * r[jj];
        }
        /* o = scale S^T q */
        double *ot = J->o + tok * V + j0;
        for (int64_t jj = 0; jj < nj; ++jj) ot[jj] = 0.0;
        for (int64_t i = 0; i < K; ++i) {
            const double qi = qt[i];
            for (int64_t jj = 0; jj < nj; ++jj) ot[jj] += S[i * nj + jj] * qi;
        }
        for (int64_t jj = 0; jj < nj; ++jj) ot[jj] *= J->scale;
    }
    double *hf = J->h_final + ((b * H + h) * K) * V;
    for (int64_t i = 0; i < K; ++i)
        for (int64_t jj = 0; jj < nj; ++jj) hf[i * V + j0 + jj] = S[i * nj + jj];
    free(S);
    free(r);
    free(dk);
}

static void *worker(void *arg) {
    job_t *J = (job_t *)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int64_t item = J->next_item++;
        pthread_mutex_unlock(&J->lock);
        if (item >= J->n_items) break;
        run_item(J, item);
    }
    return NULL;
}

/* Returns 0 on success, -1 on a bad argument. nthreads <= 0 means 1. */
int oracle_naive_forward(int64_t B, int64_t T, int64_t H, int64_t K, int64_t V, int64_t C,
                         int per_k_gate, double scale,
                         const double *q, const double *k, const double *v, const double *g,
                         const double *beta, const double *h0,
                         double *o, double *h_final, double *ckpt,
                         int64_t vblock, int nthreads) {
    if (B <= 0 || T <= 0 || H <= 0 || K <= 0 || V <= 0 || C <= 0) return -1;
    if (!q || !k || !v || !g || !beta || !o || !h_final) return -1;
    job_t J;
    memset(&J, 0, sizeof(J));
    J.B = B; J.T = T; J.H = H; J.K = K; J.V = V; J.C = C;
    J.per_k_gate = per_k_gate; J.scale = scale;
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.h0 = h0;
    J.o = o; J.h_final = h_final; J.ckpt = ckpt;
    J.vblock = (vblock <= 0 || vblock > V) ? V : vblock;
    J.n_items = B * H * ((V + J.vblock - 1) / J.vblock);
    J.next_item = 0;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads <= 1) {
        worker(&J);
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
        for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, worker, &J);
        for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&J.lock);
    return 0;
}
