/*
 * Oracle: the gradient of the gated delta rule, one token at a time, in float64.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the CPU reference that the CUDA
 * backward is checked against.  Nothing in the library links, includes or
 * calls it; only the tests, the smoke check and the benchmark's CPU legs do.
 *
 * The forward is the token recurrence of naive_recurrence.c, written here with
 * the residual r_t named (delta_t = beta_t r_t):
 *
 *     S~_t = D_t S_{t-1}            D_t = exp(g_t) or diag(exp(g_t[:]))
 *     r_t  = v_t - S~_t^T k_t
 *     S_t  = S~_t + beta_t k_t r_t^T
 *     o_t  = scale * S_t^T q_t
 *
 * The backward pass of "kernel_fun/kda/_kernels/bwd_scan.py" differentiates
 * this recurrence; here it is differentiated directly, by reverse mode over the
 * tokens.  Given dO (the loss gradient with respect to every o_t) and dS_T (with
 * respect to h_final; zero when absent), with dS the gradient with respect to
 * S_t, for t = T .. 1:
 *
 *     dS      += scale q_t do_t^T                   read-out
 *     dq_t     = scale S_t do_t
 *     dd       = dS^T k_t                           gradient of delta_t
 *     dk_t     = dS delta_t
 *     dbeta_t  = r_t . dd
 *     dr       = beta_t dd,  dv_t = dr
 *     dk_t    -= S~_t dr                            through r_t = v_t - S~_t^T k_t
 *     dS~      = dS - k_t dr^T
 *     dg_t[i]  = sum_j S~_t[i,j] dS~[i,j]           per key dim (summed over i for a scalar gate)
 *     dS       = D_t dS~                            now the gradient with respect to S_{t-1}
 *
 * and dh0 = dS after t = 1.  The states are not stored for every token: the
 * forward keeps S before every C-th token, and each stretch of C tokens is
 * replayed from its checkpoint (the same operations in the same order, so the
 * replayed states are bit-identical) before it is walked backward.  C changes
 * memory only, never a result.
 *
 * Work is split over (b, h) pairs across threads; every pair is independent.
 *
 * Layouts (all float64, contiguous, head dim last):
 *   q, k, dq, dk [B,T,H,K]; v, do, dv [B,T,H,V]; g, dg [B,T,H] or [B,T,H,K];
 *   beta, dbeta [B,T,H]; h0, dh_final, dh0 [B,H,K,V] (h0, dh_final may be NULL).
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
    const double *q, *k, *v, *g, *beta, *h0, *d_o, *dh_final;
    double *dq, *dk, *dv, *dg, *dbeta, *dh0;
    int64_t n_items, next_item;
    pthread_mutex_t lock;
} adj_t;

/* decay factors of token `tok` into dec[K] */
static void decay_of(const adj_t *J, int64_t tok, double *dec) {
    if (J->per_k_gate) {
        for (int64_t i = 0; i < J->K; ++i) dec[i] = exp(J->g[tok * J->K + i]);
    } else {
        const double a = exp(J->g[tok]);
        for (int64_t i = 0; i < J->K; ++i) dec[i] = a;
    }
}

/* One forward token: Sout = S_t from Sin = S_{t-1}.  Sdec gets S~_t, r gets r_t. */
static void step(const adj_t *J, int64_t tok, const double *Sin, double *Sout, double *Sdec, double *r,
                 double *dec) {
    const int64_t K = J->K, V = J->V;
    const double *kt = J->k + tok * K, *vt = J->v + tok * V;
    const double bt = J->beta[tok];
    decay_of(J, tok, dec);
    for (int64_t i = 0; i < K; ++i)
        for (int64_t j = 0; j < V; ++j) Sdec[i * V + j] = dec[i] * Sin[i * V + j];
    for (int64_t j = 0; j < V; ++j) r[j] = 0.0;
    for (int64_t i = 0; i < K; ++i)
        for (int64_t j = 0; j < V; ++j) r[j] += Sdec[i * V + j] * kt[i];
    for (int64_t j = 0; j < V; ++j) r[j] = vt[j] - r[j];
    for (int64_t i = 0; i < K; ++i)
        for (int64_t j = 0; j < V; ++j) Sout[i * V + j] = Sdec[i * V + j] + bt * kt[i] * r[j];
}

static void run_pair(const adj_t *J, int64_t bh) {
    const int64_t b = bh / J->H, h = bh % J->H;
    const int64_t K = J->K, V = J->V, H = J->H, T = J->T, C = J->C;
    const int64_t NT = (T + C - 1) / C, KV = K * V;
    double *ck = (double *)malloc(sizeof(double) * (size_t)(NT * KV));
    double *Ss = (double *)malloc(sizeof(double) * (size_t)((C + 1) * KV));   /* S_{t0-1} .. S_{t1-1} */
    double *Sdec = (double *)malloc(sizeof(double) * (size_t)KV);
    double *dS = (double *)malloc(sizeof(double) * (size_t)KV);
    double *dSt = (double *)malloc(sizeof(double) * (size_t)KV);
    double *r = (double *)malloc(sizeof(double) * (size_t)V);
    double *dd = (double *)malloc(sizeof(double) * (size_t)V);
    double *dr = (double *)malloc(sizeof(double) * (size_t)V);
    double *dec = (double *)malloc(sizeof(double) * (size_t)K);
    double *S = Ss;   /* forward state, walked in the first slot */

    /* forward, keeping S before every C-th token */
    if (J->h0) memcpy(S, J->h0 + (b * H + h) * KV, sizeof(double) * (size_t)KV);
    else memset(S, 0, sizeof(double) * (size_t)KV);
    for (int64_t t = 0; t < T; ++t) {
        if (t % C == 0) memcpy(ck + (t / C) * KV, S, sizeof(double) * (size_t)KV);
        step(J, (b * T + t) * H + h, S, Ss + KV, Sdec, r, dec);
        memcpy(S, Ss + KV, sizeof(double) * (size_t)KV);
    }

    /* backward */
    if (J->dh_final) memcpy(dS, J->dh_final + (b * H + h) * KV, sizeof(double) * (size_t)KV);
    else memset(dS, 0, sizeof(double) * (size_t)KV);
    for (int64_t c = NT - 1; c >= 0; --c) {
        const int64_t t0 = c * C, t1 = (t0 + C < T) ? t0 + C : T;
        memcpy(Ss, ck + c * KV, sizeof(double) * (size_t)KV);
        for (int64_t t = t0; t < t1; ++t)
            step(J, (b * T + t) * H + h, Ss + (t - t0) * KV, Ss + (t - t0 + 1) * KV, Sdec, r, dec);
        for (int64_t t = t1 - 1; t >= t0; --t) {
            const int64_t tok = (b * T + t) * H + h;
            const double *Sprev = Ss + (t - t0) * KV, *St = Ss + (t - t0 + 1) * KV;
            const double *qt = J->q + tok * K, *kt = J->k + tok * K, *dot = J->d_o + tok * V;
            const double bt = J->beta[tok];
            step(J, tok, Sprev, dSt, Sdec, r, dec);   /* S~_t and r_t again (dSt is scratch here) */

            for (int64_t i = 0; i < K; ++i)
                for (int64_t j = 0; j < V; ++j) dS[i * V + j] += J->scale * qt[i] * dot[j];
            double *dqt = J->dq + tok * K, *dkt = J->dk + tok * K;
            for (int64_t i = 0; i < K; ++i) {
                double s = 0.0;
                for (int64_t j = 0; j < V; ++j) s += St[i * V + j] * dot[j];
                dqt[i] = J->scale * s;
            }
            for (int64_t j = 0; j < V; ++j) dd[j] = 0.0;
            for (int64_t i = 0; i < K; ++i)
                for (int64_t j = 0; j < V; ++j) dd[j] += dS[i * V + j] * kt[i];
            for (int64_t i = 0; i < K; ++i) {
                double s = 0.0;
                for (int64_t j = 0; j < V; ++j) s += dS[i * V + j] * bt * r[j];
                dkt[i] = s;
            }
            double db = 0.0;
            for (int64_t j = 0; j < V; ++j) db += r[j] * dd[j];
            J->dbeta[tok] = db;
            double *dvt = J->dv + tok * V;
            for (int64_t j = 0; j < V; ++j) {
                dr[j] = bt * dd[j];
                dvt[j] = dr[j];
            }
            for (int64_t i = 0; i < K; ++i) {
                double s = 0.0;
                for (int64_t j = 0; j < V; ++j) s += Sdec[i * V + j] * dr[j];
                dkt[i] -= s;
            }
            for (int64_t i = 0; i < K; ++i)
                for (int64_t j = 0; j < V; ++j) dSt[i * V + j] = dS[i * V + j] - kt[i] * dr[j];
            if (J->per_k_gate) {
                for (int64_t i = 0; i < K; ++i) {
                    double s = 0.0;
                    for (int64_t j = 0; j < V; ++j) s += Sdec[i * V + j] * dSt[i * V + j];
                    J->dg[tok * K + i] = s;
                }
            } else {
                double s = 0.0;
                for (int64_t i = 0; i < K; ++i)
                    for (int64_t j = 0; j < V; ++j) s += Sdec[i * V + j] * dSt[i * V + j];
                J->dg[tok] = s;
            }
            for (int64_t i = 0; i < K; ++i)
                for (int64_t j = 0; j < V; ++j) dS[i * V + j] = dec[i] * dSt[i * V + j];
        }
    }
    memcpy(J->dh0 + (b * H + h) * KV, dS, sizeof(double) * (size_t)KV);
    free(ck); free(Ss); free(Sdec); free(dS); free(dSt); free(r); free(dd); free(dr); free(dec);
}

static void *adj_worker(void *arg) {
    adj_t *J = (adj_t *)arg;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        const int64_t item = J->next_item++;
        pthread_mutex_unlock(&J->lock);
        if (item >= J->n_items) break;
        run_pair(J, item);
    }
    return NULL;
}

/* Returns 0 on success, -1 on a bad argument.  nthreads <= 0 means 1. */
int oracle_naive_backward(int64_t B, int64_t T, int64_t H, int64_t K, int64_t V, int64_t C,
                          int per_k_gate, double scale,
                          const double *q, const double *k, const double *v, const double *g,
                          const double *beta, const double *h0, const double *d_o, const double *dh_final,
                          double *dq, double *dk, double *dv, double *dg, double *dbeta, double *dh0,
                          int nthreads) {
    if (B <= 0 || T <= 0 || H <= 0 || K <= 0 || V <= 0 || C <= 0) return -1;
    if (!q || !k || !v || !g || !beta || !d_o || !dq || !dk || !dv || !dg || !dbeta || !dh0) return -1;
    adj_t J;
    memset(&J, 0, sizeof(J));
    J.B = B; J.T = T; J.H = H; J.K = K; J.V = V; J.C = C;
    J.per_k_gate = per_k_gate; J.scale = scale;
    J.q = q; J.k = k; J.v = v; J.g = g; J.beta = beta; J.h0 = h0; J.d_o = d_o; J.dh_final = dh_final;
    J.dq = dq; J.dk = dk; J.dv = dv; J.dg = dg; J.dbeta = dbeta; J.dh0 = dh0;
    J.n_items = B * H;
    pthread_mutex_init(&J.lock, NULL);
    if (nthreads <= 1) {
        adj_worker(&J);
    } else {
        pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
        for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, adj_worker, &J);
        for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
        free(th);
    }
    pthread_mutex_destroy(&J.lock);
    return 0;
}
