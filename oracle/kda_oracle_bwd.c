/*
 * KDA backward oracle: the exact gradient of the forward in kda_oracle.c, by
 * reverse-mode differentiation of its token loop, written out by hand in fp64.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file; only the tests use it.  It shares no code with the CUDA library.
 *
 * The pages ship the forward only (the FlashKDA Q&A, its notes on training); the
 * backward here is the derivative of the forward those pages define (the readings
 * in kda_oracle.c), nothing more.  For a scalar loss L with dL/dout = dout and
 * dL/dS_final = dfinal, per (sequence, head) pair, with
 *   S'_t = Diag(alpha_t) S_{t-1},  w_t = v_t - S'_t^T k_t,  u_t = beta_t w_t,
 *   S_t  = S'_t + k_t u_t^T,       o_t = scale S_t^T q_t        (q, k normalised),
 * the loop runs t = L-1 .. 0 carrying dS = dL/dS_t:
 *   dq_t     = scale S_t do_t            dS += scale q_t do_t^T
 *   du       = dS^T k_t                  dk_t = dS u_t
 *   dbeta_t  = du . w_t                  dv_t = beta_t du
 *   dx       = -beta_t du                (dL/d(S'_t^T k_t))
 *   dS'      = dS + k_t dx^T             dk_t += S'_t dx
 *   dalpha_t = rowsum(dS' * S_{t-1})     dS = Diag(alpha_t) dS'
 * and dL/dS_0 = dS at the end.  The activations are then differentiated token by
 * token: the L2 norm (q_hat = q / n, n = sqrt(|q|^2 + eps): dq = dq_hat / n -
 * q (q . dq_hat) / n^3), the beta sigmoid, alpha = exp(gk), and the gate (bounded:
 * gk = lb sigmoid(z), z = exp(A_log) (g + dt_bias); without a lower bound:
 * gk = -exp(A_log) softplus(g + dt_bias)), with dA_log and ddt_bias summed over
 * every token of every sequence of the head.
 *
 * The forward states S_0 .. S_L of a pair are kept in memory (L + 1 states of
 * K x V doubles), so the oracle is for small cases only.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define KDA_ORACLE_BWD_EPS 1e-6

static double sig(double x) { return 1.0 / (1.0 + exp(-x)); }
static double splus(double x) { return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x))); }

/* Gradients of one (sequence n, head h) pair.  dq, dk, dv, dg, dbeta receive this
 * pair's tokens; part[0] += its dA_log, part[1 .. K] += its ddt_bias[h][:]. */
static void bwd_pair(const double *q, const double *k, const double *v, const double *g,
                     const double *beta_logit, double scale, const double *A_log,
                     const double *dt_bias, double lower_bound, const double *initial_state,
                     const double *dout, const double *dfinal, const int64_t *cu_seqlens,
                     int64_t n, int64_t h, int64_t T, int64_t H, int64_t K, int64_t V,
                     double *dq, double *dk, double *dv, double *dg, double *dbeta,
                     double *dinit, double *part) {
    int64_t b, t0, len;
    if (cu_seqlens) {
        b = 0;
        t0 = cu_seqlens[n];
        len = cu_seqlens[n + 1] - t0;
    } else {
        b = n;
        t0 = 0;
        len = T;
    }
    const size_t KV = (size_t)(K * V);
    const size_t soff = (size_t)((n * H + h) * V * K);
    const int unbounded = isnan(lower_bound);
    const double a = exp(A_log[h]);
    const double *dtb = dt_bias + h * K;
    /* per-token activations and the states S_0 .. S_len */
    double *qn = (double *)malloc(sizeof(double) * (size_t)(len * K + 1));
    double *kn = (double *)malloc(sizeof(double) * (size_t)(len * K + 1));
    double *al = (double *)malloc(sizeof(double) * (size_t)(len * K + 1));
    double *bt = (double *)malloc(sizeof(double) * (size_t)(len + 1));
    double *S = (double *)calloc((size_t)(len + 1) * KV, sizeof(double));
    double *Sp = (double *)malloc(sizeof(double) * KV);
    double *dS = (double *)calloc(KV, sizeof(double));
    double *dSp = (double *)malloc(sizeof(double) * KV);
    double *w = (double *)malloc(sizeof(double) * (size_t)V);
    double *du = (double *)malloc(sizeof(double) * (size_t)V);
    double *dx = (double *)malloc(sizeof(double) * (size_t)V);
    double *dqn = (double *)malloc(sizeof(double) * (size_t)K);
    double *dkn = (double *)malloc(sizeof(double) * (size_t)K);
    double *dal = (double *)malloc(sizeof(double) * (size_t)K);
    if (initial_state)
        for (int64_t j = 0; j < V; ++j)
            for (int64_t c = 0; c < K; ++c) S[c * V + j] = initial_state[soff + j * K + c];
    for (int64_t i = 0; i < len; ++i) {
        const size_t tok = (size_t)((b * T + t0 + i) * H + h);
        const double *qt = q + tok * K, *kt = k + tok * K, *gt = g + tok * K, *vt = v + tok * V;
        double sq = 0.0, sk = 0.0;
        for (int64_t c = 0; c < K; ++c) {
            sq += qt[c] * qt[c];
            sk += kt[c] * kt[c];
        }
        const double rq = 1.0 / sqrt(sq + KDA_ORACLE_BWD_EPS), rk = 1.0 / sqrt(sk + KDA_ORACLE_BWD_EPS);
        for (int64_t c = 0; c < K; ++c) {
            qn[i * K + c] = qt[c] * rq;
            kn[i * K + c] = kt[c] * rk;
            const double x = gt[c] + dtb[c];
            const double gk = unbounded ? -a * splus(x) : lower_bound * sig(a * x);
            al[i * K + c] = exp(gk);
        }
        bt[i] = sig(beta_logit[tok]);
        /* forward step: S_{i+1} from S_i */
        const double *Sprev = S + (size_t)i * KV;
        double *Snext = S + (size_t)(i + 1) * KV;
        for (int64_t c = 0; c < K; ++c)
            for (int64_t j = 0; j < V; ++j) Snext[c * V + j] = al[i * K + c] * Sprev[c * V + j];
        for (int64_t j = 0; j < V; ++j) {
            double ks = 0.0;
            for (int64_t c = 0; c < K; ++c) ks += kn[i * K + c] * Snext[c * V + j];
            w[j] = vt[j] - ks;
        }
        for (int64_t c = 0; c < K; ++c)
            for (int64_t j = 0; j < V; ++j) Snext[c * V + j] += kn[i * K + c] * bt[i] * w[j];
    }
    /* dL/dS_len from the final-state gradient (stored layout [V][K]) */
    if (dfinal)
        for (int64_t j = 0; j < V; ++j)
            for (int64_t c = 0; c < K; ++c) dS[c * V + j] = dfinal[soff + j * K + c];
    for (int64_t i = len - 1; i >= 0; --i) {
        const size_t tok = (size_t)((b * T + t0 + i) * H + h);
        const double *dot = dout + tok * V, *vt = v + tok * V;
        const double *Sprev = S + (size_t)i * KV, *St = S + (size_t)(i + 1) * KV;
        const double *qi = qn + i * K, *ki = kn + i * K, *ai = al + i * K;
        const double be = bt[i];
        /* o = scale S_t^T q */
        for (int64_t c = 0; c < K; ++c) {
            double acc = 0.0;
            for (int64_t j = 0; j < V; ++j) acc += St[c * V + j] * dot[j];
            dqn[c] = scale * acc;
            for (int64_t j = 0; j < V; ++j) dS[c * V + j] += scale * qi[c] * dot[j];
        }
        /* S' = Diag(alpha) S_{t-1};  w = v - S'^T k */
        for (int64_t c = 0; c < K; ++c)
            for (int64_t j = 0; j < V; ++j) Sp[c * V + j] = ai[c] * Sprev[c * V + j];
        for (int64_t j = 0; j < V; ++j) {
            double ks = 0.0, d = 0.0;
            for (int64_t c = 0; c < K; ++c) {
                ks += ki[c] * Sp[c * V + j];
                d += dS[c * V + j] * ki[c];
            }
            w[j] = vt[j] - ks;
            du[j] = d;
        }
        /* S_t = S' + k (beta w)^T */
        double dbe = 0.0;
        for (int64_t j = 0; j < V; ++j) {
            dbe += du[j] * w[j];
            dv[tok * V + j] = be * du[j];
            dx[j] = -be * du[j];
        }
        for (int64_t c = 0; c < K; ++c) {
            double acc = 0.0, acc2 = 0.0;
            for (int64_t j = 0; j < V; ++j) {
                acc += dS[c * V + j] * be * w[j];
                dSp[c * V + j] = dS[c * V + j] + ki[c] * dx[j];
                acc2 += Sp[c * V + j] * dx[j];
            }
            dkn[c] = acc + acc2;
        }
        for (int64_t c = 0; c < K; ++c) {
            double acc = 0.0;
            for (int64_t j = 0; j < V; ++j) acc += dSp[c * V + j] * Sprev[c * V + j];
            dal[c] = acc;
            for (int64_t j = 0; j < V; ++j) dS[c * V + j] = ai[c] * dSp[c * V + j];
        }
        /* the activations of this token */
        const double *qt = q + tok * K, *kt = k + tok * K, *gt = g + tok * K;
        double sq = 0.0, sk = 0.0, qd = 0.0, kd = 0.0;
        for (int64_t c = 0; c < K; ++c) {
            sq += qt[c] * qt[c];
            sk += kt[c] * kt[c];
            qd += qt[c] * dqn[c];
            kd += kt[c] * dkn[c];
        }
        const double nq = sqrt(sq + KDA_ORACLE_BWD_EPS), nk = sqrt(sk + KDA_ORACLE_BWD_EPS);
        for (int64_t c = 0; c < K; ++c) {
            dq[tok * K + c] = dqn[c] / nq - qt[c] * qd / (nq * nq * nq);
            dk[tok * K + c] = dkn[c] / nk - kt[c] * kd / (nk * nk * nk);
        }
        dbeta[tok] = dbe * be * (1.0 - be);
        for (int64_t c = 0; c < K; ++c) {
            const double x = gt[c] + dtb[c];
            const double dgk = dal[c] * ai[c]; /* alpha = exp(gk) */
            if (unbounded) {
                const double gk = -a * splus(x);
                const double d = dgk * (-a * sig(x));
                dg[tok * K + c] = d;
                part[1 + c] += d;
                part[0] += dgk * gk;
            } else {
                const double s = sig(a * x);
                const double dz = dgk * lower_bound * s * (1.0 - s);
                dg[tok * K + c] = dz * a;
                part[1 + c] += dz * a;
                part[0] += dz * a * x;
            }
        }
    }
    if (dinit)
        for (int64_t j = 0; j < V; ++j)
            for (int64_t c = 0; c < K; ++c) dinit[soff + j * K + c] = dS[c * V + j];
    free(qn);
    free(kn);
    free(al);
    free(bt);
    free(S);
    free(Sp);
    free(dS);
    free(dSp);
    free(w);
    free(du);
    free(dx);
    free(dqn);
    free(dkn);
    free(dal);
}

/* Gradients of L = sum(dout * out) + sum(dfinal * final_state) with respect to every
 * input of kda_oracle_fwd (same layouts; fp64).  dout [B,T,H,V]; dfinal [N,H,V,K] or
 * NULL (zero); outputs dq, dk, dg [B,T,H,K], dv [B,T,H,V], dbeta [B,T,H] (of the beta
 * logits), dA_log [H], ddt_bias [H,K], dinit [N,H,V,K] (or NULL: not written).  Token
 * rows outside every sequence are left untouched.  Returns 0, or nonzero on malformed
 * sizes or cu_seqlens. */
int kda_oracle_bwd(const double *q, const double *k, const double *v, const double *g,
                   const double *beta_logit, double scale, const double *A_log,
                   const double *dt_bias, double lower_bound, const double *initial_state,
                   const double *dout, const double *dfinal, const int64_t *cu_seqlens,
                   int64_t num_seqs, int64_t B, int64_t T, int64_t H, int64_t K, int64_t V,
                   double *dq, double *dk, double *dv, double *dg, double *dbeta, double *dA_log,
                   double *ddt_bias, double *dinit, int nthreads) {
    if (B < 0 || T < 0 || H < 0 || K <= 0 || V <= 0) return 1;
    if (cu_seqlens) {
        if (B != 1 || num_seqs < 0) return 2;
        if (cu_seqlens[0] != 0 || cu_seqlens[num_seqs] != T) return 3;
        for (int64_t n = 0; n < num_seqs; ++n)
            if (cu_seqlens[n + 1] < cu_seqlens[n]) return 3;
    }
    const int64_t N = cu_seqlens ? num_seqs : B, pairs = N * H;
    double *part = (double *)calloc((size_t)(pairs * (K + 1) + 1), sizeof(double));
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t u = 0; u < pairs; ++u)
        bwd_pair(q, k, v, g, beta_logit, scale, A_log, dt_bias, lower_bound, initial_state, dout,
                 dfinal, cu_seqlens, u / H, u % H, T, H, K, V, dq, dk, dv, dg, dbeta, dinit,
                 part + u * (K + 1));
    for (int64_t hh = 0; hh < H; ++hh) {
        dA_log[hh] = 0.0;
        for (int64_t c = 0; c < K; ++c) ddt_bias[hh * K + c] = 0.0;
    }
    for (int64_t u = 0; u < pairs; ++u) { /* in pair order: the sums do not depend on threads */
        const int64_t hh = u % H;
        dA_log[hh] += part[u * (K + 1)];
        for (int64_t c = 0; c < K; ++c) ddt_bias[hh * K + c] += part[u * (K + 1) + 1 + c];
    }
    free(part);
    (void)nthreads;
    return 0;
}
