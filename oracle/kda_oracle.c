/*
 * KDA forward oracle: a plain, slow, token-by-token fp64 recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline use it.  It shares no code with the CUDA library.
 *
 * What it computes (Kimi Delta Attention, the channel-wise gated delta rule;
 * FlashKDA README "Kernel API" table for the argument list, shapes and state
 * layout; agents-report.net "FlashKDA" article, background section, for KDA as
 * Gated DeltaNet with per-channel gating).  The pages give no formula, so the
 * recurrence and gate below are the documented readings of this project:
 *
 *   q_hat = q / sqrt(|q|^2 + eps),  k_hat likewise           (q/k L2 norm)
 *   beta  = 1 / (1 + exp(-beta_logit))                      (beta sigmoid)
 *   gk[c] = lower_bound * sigmoid(exp(A_log[h]) * (g[c] + dt_bias[h][c]))
 *           (the bounded gate, safe_gate on; lower_bound in [-5, 0]), or, when the
 *           call has no lower bound (safe_gate off; passed here as a NaN lower_bound),
 *   gk[c] = -exp(A_log[h]) * softplus(g[c] + dt_bias[h][c]),
 *           softplus(x) = log(1 + exp(x)), a log decay in (-inf, 0)
 *   S_t   = (I - beta_t k_t k_t^T) Diag(exp(gk_t)) S_{t-1} + beta_t k_t v_t^T
 *   o_t   = scale * S_t^T q_t
 *
 * S is K x V (S[c][v]); the stored state is its transpose, state[n][h][v][c]
 * ("[B,H,V,K]" in the Kernel API table).  A missing initial state means zeros.
 * Every (sequence, head) pair is an independent recurrence; with cu_seqlens the
 * sequences are the segments [cu[n], cu[n+1]) of a B=1 packed batch, otherwise
 * each batch row is a sequence.
 *
 * All arithmetic is fp64 (inputs arrive as fp64 copies of the bf16 values, which
 * is exact).  OpenMP spreads the (sequence, head) pairs over threads; each pair
 * runs the same sequential loop whatever the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define KDA_ORACLE_EPS 1e-6

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/* log(1 + exp(x)) without overflow: max(x, 0) + log1p(exp(-|x|)). */
static double softplus(double x) { return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x))); }

/* Activations of one token of one head: L2-normalised q and k, beta and the
 * per-channel log decay gk. */
static void activations(const double *q, const double *k, const double *g, double beta_logit,
                        double A_log_h, const double *dt_bias_h, double lower_bound, int64_t K,
                        double *qn, double *kn, double *beta, double *gk) {
    double sq = 0.0, sk = 0.0;
    for (int64_t c = 0; c < K; ++c) {
        sq += q[c] * q[c];
        sk += k[c] * k[c];
    }
    double rq = 1.0 / sqrt(sq + KDA_ORACLE_EPS), rk = 1.0 / sqrt(sk + KDA_ORACLE_EPS);
    for (int64_t c = 0; c < K; ++c) {
        qn[c] = q[c] * rq;
        kn[c] = k[c] * rk;
    }
    *beta = sigmoid(beta_logit);
    double a = exp(A_log_h);
    if (isnan(lower_bound)) {
        for (int64_t c = 0; c < K; ++c) gk[c] = -a * softplus(g[c] + dt_bias_h[c]);
    } else {
        for (int64_t c = 0; c < K; ++c) gk[c] = lower_bound * sigmoid(a * (g[c] + dt_bias_h[c]));
    }
}

/* One step of the recurrence on S (K x V, row-major S[c*V+v]):
 *   S <- Diag(alpha) S;  S <- S + beta k (v - S^T k)^T;  o = scale S^T q.
 * The middle line is (I - beta k k^T) S + beta k v^T written out. */
static void step(double *S, const double *qn, const double *kn, const double *vv, double beta,
                 const double *gk, double scale, int64_t K, int64_t V, double *work, double *o) {
    for (int64_t c = 0; c < K; ++c) {
        double a = exp(gk[c]);
        double *row = S + c * V;
        for (int64_t j = 0; j < V; ++j) row[j] *= a;
    }
    double *kS = work; /* kS[j] = sum_c k[c] S[c][j] */
    for (int64_t j = 0; j < V; ++j) kS[j] = 0.0;
    for (int64_t c = 0; c < K; ++c) {
        const double *row = S + c * V;
        for (int64_t j = 0; j < V; ++j) kS[j] += kn[c] * row[j];
    }
    for (int64_t c = 0; c < K; ++c) {
        double *row = S + c * V;
        double bk = beta * kn[c];
        for (int64_t j = 0; j < V; ++j) row[j] += bk * (vv[j] - kS[j]);
    }
    for (int64_t j = 0; j < V; ++j) o[j] = 0.0;
    for (int64_t c = 0; c < K; ++c) {
        const double *row = S + c * V;
        for (int64_t j = 0; j < V; ++j) o[j] += qn[c] * row[j];
    }
    for (int64_t j = 0; j < V; ++j) o[j] *= scale;
}

/* Geometry shared by both entry points: where sequence n starts and how long it is. */
static void seq_span(const int64_t *cu_seqlens, int64_t n, int64_t T, int64_t *b, int64_t *t0,
                     int64_t *len) {
    if (cu_seqlens) {
        *b = 0;
        *t0 = cu_seqlens[n];
        *len = cu_seqlens[n + 1] - cu_seqlens[n];
    } else {
        *b = n;
        *t0 = 0;
        *len = T;
    }
}

/* Runs one (sequence n, head h) pair.  `pre` selects the input form:
 *   pre == 0: raw inputs (q, k, v, g, beta logits, A_log, dt_bias, lower_bound);
 *   pre == 1: already activated inputs: q and k are used as given (no L2 norm),
 *             `g` holds the log decay gk itself and `beta` holds beta itself. */
static void run_pair(int pre, const double *q, const double *k, const double *v, const double *g,
                     const double *beta, double scale, const double *A_log, const double *dt_bias,
                     double lower_bound, const double *initial_state, double *final_state,
                     double *out, const int64_t *cu_seqlens, int64_t n, int64_t h, int64_t T,
                     int64_t H, int64_t K, int64_t V) {
    int64_t b, t0, len;
    seq_span(cu_seqlens, n, T, &b, &t0, &len);
    double *S = (double *)calloc((size_t)(K * V), sizeof(double));
    double *qn = (double *)malloc(sizeof(double) * (size_t)K);
    double *kn = (double *)malloc(sizeof(double) * (size_t)K);
    double *gk = (double *)malloc(sizeof(double) * (size_t)K);
    double *work = (double *)malloc(sizeof(double) * (size_t)V);
    const size_t state_off = (size_t)((n * H + h) * V * K);
    if (initial_state) {
        for (int64_t j = 0; j < V; ++j)
            for (int64_t c = 0; c < K; ++c) S[c * V + j] = initial_state[state_off + j * K + c];
    }
    for (int64_t t = t0; t < t0 + len; ++t) {
        const size_t tok = (size_t)((b * T + t) * H + h);
        const double *qt = q + tok * K, *kt = k + tok * K, *gt = g + tok * K, *vt = v + tok * V;
        double bt;
        if (pre) {
            memcpy(qn, qt, sizeof(double) * (size_t)K);
            memcpy(kn, kt, sizeof(double) * (size_t)K);
            memcpy(gk, gt, sizeof(double) * (size_t)K);
            bt = beta[tok];
        } else {
            activations(qt, kt, gt, beta[tok], A_log[h], dt_bias + h * K, lower_bound, K, qn, kn,
                        &bt, gk);
        }
        step(S, qn, kn, vt, bt, gk, scale, K, V, work, out + tok * V);
    }
    if (final_state) {
        for (int64_t j = 0; j < V; ++j)
            for (int64_t c = 0; c < K; ++c) final_state[state_off + j * K + c] = S[c * V + j];
    }
    free(S);
    free(qn);
    free(kn);
    free(gk);
    free(work);
}

static int check_args(const int64_t *cu_seqlens, int64_t num_seqs, int64_t B, int64_t T, int64_t H,
                      int64_t K, int64_t V) {
    if (B < 0 || T < 0 || H < 0 || K <= 0 || V <= 0) return 1;
    if (cu_seqlens) {
        if (B != 1 || num_seqs < 0) return 2;
        if (cu_seqlens[0] != 0 || cu_seqlens[num_seqs] != T) return 3;
        for (int64_t n = 0; n < num_seqs; ++n)
            if (cu_seqlens[n + 1] < cu_seqlens[n]) return 3;
    }
    return 0;
}

static int run_all(int pre, const double *q, const double *k, const double *v, const double *g,
                   const double *beta, double scale, const double *A_log, const double *dt_bias,
                   double lower_bound, const double *initial_state, double *final_state,
                   double *out, const int64_t *cu_seqlens, int64_t num_seqs, int64_t B, int64_t T,
                   int64_t H, int64_t K, int64_t V, const int64_t *pairs, int64_t n_pairs,
                   int nthreads) {
    int rc = check_args(cu_seqlens, num_seqs, B, T, H, K, V);
    if (rc) return rc;
    const int64_t N = cu_seqlens ? num_seqs : B;
    const int64_t total = pairs ? n_pairs : N * H;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t u = 0; u < total; ++u) {
        int64_t n = pairs ? pairs[2 * u] : u / H;
        int64_t h = pairs ? pairs[2 * u + 1] : u % H;
        run_pair(pre, q, k, v, g, beta, scale, A_log, dt_bias, lower_bound, initial_state,
                 final_state, out, cu_seqlens, n, h, T, H, K, V);
    }
    (void)nthreads;
    return 0;
}

/* Full forward from raw inputs.  All arrays are fp64, contiguous, in the layouts
 * of the Kernel API table: q,k,g [B,T,H,K]; v,out [B,T,H,V]; beta [B,T,H];
 * A_log [H]; dt_bias [H,K]; states [N,H,V,K] (N = num_seqs with cu_seqlens,
 * else B), either may be NULL.  `pairs` (optional) restricts the work to the
 * listed (n, h) pairs; outputs of other pairs are left untouched.  Returns 0 on
 * success, nonzero on malformed sizes or cu_seqlens. */
int kda_oracle_fwd(const double *q, const double *k, const double *v, const double *g,
                   const double *beta_logit, double scale, const double *A_log,
                   const double *dt_bias, double lower_bound, const double *initial_state,
                   double *final_state, double *out, const int64_t *cu_seqlens, int64_t num_seqs,
                   int64_t B, int64_t T, int64_t H, int64_t K, int64_t V, const int64_t *pairs,
                   int64_t n_pairs, int nthreads) {
    return run_all(0, q, k, v, g, beta_logit, scale, A_log, dt_bias, lower_bound, initial_state,
                   final_state, out, cu_seqlens, num_seqs, B, T, H, K, V, pairs, n_pairs, nthreads);
}

/* The recurrence alone, on activated inputs: q and k used as given, gk [B,T,H,K]
 * the per-channel log decay, beta [B,T,H] the (post-sigmoid) beta. */
int kda_oracle_recurrence(const double *q, const double *k, const double *v, const double *gk,
                          const double *beta, double scale, const double *initial_state,
                          double *final_state, double *out, const int64_t *cu_seqlens,
                          int64_t num_seqs, int64_t B, int64_t T, int64_t H, int64_t K, int64_t V,
                          int nthreads) {
    return run_all(1, q, k, v, gk, beta, scale, NULL, NULL, 0.0, initial_state, final_state, out,
                   cu_seqlens, num_seqs, B, T, H, K, V, NULL, 0, nthreads);
}

/* The activations alone (for pins of the gate, beta and norm readings). Outputs
 * qn, kn, gk [B,T,H,K] and beta [B,T,H], fp64. */
int kda_oracle_activations(const double *q, const double *k, const double *g,
                           const double *beta_logit, const double *A_log, const double *dt_bias,
                           double lower_bound, int64_t B, int64_t T, int64_t H, int64_t K,
                           double *qn, double *kn, double *gk, double *beta) {
    if (B < 0 || T < 0 || H < 0 || K <= 0) return 1;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t t = 0; t < T; ++t)
            for (int64_t h = 0; h < H; ++h) {
                size_t tok = (size_t)((b * T + t) * H + h);
                activations(q + tok * K, k + tok * K, g + tok * K, beta_logit[tok], A_log[h],
                            dt_bias + h * K, lower_bound, K, qn + tok * K, kn + tok * K,
                            beta + tok, gk + tok * K);
            }
    return 0;
}

int kda_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
