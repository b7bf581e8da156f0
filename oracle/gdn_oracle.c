/*
 * gdn_oracle.c -- plain fp64 CPU oracle of the Kimi Delta Attention (KDA) /
 * Gated DeltaNet (GDN) per-token step.
 *
 * TEST INFRASTRUCTURE ONLY.  The tests, the package's smoke check and the
 * benchmark's CPU-baseline leg may load this library; the product path never
 * does.  It shares no code, header, table or constant with the CUDA path.
 *
 * What it follows ("Thirty tiny kernels per layer", the decode-step list and
 * the pure step function `_decode_step_pure`; the delta-rule definition of the
 * step; "llama.cpp PR #84", the chunk_kda description of the chunked form):
 *
 *   a1  X = [conv_state (K-1 rows, oldest first); qkv_t];
 *       xhat[c] = silu(sum_j w[c][j] X[j][c]); conv_state <- X[1..K-1]
 *   a2  split xhat into q [H_qk,d_k], k [H_qk,d_k], v [H_v,d_v];
 *       q <- q * s / sqrt(sum q^2 + eps_l2),  k <- k / sqrt(sum k^2 + eps_l2)
 *   a3  g = -exp(A_log[h]) * softplus(f + dt_bias)   (per key channel: KDA;
 *       one per head: GDN);  alpha = exp(g).  Lower-bound ("safe") gate of the
 *       GLM KDA ("llama.cpp PR #84", the KDA decay precompute):
 *       g = lb[h] * sigmoid(-a[h] f) per key channel, lb <= 0 bounding g from below
 *   a4  beta = sigmoid(beta_logit)
 *   a5  S <- (I - beta k k^T) Diag(alpha) S + beta k v^T, written as
 *       St = Diag(alpha) S;  u = beta (v - St^T k);  S = St + k u^T
 *   a6  o = S^T q (with the updated S)
 *   a7  y = o / sqrt(mean(o^2) + eps_norm) * w * silu(z)   (or * sigmoid(z), the
 *       output gate of the GLM KDA: "llama.cpp PR #84", the gated-norm fusion)
 *
 * Readings where the pages are silent (listed with the other readings in the
 * design notes): softplus(x) = max(x,0) + log1p(exp(-|x|)) with no cut-off;
 * causal conv with tap K-1 on the current token and no bias; value head h
 * reads qk head h / (H_v / H_qk); A_log is per value head, dt_bias is
 * [H_v, d_k] (KDA) or [H_v] (GDN); the norm weight is one [d_v] vector.
 *
 * Parity pins for every function here live in the CPU test suite (closed
 * forms, special cases, brute-force matrix products on tiny sizes, and
 * sequential == chunked == verify).
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int B, T, H_qk, H_v, d_k, d_v, K;
    int gate;         /* 0: one decay per head (GDN); 1: per key channel (KDA);
                         2: per key channel, lower-bound form (A_log holds a, dt_bias lb) */
    int out_gate;     /* 0: silu(z); 1: sigmoid(z) */
    double q_scale;   /* d_k^-1/2 as the caller rounded it */
    double eps_l2, eps_norm;
} gdn_oracle_shape;

/* ---------------------------------------------------------------- scalars */

double gdn_oracle_silu(double x) { return x / (1.0 + exp(-x)); }

double gdn_oracle_sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

double gdn_oracle_softplus(double x)
{
    return (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
}

/* ---------------------------------------------------------------- a2 */

/* out = x * scale / sqrt(sum x^2 + eps) over n entries. */
void gdn_oracle_l2norm(int n, const double *x, double scale, double eps, double *out)
{
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double r = scale / sqrt(ss + eps);
    for (int i = 0; i < n; ++i) out[i] = x[i] * r;
}

/* ---------------------------------------------------------------- a3 */

/* Log-decay g[i] = -exp(A_log) * softplus(f[i] + dt_bias[i]) for n channels. */
void gdn_oracle_log_decay(int n, const double *f, const double *dt_bias, double A_log,
                          double *g)
{
    double a = exp(A_log);
    for (int i = 0; i < n; ++i) g[i] = -a * gdn_oracle_softplus(f[i] + dt_bias[i]);
}

/* Lower-bound log-decay g[i] = lb * sigmoid(-a * f[i]) for n channels. */
void gdn_oracle_log_decay_lb(int n, const double *f, double a, double lb, double *g)
{
    for (int i = 0; i < n; ++i) g[i] = lb * gdn_oracle_sigmoid(-a * f[i]);
}

/* ---------------------------------------------------------------- a5 + a6 */

/*
 * One delta-rule update of a [d_k, d_v] state (row i = key channel, column
 * j = value channel, S[i*d_v + j]) followed by the readout o = S^T q.
 */
void gdn_oracle_delta_step(int d_k, int d_v, double *S, const double *alpha, double beta,
                           const double *k, const double *v, const double *q, double *o)
{
    double *u = (double *)malloc(sizeof(double) * (size_t)d_v);
    for (int i = 0; i < d_k; ++i)
        for (int j = 0; j < d_v; ++j) S[(size_t)i * d_v + j] *= alpha[i];
    for (int j = 0; j < d_v; ++j) {
        double kS = 0.0;
        for (int i = 0; i < d_k; ++i) kS += S[(size_t)i * d_v + j] * k[i];
        u[j] = beta * (v[j] - kS);
    }
    for (int i = 0; i < d_k; ++i)
        for (int j = 0; j < d_v; ++j) S[(size_t)i * d_v + j] += k[i] * u[j];
    for (int j = 0; j < d_v; ++j) {
        double acc = 0.0;
        for (int i = 0; i < d_k; ++i) acc += S[(size_t)i * d_v + j] * q[i];
        o[j] = acc;
    }
    free(u);
}

/* ---------------------------------------------------------------- a7 */

/* sigmoid_gate: 0 multiplies by silu(z), 1 by sigmoid(z). */
void gdn_oracle_gated_rmsnorm(int n, const double *o, const double *z, const double *w,
                              double eps, int sigmoid_gate, double *y)
{
    double ms = 0.0;
    for (int j = 0; j < n; ++j) ms += o[j] * o[j];
    ms /= (double)n;
    double r = 1.0 / sqrt(ms + eps);
    for (int j = 0; j < n; ++j)
        y[j] = o[j] * r * w[j] * (sigmoid_gate ? gdn_oracle_sigmoid(z[j]) : gdn_oracle_silu(z[j]));
}

/* ---------------------------------------------------------------- a1 */

static size_t n_channels(const gdn_oracle_shape *s)
{
    return (size_t)2 * s->H_qk * s->d_k + (size_t)s->H_v * s->d_v;
}

/* Row r of X = [conv_state[b] (K-1 rows); qkv[b, 0..T-1]] at channel c. */
static double x_row(const gdn_oracle_shape *s, const float *qkv, const double *conv_state0,
                    int b, int r, size_t c)
{
    size_t C = n_channels(s);
    if (r < s->K - 1) return conv_state0[((size_t)b * (s->K - 1) + r) * C + c];
    return (double)qkv[((size_t)b * s->T + (r - (s->K - 1))) * C + c];
}

/* Post-conv, post-SiLU value of channel c at token t. */
static double conv_at(const gdn_oracle_shape *s, const float *qkv, const float *conv_w,
                      const double *conv_state0, int b, int t, size_t c)
{
    double acc = 0.0;
    for (int j = 0; j < s->K; ++j)
        acc += (double)conv_w[c * s->K + j] * x_row(s, qkv, conv_state0, b, t + j, c);
    return gdn_oracle_silu(acc);
}

/* a1 alone: xhat [B,T,C]; conv_state [B,K-1,C] is advanced in place. */
void gdn_oracle_conv(const gdn_oracle_shape *s, const float *qkv, const float *conv_w,
                     double *conv_state, double *xhat)
{
    size_t C = n_channels(s);
    size_t nstate = (size_t)s->B * (s->K - 1) * C;
    double *cs0 = (double *)malloc(sizeof(double) * (nstate ? nstate : 1));
    memcpy(cs0, conv_state, sizeof(double) * nstate);
    for (int b = 0; b < s->B; ++b)
        for (int t = 0; t < s->T; ++t)
            for (size_t c = 0; c < C; ++c)
                xhat[((size_t)b * s->T + t) * C + c] = conv_at(s, qkv, conv_w, cs0, b, t, c);
    for (int b = 0; b < s->B; ++b)
        for (int r = 0; r < s->K - 1; ++r)
            for (size_t c = 0; c < C; ++c)
                conv_state[((size_t)b * (s->K - 1) + r) * C + c] =
                    x_row(s, qkv, cs0, b, s->T + r, c);
    free(cs0);
}

/* ---------------------------------------------------------------- per-unit inputs */

typedef struct {
    const gdn_oracle_shape *s;
    const float *qkv, *f, *beta, *z, *conv_w, *A_log, *dt_bias, *norm_w;
    const double *conv_state0;
    double *state, *y, *o_raw, *state_hist;
    int chunk;          /* 0: sequential; > 0: chunked form with this chunk size */
    int nthreads;
    int tid;
} job_t;

/* q, k, v (a1 + a2), log-decay g (a3) and beta (a4) of unit (b, h) at token t. */
static void token_inputs(const job_t *J, int b, int h, int t, double *q, double *k, double *v,
                         double *g, double *beta)
{
    const gdn_oracle_shape *s = J->s;
    int group = s->H_v / s->H_qk;
    int hq = h / group;
    size_t qoff = (size_t)hq * s->d_k;
    size_t koff = (size_t)s->H_qk * s->d_k + (size_t)hq * s->d_k;
    size_t voff = (size_t)2 * s->H_qk * s->d_k + (size_t)h * s->d_v;
    double *tmp = (double *)malloc(sizeof(double) * (size_t)(s->d_k > s->d_v ? s->d_k : s->d_v));

    for (int i = 0; i < s->d_k; ++i)
        tmp[i] = conv_at(s, J->qkv, J->conv_w, J->conv_state0, b, t, qoff + i);
    gdn_oracle_l2norm(s->d_k, tmp, s->q_scale, s->eps_l2, q);
    for (int i = 0; i < s->d_k; ++i)
        tmp[i] = conv_at(s, J->qkv, J->conv_w, J->conv_state0, b, t, koff + i);
    gdn_oracle_l2norm(s->d_k, tmp, 1.0, s->eps_l2, k);
    for (int j = 0; j < s->d_v; ++j)
        v[j] = conv_at(s, J->qkv, J->conv_w, J->conv_state0, b, t, voff + j);

    size_t bth = ((size_t)b * s->T + t) * s->H_v + h;
    if (s->gate == 2) {
        double *fi = (double *)malloc(sizeof(double) * (size_t)s->d_k);
        for (int i = 0; i < s->d_k; ++i) fi[i] = (double)J->f[bth * s->d_k + i];
        gdn_oracle_log_decay_lb(s->d_k, fi, (double)J->A_log[h], (double)J->dt_bias[h], g);
        free(fi);
    } else if (s->gate == 1) {
        double *fi = (double *)malloc(sizeof(double) * (size_t)s->d_k);
        double *di = (double *)malloc(sizeof(double) * (size_t)s->d_k);
        for (int i = 0; i < s->d_k; ++i) {
            fi[i] = (double)J->f[bth * s->d_k + i];
            di[i] = (double)J->dt_bias[(size_t)h * s->d_k + i];
        }
        gdn_oracle_log_decay(s->d_k, fi, di, (double)J->A_log[h], g);
        free(fi);
        free(di);
    } else {
        double fi = (double)J->f[bth], di = (double)J->dt_bias[h], g0;
        gdn_oracle_log_decay(1, &fi, &di, (double)J->A_log[h], &g0);
        for (int i = 0; i < s->d_k; ++i) g[i] = g0;
    }
    *beta = gdn_oracle_sigmoid((double)J->beta[bth]);
    free(tmp);
}

static void emit_output(const job_t *J, int b, int h, int t, const double *o)
{
    const gdn_oracle_shape *s = J->s;
    size_t row = (((size_t)b * s->T + t) * s->H_v + h) * s->d_v;
    double *z = (double *)malloc(sizeof(double) * (size_t)s->d_v);
    double *w = (double *)malloc(sizeof(double) * (size_t)s->d_v);
    for (int j = 0; j < s->d_v; ++j) {
        z[j] = (double)J->z[row + j];
        w[j] = (double)J->norm_w[j];
    }
    gdn_oracle_gated_rmsnorm(s->d_v, o, z, w, s->eps_norm, s->out_gate, J->y + row);
    if (J->o_raw) memcpy(J->o_raw + row, o, sizeof(double) * (size_t)s->d_v);
    free(z);
    free(w);
}

/* ---------------------------------------------------------------- sequential unit */

static void run_unit_sequential(const job_t *J, int b, int h)
{
    const gdn_oracle_shape *s = J->s;
    size_t dd = (size_t)s->d_k * s->d_v;
    double *S = J->state + ((size_t)b * s->H_v + h) * dd;
    double *q = malloc(sizeof(double) * s->d_k), *k = malloc(sizeof(double) * s->d_k);
    double *g = malloc(sizeof(double) * s->d_k), *alpha = malloc(sizeof(double) * s->d_k);
    double *v = malloc(sizeof(double) * s->d_v), *o = malloc(sizeof(double) * s->d_v);
    double beta;
    for (int t = 0; t < s->T; ++t) {
        token_inputs(J, b, h, t, q, k, v, g, &beta);
        for (int i = 0; i < s->d_k; ++i) alpha[i] = exp(g[i]);
        gdn_oracle_delta_step(s->d_k, s->d_v, S, alpha, beta, k, v, q, o);
        emit_output(J, b, h, t, o);
        if (J->state_hist)
            memcpy(J->state_hist + (((size_t)t * s->B + b) * s->H_v + h) * dd, S,
                   sizeof(double) * dd);
    }
    free(q); free(k); free(g); free(alpha); free(v); free(o);
}

/* ---------------------------------------------------------------- chunked unit */

/*
 * The same recurrence in the chunked WY/UT form ("llama.cpp PR #84", chunked
 * KDA prefill): inside a chunk of n tokens with start state S0 and
 * per-channel cumulative log-decay G_t = sum_{r<=t} g_r,
 *   L[t][s] = sum_i k_t,i k_s,i exp(G_t,i - G_s,i)              (s < t)
 *   (I + diag(beta) L) W  = diag(beta) (exp(G) . K)      (forward substitution)
 *   (I + diag(beta) L) Ut = diag(beta) V
 *   Vn = Ut - W S0
 *   O_t = S0^T (exp(G_t) . q_t) + sum_{s<=t} M[t][s] Vn_s,
 *        M[t][s] = sum_i q_t,i k_s,i exp(G_t,i - G_s,i)
 *   S  <- Diag(exp(G_n)) S0 + sum_s (k_s . exp(G_n - G_s)) Vn_s^T
 * Every exponent is <= 0.  Used only to check chunked == sequential.
 */
static void run_unit_chunked(const job_t *J, int b, int h)
{
    const gdn_oracle_shape *s = J->s;
    const int dk = s->d_k, dv = s->d_v, CS = J->chunk;
    size_t dd = (size_t)dk * dv;
    double *S = J->state + ((size_t)b * s->H_v + h) * dd;
    double *Q = malloc(sizeof(double) * CS * dk), *Kc = malloc(sizeof(double) * CS * dk);
    double *V = malloc(sizeof(double) * CS * dv), *G = malloc(sizeof(double) * CS * dk);
    double *Bt = malloc(sizeof(double) * CS);
    double *L = malloc(sizeof(double) * CS * CS);
    double *W = malloc(sizeof(double) * CS * dk), *Ut = malloc(sizeof(double) * CS * dv);
    double *Vn = malloc(sizeof(double) * CS * dv), *o = malloc(sizeof(double) * dv);
    double *Snew = malloc(sizeof(double) * dd), *g = malloc(sizeof(double) * dk);

    for (int c0 = 0; c0 < s->T; c0 += CS) {
        int n = s->T - c0 < CS ? s->T - c0 : CS;
        for (int t = 0; t < n; ++t) {
            token_inputs(J, b, h, c0 + t, Q + t * dk, Kc + t * dk, V + t * dv, g, Bt + t);
            for (int i = 0; i < dk; ++i) G[t * dk + i] = g[i] + (t ? G[(t - 1) * dk + i] : 0.0);
        }
        for (int t = 0; t < n; ++t)
            for (int r = 0; r < t; ++r) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i)
                    acc += Kc[t * dk + i] * Kc[r * dk + i] * exp(G[t * dk + i] - G[r * dk + i]);
                L[t * CS + r] = acc;
            }
        for (int t = 0; t < n; ++t) {
            for (int i = 0; i < dk; ++i) {
                double acc = Bt[t] * exp(G[t * dk + i]) * Kc[t * dk + i];
                for (int r = 0; r < t; ++r) acc -= Bt[t] * L[t * CS + r] * W[r * dk + i];
                W[t * dk + i] = acc;
            }
            for (int j = 0; j < dv; ++j) {
                double acc = Bt[t] * V[t * dv + j];
                for (int r = 0; r < t; ++r) acc -= Bt[t] * L[t * CS + r] * Ut[r * dv + j];
                Ut[t * dv + j] = acc;
            }
        }
        for (int t = 0; t < n; ++t)
            for (int j = 0; j < dv; ++j) {
                double ws = 0.0;
                for (int i = 0; i < dk; ++i) ws += W[t * dk + i] * S[(size_t)i * dv + j];
                Vn[t * dv + j] = Ut[t * dv + j] - ws;
            }
        for (int t = 0; t < n; ++t) {
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i)
                    acc += exp(G[t * dk + i]) * Q[t * dk + i] * S[(size_t)i * dv + j];
                o[j] = acc;
            }
            for (int r = 0; r <= t; ++r) {
                double m = 0.0;
                for (int i = 0; i < dk; ++i)
                    m += Q[t * dk + i] * Kc[r * dk + i] * exp(G[t * dk + i] - G[r * dk + i]);
                for (int j = 0; j < dv; ++j) o[j] += m * Vn[r * dv + j];
            }
            emit_output(J, b, h, c0 + t, o);
        }
        for (int i = 0; i < dk; ++i) {
            double gl = G[(n - 1) * dk + i];
            for (int j = 0; j < dv; ++j) {
                double acc = exp(gl) * S[(size_t)i * dv + j];
                for (int r = 0; r < n; ++r)
                    acc += Kc[r * dk + i] * exp(gl - G[r * dk + i]) * Vn[r * dv + j];
                Snew[(size_t)i * dv + j] = acc;
            }
        }
        memcpy(S, Snew, sizeof(double) * dd);
    }
    free(Q); free(Kc); free(V); free(G); free(Bt); free(L); free(W); free(Ut);
    free(Vn); free(o); free(Snew); free(g);
}

/* ---------------------------------------------------------------- driver */

static void *worker(void *arg)
{
    const job_t *J = (const job_t *)arg;
    int units = J->s->B * J->s->H_v;
    for (int u = J->tid; u < units; u += J->nthreads) {
        int b = u / J->s->H_v, h = u % J->s->H_v;
        if (J->chunk > 0) run_unit_chunked(J, b, h);
        else run_unit_sequential(J, b, h);
    }
    return NULL;
}

static int check_shape(const gdn_oracle_shape *s)
{
    if (s->B < 0 || s->T < 0 || s->H_qk <= 0 || s->H_v <= 0 || s->d_k <= 0 || s->d_v <= 0 ||
        s->K < 1 || s->H_v % s->H_qk != 0)
        return -3;
    return 0;
}

static int drive(const gdn_oracle_shape *s, const float *qkv, const float *f, const float *beta,
                 const float *z, const float *conv_w, const float *A_log, const float *dt_bias,
                 const float *norm_w, double *conv_state, double *state, double *y,
                 double *o_raw, double *state_hist, int chunk, int nthreads)
{
    int rc = check_shape(s);
    if (rc) return rc;
    size_t C = n_channels(s);
    size_t nstate = (size_t)s->B * (s->K - 1) * C;
    double *cs0 = (double *)malloc(sizeof(double) * (nstate ? nstate : 1));
    memcpy(cs0, conv_state, sizeof(double) * nstate);

    int units = s->B * s->H_v;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > units) nthreads = units > 0 ? units : 1;
    job_t *jobs = (job_t *)calloc((size_t)nthreads, sizeof(job_t));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int i = 0; i < nthreads; ++i) {
        job_t J = {s, qkv, f, beta, z, conv_w, A_log, dt_bias, norm_w, cs0,
                   state, y, o_raw, state_hist, chunk, nthreads, i};
        jobs[i] = J;
    }
    for (int i = 1; i < nthreads; ++i) pthread_create(&th[i], NULL, worker, &jobs[i]);
    worker(&jobs[0]);
    for (int i = 1; i < nthreads; ++i) pthread_join(th[i], NULL);

    /* a1's state update: the last K-1 rows of [conv_state; qkv]. */
    for (int b = 0; b < s->B; ++b)
        for (int r = 0; r < s->K - 1; ++r)
            for (size_t c = 0; c < C; ++c)
                conv_state[((size_t)b * (s->K - 1) + r) * C + c] =
                    x_row(s, qkv, cs0, b, s->T + r, c);
    free(cs0);
    free(jobs);
    free(th);
    return 0;
}

/*
 * T sequential steps (a1..a7) for every sequence and value head.
 *   qkv [B,T,C], f [B,T,H_v,d_k] (KDA) or [B,T,H_v] (GDN), beta [B,T,H_v] logits,
 *   z [B,T,H_v,d_v]; conv_w [C,K], A_log [H_v], dt_bias [H_v,d_k] / [H_v], norm_w [d_v];
 *   conv_state [B,K-1,C] and state [B,H_v,d_k,d_v] advanced in place;
 *   y [B,T,H_v,d_v]; o_raw (optional) the readout before the norm;
 *   state_hist (optional) [T,B,H_v,d_k,d_v] = state after each token.
 * Returns 0, or -3 for an impossible shape.
 */
int gdn_oracle_run(const gdn_oracle_shape *s, const float *qkv, const float *f,
                   const float *beta, const float *z, const float *conv_w, const float *A_log,
                   const float *dt_bias, const float *norm_w, double *conv_state, double *state,
                   double *y, double *o_raw, double *state_hist, int nthreads)
{
    return drive(s, qkv, f, beta, z, conv_w, A_log, dt_bias, norm_w, conv_state, state, y, o_raw,
                 state_hist, 0, nthreads);
}

/* The chunked WY/UT form of the same T tokens (no per-token states). */
int gdn_oracle_run_chunked(const gdn_oracle_shape *s, int chunk, const float *qkv,
                           const float *f, const float *beta, const float *z,
                           const float *conv_w, const float *A_log, const float *dt_bias,
                           const float *norm_w, double *conv_state, double *state, double *y,
                           double *o_raw, int nthreads)
{
    if (chunk < 1) return -3;
    return drive(s, qkv, f, beta, z, conv_w, A_log, dt_bias, norm_w, conv_state, state, y, o_raw,
                 NULL, chunk, nthreads);
}
