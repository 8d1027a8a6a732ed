/*
 * gdn_oracle.c -- fp64 CPU oracle for the Gated DeltaNet verify path.
 *
 * TEST INFRASTRUCTURE ONLY (see gdn_oracle.h).  Plain, slow and literal: every
 * step is written out in the order of the gated delta rule, in fp64, with no
 * blocking, fusion or reordering.  Built with -ffp-contract=off so the
 * results are the same on x86-64 and aarch64.
 */
#include "gdn_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }
static double silu(double x) { return x * sigmoid(x); }

/* ---------------------------------------------------------------------- */
/* stages                                                                 */
/* ---------------------------------------------------------------------- */

/* Depthwise causal conv: the window is concat(old conv state, new tokens) in
 * time order (internal.h, DeltaNetCapture: "concat(old_conv_state,
 * qkv_new_tokens) fed to ggml_ssm_conv"); weights are [kernel, dim]
 * (internal.h, TargetLayer::ssm_conv1d).  Tap j multiplies window row t+j, so
 * the last tap meets the current token.  No bias.  SiLU follows the conv. */
void gdno_conv_silu(int W, int T, int C, const double *conv_w, const double *win, double *y)
{
    for (int t = 0; t < T; ++t)
        for (int c = 0; c < C; ++c) {
            double acc = 0.0;
            for (int j = 0; j < W; ++j)
                acc += conv_w[(size_t)j * C + c] * win[(size_t)(t + j) * C + c];
            y[(size_t)t * C + c] = silu(acc);
        }
}

void gdno_l2norm(int n, const double *x, double eps, double *xhat)
{
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    double inv = 1.0 / sqrt(ss + eps);
    for (int i = 0; i < n; ++i) xhat[i] = x[i] * inv;
}

double gdno_softplus(double x)
{
    if (x > 30.0) return x;         /* log1p(exp(x)) == x to fp64 precision */
    return log1p(exp(x));
}

/* log of the decay gate: -exp(A_log) * softplus(alpha + dt_bias).  ssm_a in
 * internal.h is the per-head "-A" parameter; A_log is its log-magnitude. */
static double log_gate(double A_log, double dt_bias, double alpha)
{
    return -exp(A_log) * gdno_softplus(alpha + dt_bias);
}

void gdno_gates(double A_log, double dt_bias, double alpha, double beta_raw,
                double *g, double *beta)
{
    *g = exp(log_gate(A_log, dt_bias, alpha));
    *beta = sigmoid(beta_raw);
}

/* One step of the gated delta rule on logical S[i][j] (i over d_k, j over d_v):
 * decay, read the current association for k, write beta*(v - read), then read
 * out with q. */
void gdno_delta_step(int dk, int dv, double *S, const double *k, const double *v,
                     const double *q, double g, double beta, double q_scale, double *o)
{
    double u[dv];
    for (int i = 0; i < dk; ++i)                       /* S~ = g S */
        for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= g;
    for (int j = 0; j < dv; ++j) {                     /* u = S~^T k */
        double acc = 0.0;
        for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * k[i];
        u[j] = acc;
    }
    for (int i = 0; i < dk; ++i)                       /* S = S~ + beta k (v - u)^T */
        for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] += beta * k[i] * (v[j] - u[j]);
    for (int j = 0; j < dv; ++j) {                     /* o = q_scale S^T q */
        double acc = 0.0;
        for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * q[i];
        o[j] = q_scale * acc;
    }
}

/* Gated RMSNorm: internal.h TargetLayer::ssm_norm is one [head_v_dim] weight
 * and wqkv_gate is the "z" projection; eps is TargetWeights::rms_eps. */
void gdno_rmsnorm_gate(int dv, const double *o, const double *z, const double *w,
                       double eps, double *out)
{
    double ss = 0.0;
    for (int j = 0; j < dv; ++j) ss += o[j] * o[j];
    double inv = 1.0 / sqrt(ss / dv + eps);
    for (int j = 0; j < dv; ++j) out[j] = o[j] * inv * w[j] * silu(z[j]);
}

/* ---------------------------------------------------------------------- */
/* helpers shared by the composites                                       */
/* ---------------------------------------------------------------------- */

static int dims_ok(const gdno_dims *d)
{
    return d && d->n_slots >= 0 && d->n_qk_heads > 0 && d->n_v_heads > 0 &&
           d->n_v_heads % d->n_qk_heads == 0 && d->d_k > 0 && d->d_v > 0 &&
           d->conv_width >= 1 && d->n_tokens >= 0;
}

static size_t n_channels(const gdno_dims *d)
{
    return (size_t)2 * d->n_qk_heads * d->d_k + (size_t)d->n_v_heads * d->d_v;
}

/* Per slot: build the window, run conv+SiLU, store the window capture and the
 * new conv state.  y_all is [B][T][C]. */
static void conv_all_slots(const gdno_dims *d, const double *conv_w, const double *qkv,
                           double *conv_state, double *cap_conv, double *y_all)
{
    const int W = d->conv_width, T = d->n_tokens;
    const size_t C = n_channels(d);
    double *win = (double *)malloc(sizeof(double) * (size_t)(W - 1 + T) * C + 1);
    for (int s = 0; s < d->n_slots; ++s) {
        memcpy(win, conv_state + (size_t)s * (W - 1) * C, sizeof(double) * (W - 1) * C);
        memcpy(win + (size_t)(W - 1) * C, qkv + (size_t)s * T * C, sizeof(double) * T * C);
        gdno_conv_silu(W, T, (int)C, conv_w, win, y_all + (size_t)s * T * C);
        if (cap_conv)
            memcpy(cap_conv + (size_t)s * (W - 1 + T) * C, win, sizeof(double) * (W - 1 + T) * C);
        memcpy(conv_state + (size_t)s * (W - 1) * C, win + (size_t)T * C,
               sizeof(double) * (W - 1) * C);
    }
    free(win);
}

/* state storage [B][H_v][d_v][d_k] <-> logical S[i][j] */
static void load_state(const gdno_dims *d, const double *state, int s, int h, double *S)
{
    const int dk = d->d_k, dv = d->d_v;
    const double *src = state + ((size_t)s * d->n_v_heads + h) * dv * dk;
    for (int j = 0; j < dv; ++j)
        for (int i = 0; i < dk; ++i) S[(size_t)i * dv + j] = src[(size_t)j * dk + i];
}

static void store_state(const gdno_dims *d, double *dst_head, const double *S)
{
    const int dk = d->d_k, dv = d->d_v;
    for (int j = 0; j < dv; ++j)
        for (int i = 0; i < dk; ++i) dst_head[(size_t)j * dk + i] = S[(size_t)i * dv + j];
}

typedef struct {
    const gdno_dims *d;
    const double *conv_w, *A_log, *dt_bias, *norm_w, *z, *alpha, *beta_raw, *y_all;
    double *state, *cap_state, *out;
    const unsigned char *head_mask;
    int chunk;                 /* 0 = sequential form */
    int tid, n_threads;
    const int *parent;         /* tree verify: [B][T] parent of each token, else NULL */
} job_t;

/* q^, k^, v of token t for (slot s, value head h) from the post-SiLU stream.
 * V head h reads key head floor(h / r): consecutive value heads share a key head. */
static void token_qkv(const job_t *J, int s, int h, int t, double *qn, double *kn, const double **v)
{
    const gdno_dims *d = J->d;
    const int r = d->n_v_heads / d->n_qk_heads, kh = h / r;
    const size_t C = n_channels(d);
    const double *y = J->y_all + ((size_t)s * d->n_tokens + t) * C;
    gdno_l2norm(d->d_k, y + (size_t)kh * d->d_k, d->l2_eps, qn);
    gdno_l2norm(d->d_k, y + (size_t)d->n_qk_heads * d->d_k + (size_t)kh * d->d_k, d->l2_eps, kn);
    *v = y + (size_t)2 * d->n_qk_heads * d->d_k + (size_t)h * d->d_v;
}

static void run_head_sequential(const job_t *J, int s, int h)
{
    const gdno_dims *d = J->d;
    const int dk = d->d_k, dv = d->d_v, T = d->n_tokens, Hv = d->n_v_heads;
    double *S = (double *)malloc(sizeof(double) * dk * dv);
    double qn[dk], kn[dk], o[dv];
    load_state(d, J->state, s, h, S);
    for (int t = 0; t < T; ++t) {
        const double *v;
        token_qkv(J, s, h, t, qn, kn, &v);
        const size_t st = (size_t)s * T + t;
        double g, beta;
        gdno_gates(J->A_log[h], J->dt_bias[h], J->alpha[st * Hv + h], J->beta_raw[st * Hv + h], &g, &beta);
        gdno_delta_step(dk, dv, S, kn, v, qn, g, beta, d->q_scale, o);
        if (J->cap_state)
            store_state(d, J->cap_state + (st * Hv + h) * dv * dk, S);
        gdno_rmsnorm_gate(dv, o, J->z + st * Hv * dv + (size_t)h * dv, J->norm_w, d->rms_eps,
                          J->out + st * Hv * dv + (size_t)h * dv);
    }
    store_state(d, J->state + ((size_t)s * Hv + h) * dv * dk, S);
    free(S);
}

/* Chunkwise form.  With Gamma_r the decay accumulated inside the chunk up to
 * and including token r, unrolling the recurrence from the chunk's initial
 * state S0 gives u_r = beta_r (v_r - Gamma_r S0^T k_r - sum_{s<r} (Gamma_r /
 * Gamma_s)(k_r.k_s) u_s), i.e. (I + A) U = diag(beta)(V - diag(Gamma) K S0)
 * with A strictly lower triangular (the WY / UT transform of Yang et al.,
 * "Parallelizing Linear Transformers with the Delta Rule over Sequence
 * Length", NeurIPS 2024, extended by the gate as in Gated Delta Networks). */
static void run_head_chunked(const job_t *J, int s, int h)
{
    const gdno_dims *d = J->d;
    const int dk = d->d_k, dv = d->d_v, L = d->n_tokens, Hv = d->n_v_heads, Cn = J->chunk;
    double *S = (double *)malloc(sizeof(double) * dk * dv);
    double *Q = (double *)malloc(sizeof(double) * Cn * dk);
    double *K = (double *)malloc(sizeof(double) * Cn * dk);
    double *V = (double *)malloc(sizeof(double) * Cn * dv);
    double *A = (double *)malloc(sizeof(double) * Cn * Cn);
    double *Tm = (double *)malloc(sizeof(double) * Cn * Cn);
    double *Wm = (double *)malloc(sizeof(double) * Cn * dk);
    double *Ut = (double *)malloc(sizeof(double) * Cn * dv);
    double *U = (double *)malloc(sizeof(double) * Cn * dv);
    double *O = (double *)malloc(sizeof(double) * Cn * dv);
    double *Snew = (double *)malloc(sizeof(double) * dk * dv);
    double logG[Cn], G[Cn], beta[Cn], o[dv];
    load_state(d, J->state, s, h, S);

    for (int c0 = 0; c0 < L; c0 += Cn) {
        const int n = (L - c0 < Cn) ? L - c0 : Cn;
        double acc_log = 0.0;
        for (int r = 0; r < n; ++r) {
            const double *v;
            const size_t st = (size_t)s * L + c0 + r;
            token_qkv(J, s, h, c0 + r, Q + (size_t)r * dk, K + (size_t)r * dk, &v);
            memcpy(V + (size_t)r * dv, v, sizeof(double) * dv);
            acc_log += log_gate(J->A_log[h], J->dt_bias[h], J->alpha[st * Hv + h]);
            logG[r] = acc_log;                          /* Gamma = exp(cumsum(log g)) */
            G[r] = exp(acc_log);
            beta[r] = sigmoid(J->beta_raw[st * Hv + h]);
        }
        /* A[r][s] = beta_r (Gamma_r / Gamma_s) k_r . k_s for s < r */
        for (int r = 0; r < n; ++r)
            for (int c = 0; c < n; ++c) {
                double a = 0.0;
                if (c < r) {
                    double kk = 0.0;
                    for (int i = 0; i < dk; ++i) kk += K[(size_t)r * dk + i] * K[(size_t)c * dk + i];
                    a = beta[r] * exp(logG[r] - logG[c]) * kk;
                }
                A[(size_t)r * n + c] = a;
            }
        /* Tm = (I + A)^-1 by forward substitution, one column at a time */
        for (int c = 0; c < n; ++c)
            for (int r = 0; r < n; ++r) {
                double x = (r == c) ? 1.0 : 0.0;
                for (int m = 0; m < r; ++m) x -= A[(size_t)r * n + m] * Tm[(size_t)m * n + c];
                Tm[(size_t)r * n + c] = x;
            }
        /* W = Tm diag(beta Gamma) K,  Ut = Tm diag(beta) V */
        for (int r = 0; r < n; ++r) {
            for (int i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (int m = 0; m < n; ++m) acc += Tm[(size_t)r * n + m] * beta[m] * G[m] * K[(size_t)m * dk + i];
                Wm[(size_t)r * dk + i] = acc;
            }
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int m = 0; m < n; ++m) acc += Tm[(size_t)r * n + m] * beta[m] * V[(size_t)m * dv + j];
                Ut[(size_t)r * dv + j] = acc;
            }
        }
        /* U = Ut - W S */
        for (int r = 0; r < n; ++r)
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += Wm[(size_t)r * dk + i] * S[(size_t)i * dv + j];
                U[(size_t)r * dv + j] = Ut[(size_t)r * dv + j] - acc;
            }
        /* O = diag(Gamma) Q S + (Q K^T (.) M) U, M[r][s] = Gamma_r / Gamma_s for s <= r */
        for (int r = 0; r < n; ++r)
            for (int j = 0; j < dv; ++j) {
                double inter = 0.0;
                for (int i = 0; i < dk; ++i) inter += Q[(size_t)r * dk + i] * S[(size_t)i * dv + j];
                double intra = 0.0;
                for (int m = 0; m <= r; ++m) {
                    double qk = 0.0;
                    for (int i = 0; i < dk; ++i) qk += Q[(size_t)r * dk + i] * K[(size_t)m * dk + i];
                    intra += qk * exp(logG[r] - logG[m]) * U[(size_t)m * dv + j];
                }
                O[(size_t)r * dv + j] = G[r] * inter + intra;
            }
        /* S <- Gamma_C S + (diag(Gamma_C / Gamma) K)^T U */
        for (int i = 0; i < dk; ++i)
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int m = 0; m < n; ++m)
                    acc += exp(logG[n - 1] - logG[m]) * K[(size_t)m * dk + i] * U[(size_t)m * dv + j];
                Snew[(size_t)i * dv + j] = G[n - 1] * S[(size_t)i * dv + j] + acc;
            }
        memcpy(S, Snew, sizeof(double) * dk * dv);
        for (int r = 0; r < n; ++r) {
            const size_t st = (size_t)s * L + c0 + r;
            for (int j = 0; j < dv; ++j) o[j] = d->q_scale * O[(size_t)r * dv + j];
            gdno_rmsnorm_gate(dv, o, J->z + st * Hv * dv + (size_t)h * dv, J->norm_w, d->rms_eps,
                              J->out + st * Hv * dv + (size_t)h * dv);
        }
    }
    store_state(d, J->state + ((size_t)s * Hv + h) * dv * dk, S);
    free(S); free(Q); free(K); free(V); free(A); free(Tm); free(Wm); free(Ut); free(U);
    free(O); free(Snew);
}

/* Tree verify for (slot s, value head h): token t starts from the state after
 * its parent (the state before the batch when the parent is -1), so along any
 * path from the root the recurrence is the chain recurrence over that path. */
static void run_head_tree(const job_t *J, int s, int h)
{
    const gdno_dims *d = J->d;
    const int dk = d->d_k, dv = d->d_v, T = d->n_tokens, Hv = d->n_v_heads;
    double *S = (double *)malloc(sizeof(double) * dk * dv);
    double qn[dk], kn[dk], o[dv];
    for (int t = 0; t < T; ++t) {
        const int p = J->parent[(size_t)s * T + t];
        if (p < 0) load_state(d, J->state, s, h, S);
        else {
            /* cap_state[s][p] has the layout of one slot of `state` */
            const double *src = J->cap_state + (((size_t)s * T + p) * Hv + h) * dv * dk;
            for (int j = 0; j < dv; ++j)
                for (int i = 0; i < dk; ++i) S[(size_t)i * dv + j] = src[(size_t)j * dk + i];
        }
        const double *v;
        token_qkv(J, s, h, t, qn, kn, &v);
        const size_t st = (size_t)s * T + t;
        double g, beta;
        gdno_gates(J->A_log[h], J->dt_bias[h], J->alpha[st * Hv + h], J->beta_raw[st * Hv + h], &g, &beta);
        gdno_delta_step(dk, dv, S, kn, v, qn, g, beta, d->q_scale, o);
        store_state(d, J->cap_state + (st * Hv + h) * dv * dk, S);
        gdno_rmsnorm_gate(dv, o, J->z + st * Hv * dv + (size_t)h * dv, J->norm_w, d->rms_eps,
                          J->out + st * Hv * dv + (size_t)h * dv);
    }
    free(S);
}

static void *worker(void *arg)
{
    const job_t *J = (const job_t *)arg;
    const int Hv = J->d->n_v_heads, n_items = J->d->n_slots * Hv;
    for (int it = J->tid; it < n_items; it += J->n_threads) {
        const int s = it / Hv, h = it % Hv;
        if (J->head_mask && !J->head_mask[h]) continue;
        if (J->parent) run_head_tree(J, s, h);
        else if (J->chunk > 0) run_head_chunked(J, s, h);
        else run_head_sequential(J, s, h);
    }
    return NULL;
}

static void run_items(job_t *proto, int n_threads)
{
    if (n_threads < 1) n_threads = 1;
    if (n_threads == 1) {
        proto->tid = 0; proto->n_threads = 1;
        worker(proto);
        return;
    }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * n_threads);
    job_t *jobs = (job_t *)malloc(sizeof(job_t) * n_threads);
    for (int i = 0; i < n_threads; ++i) {
        jobs[i] = *proto;
        jobs[i].tid = i;
        jobs[i].n_threads = n_threads;
        pthread_create(&th[i], NULL, worker, &jobs[i]);
    }
    for (int i = 0; i < n_threads; ++i) pthread_join(th[i], NULL);
    free(th); free(jobs);
}

/* ---------------------------------------------------------------------- */
/* composites                                                             */
/* ---------------------------------------------------------------------- */

int gdno_verify(const gdno_dims *d, const double *conv_w, const double *A_log,
                const double *dt_bias, const double *norm_w,
                const double *qkv, const double *z, const double *alpha, const double *beta_raw,
                double *state, double *conv_state, double *cap_state, double *cap_conv,
                double *out, const unsigned char *head_mask, int n_threads)
{
    if (!dims_ok(d)) return -1;
    const size_t C = n_channels(d);
    double *y_all = (double *)malloc(sizeof(double) * (size_t)d->n_slots * d->n_tokens * C + 1);
    conv_all_slots(d, conv_w, qkv, conv_state, cap_conv, y_all);
    job_t J = {d, conv_w, A_log, dt_bias, norm_w, z, alpha, beta_raw, y_all,
               state, cap_state, out, head_mask, 0, 0, 1, NULL};
    run_items(&J, n_threads);
    free(y_all);
    return 0;
}

int gdno_prefill_chunked(const gdno_dims *d, int chunk, const double *conv_w,
                         const double *A_log, const double *dt_bias, const double *norm_w,
                         const double *qkv, const double *z, const double *alpha,
                         const double *beta_raw, double *state, double *conv_state,
                         double *out, const unsigned char *head_mask, int n_threads)
{
    if (!dims_ok(d) || chunk < 1) return -1;
    const size_t C = n_channels(d);
    double *y_all = (double *)malloc(sizeof(double) * (size_t)d->n_slots * d->n_tokens * C + 1);
    conv_all_slots(d, conv_w, qkv, conv_state, NULL, y_all);
    job_t J = {d, conv_w, A_log, dt_bias, norm_w, z, alpha, beta_raw, y_all,
               state, NULL, out, head_mask, chunk, 0, 1, NULL};
    run_items(&J, n_threads);
    free(y_all);
    return 0;
}

int gdno_rollback(const gdno_dims *d, const int *trim, double *state, double *conv_state,
                  const double *cap_state, const double *cap_conv, int *slot_status)
{
    if (!dims_ok(d)) return -1;
    const int T = d->n_tokens, W = d->conv_width;
    const size_t C = n_channels(d);
    const size_t per_state = (size_t)d->n_v_heads * d->d_v * d->d_k;
    int refused = 0;
    for (int s = 0; s < d->n_slots; ++s) {
        slot_status[s] = 0;
        if (trim[s] == 0) continue;                     /* nothing to discard */
        if (trim[s] < 0 || trim[s] >= T) {              /* would discard more than was verified */
            slot_status[s] = 1;
            ++refused;
            continue;
        }
        const int accepted_idx = T - 1 - trim[s];
        const int commit_n = accepted_idx + 1;
        memcpy(state + (size_t)s * per_state,
               cap_state + ((size_t)s * T + accepted_idx) * per_state, sizeof(double) * per_state);
        memcpy(conv_state + (size_t)s * (W - 1) * C,
               cap_conv + ((size_t)s * (W - 1 + T) + commit_n) * C, sizeof(double) * (W - 1) * C);
    }
    return refused;
}

/* ---------------------------------------------------------------------- */
/* tree (DDTree) verify                                                   */
/* ---------------------------------------------------------------------- */

/* The raw input row of node n for slot s: a token of the batch for n >= 0,
 * else the old conv state, most recent row first (n = -1 is row W-2). */
static const double *node_input(const gdno_dims *d, const double *qkv, const double *conv_state, int s, int n)
{
    const int W = d->conv_width, T = d->n_tokens;
    const size_t C = n_channels(d);
    if (n >= 0) return qkv + ((size_t)s * T + n) * C;
    return conv_state + ((size_t)s * (W - 1) + (W - 1) + n) * C;
}

int gdno_verify_tree(const gdno_dims *d, const int *parent, const double *conv_w, const double *A_log,
                     const double *dt_bias, const double *norm_w,
                     const double *qkv, const double *z, const double *alpha, const double *beta_raw,
                     const double *state, const double *conv_state, double *cap_state, double *cap_conv,
                     double *out, const unsigned char *head_mask, int n_threads)
{
    if (!dims_ok(d) || !parent || !cap_state || !cap_conv) return -1;
    const int W = d->conv_width, T = d->n_tokens;
    const size_t C = n_channels(d);
    for (int s = 0; s < d->n_slots; ++s)
        for (int t = 0; t < T; ++t) {
            const int p = parent[(size_t)s * T + t];
            if (p < -1 || p >= t) return -2;            /* not a tree in token order */
        }
    double *y_all = (double *)malloc(sizeof(double) * (size_t)d->n_slots * T * C + 1);
    double *win = (double *)malloc(sizeof(double) * (size_t)W * C + 1);
    for (int s = 0; s < d->n_slots; ++s)
        for (int t = 0; t < T; ++t) {
            /* window of t: its W-1 nearest ancestors (oldest first), then t; past the
             * root the ancestors continue into the old conv state */
            int anc = t;
            for (int j = W - 1; j >= 0; --j) {
                memcpy(win + (size_t)j * C, node_input(d, qkv, conv_state, s, anc), sizeof(double) * C);
                anc = anc >= 0 ? parent[(size_t)s * T + anc] : anc - 1;
            }
            gdno_conv_silu(W, 1, (int)C, conv_w, win, y_all + ((size_t)s * T + t) * C);
            memcpy(cap_conv + ((size_t)s * T + t) * (W - 1) * C, win + C, sizeof(double) * (W - 1) * C);
        }
    free(win);
    job_t J = {d, conv_w, A_log, dt_bias, norm_w, z, alpha, beta_raw, y_all,
               (double *)state, cap_state, out, head_mask, 0, 0, 1, parent};
    run_items(&J, n_threads);
    free(y_all);
    return 0;
}

int gdno_rollback_tree(const gdno_dims *d, const int *accept, double *state, double *conv_state,
                       const double *cap_state, const double *cap_conv, int *slot_status)
{
    if (!dims_ok(d)) return -1;
    const int T = d->n_tokens, W = d->conv_width;
    const size_t C = n_channels(d);
    const size_t per_state = (size_t)d->n_v_heads * d->d_v * d->d_k;
    int refused = 0;
    for (int s = 0; s < d->n_slots; ++s) {
        slot_status[s] = 0;
        if (accept[s] == -1) continue;                  /* nothing accepted: keep the state before the batch */
        if (accept[s] < -1 || accept[s] >= T) {
            slot_status[s] = 1;
            ++refused;
            continue;
        }
        memcpy(state + (size_t)s * per_state, cap_state + ((size_t)s * T + accept[s]) * per_state,
               sizeof(double) * per_state);
        memcpy(conv_state + (size_t)s * (W - 1) * C, cap_conv + ((size_t)s * T + accept[s]) * (W - 1) * C,
               sizeof(double) * (W - 1) * C);
    }
    return refused;
}
