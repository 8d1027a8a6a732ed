/*
 * gdn_oracle.h -- fp64 CPU oracle for the Gated DeltaNet verify path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline / reference arm may load this library.  The CUDA library never
 * includes, links or calls it, and it shares no header, helper or constant
 * with the CUDA library.
 *
 * What it computes, in the notation of the gated delta rule (Yang, Kautz &
 * Hatamizadeh, "Gated Delta Networks: Improving Mamba2 with Delta Rule",
 * ICLR 2025), for one slot and one value head h whose key head is
 * kh = floor(h / (H_v / H_k)):
 *
 *   win  = concat(conv_state (W-1 rows), x_0 .. x_{T-1})          (time order)
 *   y_t  = SiLU( sum_{j<W} w[j] * win[t+j] )     per channel, tap W-1 = x_t
 *   q_t, k_t, v_t = channel slices of y_t; q^ = q/sqrt(|q|^2+eps), same for k
 *   g_t  = exp(-exp(A_log) * softplus(alpha_t + dt_bias)),  beta_t = sigmoid(beta_raw_t)
 *   S~   = g_t S;   u = S~^T k^;   S = S~ + beta_t k^ (v - u)^T;   o = q_scale * S^T q^
 *   cap[t] = S (state after token t)
 *   out_t = o / sqrt(mean(o^2) + eps_rms) * norm_w * SiLU(z_t)
 *   conv_state <- win[T .. T+W-2];  state <- S
 *
 * Storage conventions follow the lucebox-hub page "server/src/internal.h",
 * section "Target cache": the recurrent state of one layer is square per value
 * head, [S_v, S_v, H_v] f32; the conv state holds the last (kernel-1) raw
 * inputs of every conv channel; the verify capture holds one full state per
 * verify position ("element t ... holds the DeltaNet recurrent state after
 * processing verify token t") and the conv capture is the whole concatenated
 * window fed to the convolution.  The reading used here:
 *   qkv        [B][T][C]            C = 2*H_k*d_k + H_v*d_v, channels [q | k | v], head-major
 *   z          [B][T][H_v*d_v]
 *   alpha, beta_raw [B][T][H_v]
 *   conv_w     [W][C];  A_log, dt_bias [H_v];  norm_w [d_v] (shared by all value heads)
 *   state      [B][H_v][d_v][d_k]   element (j, i) is logical S[i][j], i in d_k, j in d_v
 *   conv_state [B][W-1][C]
 *   cap_state  [B][T][H_v][d_v][d_k]
 *   cap_conv   [B][W-1+T][C]
 *   out        [B][T][H_v*d_v]
 *
 * Rollback follows the hf2q page "qwen35_target.rs", rollback_kv: trim 0 is a
 * no-op; accepted_idx = n_tokens_max - 1 - trim; the state becomes
 * capture[accepted_idx]; and per the internal.h DeltaNetCapture comment the
 * conv state becomes window rows [commit_n .. commit_n + W - 2] with
 * commit_n = accepted_idx + 1.  A trim >= T is refused and leaves the slot
 * untouched (the page skips it).
 *
 * Parity pins: see tests/test_oracle_pins.py.  No function here is unpinned.
 */
#ifndef GDN_ORACLE_H
#define GDN_ORACLE_H

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int n_slots, n_qk_heads, n_v_heads, d_k, d_v, conv_width, n_tokens;
    double rms_eps, l2_eps, q_scale;
} gdno_dims;

/* ---- stages (each pinned on its own) ---------------------------------- */

/* Depthwise causal conv over a window win[W-1+T][C]; y[t][c] = SiLU(sum_j w[j][c] win[t+j][c]). */
void gdno_conv_silu(int W, int T, int C, const double *conv_w, const double *win, double *y);

/* xhat = x / sqrt(sum x^2 + eps). */
void gdno_l2norm(int n, const double *x, double eps, double *xhat);

/* softplus(x) = log(1 + exp(x)), returned as x for x > 30. */
double gdno_softplus(double x);

/* g = exp(-exp(A_log) * softplus(alpha + dt_bias)), beta = 1 / (1 + exp(-beta_raw)). */
void gdno_gates(double A_log, double dt_bias, double alpha, double beta_raw,
                double *g, double *beta);

/* One gated delta-rule step on S[d_k][d_v] (row-major, S[i*dv + j]) with the
 * gate values given directly; o (length dv) = q_scale * S_new^T q. */
void gdno_delta_step(int dk, int dv, double *S, const double *k, const double *v,
                     const double *q, double g, double beta, double q_scale, double *o);

/* out = o / sqrt(mean(o^2) + eps) * w * z * sigmoid(z), length dv. */
void gdno_rmsnorm_gate(int dv, const double *o, const double *z, const double *w,
                       double eps, double *out);

/* ---- composites --------------------------------------------------------- */

/* Verify forward over T tokens for all slots.  state/conv_state are updated in
 * place.  cap_state / cap_conv may be NULL (no capture).  head_mask (length
 * H_v, may be NULL = all) restricts which value heads are computed: state,
 * captures and outputs of masked-out heads are left untouched, and the conv
 * state / window are still written for every channel.  n_threads >= 1 workers
 * over (slot, head) pairs.  Returns 0, or -1 on bad dims. */
int gdno_verify(const gdno_dims *d, const double *conv_w, const double *A_log,
                const double *dt_bias, const double *norm_w,
                const double *qkv, const double *z, const double *alpha, const double *beta_raw,
                double *state, double *conv_state, double *cap_state, double *cap_conv,
                double *out, const unsigned char *head_mask, int n_threads);

/* Rollback per slot.  slot_status[s] = 0 applied / no-op, 1 = trim out of
 * range (slot untouched).  Returns the number of refused slots. */
int gdno_rollback(const gdno_dims *d, const int *trim, double *state, double *conv_state,
                  const double *cap_state, const double *cap_conv, int *slot_status);

/* The chunkwise (WY / UT-transform) form of the same recurrence over
 * d->n_tokens tokens, chunk length `chunk` (last chunk may be partial), no
 * capture.  A second, independent implementation used to pin the sequential
 * one; same arguments as gdno_verify minus the captures. */
int gdno_prefill_chunked(const gdno_dims *d, int chunk, const double *conv_w,
                         const double *A_log, const double *dt_bias, const double *norm_w,
                         const double *qkv, const double *z, const double *alpha,
                         const double *beta_raw, double *state, double *conv_state,
                         double *out, const unsigned char *head_mask, int n_threads);

/* Tree (DDTree) verify.  parent[s][t] in [-1, t-1] is the parent of token t
 * (-1: the state before the batch).  Token t runs from its parent's state, and
 * its conv window is the raw input of its W-1 nearest ancestors and itself,
 * the ancestors continuing into the old conv state rows past the root.
 * state / conv_state are read only.  cap_state[s][t] = state after t;
 * cap_conv[s][t] = the conv state after t (W-1 rows: its W-2 nearest ancestors
 * and t, oldest first).  Returns 0, -1 on bad dims / missing captures, -2 when
 * parent is not a tree in token order. */
int gdno_verify_tree(const gdno_dims *d, const int *parent, const double *conv_w, const double *A_log,
                     const double *dt_bias, const double *norm_w,
                     const double *qkv, const double *z, const double *alpha, const double *beta_raw,
                     const double *state, const double *conv_state, double *cap_state, double *cap_conv,
                     double *out, const unsigned char *head_mask, int n_threads);

/* Rollback after a tree verify: accept[s] = the accepted node (-1 = none, the
 * slot keeps its state); state and conv state are copied from its captures.
 * slot_status[s] = 1 for an index out of range (slot untouched).  Returns the
 * number of refused slots. */
int gdno_rollback_tree(const gdno_dims *d, const int *accept, double *state, double *conv_state,
                       const double *cap_state, const double *cap_conv, int *slot_status);

#ifdef __cplusplus
}
#endif
#endif
