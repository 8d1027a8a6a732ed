/*
 * gdn_verify.h -- C ABI of the GB300 (sm_103a) Gated DeltaNet verify library.
 *
 * The library runs the Gated DeltaNet linear-attention block of a hybrid
 * (full-attention + GDN) model over a speculative-decode verify batch of T =
 * K+1 tokens, captures the recurrent and conv state after every position, and
 * rolls a slot back to the state after its last accepted token.  It also runs
 * a chunkwise prefill of the same block over a long prompt.
 *
 * Math (gated delta rule; Yang, Kautz & Hatamizadeh, "Gated Delta Networks",
 * ICLR 2025), per slot and value head h with key head kh = h / (H_v / H_k):
 *   window  = concat(conv_state, qkv tokens); y_t = SiLU(sum_j conv_w[j] * window[t+j])
 *   q^, k^  = L2-normalised (eps l2_eps) key-head slices of y_t; v = value-head slice
 *   g_t     = exp(-exp(A_log[h]) * softplus(alpha_t + dt_bias[h])), beta_t = sigmoid(beta_raw_t)
 *   S_t     = g_t S_{t-1} + beta_t k^ (v - (g_t S_{t-1})^T k^)^T,   o_t = q_scale * S_t^T q^
 *   out_t   = o_t / sqrt(mean(o_t^2) + rms_eps) * norm_w * SiLU(z_t)
 *
 * Structure and storage follow the lucebox-hub page server/src/internal.h:
 * "Target cache" (GDN recurrent state [S_v,S_v,H_v] f32 and conv state
 * [(kernel-1), conv_channels] f32 per layer, persistent and pre-allocated),
 * the per-step capture buffers ssm_intermediate / conv_input_cache (state
 * after verify token t; the concatenated conv window), TargetWeights GDN dims
 * (ssm_d_conv 4, rms_eps 1e-6), and TargetLayer's GDN tensors (fused wqkv
 * stream, z gate, ssm_conv1d [kernel,dim], per-head A and dt bias, ssm_norm
 * [head_v_dim]).  Rollback follows the hf2q page qwen35_target.rs,
 * DFlashTarget::rollback_kv (trim 0 is a no-op; accepted_idx = n_tokens_max
 * - 1 - trim; per-slot isolation).
 *
 * Conventions
 *  - Every buffer is caller-owned device memory (except the dims / params
 *    structs, which are host memory read during the call).  The library never
 *    allocates, frees or synchronises; work is enqueued on `stream` (a
 *    cudaStream_t passed as void*; NULL = the legacy default stream) and the
 *    call returns as soon as it is enqueued.  Calls may be captured into a
 *    CUDA graph.
 *  - Every device pointer must be 16-byte aligned (GDN_ERR_ALIGN otherwise).
 *  - A non-OK return means nothing was enqueued; gdn_last_error() (per
 *    thread) then describes the problem.  Problems only the device can see
 *    are written to *d_status (a device int the caller zeroes; may be NULL):
 *    the first error code wins.  No kernel traps, asserts or waits unbounded.
 *
 * Layouts (row-major, last index fastest; B = n_slots, T = n_tokens,
 * C = 2*H_k*d_k + H_v*d_v conv channels ordered [q | k | v], head-major):
 *   qkv        [B][T][C]            act_dtype   (projected, pre-conv)
 *   z          [B][T][H_v*d_v]      act_dtype
 *   alpha      [B][T][H_v]          act_dtype
 *   beta_raw   [B][T][H_v]          act_dtype
 *   out        [B][T][H_v*d_v]      act_dtype
 *   conv_w     [W][C] f32, A_log [H_v] f32, dt_bias [H_v] f32, norm_w [d_v] f32
 *   state      [B][H_v][d_v][d_k] f32   (element (j,i) = S[i][j]; d_k contiguous)
 *   conv_state [B][W-1][C] f32          (last W-1 raw qkv inputs per channel)
 *   cap_state  [B][T][H_v][d_v][d_k] f32   (state after token t)
 *   cap_conv   [B][W-1+T][C] f32        (concat(conv_state, qkv) window)
 */
#ifndef GDN_VERIFY_H
#define GDN_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GDN_OK = 0,
    GDN_ERR_ARG = 1,         /* a required pointer is NULL or an enum is invalid */
    GDN_ERR_SHAPE = 2,       /* dims outside what the kernels support (see each call) */
    GDN_ERR_ALIGN = 3,       /* a device pointer is not 16-byte aligned */
    GDN_ERR_DTYPE = 4,       /* act_dtype not supported for this call */
    GDN_ERR_TRIM_RANGE = 5,  /* (device) a slot's trim is outside [0, T-1]; slot left untouched */
    GDN_ERR_NO_CAPTURE = 6,  /* rollback asked without capture buffers */
    GDN_ERR_LAUNCH = 7,      /* the CUDA launch itself failed (message in gdn_last_error) */
    GDN_ERR_TIMEOUT = 8,     /* (device) a bounded wait gave up */
    GDN_ERR_WORKSPACE = 9,   /* workspace missing or smaller than the query returned */
    GDN_ERR_TREE = 10,       /* (device) a parent id is outside [-1, t-1]; that token ran from the root */
    GDN_ERR_BOUNDS = 11      /* (device, checked builds only) an access fell outside its buffer and was skipped */
} gdn_status;

typedef enum { GDN_F32 = 0, GDN_BF16 = 1 } gdn_dtype;

typedef struct {
    int n_slots;       /* B >= 1: independent sequences ("slots"), each with its own state */
    int n_qk_heads;    /* H_k >= 1 */
    int n_v_heads;     /* H_v, a multiple of H_k; value head h reads key head h / (H_v/H_k) */
    int d_k;           /* key head dim: 32, 64 or 128 */
    int d_v;           /* value head dim: a multiple of 8, 8..256 */
    int conv_width;    /* W: must be 4 (ssm_d_conv) */
    int n_tokens;      /* T: verify positions (K+1), or prompt length for prefill */
    gdn_dtype act_dtype;
    float rms_eps;     /* gated RMSNorm epsilon (1e-6) */
    float l2_eps;      /* q/k L2-norm epsilon (1e-6) */
    float q_scale;     /* read-out scale on q (1.0 = none; 1/sqrt(d_k) is common) */
} gdn_dims;

typedef struct {
    const float *conv_w;   /* [W][C] depthwise conv weights, tap W-1 meets the current token */
    const float *A_log;    /* [H_v] log of the decay rate magnitude */
    const float *dt_bias;  /* [H_v] bias added to alpha before softplus */
    const float *norm_w;   /* [d_v] RMSNorm weight shared by all value heads */
} gdn_layer_params;

/*
 * Verify forward over T positions.  Reads qkv/z/alpha/beta_raw and the layer
 * params; updates state and conv_state IN PLACE to "after all T tokens";
 * writes out.  If cap_state is non-NULL it receives, for every position t,
 * the state after token t (internal.h, "Target cache", the ssm_intermediate
 * comment: entry t of that per-layer buffer is the recurrent state once the
 * verify has run token t), so
 * cap_state[:, T-1] equals the new state bit for bit.  If cap_conv is non-NULL
 * it receives the concat(old conv_state, qkv) window (internal.h,
 * conv_input_cache).  Supported: 1 <= T <= 64, d_k in {32,64,128}, d_v % 8 ==
 * 0 and d_v <= 256, (H_v/H_k) * ceil(d_v / 64) <= 16 (the value heads of a key
 * head share one thread-block cluster, a CTA holding at most 64 value rows;
 * GDN_ERR_SHAPE otherwise), W == 4, act_dtype f32 or bf16.
 * d_status may be NULL (the verify kernel reports nothing through it).
 */
int gdn_verify_forward(const gdn_dims *dims, const gdn_layer_params *params,
                       const void *qkv, const void *z, const void *alpha, const void *beta_raw,
                       float *state, float *conv_state, float *cap_state, float *cap_conv,
                       void *out, int *d_status, void *stream);

/*
 * Rollback after a verify of T = dims->n_tokens positions (hf2q qwen35_target.rs,
 * rollback_kv).  d_trim is a DEVICE int32[B] (so the call can sit in a CUDA
 * graph).  Per slot s: trim 0 = no-op (no bytes moved); 1 <= trim <= T-1:
 * accepted_idx = T-1-trim, state[s] = cap_state[s][accepted_idx] and
 * conv_state[s] = cap_conv[s][accepted_idx+1 .. accepted_idx+W-1] (the window
 * rows [commit_n .. commit_n+kernel-2] of internal.h with commit_n =
 * accepted_idx+1); any other trim leaves the slot untouched and writes
 * GDN_ERR_TRIM_RANGE to *d_status.  Slots are independent.  cap_state or
 * cap_conv NULL -> GDN_ERR_NO_CAPTURE (the page skips silently; this ABI
 * reports).  Only state/conv_state of the rolled-back slots change.
 */
int gdn_rollback(const gdn_dims *dims, const int32_t *d_trim, float *state, float *conv_state,
                 const float *cap_state, const float *cap_conv, int *d_status, void *stream);

/*
 * gdn_rollback of n_layers layers in one launch, with the same trims: the
 * target cache keeps one DeltaNetCapture per DeltaNet layer (internal.h,
 * Target cache, create_target_cache), and a serving step rolls every layer
 * back once the verify of the whole pass has decided how many tokens each
 * slot accepted (hf2q qwen35_target.rs, rollback_kv).  d_state,
 * d_conv_state, d_cap_state and d_cap_conv are DEVICE arrays of n_layers
 * pointers (8-byte aligned), entry l being layer l's buffer as gdn_rollback
 * takes it (same dims for every layer); the tables are read on the device, so
 * the call can sit in a CUDA graph.  Per layer and slot exactly gdn_rollback
 * (bit-identical); a table entry that is NULL or not 16-byte aligned skips
 * that layer and writes GDN_ERR_ARG to *d_status.  The caller owns the tables.
 */
int gdn_rollback_layers(const gdn_dims *dims, int n_layers, const int32_t *d_trim, float *const *d_state,
                        float *const *d_conv_state, const float *const *d_cap_state, const float *const *d_cap_conv,
                        int *d_status, void *stream);

/*
 * Tree (DDTree) verify: the T = dims->n_tokens tokens of each slot form a
 * draft tree in token order (internal.h, Target forward graph:
 * QwenGraphInputs::parent_ids, "tree mode when non-null"; the capture is sized
 * for the tree: create_target_cache, max_verify_tokens).  d_parent is a DEVICE
 * int32[B][T]; parent t' of token t is in [-1, t-1], -1 meaning the state
 * before the batch.  Token t runs from its parent's state, and its conv window
 * is the raw input of t and of its three nearest ancestors, continuing into
 * the old conv-state rows past the root; along any root-to-node path this is
 * the chain verify of that path's tokens.  state and conv_state are only read
 * (a tree has no single "after all tokens" state): gdn_rollback_tree moves a
 * slot to its accepted node.  cap_state [B][T][H_v][d_v][d_k] receives the
 * state after every node; cap_conv [B][T][W-1][C] the conv state after every
 * node (its two nearest ancestors' raw inputs and its own, oldest first); both
 * are required (GDN_ERR_NO_CAPTURE).  out as gdn_verify_forward.  A parent id
 * out of range writes GDN_ERR_TREE to *d_status and that token runs from the
 * root.  Same shapes as gdn_verify_forward.
 */
int gdn_verify_tree(const gdn_dims *dims, const gdn_layer_params *params,
                    const void *qkv, const void *z, const void *alpha, const void *beta_raw,
                    const int32_t *d_parent, const float *state, const float *conv_state,
                    float *cap_state, float *cap_conv, void *out, int *d_status, void *stream);

/*
 * Rollback after a tree verify: d_accept is a DEVICE int32[B], the accepted
 * node of each slot (-1: nothing accepted, no-op).  state[s] = cap_state[s][a]
 * and conv_state[s] = cap_conv[s][a] (the gdn_verify_tree layouts); an index
 * outside [-1, T-1] leaves the slot untouched and writes GDN_ERR_TRIM_RANGE to
 * *d_status.  Same launch and error behaviour as gdn_rollback.
 */
int gdn_rollback_tree(const gdn_dims *dims, const int32_t *d_accept, float *state, float *conv_state,
                      const float *cap_state, const float *cap_conv, int *d_status, void *stream);

/*
 * gdn_rollback_tree of n_layers layers in one launch, with the same accepted
 * nodes: the tables as for gdn_rollback_layers (each layer's cap_conv holding
 * its per-node conv states, as gdn_verify_tree writes them).  Per layer and
 * slot exactly gdn_rollback_tree (bit-identical); a bad table entry skips that
 * layer and writes GDN_ERR_ARG to *d_status.
 */
int gdn_rollback_tree_layers(const gdn_dims *dims, int n_layers, const int32_t *d_accept, float *const *d_state,
                             float *const *d_conv_state, const float *const *d_cap_state,
                             const float *const *d_cap_conv, int *d_status, void *stream);

/*
 * gdn_verify_after_rollback: a verify step with the previous step's rollback
 * folded in (one launch per step instead of a verify and a rollback).
 * cap_state / cap_conv hold the previous gdn_verify_forward (or
 * gdn_verify_after_rollback) of the same dims, not yet rolled back; d_prev_trim
 * is a DEVICE int32[B] with gdn_rollback's meaning.  Per slot the batch starts
 * from exactly what gdn_rollback(d_prev_trim) would leave -- the captured
 * state cap_state[s][T-1-trim] and the window rows after that token -- and
 * state / conv_state are not read.  Everything else is gdn_verify_forward:
 * outputs, the new captures (overwriting the old ones), state and conv_state
 * after all T tokens, bit-identical to gdn_rollback followed by
 * gdn_verify_forward.  A trim outside [0, T-1] leaves the slot untouched (no
 * outputs) and writes GDN_ERR_TRIM_RANGE to *d_status.  Without capture
 * buffers: GDN_ERR_NO_CAPTURE.
 */
int gdn_verify_after_rollback(const gdn_dims *dims, const gdn_layer_params *params, const int32_t *d_prev_trim,
                              const void *qkv, const void *z, const void *alpha, const void *beta_raw,
                              float *state, float *conv_state, float *cap_state, float *cap_conv,
                              void *out, int *d_status, void *stream);

/*
 * Lazy capture: the byte-saving alternative to per-position capture.  Instead
 * of writing the state after every token and copying one back, a lazy verify
 * writes only its outputs and leaves the batch "pending": state and
 * conv_state keep the state before it.  Once the acceptance is known, the
 * pending batch is committed by re-running its accepted tokens from that
 * state -- inside the next lazy verify (one launch per step), or by
 * gdn_commit_lazy.  The single-snapshot rollback of the lucebox-hub page
 * (internal.h, "Target cache" and its snapshot tensors) keeps the same one
 * state per slot; the re-run rests on the prefix property of the recurrence
 * (the state after token t depends only on tokens 0..t).
 *
 * gdn_verify_lazy: d_prev_trim == NULL: no batch is pending; as
 * gdn_verify_forward with no capture, except that state and conv_state are
 * only read.  d_prev_trim != NULL: a DEVICE int32[B], the trims of the pending
 * batch whose qkv, alpha and beta_raw are prev_qkv / prev_alpha /
 * prev_beta_raw (same dims and layouts as the new batch; z is not needed).
 * Per slot the launch first runs the pending batch's tokens 0..T-1-trim from
 * state / conv_state and writes the state and conv state after them in place
 * (what gdn_commit_lazy would write), then runs the new batch from there and
 * writes its outputs; the new batch is then the pending one.  Outputs and
 * committed states are bit-identical to gdn_verify_forward with capture +
 * gdn_rollback.  A pending trim outside [0, T-1] leaves the slot untouched
 * (no outputs either) and writes GDN_ERR_TRIM_RANGE to *d_status.  With a
 * pending batch the shared memory holds 2T tokens, so T is limited by the
 * device's shared memory (GDN_ERR_SHAPE).
 */
int gdn_verify_lazy(const gdn_dims *dims, const gdn_layer_params *params,
                    const int32_t *d_prev_trim, const void *prev_qkv, const void *prev_alpha,
                    const void *prev_beta_raw,
                    const void *qkv, const void *z, const void *alpha, const void *beta_raw,
                    float *state, float *conv_state, void *out, int *d_status, void *stream);

/*
 * gdn_commit_lazy: commits a pending batch on its own (e.g. at the end of a
 * generation).  d_trim is a DEVICE int32[B] with gdn_rollback's meaning (trim
 * in 0..T-1; the slot keeps tokens 0..T-1-trim).  For every slot it runs those
 * T - trim tokens of the batch's qkv, alpha and beta_raw (z and the outputs
 * are not needed) from state / conv_state -- which must still hold the state
 * before the batch -- and writes the state and conv state after them in
 * place.  Bit-identical to gdn_verify_forward with capture followed by
 * gdn_rollback with the same trims.  A trim outside [0, T-1] leaves the slot
 * untouched and writes GDN_ERR_TRIM_RANGE to *d_status.  Same shapes and
 * limits as gdn_verify_forward.
 */
int gdn_commit_lazy(const gdn_dims *dims, const gdn_layer_params *params, const int32_t *d_trim,
                    const void *qkv, const void *alpha, const void *beta_raw,
                    float *state, float *conv_state, int *d_status, void *stream);

/*
 * The projections either side of the block, as bf16 GEMMs with fp32
 * accumulation (this library's own tensor-core kernel: the weight rows
 * stream through shared memory while the B*T activation rows stay resident),
 * and the layer step that chains them around the verify.  They follow the GDN tensors of internal.h, Target weights
 * (TargetLayer: wqkv, the fused Q/K/V projection; wqkv_gate, the z
 * projection; ssm_alpha and ssm_beta, the per-token gate inputs; ssm_out, the
 * output projection), each weight stored as its output rows with n_embd
 * contiguous (the K-major "TN" layout of the tensor cores):
 *   w_in  [C + H_v*d_v + 2*H_v][n_embd] bf16: the wqkv rows (C, channels
 *         [q | k | v] as in qkv), then the wqkv_gate rows (H_v*d_v), then
 *         ssm_alpha (H_v), then ssm_beta (H_v) -- the four input projections
 *         fused so that one GEMM streams them all;
 *   w_out [n_embd][H_v*d_v] bf16 (ssm_out).
 * x and y are [B][T][n_embd] bf16.  The norm before the block, the residual
 * add after it and the rest of the model are not part of this library.
 * Limits: act_dtype GDN_BF16, n_embd a multiple of 8, n_v_heads a multiple of
 * 8 (GDN_ERR_DTYPE / GDN_ERR_SHAPE).
 */
typedef struct {
    int n_embd;            /* hidden size */
    const void *w_in;      /* [C + H_v*d_v + 2*H_v][n_embd] bf16 */
    const void *w_out;     /* [n_embd][H_v*d_v] bf16 */
} gdn_proj_weights;

/* Row stride (elements) of gdn_project_in's output: C + H_v*d_v + 2*H_v rounded up to 8. */
long long gdn_proj_in_ld(const gdn_dims *dims);

/* Device workspace of gdn_layer_verify: the activation matrix and the block's
 * output (0 on bad arguments).  The GEMMs themselves need no scratch. */
size_t gdn_layer_workspace_bytes(const gdn_dims *dims, int n_embd);

/* act[B*T][gdn_proj_in_ld] = x @ w_in^T: columns [0, C) are qkv, then z, then
 * alpha, then beta_raw, per row (bf16).  workspace / ws_bytes are not used (the
 * GEMM needs no scratch; pass NULL, 0). */
int gdn_project_in(const gdn_dims *dims, const gdn_proj_weights *w, const void *x, void *act,
                   void *workspace, size_t ws_bytes, void *stream);

/* y[B*T][n_embd] = out @ w_out^T (bf16).  workspace / ws_bytes are not used. */
int gdn_project_out(const gdn_dims *dims, const gdn_proj_weights *w, const void *out, void *y,
                    void *workspace, size_t ws_bytes, void *stream);

/*
 * One GDN layer of a verify step: gdn_project_in into the workspace, the
 * verify of gdn_verify_forward reading qkv, z, alpha and beta_raw as column
 * blocks of that matrix (state, conv_state and the optional captures as
 * there), its output into the workspace, then gdn_project_out into y.  Roll
 * back with gdn_rollback as usual.  workspace: gdn_layer_workspace_bytes,
 * 256-byte aligned; the activation matrix sits at its start (row stride
 * gdn_proj_in_ld) and the block's output [B*T][H_v*d_v] right after it (at
 * the next 256-byte boundary).  While it runs, the verify also brings
 * w_out into L2 (bulk prefetches; nothing is written) for the output GEMM.
 */
int gdn_layer_verify(const gdn_dims *dims, const gdn_layer_params *params, const gdn_proj_weights *w,
                     const void *x, float *state, float *conv_state, float *cap_state, float *cap_conv,
                     void *y, void *workspace, size_t ws_bytes, int *d_status, void *stream);

/*
 * One verify step from host memory: the inputs of the step arrive as one
 * packed host block, the outputs leave as one host block, and everything in
 * between is enqueued on `stream` by this one call (the caller synchronises
 * the stream when it needs h_out).  The packed input block holds qkv, z,
 * alpha, beta_raw (the layouts above, act_dtype) and the int32 trims [B], each
 * section starting at the offset gdn_step_io_layout gives (256-byte aligned);
 * the output block is out.  d_io is caller-owned device staging of
 * in_bytes + out_bytes (256-byte aligned).  rollback_first = 0: verify with
 * capture, then gdn_rollback with the staged trims (the trims of this batch);
 * rollback_first = 1: gdn_verify_after_rollback (the trims of the previous
 * batch, whose captures cap_state / cap_conv still hold).  h_in and h_out
 * should be pinned for the copies to be asynchronous.  Errors as the calls it
 * makes; a copy that cannot be enqueued is GDN_ERR_LAUNCH.
 */
typedef struct {
    size_t qkv, z, alpha, beta_raw, trim;   /* byte offsets in the packed input block */
    size_t in_bytes, out_bytes;             /* sizes of the input and output blocks */
} gdn_step_io;

int gdn_step_io_layout(const gdn_dims *dims, gdn_step_io *io);

int gdn_verify_step_host(const gdn_dims *dims, const gdn_layer_params *params, int rollback_first,
                         const void *h_in, void *h_out, void *d_io, size_t d_io_bytes,
                         float *state, float *conv_state, float *cap_state, float *cap_conv,
                         int *d_status, void *stream);

/*
 * Bytes of device workspace gdn_prefill_chunked needs for these dims (0 on bad
 * dims).  internal.h, "Target cache", create_target_cache: a cache made with
 * prefill_only holds only the persistent recurrent and conv state (the
 * rollback tensors -- snapshots, per-step intermediates -- are skipped), and
 * migrate_prefill_cache later promotes it to a full decode cache.  The
 * prefill therefore runs over exactly the state / conv_state buffers that
 * gdn_verify_forward and gdn_rollback use; the workspace sized here is
 * transient scratch of the chunkwise form (operand rings, flags, a work
 * counter), which has no counterpart on the pages: the caller owns it, as the
 * page's caller owns the cache.
 */
size_t gdn_prefill_workspace_bytes(const gdn_dims *dims);

/*
 * Chunkwise prefill of a prompt of L = dims->n_tokens tokens per slot (any
 * L >= 1; chunks of 64, the last one may be partial).  Same inputs/outputs as
 * gdn_verify_forward with T = L, no capture (a prefill-only cache skips the
 * rollback tensors: internal.h, create_target_cache, prefill_only).  Updates
 * state and conv_state in place.  workspace: caller-owned device scratch of
 * at least gdn_prefill_workspace_bytes(dims) bytes, 256-byte aligned (1 MiB
 * per (slot, value head): a ring of operand slots, plus its flags and a work
 * counter per launch); its contents need no initialisation and are garbage
 * afterwards.  The call enqueues, on `stream`, a memset of the ring
 * flags, one cooperative launch per group of slots that fits on the device
 * at once, and a small kernel that advances conv_state; calls sharing a
 * workspace must be ordered.  Supported:
 * d_k == d_v == 128, W == 4, act_dtype bf16 or f32.
 */
int gdn_prefill_chunked(const gdn_dims *dims, const gdn_layer_params *params,
                        const void *qkv, const void *z, const void *alpha, const void *beta_raw,
                        float *state, float *conv_state, void *out,
                        void *workspace, size_t ws_bytes, int *d_status, void *stream);

/*
 * gdn_prefill_chunked without a caller workspace: the same computation, with
 * its scratch taken from a fixed array inside this library.  The method itself
 * has no such call; it exists for callers that cannot allocate device memory
 * at the point where they prefill -- a host program that only holds the
 * buffers it was handed, or a server running under a fixed device-memory
 * budget whose allocator must not grow -- and so have no workspace to pass.
 *
 * Limit: the call needs gdn_prefill_workspace_bytes(dims) bytes of scratch and
 * the built-in array holds GDN_PREFILL_STATIC_SCRATCH_BYTES (16 MiB; also
 * returned by gdn_prefill_static_scratch_bytes); larger dims are rejected with
 * GDN_ERR_WORKSPACE before anything is enqueued.  The scratch needs no
 * initialisation.  The array is reserved on a device when this library's
 * device code is loaded into a context there: under CUDA's default lazy
 * module loading that is the first call into the library that runs its
 * device code on the device; with CUDA_MODULE_LOADING=EAGER it is when the
 * context is created.  Each context holds its own copy until it is destroyed
 * (and the bounds-checked build of the library holds another).
 *
 * The first call in a context (normally: the first call on a device, with
 * that device current) looks the array's device address up and caches it
 * under the context's id, so make that first call before any stream capture
 * on the device.  After cudaDeviceReset, or in another context, the address
 * is looked up again.  Calls that overlap on one device -- different
 * streams, or host threads, with no ordering between them -- share the one
 * array and race: order them (one stream, or events).  Everything else,
 * including the error codes, is as for gdn_prefill_chunked.
 */
#define GDN_PREFILL_STATIC_SCRATCH_BYTES ((size_t)16 << 20)
/* The size of that built-in array (GDN_PREFILL_STATIC_SCRATCH_BYTES), for
 * bindings that cannot read the macro. */
size_t gdn_prefill_static_scratch_bytes(void);
int gdn_prefill_chunked_static(const gdn_dims *dims, const gdn_layer_params *params,
                               const void *qkv, const void *z, const void *alpha, const void *beta_raw,
                               float *state, float *conv_state, void *out, int *d_status, void *stream);

/*
 * Message for the last non-OK return on this thread ("" if none).  internal.h,
 * top of the file: one error channel for the whole library, into which every
 * loader and graph builder writes through set_last_error(...), and whose
 * builders "return false and set last_error on failure" ("Target forward
 * graph").  Here every call returns a gdn_status and, when it is not GDN_OK,
 * leaves the reason in this per-thread string (valid until the thread's next
 * call into the library).
 */
const char *gdn_last_error(void);

/* Library version string. */
const char *gdn_version(void);

#ifdef __cplusplus
}
#endif
#endif /* GDN_VERIFY_H */
