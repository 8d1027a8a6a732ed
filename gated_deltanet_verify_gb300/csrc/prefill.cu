// prefill.cu -- prefill of a long prompt through the same GDN block.
//
// First correct path: the prompt is processed as consecutive 64-token
// segments by the fused verify kernel with capture disabled; state and conv
// state are carried in place from one segment to the next.  This is the
// sequential recurrence (bit-for-bit what verify computes), launched L/64
// times.  No workspace is needed.
#include "internal.cuh"

#include <string>

namespace gdn {
size_t verify_smem_bytes(int T, int dk, int dv, int P, int act_bytes);

namespace {
constexpr int kSegment = 64;
}

int prefill_check(const gdn_dims &d, std::string &why) {
    if (d.d_k != 32 && d.d_k != 64 && d.d_k != 128) {
        why = "prefill: d_k must be 32, 64 or 128";
        return GDN_ERR_SHAPE;
    }
    if (d.d_v % 8 || d.d_v > 256) {
        why = "prefill: d_v must be a multiple of 8 up to 256";
        return GDN_ERR_SHAPE;
    }
    if (d.n_slots > 65535) {
        why = "prefill: n_slots must be <= 65535";
        return GDN_ERR_SHAPE;
    }
    const int r = d.n_v_heads / d.n_qk_heads;
    if (verify_parts_per_head(d.n_slots, d.n_v_heads, r, d.d_v, 0) == 0) {
        why = "prefill: H_v/H_k too large for one thread-block cluster";
        return GDN_ERR_SHAPE;
    }
    return GDN_OK;
}

size_t prefill_workspace_bytes(const gdn_dims &d) {
    (void)d;
    return 0;
}

cudaError_t launch_prefill(const gdn_dims &d, const gdn_layer_params &p, const void *qkv, const void *z,
                           const void *alpha, const void *beta_raw, float *state, float *conv_state,
                           void *out, void *workspace, int *d_status, cudaStream_t stream) {
    (void)workspace;
    const int act_bytes = d.act_dtype == GDN_BF16 ? 2 : 4;
    const int r = d.n_v_heads / d.n_qk_heads;
    VerifyArgs a{};
    a.B = d.n_slots; a.Hk = d.n_qk_heads; a.Hv = d.n_v_heads; a.dk = d.d_k; a.dv = d.d_v;
    a.C = 2 * d.n_qk_heads * d.d_k + d.n_v_heads * d.d_v; a.r = r;
    a.P = verify_parts_per_head(d.n_slots, d.n_v_heads, r, d.d_v, 0);
    a.Ts = d.n_tokens;
    a.rms_eps = d.rms_eps; a.l2_eps = d.l2_eps; a.q_scale = d.q_scale;
    a.conv_w = p.conv_w; a.A_log = p.A_log; a.dt_bias = p.dt_bias; a.norm_w = p.norm_w;
    a.state = state; a.conv_state = conv_state; a.cap_state = nullptr; a.cap_conv = nullptr;
    a.d_status = d_status;
    const size_t Cb = size_t(a.C) * act_bytes, Zb = size_t(d.n_v_heads) * d.d_v * act_bytes,
                 Gb = size_t(d.n_v_heads) * act_bytes;
    for (int t0 = 0; t0 < d.n_tokens; t0 += kSegment) {
        a.T = (d.n_tokens - t0 < kSegment) ? d.n_tokens - t0 : kSegment;
        a.qkv = static_cast<const char *>(qkv) + t0 * Cb;
        a.z = static_cast<const char *>(z) + t0 * Zb;
        a.alpha = static_cast<const char *>(alpha) + t0 * Gb;
        a.beta_raw = static_cast<const char *>(beta_raw) + t0 * Gb;
        a.out = static_cast<char *>(out) + t0 * Zb;
        cudaError_t e = launch_verify(a, d.act_dtype, stream);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace gdn
