// internal.cuh -- argument blocks shared by the C-ABI layer and the kernels.
// Not part of the public interface (that is include/gdn_verify.h).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>
#include <mutex>
#include <string>

#include "gdn_verify.h"
#include "check.cuh"

namespace gdn {

// Verify kernel modes: the chain, a draft tree, lazy (outputs only), the
// lazy commit (re-run of each slot's accepted tokens), and the chain started
// from the previous batch's captures (its rollback folded in).
enum VerifyMode { kChain = 0, kTree = 1, kLazy = 2, kCommit = 3, kRolled = 4 };

// Everything one verify launch needs, validated on the host.
struct VerifyArgs {
    CUtensorMap qk_map;               // the q|k|v channels as a 2-D tensor [B*Ts rows][C], box d_k x T tokens
    CUtensorMap v_map;                // the same tensor, box (d_v / P) x T: a CTA's value rows
    CUtensorMap z_map;                // z as [B*Ts rows][H_v*d_v], box (d_v / P) x T (not used by a commit)
    int B, Hk, Hv, dk, dv, T, C, r;   // C: conv channels; r = Hv / Hk
    int Ts;                           // tokens per slot in the activation buffers (>= T)
    int Tm;                           // tokens the shared memory holds (T; 2T for a lazy verify with a pending batch)
    long long ld_qkv, ld_z, ld_ab;    // row strides (elements) of qkv, z and alpha / beta_raw (C, H_v*d_v, H_v
                                      // when separate; one shared stride when they are column blocks of one matrix)
    int P;                            // CTAs per value head (each owns d_v / P rows)
    float rms_eps, l2_eps, q_scale;
    const float *conv_w, *A_log, *dt_bias, *norm_w;
    const void *qkv, *z, *alpha, *beta_raw;
    float *state, *conv_state, *cap_state, *cap_conv;
    void *out;
    int *d_status;                    // device status word (may be NULL)
    const int32_t *parent;            // tree verify: [B][T] parent of each token
    const int32_t *trim;              // [B] trims, 0 .. T-1: lazy commit, a lazy verify's pending batch, or the
                                      // previous batch's rollback folded into a verify
    const void *qkv_prev, *alpha_prev, *beta_prev;   // lazy verify: the pending batch (same layouts)
    int mode;                         // VerifyMode
    // optional: a region the next kernel in the stream streams (the layer call's output-projection
    // weights), brought into L2 by bulk prefetches once each CTA's own loads have landed (NULL: none)
    const void *l2_next;
    size_t l2_next_bytes;
    // buffer extents in bytes, for the bounds checks of a checked build
    size_t ext_qkv, ext_z, ext_ab, ext_state, ext_conv_state, ext_cap_state, ext_cap_conv, ext_out;
    size_t ext_conv_w, ext_head, ext_norm_w, ext_parent, ext_trim;
};

struct RollbackArgs {
    int B, T, W1;                 // W1 = conv_width - 1
    long long state_elems;        // floats per slot state (H_v * d_v * d_k)
    long long conv_elems;         // floats per slot conv state (W1 * C)
    long long C;
    const int32_t *trim;              // per slot: trim (chain) or the accepted node (tree)
    float *state, *conv_state;
    const float *cap_state, *cap_conv;
    int *d_status;
    int tree;                         // 1: cap_conv holds per-node conv states [B][T][W-1][C]
    size_t ext_state, ext_conv_state, ext_cap_state, ext_cap_conv;   // bytes, for a checked build
    // several layers in one launch (grid z = layer): device tables of n_layers pointers replace the four
    // buffers above (NULL tables: one layer, the buffers above)
    int n_layers;
    float *const *tab_state;
    float *const *tab_conv_state;
    const float *const *tab_cap_state;
    const float *const *tab_cap_conv;
};

// Everything one chunkwise prefill launch needs (d_k = d_v = 128, W = 4).
struct PrefillArgs {
    CUtensorMap qkv_map;              // qkv as a 2-D tensor [B*L rows][C channels], box 128 x 67
    CUtensorMap z_map;                // z as a 2-D tensor [B*L rows][H_v*d_v], box 128 x 64
    int B, Hk, Hv, L, C, r;           // L: prompt tokens per slot; C: conv channels; r = Hv / Hk
    int slot0, ns;                    // slots of this launch: slot0 .. slot0 + ns - 1
    int n_prep;                       // preparation CTAs of this launch
    int *counter;                     // work counter of this launch (zeroed before the launch)
    int drop_chunk;                   // fault injection: this chunk is never published (-1: none)
    float rms_eps, l2_eps, q_scale;
    const float *conv_w, *A_log, *dt_bias, *norm_w;
    const void *qkv, *z, *alpha, *beta_raw;
    float *state, *conv_state;
    void *out;
    float *scratch;                   // the caller's workspace (ring flags first), prefill_workspace_bytes
    size_t ring_offset;               // bytes from the workspace start to the ring slots
    int *d_status;
};

// Returns a cudaError_t of the launch (cudaSuccess when enqueued).
cudaError_t launch_verify(const VerifyArgs &a, gdn_dtype act, int sm_count, cudaStream_t stream);
cudaError_t launch_rollback(const RollbackArgs &a, cudaStream_t stream);

// Prefill: shape check (GDN_OK or a status, reason in why), workspace size,
// and the launch.
int prefill_check(const gdn_dims &d, std::string &why);
size_t prefill_workspace_bytes(const gdn_dims &d);
cudaError_t launch_prefill(const gdn_dims &d, const gdn_layer_params &p, const void *qkv, const void *z,
                           const void *alpha, const void *beta_raw, float *state, float *conv_state,
                           void *out, void *workspace, int *d_status, cudaStream_t stream);

// Row-major C[M][N] (row stride ldc) = X[M][K] @ W[N][K]^T, bf16 in and out,
// fp32 accumulation (proj.cu; no scratch).  d_status (may be NULL) receives
// GDN_ERR_TIMEOUT if a bounded wait gave up.  false with the reason in why.
bool gemm_xwt_bf16(const void *W, const void *X, void *C, int M, int N, int K, long long ldc, int *d_status,
                   cudaStream_t stream, std::string &why);

// cuTensorMapEncodeTiled from the driver, looked up once (NULL if unavailable).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// Choice of CTAs per value head for a verify launch (host heuristic).
int verify_parts_per_head(int B, int Hv, int r, int dv, int sm_count);

// Identity of the CUDA context current on the calling thread (cuCtxGetId: unique for the life of the
// process).  Host-side caches of per-context facts -- function attributes, device-symbol addresses --
// are keyed on it, so that a device reset or another context on the same device never reads an entry
// made for a context that no longer exists.  false if no context is current (or the driver lacks the
// entry points).
bool current_context_id(unsigned long long *id);

// A small thread-safe map from context id to one cached value; the oldest entry gives way when full.
template <typename V, int N = 16>
class PerContext {
  public:
    bool get(unsigned long long id, V *v) {
        std::lock_guard<std::mutex> lock(mu_);
        for (int i = 0; i < N; ++i)
            if (used_[i] && ids_[i] == id) {
                *v = vals_[i];
                return true;
            }
        return false;
    }
    void put(unsigned long long id, const V &v) {
        std::lock_guard<std::mutex> lock(mu_);
        for (int i = 0; i < N; ++i)
            if (used_[i] && ids_[i] == id) {
                vals_[i] = v;
                return;
            }
        ids_[next_] = id;
        vals_[next_] = v;
        used_[next_] = true;
        next_ = (next_ + 1) % N;
    }

  private:
    std::mutex mu_;
    unsigned long long ids_[N] = {};
    V vals_[N] = {};
    bool used_[N] = {};
    int next_ = 0;
};

}  // namespace gdn
