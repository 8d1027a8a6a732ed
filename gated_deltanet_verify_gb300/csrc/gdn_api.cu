// gdn_api.cu -- the C ABI declared in include/gdn_verify.h: argument
// validation, launch-shape choice and error reporting.  No allocation, no
// synchronisation: every call only enqueues work on the caller's stream.
#include "internal.cuh"

#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>
#include <string>

#include <cudaTypedefs.h>

namespace gdn {
size_t verify_smem_bytes(int Tm, int T, int dk, int dv, int P, int act_bytes, bool tree);
int verify_part_rows(int dv, int P);
}  // namespace gdn

namespace {

thread_local std::string g_err;

int fail(int code, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

struct DevInfo {
    int sms = 0, smem_optin = 0;
};

DevInfo dev_info() {
    int dev = 0;
    DevInfo d;
    if (cudaGetDevice(&dev) != cudaSuccess) return d;
    cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    return d;
}

// Basic shape checks common to every call.
int check_common(const gdn_dims *d) {
    if (!d) return fail(GDN_ERR_ARG, "dims is NULL");
    if (d->n_slots < 1 || d->n_qk_heads < 1 || d->n_v_heads < 1 || d->d_k < 1 || d->d_v < 1 ||
        d->n_tokens < 1)
        return fail(GDN_ERR_SHAPE, "dims must be positive (slots %d, H_k %d, H_v %d, d_k %d, d_v %d, T %d)",
                    d->n_slots, d->n_qk_heads, d->n_v_heads, d->d_k, d->d_v, d->n_tokens);
    if (d->n_v_heads % d->n_qk_heads != 0)
        return fail(GDN_ERR_SHAPE, "n_v_heads (%d) must be a multiple of n_qk_heads (%d)", d->n_v_heads,
                    d->n_qk_heads);
    if (d->conv_width != 4) return fail(GDN_ERR_SHAPE, "conv_width must be 4 (got %d)", d->conv_width);
    if (d->act_dtype != GDN_F32 && d->act_dtype != GDN_BF16)
        return fail(GDN_ERR_DTYPE, "act_dtype %d is neither GDN_F32 nor GDN_BF16", int(d->act_dtype));
    if (!(d->rms_eps >= 0.f) || !(d->l2_eps >= 0.f)) return fail(GDN_ERR_ARG, "eps must be >= 0");
    return GDN_OK;
}

long long conv_channels(const gdn_dims *d) {
    return 2LL * d->n_qk_heads * d->d_k + (long long)d->n_v_heads * d->d_v;
}

int check_params(const gdn_layer_params *p) {
    if (!p) return fail(GDN_ERR_ARG, "params is NULL");
    if (!p->conv_w || !p->A_log || !p->dt_bias || !p->norm_w)
        return fail(GDN_ERR_ARG, "a layer parameter pointer is NULL");
    if (!aligned16(p->conv_w) || !aligned16(p->A_log) || !aligned16(p->dt_bias) || !aligned16(p->norm_w))
        return fail(GDN_ERR_ALIGN, "layer parameter pointers must be 16-byte aligned");
    return GDN_OK;
}

}  // namespace

namespace gdn {

// CTAs per value head: as many equal parts (a power of two) as the cluster
// allows (portable size 8) while a CTA keeps at most 8 warps of 8 rows; more
// CTAs spread a small batch over more SMs.  Failing that, equal parts within a
// non-portable cluster of up to 16; failing that (d_v/8 warps with no such
// divisor, e.g. 9 or 30), the fewest parts of unequal width (floor or ceil of
// d_v/8 / P warps) that keep a CTA at 8 warps and the cluster at 16.
int verify_parts_per_head(int B, int Hv, int r, int dv, int sm_count) {
    (void)B; (void)Hv; (void)sm_count;
    const int warps_head = dv / 8;
    int best = 0;
    for (int P = 1; P <= warps_head; P *= 2) {
        if (warps_head % P) continue;
        if (warps_head / P > 8) continue;
        if (r * P <= 8) best = P;
    }
    if (best) return best;
    for (int P = 1; P <= warps_head; P *= 2) {             // non-portable cluster sizes up to 16
        if (warps_head % P || warps_head / P > 8) continue;
        if (r * P <= 16) return P;
    }
    const int P = (warps_head + 7) / 8;
    return r * P <= 16 ? P : 0;
}

}  // namespace gdn

namespace gdn {

// cuCtxGetCurrent / cuCtxGetId from the driver, looked up once (the library links only the runtime)
bool current_context_id(unsigned long long *id) {
    static std::once_flag once;
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    if (!get_current || !get_id) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace gdn

// ---- prefill with library-owned scratch -----------------------------------
// One fixed scratch array, which every context that loads this library's
// device code holds (module globals are per context).  Its device address is
// looked up with cudaGetSymbolAddress once per context -- in practice once per
// device, on the first static call with that device current -- and cached
// under the context's id, so a reset device (a new context, a new address) is
// looked up again instead of being handed a stale pointer.
namespace {
__device__ __align__(256) unsigned char g_prefill_scratch[GDN_PREFILL_STATIC_SCRATCH_BYTES];
gdn::PerContext<void *> g_scratch_addr;

int static_scratch(void **addr) {
    unsigned long long ctx = 0;
    const bool known = gdn::current_context_id(&ctx);
    if (known && g_scratch_addr.get(ctx, addr)) return GDN_OK;
    void *p = nullptr;
    // initialises the runtime's context on the current device if none is current yet
    cudaError_t e = cudaGetSymbolAddress(&p, g_prefill_scratch);
    if (e != cudaSuccess || !p)
        return fail(GDN_ERR_LAUNCH, "looking up the prefill scratch array failed: %s", cudaGetErrorString(e));
    if (gdn::current_context_id(&ctx)) g_scratch_addr.put(ctx, p);
    *addr = p;
    return GDN_OK;
}
}  // namespace

extern "C" {

const char *gdn_last_error(void) { return g_err.c_str(); }

const char *gdn_version(void) { return GDN_CHECKED ? "gdn-verify 0.1.0 (sm_103a, checked)" : "gdn-verify 0.1.0 (sm_103a)"; }

static int verify_impl(const gdn_dims *dims, const gdn_layer_params *params, const void *qkv, const void *z,
                       const void *alpha, const void *beta_raw, const int32_t *d_parent, float *state,
                       float *conv_state, float *cap_state, float *cap_conv, void *out, int *d_status,
                       void *stream, int mode = gdn::kChain, const int32_t *d_trim = nullptr,
                       const void *qkv_prev = nullptr, const void *alpha_prev = nullptr,
                       const void *beta_prev = nullptr, long long ld_act = 0, const void *l2_next = nullptr,
                       size_t l2_next_bytes = 0) {
    g_err.clear();
    int rc = check_common(dims);
    if (rc) return rc;
    if ((rc = check_params(params))) return rc;
    const gdn_dims &d = *dims;
    if (d.d_k != 32 && d.d_k != 64 && d.d_k != 128)
        return fail(GDN_ERR_SHAPE, "d_k must be 32, 64 or 128 (got %d)", d.d_k);
    if (d.d_v % 8 || d.d_v > 256) return fail(GDN_ERR_SHAPE, "d_v must be a multiple of 8 up to 256 (got %d)", d.d_v);
    if (d.n_tokens > 64) return fail(GDN_ERR_SHAPE, "n_tokens must be <= 64 for verify (got %d)", d.n_tokens);
    if (d.n_slots > 65535) return fail(GDN_ERR_SHAPE, "n_slots must be <= 65535");
    const bool commit = mode == gdn::kCommit;
    const bool pending = mode == gdn::kLazy && d_trim != nullptr;
    if (!qkv || (!z && !commit) || !alpha || !beta_raw || !state || !conv_state || (!out && !commit))
        return fail(GDN_ERR_ARG, "a required buffer pointer is NULL");
    if (pending && (!qkv_prev || !alpha_prev || !beta_prev))
        return fail(GDN_ERR_ARG, "a pending batch needs its qkv, alpha and beta_raw");
    const void *ptrs[] = {qkv, z, alpha, beta_raw, state, conv_state, cap_state, cap_conv, out, qkv_prev,
                          alpha_prev, beta_prev};
    for (const void *p : ptrs)
        if (p && !aligned16(p)) return fail(GDN_ERR_ALIGN, "buffer %p is not 16-byte aligned", p);
    const int r = d.n_v_heads / d.n_qk_heads;
    const DevInfo info = dev_info();
    const int P = gdn::verify_parts_per_head(d.n_slots, d.n_v_heads, r, d.d_v, info.sms);
    if (P == 0)
        return fail(GDN_ERR_SHAPE, "H_v/H_k = %d heads of d_v = %d need more than 16 CTAs per thread-block cluster "
                    "(at most 8 warps of 8 value rows per CTA)", r, d.d_v);
    const int act_bytes = d.act_dtype == GDN_BF16 ? 2 : 4;
    // a lazy verify with a pending batch runs up to 2T tokens through shared memory
    const int Tm = pending ? 2 * d.n_tokens : d.n_tokens;
    const size_t smem = gdn::verify_smem_bytes(Tm, d.n_tokens, d.d_k, d.d_v, P, act_bytes, mode == gdn::kTree);
    if (info.smem_optin > 0 && smem > size_t(info.smem_optin))
        return fail(GDN_ERR_SHAPE, "verify needs %zu bytes of shared memory per CTA (max %d)", smem,
                    info.smem_optin);

    gdn::VerifyArgs a{};
    a.B = d.n_slots; a.Hk = d.n_qk_heads; a.Hv = d.n_v_heads; a.dk = d.d_k; a.dv = d.d_v;
    a.T = d.n_tokens; a.Ts = d.n_tokens; a.Tm = Tm; a.C = int(conv_channels(&d)); a.r = r; a.P = P;
    a.ld_qkv = a.C; a.ld_z = (long long)d.n_v_heads * d.d_v; a.ld_ab = d.n_v_heads;
    if (ld_act) a.ld_qkv = a.ld_z = a.ld_ab = ld_act;     // column blocks of one activation matrix
    a.l2_next = l2_next;
    a.l2_next_bytes = l2_next ? l2_next_bytes : 0;
    a.rms_eps = d.rms_eps; a.l2_eps = d.l2_eps; a.q_scale = d.q_scale;
    a.conv_w = params->conv_w; a.A_log = params->A_log; a.dt_bias = params->dt_bias; a.norm_w = params->norm_w;
    a.qkv = qkv; a.z = z; a.alpha = alpha; a.beta_raw = beta_raw;
    a.state = state; a.conv_state = conv_state; a.cap_state = cap_state; a.cap_conv = cap_conv; a.out = out;
    a.d_status = d_status;
    a.parent = d_parent;
    a.trim = d_trim;
    a.qkv_prev = qkv_prev; a.alpha_prev = alpha_prev; a.beta_prev = beta_prev;
    a.mode = mode;
    {   // extents in bytes (the bounds checks of a checked build)
        const size_t ab = size_t(act_bytes), M = size_t(d.n_slots) * d.n_tokens;
        const size_t st = size_t(d.n_slots) * d.n_v_heads * d.d_v * d.d_k * 4, V = size_t(d.n_v_heads) * d.d_v;
        a.ext_qkv = ((M - 1) * size_t(a.ld_qkv) + size_t(a.C)) * ab;
        a.ext_z = ((M - 1) * size_t(a.ld_z) + V) * ab;
        a.ext_ab = ((M - 1) * size_t(a.ld_ab) + size_t(d.n_v_heads)) * ab;
        a.ext_state = st;
        a.ext_conv_state = size_t(d.n_slots) * 3 * size_t(a.C) * 4;
        a.ext_cap_state = st * size_t(d.n_tokens);
        a.ext_cap_conv = size_t(d.n_slots) * (mode == gdn::kTree ? 3 * size_t(d.n_tokens) : 3 + size_t(d.n_tokens)) *
                         size_t(a.C) * 4;
        a.ext_out = M * V * ab;
        a.ext_conv_w = 4 * size_t(a.C) * 4;
        a.ext_head = size_t(d.n_v_heads) * 4;
        a.ext_norm_w = size_t(d.d_v) * 4;
        a.ext_parent = M * 4;
        a.ext_trim = size_t(d.n_slots) * 4;
    }
    {   // the batch's activations as 2-D tensors for the kernel's TMA boxes (T tokens of a slot per box); the v
        // and z boxes are as wide as the widest part of a head (the last), so a narrower part also reads the
        // first rows of the next part of its own head
        PFN_cuTensorMapEncodeTiled_v12000 encode = gdn::tensor_map_encoder();
        if (!encode) return fail(GDN_ERR_LAUNCH, "the driver's tensor-map encoder is unavailable");
        const CUtensorMapDataType dt = d.act_dtype == GDN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                               : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
        const cuuint32_t estr[2] = {1, 1};
        const cuuint64_t rows = cuuint64_t(d.n_slots) * cuuint64_t(d.n_tokens);
        auto make = [&](CUtensorMap *map, const void *base, cuuint64_t cols, long long ld, int box_x) {
            const cuuint64_t dims[2] = {cols, rows};
            const cuuint64_t strides[1] = {cuuint64_t(ld) * cuuint64_t(act_bytes)};
            const cuuint32_t box[2] = {cuuint32_t(box_x), cuuint32_t(d.n_tokens)};
            return encode(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
        };
        if (!make(&a.qk_map, qkv, cuuint64_t(a.C), a.ld_qkv, d.d_k) ||
            !make(&a.v_map, qkv, cuuint64_t(a.C), a.ld_qkv, gdn::verify_part_rows(d.d_v, P)) ||
            (z && !make(&a.z_map, z, cuuint64_t(d.n_v_heads) * d.d_v, a.ld_z, gdn::verify_part_rows(d.d_v, P))))
            return fail(GDN_ERR_LAUNCH, "encoding the activation tensor maps failed");
    }
    cudaError_t e = gdn::launch_verify(a, d.act_dtype, info.sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(GDN_ERR_LAUNCH, "verify launch failed: %s", cudaGetErrorString(e));
    return GDN_OK;
}

int gdn_verify_forward(const gdn_dims *dims, const gdn_layer_params *params, const void *qkv,
                       const void *z, const void *alpha, const void *beta_raw, float *state,
                       float *conv_state, float *cap_state, float *cap_conv, void *out, int *d_status,
                       void *stream) {
    return verify_impl(dims, params, qkv, z, alpha, beta_raw, nullptr, state, conv_state, cap_state, cap_conv, out,
                       d_status, stream);
}

int gdn_verify_tree(const gdn_dims *dims, const gdn_layer_params *params, const void *qkv, const void *z,
                    const void *alpha, const void *beta_raw, const int32_t *d_parent, const float *state,
                    const float *conv_state, float *cap_state, float *cap_conv, void *out, int *d_status,
                    void *stream) {
    g_err.clear();
    if (!d_parent) return fail(GDN_ERR_ARG, "parent ids are NULL");
    if (!cap_state || !cap_conv) return fail(GDN_ERR_NO_CAPTURE, "a tree verify needs cap_state and cap_conv");
    // state and conv_state are only read (the kernel takes them through the shared argument block)
    return verify_impl(dims, params, qkv, z, alpha, beta_raw, d_parent, const_cast<float *>(state),
                       const_cast<float *>(conv_state), cap_state, cap_conv, out, d_status, stream, gdn::kTree);
}

int gdn_verify_after_rollback(const gdn_dims *dims, const gdn_layer_params *params, const int32_t *d_prev_trim,
                              const void *qkv, const void *z, const void *alpha, const void *beta_raw,
                              float *state, float *conv_state, float *cap_state, float *cap_conv, void *out,
                              int *d_status, void *stream) {
    g_err.clear();
    if (!d_prev_trim) return fail(GDN_ERR_ARG, "trim is NULL");
    if (!cap_state || !cap_conv)
        return fail(GDN_ERR_NO_CAPTURE, "the previous batch's captures (cap_state, cap_conv) are needed");
    return verify_impl(dims, params, qkv, z, alpha, beta_raw, nullptr, state, conv_state, cap_state, cap_conv, out,
                       d_status, stream, gdn::kRolled, d_prev_trim);
}

int gdn_verify_lazy(const gdn_dims *dims, const gdn_layer_params *params, const int32_t *d_prev_trim,
                    const void *prev_qkv, const void *prev_alpha, const void *prev_beta_raw, const void *qkv,
                    const void *z, const void *alpha, const void *beta_raw, float *state, float *conv_state,
                    void *out, int *d_status, void *stream) {
    return verify_impl(dims, params, qkv, z, alpha, beta_raw, nullptr, state, conv_state, nullptr, nullptr, out,
                       d_status, stream, gdn::kLazy, d_prev_trim, prev_qkv, prev_alpha, prev_beta_raw);
}

int gdn_commit_lazy(const gdn_dims *dims, const gdn_layer_params *params, const int32_t *d_trim,
                    const void *qkv, const void *alpha, const void *beta_raw, float *state, float *conv_state,
                    int *d_status, void *stream) {
    g_err.clear();
    if (!d_trim) return fail(GDN_ERR_ARG, "trim is NULL");
    return verify_impl(dims, params, qkv, nullptr, alpha, beta_raw, nullptr, state, conv_state, nullptr, nullptr,
                       nullptr, d_status, stream, gdn::kCommit, d_trim);
}

static int rollback_impl(const gdn_dims *dims, const int32_t *d_trim, float *state, float *conv_state,
                         const float *cap_state, const float *cap_conv, int *d_status, void *stream, int tree) {
    g_err.clear();
    int rc = check_common(dims);
    if (rc) return rc;
    const gdn_dims &d = *dims;
    if (d.n_slots > 65535) return fail(GDN_ERR_SHAPE, "n_slots must be <= 65535");
    if ((d.d_k % 4) || (d.d_v % 8)) return fail(GDN_ERR_SHAPE, "d_k must be a multiple of 4 and d_v of 8");
    if (!d_trim || !state || !conv_state) return fail(GDN_ERR_ARG, "trim, state or conv_state is NULL");
    if (!cap_state || !cap_conv) return fail(GDN_ERR_NO_CAPTURE, "rollback needs both capture buffers");
    const void *ptrs[] = {d_trim, state, conv_state, cap_state, cap_conv};
    for (const void *p : ptrs)
        if (!aligned16(p)) return fail(GDN_ERR_ALIGN, "buffer %p is not 16-byte aligned", p);
    gdn::RollbackArgs a{};
    a.B = d.n_slots; a.T = d.n_tokens; a.W1 = d.conv_width - 1;
    a.C = conv_channels(&d);
    a.state_elems = (long long)d.n_v_heads * d.d_v * d.d_k;
    a.conv_elems = (long long)a.W1 * a.C;
    a.trim = d_trim; a.state = state; a.conv_state = conv_state; a.cap_state = cap_state; a.cap_conv = cap_conv;
    a.d_status = d_status;
    a.tree = tree;
    a.ext_state = size_t(a.B) * size_t(a.state_elems) * 4;
    a.ext_conv_state = size_t(a.B) * size_t(a.conv_elems) * 4;
    a.ext_cap_state = size_t(a.B) * a.T * size_t(a.state_elems) * 4;
    a.ext_cap_conv = size_t(a.B) * (tree ? size_t(a.T) * a.W1 : size_t(a.W1 + a.T)) * size_t(a.C) * 4;
    cudaError_t e = gdn::launch_rollback(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(GDN_ERR_LAUNCH, "rollback launch failed: %s", cudaGetErrorString(e));
    return GDN_OK;
}

int gdn_rollback(const gdn_dims *dims, const int32_t *d_trim, float *state, float *conv_state,
                 const float *cap_state, const float *cap_conv, int *d_status, void *stream) {
    return rollback_impl(dims, d_trim, state, conv_state, cap_state, cap_conv, d_status, stream, 0);
}

int gdn_rollback_tree(const gdn_dims *dims, const int32_t *d_accept, float *state, float *conv_state,
                      const float *cap_state, const float *cap_conv, int *d_status, void *stream) {
    return rollback_impl(dims, d_accept, state, conv_state, cap_state, cap_conv, d_status, stream, 1);
}

static int rollback_layers_impl(const gdn_dims *dims, int n_layers, const int32_t *d_trim, float *const *d_state,
                                float *const *d_conv_state, const float *const *d_cap_state,
                                const float *const *d_cap_conv, int *d_status, void *stream, int tree) {
    g_err.clear();
    int rc = check_common(dims);
    if (rc) return rc;
    const gdn_dims &d = *dims;
    if (n_layers < 1 || n_layers > 65535) return fail(GDN_ERR_SHAPE, "n_layers must be in [1, 65535] (got %d)", n_layers);
    if (d.n_slots > 65535) return fail(GDN_ERR_SHAPE, "n_slots must be <= 65535");
    if ((d.d_k % 4) || (d.d_v % 8)) return fail(GDN_ERR_SHAPE, "d_k must be a multiple of 4 and d_v of 8");
    if (!d_trim || !d_state || !d_conv_state) return fail(GDN_ERR_ARG, "trim or a state table is NULL");
    if (!d_cap_state || !d_cap_conv) return fail(GDN_ERR_NO_CAPTURE, "rollback needs both capture tables");
    if (!aligned16(d_trim)) return fail(GDN_ERR_ALIGN, "d_trim is not 16-byte aligned");
    const void *tabs[] = {d_state, d_conv_state, d_cap_state, d_cap_conv};
    for (const void *p : tabs)
        if (reinterpret_cast<uintptr_t>(p) & 7u) return fail(GDN_ERR_ALIGN, "pointer table %p is not 8-byte aligned", p);
    gdn::RollbackArgs a{};
    a.B = d.n_slots; a.T = d.n_tokens; a.W1 = d.conv_width - 1;
    a.C = conv_channels(&d);
    a.state_elems = (long long)d.n_v_heads * d.d_v * d.d_k;
    a.conv_elems = (long long)a.W1 * a.C;
    a.trim = d_trim;
    a.d_status = d_status;
    a.tree = tree;
    a.ext_state = size_t(a.B) * size_t(a.state_elems) * 4;
    a.ext_conv_state = size_t(a.B) * size_t(a.conv_elems) * 4;
    a.ext_cap_state = size_t(a.B) * a.T * size_t(a.state_elems) * 4;
    a.ext_cap_conv = size_t(a.B) * (tree ? size_t(a.T) * a.W1 : size_t(a.W1 + a.T)) * size_t(a.C) * 4;
    a.n_layers = n_layers;
    a.tab_state = d_state; a.tab_conv_state = d_conv_state; a.tab_cap_state = d_cap_state; a.tab_cap_conv = d_cap_conv;
    cudaError_t e = gdn::launch_rollback(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(GDN_ERR_LAUNCH, "rollback launch failed: %s", cudaGetErrorString(e));
    return GDN_OK;
}

int gdn_rollback_layers(const gdn_dims *dims, int n_layers, const int32_t *d_trim, float *const *d_state,
                        float *const *d_conv_state, const float *const *d_cap_state, const float *const *d_cap_conv,
                        int *d_status, void *stream) {
    return rollback_layers_impl(dims, n_layers, d_trim, d_state, d_conv_state, d_cap_state, d_cap_conv, d_status,
                                stream, 0);
}

int gdn_rollback_tree_layers(const gdn_dims *dims, int n_layers, const int32_t *d_accept, float *const *d_state,
                             float *const *d_conv_state, const float *const *d_cap_state,
                             const float *const *d_cap_conv, int *d_status, void *stream) {
    return rollback_layers_impl(dims, n_layers, d_accept, d_state, d_conv_state, d_cap_state, d_cap_conv, d_status,
                                stream, 1);
}

size_t gdn_prefill_workspace_bytes(const gdn_dims *dims) {
    if (!dims) return 0;
    std::string why;
    if (check_common(dims) != GDN_OK || gdn::prefill_check(*dims, why) != GDN_OK) return 0;
    return gdn::prefill_workspace_bytes(*dims);
}

int gdn_prefill_chunked(const gdn_dims *dims, const gdn_layer_params *params, const void *qkv, const void *z,
                        const void *alpha, const void *beta_raw, float *state, float *conv_state, void *out,
                        void *workspace, size_t ws_bytes, int *d_status, void *stream) {
    g_err.clear();
    int rc = check_common(dims);
    if (rc) return rc;
    if ((rc = check_params(params))) return rc;
    std::string why;
    if ((rc = gdn::prefill_check(*dims, why))) return fail(rc, "%s", why.c_str());
    if (!qkv || !z || !alpha || !beta_raw || !state || !conv_state || !out)
        return fail(GDN_ERR_ARG, "a required buffer pointer is NULL");
    const void *ptrs[] = {qkv, z, alpha, beta_raw, state, conv_state, out};
    for (const void *p : ptrs)
        if (!aligned16(p)) return fail(GDN_ERR_ALIGN, "buffer %p is not 16-byte aligned", p);
    const size_t need = gdn::prefill_workspace_bytes(*dims);
    if (need > 0 && (!workspace || ws_bytes < need))
        return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes needed (got %zu)", need, ws_bytes);
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return fail(GDN_ERR_ALIGN, "workspace must be 256-byte aligned");
    cudaError_t e = gdn::launch_prefill(*dims, *params, qkv, z, alpha, beta_raw, state, conv_state, out,
                                        workspace, d_status, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail(GDN_ERR_LAUNCH, "prefill launch failed: %s", cudaGetErrorString(e));
    return GDN_OK;
}

size_t gdn_prefill_static_scratch_bytes(void) { return GDN_PREFILL_STATIC_SCRATCH_BYTES; }

#if GDN_CHECKED
// Test build only: the scratch address gdn_prefill_chunked_static would use in the current context
// (NULL on failure), so a test can check that each context gets its own.
void *gdn_test_static_scratch_address(void) {
    void *p = nullptr;
    return static_scratch(&p) == GDN_OK ? p : nullptr;
}
#endif

int gdn_prefill_chunked_static(const gdn_dims *dims, const gdn_layer_params *params, const void *qkv,
                               const void *z, const void *alpha, const void *beta_raw, float *state,
                               float *conv_state, void *out, int *d_status, void *stream) {
    g_err.clear();
    int rc = check_common(dims);
    if (rc) return rc;
    std::string why;
    if ((rc = gdn::prefill_check(*dims, why))) return fail(rc, "%s", why.c_str());
    const size_t need = gdn::prefill_workspace_bytes(*dims);
    if (need > GDN_PREFILL_STATIC_SCRATCH_BYTES)
        return fail(GDN_ERR_WORKSPACE, "prefill needs %zu bytes of scratch; the built-in array holds %zu", need,
                    (size_t)GDN_PREFILL_STATIC_SCRATCH_BYTES);
    void *scratch = nullptr;
    if (need > 0 && (rc = static_scratch(&scratch))) return rc;
    return gdn_prefill_chunked(dims, params, qkv, z, alpha, beta_raw, state, conv_state, out, scratch,
                               need > 0 ? (size_t)GDN_PREFILL_STATIC_SCRATCH_BYTES : 0, d_status, stream);
}

// ---- one verify step from host memory ---------------------------------------

int gdn_step_io_layout(const gdn_dims *dims, gdn_step_io *io) {
    g_err.clear();
    int rc = check_common(dims);
    if (rc) return rc;
    if (!io) return fail(GDN_ERR_ARG, "io is NULL");
    const gdn_dims &d = *dims;
    const size_t ab = d.act_dtype == GDN_BF16 ? 2 : 4, M = size_t(d.n_slots) * d.n_tokens;
    const size_t V = size_t(d.n_v_heads) * d.d_v;
    auto up = [](size_t n) { return (n + 255) & ~size_t(255); };
    size_t off = 0;
    io->qkv = off; off += up(M * size_t(conv_channels(&d)) * ab);
    io->z = off; off += up(M * V * ab);
    io->alpha = off; off += up(M * size_t(d.n_v_heads) * ab);
    io->beta_raw = off; off += up(M * size_t(d.n_v_heads) * ab);
    io->trim = off; off += up(size_t(d.n_slots) * 4);
    io->in_bytes = off;
    io->out_bytes = up(M * V * ab);
    return GDN_OK;
}

int gdn_verify_step_host(const gdn_dims *dims, const gdn_layer_params *params, int rollback_first,
                         const void *h_in, void *h_out, void *d_io, size_t d_io_bytes, float *state,
                         float *conv_state, float *cap_state, float *cap_conv, int *d_status, void *stream) {
    gdn_step_io io;
    int rc = gdn_step_io_layout(dims, &io);
    if (rc) return rc;
    if (!h_in || !h_out || !d_io) return fail(GDN_ERR_ARG, "h_in, h_out or d_io is NULL");
    if (d_io_bytes < io.in_bytes + io.out_bytes)
        return fail(GDN_ERR_WORKSPACE, "d_io of %zu bytes needed (got %zu)", io.in_bytes + io.out_bytes, d_io_bytes);
    if (reinterpret_cast<uintptr_t>(d_io) & 255u) return fail(GDN_ERR_ALIGN, "d_io must be 256-byte aligned");
    if (rollback_first != 0 && rollback_first != 1) return fail(GDN_ERR_ARG, "rollback_first must be 0 or 1");
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned char *din = static_cast<unsigned char *>(d_io), *dout = din + io.in_bytes;
    cudaError_t e = cudaMemcpyAsync(din, h_in, io.in_bytes, cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return fail(GDN_ERR_LAUNCH, "input copy failed: %s", cudaGetErrorString(e));
    const int32_t *trim = reinterpret_cast<const int32_t *>(din + io.trim);
    if (rollback_first) {
        rc = gdn_verify_after_rollback(dims, params, trim, din + io.qkv, din + io.z, din + io.alpha,
                                       din + io.beta_raw, state, conv_state, cap_state, cap_conv, dout, d_status,
                                       stream);
    } else {
        rc = gdn_verify_forward(dims, params, din + io.qkv, din + io.z, din + io.alpha, din + io.beta_raw, state,
                                conv_state, cap_state, cap_conv, dout, d_status, stream);
        if (rc == GDN_OK) rc = gdn_rollback(dims, trim, state, conv_state, cap_state, cap_conv, d_status, stream);
    }
    if (rc) return rc;
    e = cudaMemcpyAsync(h_out, dout, io.out_bytes, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return fail(GDN_ERR_LAUNCH, "output copy failed: %s", cudaGetErrorString(e));
    return GDN_OK;
}

// ---- projections around the block and the layer step ----------------------

static long long proj_in_cols(const gdn_dims &d) {
    return conv_channels(&d) + (long long)d.n_v_heads * d.d_v + 2LL * d.n_v_heads;
}

static size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

// checks shared by the projection calls; M = B * T rows
static int check_proj(const gdn_dims *dims, const gdn_proj_weights *w) {
    int rc = check_common(dims);
    if (rc) return rc;
    if (!w) return fail(GDN_ERR_ARG, "projection weights are NULL");
    if (dims->act_dtype != GDN_BF16) return fail(GDN_ERR_DTYPE, "the projections run in bf16 (act_dtype GDN_BF16)");
    if (w->n_embd < 8 || w->n_embd % 8)
        return fail(GDN_ERR_SHAPE, "n_embd must be a positive multiple of 8 (got %d)", w->n_embd);
    if (dims->n_v_heads % 8)
        return fail(GDN_ERR_SHAPE, "the layer step needs n_v_heads to be a multiple of 8 (got %d)", dims->n_v_heads);
    if (!w->w_in || !w->w_out) return fail(GDN_ERR_ARG, "a projection weight pointer is NULL");
    if (!aligned16(w->w_in) || !aligned16(w->w_out)) return fail(GDN_ERR_ALIGN, "weights must be 16-byte aligned");
    const long long M = (long long)dims->n_slots * dims->n_tokens;
    if (M > (1LL << 30) || proj_in_cols(*dims) > (1LL << 30))
        return fail(GDN_ERR_SHAPE, "projection sizes out of range");
    return GDN_OK;
}

long long gdn_proj_in_ld(const gdn_dims *dims) {
    if (!dims) return 0;
    return (proj_in_cols(*dims) + 7) / 8 * 8;
}

size_t gdn_layer_workspace_bytes(const gdn_dims *dims, int n_embd) {
    if (!dims || n_embd < 1) return 0;
    const size_t M = size_t(dims->n_slots) * size_t(dims->n_tokens);
    return align256(M * size_t(gdn_proj_in_ld(dims)) * 2) + align256(M * size_t(dims->n_v_heads) * dims->d_v * 2);
}

static int project_in(const gdn_dims *dims, const gdn_proj_weights *w, const void *x, void *act, int *d_status,
                      void *stream) {
    int rc = check_proj(dims, w);
    if (rc) return rc;
    if (!x || !act) return fail(GDN_ERR_ARG, "x or act is NULL");
    if (!aligned16(x) || !aligned16(act)) return fail(GDN_ERR_ALIGN, "x and act must be 16-byte aligned");
    std::string why;
    const int M = dims->n_slots * dims->n_tokens;
    if (!gdn::gemm_xwt_bf16(w->w_in, x, act, M, int(proj_in_cols(*dims)), w->n_embd, gdn_proj_in_ld(dims), d_status,
                            static_cast<cudaStream_t>(stream), why))
        return fail(GDN_ERR_LAUNCH, "input projection: %s", why.c_str());
    return GDN_OK;
}

static int project_out(const gdn_dims *dims, const gdn_proj_weights *w, const void *out, void *y, int *d_status,
                       void *stream) {
    int rc = check_proj(dims, w);
    if (rc) return rc;
    if (!out || !y) return fail(GDN_ERR_ARG, "out or y is NULL");
    if (!aligned16(out) || !aligned16(y)) return fail(GDN_ERR_ALIGN, "out and y must be 16-byte aligned");
    std::string why;
    const int M = dims->n_slots * dims->n_tokens;
    if (!gdn::gemm_xwt_bf16(w->w_out, out, y, M, w->n_embd, dims->n_v_heads * dims->d_v, w->n_embd, d_status,
                            static_cast<cudaStream_t>(stream), why))
        return fail(GDN_ERR_LAUNCH, "output projection: %s", why.c_str());
    return GDN_OK;
}

int gdn_project_in(const gdn_dims *dims, const gdn_proj_weights *w, const void *x, void *act, void *workspace,
                   size_t ws_bytes, void *stream) {
    g_err.clear();
    (void)workspace; (void)ws_bytes;            // the GEMM needs no scratch
    return project_in(dims, w, x, act, nullptr, stream);
}

int gdn_project_out(const gdn_dims *dims, const gdn_proj_weights *w, const void *out, void *y, void *workspace,
                    size_t ws_bytes, void *stream) {
    g_err.clear();
    (void)workspace; (void)ws_bytes;
    return project_out(dims, w, out, y, nullptr, stream);
}

int gdn_layer_verify(const gdn_dims *dims, const gdn_layer_params *params, const gdn_proj_weights *w,
                     const void *x, float *state, float *conv_state, float *cap_state, float *cap_conv, void *y,
                     void *workspace, size_t ws_bytes, int *d_status, void *stream) {
    g_err.clear();
    int rc = check_proj(dims, w);
    if (rc) return rc;
    const size_t need = gdn_layer_workspace_bytes(dims, w->n_embd);
    if (!workspace || ws_bytes < need)
        return fail(GDN_ERR_WORKSPACE, "workspace of %zu bytes needed (got %zu)", need, ws_bytes);
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return fail(GDN_ERR_ALIGN, "workspace must be 256-byte aligned");
    const gdn_dims &d = *dims;
    const size_t M = size_t(d.n_slots) * d.n_tokens;
    const long long ld = gdn_proj_in_ld(dims);
    unsigned char *act = static_cast<unsigned char *>(workspace);
    unsigned char *out = act + align256(M * size_t(ld) * 2);
    if ((rc = project_in(dims, w, x, act, d_status, stream))) return rc;
    // the verify reads q|k|v, z, alpha and beta_raw as column blocks of the activation matrix
    const long long C = conv_channels(dims), V = (long long)d.n_v_heads * d.d_v;
    unsigned char *z = act + C * 2, *alpha = act + (C + V) * 2, *beta = alpha + size_t(d.n_v_heads) * 2;
    // the verify also warms L2 with the output projection's weights (read by the next launch)
    const size_t w_out_bytes = size_t(w->n_embd) * size_t(V) * 2;
    if ((rc = verify_impl(dims, params, act, z, alpha, beta, nullptr, state, conv_state, cap_state, cap_conv, out,
                          d_status, stream, gdn::kChain, nullptr, nullptr, nullptr, nullptr, ld, w->w_out,
                          reinterpret_cast<uintptr_t>(w->w_out) % 16 ? 0 : w_out_bytes & ~size_t(15))))
        return rc;
    return project_out(dims, w, out, y, d_status, stream);
}

}  // extern "C"
