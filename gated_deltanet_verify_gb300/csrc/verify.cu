// verify.cu -- fused Gated DeltaNet verify forward for sm_103a.
//
// One launch runs, for every slot and value head, the whole verify path over
// T = K+1 tokens: conv window + depthwise causal conv + SiLU, q/k L2 norm,
// gates, the gated delta-rule recurrence with the state held in registers,
// per-position state capture, gated RMSNorm, conv-state advance.
//
// Work decomposition
//   * A thread-block cluster covers one (slot, key-head group): the r = H_v/H_k
//     value heads that share key head kh, each split into P CTAs along d_v.
//     Columns j of S (value dims) evolve independently, so a CTA owns d_v/P
//     of them; only the per-head RMSNorm needs all d_v, and its partial sums
//     are exchanged through distributed shared memory inside the cluster.
//     The cluster also orders the in-place conv_state update: the q/k conv
//     channels are read by every CTA of the group and are rewritten only after
//     a cluster barrier.
//   * Inside a CTA each warp owns 8 value rows j; lane l holds S[i][j] for
//     i in [l*EPL, (l+1)*EPL) (EPL = d_k/32), so one warp-wide 16-byte store
//     writes a whole 512-byte row of the captured state.
//   * Per token the two reductions over d_k -- k^T S and q^T S, taken on the
//     state *before* the update -- are done together by one reduce-scatter
//     butterfly (16 shuffles for 8 rows x 2 vectors).  The update then reads
//     S_t^T q = g S^T q + (k.q) w, with w = beta (v - g S^T k), so a token
//     costs one reduction phase, not two.
//   * Reduction orders are fixed by the lane layout only, never by P or T, so
//     the state after token t is bit-identical whatever the launch shape and
//     however many tokens follow it.
#include "internal.cuh"

#include <cooperative_groups.h>
#include <cuda_bf16.h>

namespace cg = cooperative_groups;

namespace gdn {
namespace {

constexpr int kRowsPerWarp = 8;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kMaxDevices = 64;

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename Act> __device__ __forceinline__ Act from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float silu(float x) { return x / (1.0f + expf(-x)); }

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_group 0;\n" ::: "memory");
}

// 16-byte streaming store (evict-first): captured states are written once and
// read back at most once, by a rollback.
__device__ __forceinline__ void st_stream4(float *p, float a, float b, float c, float d) {
    asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"l"(p), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

// The state is rewritten by this kernel, so it is read through the coherent
// path (no .nc), only without allocating in L1.
__device__ __forceinline__ float4 ld_stream4(const float *p) {
    float4 v;
    asm volatile("ld.global.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];\n"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

// Shared-memory carve-up; identical on host and device.
struct Smem {
    int T, NCH, ROWS, WARPS, act_bytes;
    size_t xs, zs, cw, cs, nw, ys, tail, os, gs, bs, kqs, rinv, part, total;
    __host__ __device__ Smem(int T_, int dk, int rows, int warps, int act_bytes_)
        : T(T_), NCH(2 * dk + rows), ROWS(rows), WARPS(warps), act_bytes(act_bytes_) {
        size_t off = 0;
        auto take = [&](size_t bytes) {
            size_t o = off;
            off += (bytes + 15) & ~size_t(15);
            return o;
        };
        xs = take(size_t(T) * NCH * act_bytes);    // raw q | k | v inputs
        zs = take(size_t(T) * ROWS * act_bytes);   // raw z for own rows
        cw = take(size_t(4) * NCH * 4);             // conv weights
        cs = take(size_t(3) * NCH * 4);             // old conv state
        nw = take(size_t(ROWS) * 4);                // norm weight for own rows
        ys = take(size_t(T) * NCH * 4);             // post conv+SiLU (q, k normalised in place)
        tail = take(size_t(3) * NCH * 4);           // new conv state (window rows T..T+2)
        os = take(size_t(T) * ROWS * 4);            // o before the RMSNorm
        gs = take(size_t(T) * 4);
        bs = take(size_t(T) * 4);
        kqs = take(size_t(T) * 4);
        rinv = take(size_t(T) * 4);
        part = take(size_t(T) * WARPS * 4);         // per-warp sums of o^2
        total = off;
    }
};

template <int DK, typename Act>
__global__ void __launch_bounds__(512) verify_kernel(const VerifyArgs a) {
    constexpr int EPL = DK / 32;
    static_assert(EPL == 1 || EPL == 2 || EPL == 4, "d_k must be 32, 64 or 128");

    cg::cluster_group cluster = cg::this_cluster();
    extern __shared__ __align__(16) unsigned char smem_raw[];

    const int tid = threadIdx.x, nthr = blockDim.x;
    const int lane = tid & 31, wid = tid >> 5, WARPS = nthr >> 5;
    const int ROWS = WARPS * kRowsPerWarp;
    const int T = a.T, Hv = a.Hv, Hk = a.Hk, DV = a.dv, C = a.C;
    const int s = blockIdx.y;
    const int h = blockIdx.x / a.P, p = blockIdx.x % a.P;
    const int kh = h / a.r;
    const int j0 = p * ROWS;                                   // first value row of this CTA
    const bool qk_writer = (h % a.r == 0) && (p == 0);        // writes the shared q/k conv channels

    const Smem L(T, DK, ROWS, WARPS, sizeof(Act));
    Act *xs = reinterpret_cast<Act *>(smem_raw + L.xs);
    Act *zs = reinterpret_cast<Act *>(smem_raw + L.zs);
    float *cw = reinterpret_cast<float *>(smem_raw + L.cw);
    float *cs = reinterpret_cast<float *>(smem_raw + L.cs);
    float *nw = reinterpret_cast<float *>(smem_raw + L.nw);
    float *ys = reinterpret_cast<float *>(smem_raw + L.ys);
    float *tail = reinterpret_cast<float *>(smem_raw + L.tail);
    float *os = reinterpret_cast<float *>(smem_raw + L.os);
    float *gs = reinterpret_cast<float *>(smem_raw + L.gs);
    float *bs = reinterpret_cast<float *>(smem_raw + L.bs);
    float *kqs = reinterpret_cast<float *>(smem_raw + L.kqs);
    float *rinv = reinterpret_cast<float *>(smem_raw + L.rinv);
    float *part = reinterpret_cast<float *>(smem_raw + L.part);
    const int NCH = L.NCH;

    // local channel c -> global conv channel
    auto gchan = [&](int c) -> int {
        if (c < DK) return kh * DK + c;                                  // q of key head kh
        if (c < 2 * DK) return Hk * DK + kh * DK + (c - DK);            // k of key head kh
        return 2 * Hk * DK + h * DV + j0 + (c - 2 * DK);                 // v rows of this CTA
    };

    // ---------------------------------------------------------------- loads
    // (1) the state rows this warp owns, straight into registers
    const int rbase = wid * kRowsPerWarp;
    float S[kRowsPerWarp][EPL];
    {
        const float *src = a.state + ((size_t(s) * Hv + h) * DV + j0 + rbase) * DK + lane * EPL;
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            if constexpr (EPL == 4) {
                float4 v = ld_stream4(src + size_t(r) * DK);
                S[r][0] = v.x; S[r][1] = v.y; S[r][2] = v.z; S[r][3] = v.w;
            } else {
#pragma unroll
                for (int e = 0; e < EPL; ++e) S[r][e] = src[size_t(r) * DK + e];
            }
        }
    }
    // (2) activations, conv weights / state, norm weight: 16-byte async copies to smem
    {
        constexpr int kPer16 = 16 / sizeof(Act);
        const int vq = DK / kPer16, vv = ROWS / kPer16;     // 16-byte vectors per segment
        const int per_t = 2 * vq + 2 * vv;                  // q, k, v, z
        const Act *qkv = static_cast<const Act *>(a.qkv);
        const Act *z = static_cast<const Act *>(a.z);
        for (int i = tid; i < T * per_t; i += nthr) {
            const int t = i / per_t, w = i % per_t;
            const size_t row = size_t(s) * a.Ts + t;
            const Act *src;
            Act *dst;
            if (w < vq) {
                src = qkv + row * C + size_t(kh) * DK + w * kPer16;
                dst = xs + size_t(t) * NCH + w * kPer16;
            } else if (w < 2 * vq) {
                src = qkv + row * C + size_t(Hk + kh) * DK + (w - vq) * kPer16;
                dst = xs + size_t(t) * NCH + DK + (w - vq) * kPer16;
            } else if (w < 2 * vq + vv) {
                src = qkv + row * C + size_t(2 * Hk) * DK + size_t(h) * DV + j0 + (w - 2 * vq) * kPer16;
                dst = xs + size_t(t) * NCH + 2 * DK + (w - 2 * vq) * kPer16;
            } else {
                src = z + row * size_t(Hv) * DV + size_t(h) * DV + j0 + (w - 2 * vq - vv) * kPer16;
                dst = zs + size_t(t) * ROWS + (w - 2 * vq - vv) * kPer16;
            }
            cp_async16(dst, src);
        }
        // conv weights (4 rows) and old conv state (3 rows), per segment in float4s
        const int fq = DK / 4, fv = ROWS / 4, per_row = 2 * fq + fv;
        for (int i = tid; i < 7 * per_row; i += nthr) {
            const int rrow = i / per_row, w = i % per_row;
            int c0;
            if (w < fq) c0 = w * 4;
            else if (w < 2 * fq) c0 = DK + (w - fq) * 4;
            else c0 = 2 * DK + (w - 2 * fq) * 4;
            const int g0 = gchan(c0);
            if (rrow < 4) cp_async16(cw + rrow * NCH + c0, a.conv_w + size_t(rrow) * C + g0);
            else cp_async16(cs + (rrow - 4) * NCH + c0, a.conv_state + (size_t(s) * 3 + (rrow - 4)) * C + g0);
        }
        for (int i = tid; i < ROWS / 4; i += nthr) cp_async16(nw + i * 4, a.norm_w + j0 + i * 4);
    }
    // (3) gates for this head, one token per thread
    for (int t = tid; t < T; t += nthr) {
        const size_t idx = (size_t(s) * a.Ts + t) * Hv + h;
        const float al = to_f32(static_cast<const Act *>(a.alpha)[idx]);
        const float br = to_f32(static_cast<const Act *>(a.beta_raw)[idx]);
        const float x = al + __ldg(a.dt_bias + h);
        const float sp = x > 20.0f ? x : log1pf(expf(x));               // softplus
        gs[t] = expf(-expf(__ldg(a.A_log + h)) * sp);
        bs[t] = 1.0f / (1.0f + expf(-br));
    }
    cp_async_wait_all();
    __syncthreads();

    // ------------------------------------------------ conv + SiLU (+ capture)
    const bool cap_conv = a.cap_conv != nullptr;
    for (int c = tid; c < NCH; c += nthr) {
        const float w0 = cw[c], w1 = cw[NCH + c], w2 = cw[2 * NCH + c], w3 = cw[3 * NCH + c];
        float x0 = cs[c], x1 = cs[NCH + c], x2 = cs[2 * NCH + c];
        const int g = gchan(c);
        const bool writer = (c >= 2 * DK) || qk_writer;
        float *wcap = cap_conv ? a.cap_conv + size_t(s) * (3 + T) * C + g : nullptr;
        if (cap_conv && writer) {
            wcap[0] = x0;
            wcap[size_t(C)] = x1;
            wcap[2 * size_t(C)] = x2;
        }
        for (int t = 0; t < T; ++t) {
            const float x3 = to_f32(xs[size_t(t) * NCH + c]);
            const float pre = fmaf(w3, x3, fmaf(w2, x2, fmaf(w1, x1, w0 * x0)));
            ys[size_t(t) * NCH + c] = silu(pre);
            if (cap_conv && writer) wcap[size_t(3 + t) * C] = x3;
            x0 = x1; x1 = x2; x2 = x3;
        }
        tail[c] = x0; tail[NCH + c] = x1; tail[2 * NCH + c] = x2;
    }
    __syncthreads();

    // ------------------------------------------- q/k L2 norm, k.q per token
    for (int t = wid; t < T; t += WARPS) {
        float *q = ys + size_t(t) * NCH + lane * EPL;
        float *k = ys + size_t(t) * NCH + DK + lane * EPL;
        float qv[EPL], kv[EPL];
        float sq = 0.f, sk = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            qv[e] = q[e]; kv[e] = k[e];
            sq = fmaf(qv[e], qv[e], sq);
            sk = fmaf(kv[e], kv[e], sk);
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) {
            sq += __shfl_xor_sync(kFull, sq, m);
            sk += __shfl_xor_sync(kFull, sk, m);
        }
        const float iq = 1.0f / sqrtf(sq + a.l2_eps), ik = 1.0f / sqrtf(sk + a.l2_eps);
        float kq = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            qv[e] *= iq; kv[e] *= ik;
            q[e] = qv[e]; k[e] = kv[e];
            kq = fmaf(kv[e], qv[e], kq);
        }
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) kq += __shfl_xor_sync(kFull, kq, m);
        if (lane == 0) kqs[t] = kq;
    }
    __syncthreads();

    // ------------------------------------------------------------ recurrence
    const bool hi16 = (lane & 16) != 0;
    const int rr = ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
    const bool o_writer = !hi16 && !(lane & 1);
    const bool capture = a.cap_state != nullptr;
    float *cap_row0 = capture ? a.cap_state + (size_t(h) * DV + j0 + rbase) * DK + lane * EPL : nullptr;
    const float q_scale = a.q_scale;

    for (int t = 0; t < T; ++t) {
        const float *yt = ys + size_t(t) * NCH;
        float kk[EPL], qq[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) {
            qq[e] = yt[lane * EPL + e];
            kk[e] = yt[DK + lane * EPL + e];
        }
        const float g = gs[t], beta = bs[t], kq = kqs[t];

        // per-lane partial dot products over this lane's d_k slice
        float v16[16];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            float dk_ = S[r][0] * kk[0], dq_ = S[r][0] * qq[0];
#pragma unroll
            for (int e = 1; e < EPL; ++e) {
                dk_ = fmaf(S[r][e], kk[e], dk_);
                dq_ = fmaf(S[r][e], qq[e], dq_);
            }
            v16[r] = dk_;
            v16[8 + r] = dq_;
        }
        // reduce-scatter butterfly: after the masks 16, 8, 4, 2 each lane keeps
        // one value (kind = lane bit 4, row = lane bits 3..1); mask 1 completes it
#pragma unroll
        for (int lvl = 0; lvl < 4; ++lvl) {
            const int m = 16 >> lvl, half = 8 >> lvl;
            const bool up = (lane & m) != 0;
#pragma unroll
            for (int i = 0; i < half; ++i) {
                const float keep = up ? v16[i + half] : v16[i];
                const float send = up ? v16[i] : v16[i + half];
                v16[i] = keep + __shfl_xor_sync(kFull, send, m);
            }
        }
        const float mine = v16[0] + __shfl_xor_sync(kFull, v16[0], 1);
        const float other = __shfl_xor_sync(kFull, mine, 16);
        const float kd = hi16 ? other : mine;     // (S^T k)_j for row rr
        const float qd = hi16 ? mine : other;     // (S^T q)_j for row rr
        const float vj = yt[2 * DK + rbase + rr];
        const float w = beta * (vj - g * kd);     // beta (v - (g S)^T k)
        if (o_writer) os[size_t(t) * ROWS + rbase + rr] = q_scale * fmaf(g, qd, kq * w);

        // S <- g S + k w^T for the 8 rows
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            const float wr = __shfl_sync(kFull, w, 2 * r);
#pragma unroll
            for (int e = 0; e < EPL; ++e) S[r][e] = fmaf(kk[e], wr, g * S[r][e]);
        }
        if (capture) {
            float *dst = cap_row0 + (size_t(s) * T + t) * size_t(Hv) * DV * DK;
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r) {
                if constexpr (EPL == 4) st_stream4(dst + size_t(r) * DK, S[r][0], S[r][1], S[r][2], S[r][3]);
                else {
#pragma unroll
                    for (int e = 0; e < EPL; ++e) __stcs(dst + size_t(r) * DK + e, S[r][e]);
                }
            }
        }
    }

    // ------------------------------------------------------------- epilogue
    {
        float *dst = a.state + ((size_t(s) * Hv + h) * DV + j0 + rbase) * DK + lane * EPL;
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
            if constexpr (EPL == 4)
                *reinterpret_cast<float4 *>(dst + size_t(r) * DK) = make_float4(S[r][0], S[r][1], S[r][2], S[r][3]);
            else {
#pragma unroll
                for (int e = 0; e < EPL; ++e) dst[size_t(r) * DK + e] = S[r][e];
            }
        }
    }
    __syncthreads();
    for (int i = tid; i < T * WARPS; i += nthr) {
        const int t = i / WARPS, w = i % WARPS;
        const float *o = os + size_t(t) * ROWS + w * kRowsPerWarp;
        float acc = o[0] * o[0];
#pragma unroll
        for (int r = 1; r < kRowsPerWarp; ++r) acc = fmaf(o[r], o[r], acc);
        part[i] = acc;
    }
    // every CTA of the cluster has read the old conv state and published its partials
    cluster.sync();
    {
        const int first_rank = (h - kh * a.r) * a.P;        // rank of (h, part 0) in the cluster
        for (int t = tid; t < T; t += nthr) {
            float tot = 0.f;
            for (int pp = 0; pp < a.P; ++pp) {               // head-level warp order: fixed
                const float *rp = cluster.map_shared_rank(part, first_rank + pp);
                for (int w = 0; w < WARPS; ++w) tot += rp[t * WARPS + w];
            }
            rinv[t] = 1.0f / sqrtf(tot / float(DV) + a.rms_eps);
        }
    }
    __syncthreads();
    {
        Act *out = static_cast<Act *>(a.out);
        for (int i = tid; i < T * ROWS; i += nthr) {
            const int t = i / ROWS, c = i % ROWS;
            const float zz = to_f32(zs[size_t(t) * ROWS + c]);
            const float y = os[size_t(t) * ROWS + c] * rinv[t] * nw[c] * silu(zz);
            out[(size_t(s) * a.Ts + t) * size_t(Hv) * DV + size_t(h) * DV + j0 + c] = from_f32<Act>(y);
        }
    }
    for (int c = tid; c < NCH; c += nthr) {
        if (c < 2 * DK && !qk_writer) continue;
        float *dst = a.conv_state + size_t(s) * 3 * C + gchan(c);
        dst[0] = tail[c];
        dst[size_t(C)] = tail[NCH + c];
        dst[2 * size_t(C)] = tail[2 * NCH + c];
    }
    // keep this CTA's shared memory alive until every peer has read its partials
    cluster.sync();
}

template <int DK, typename Act>
cudaError_t launch_t(const VerifyArgs &a, cudaStream_t stream) {
    const int rows = a.dv / a.P;
    const int warps = rows / kRowsPerWarp;
    const Smem L(a.T, DK, rows, warps, sizeof(Act));
    auto kern = verify_kernel<DK, Act>;
    // Function attributes are set once per device (and raised when a launch needs more).
    static int smem_set[kMaxDevices] = {};
    static bool nonportable_set[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int slot = dev < kMaxDevices ? dev : kMaxDevices - 1;
    if (int(L.total) > smem_set[slot] || dev >= kMaxDevices) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(L.total));
        if (e != cudaSuccess) return e;
        smem_set[slot] = int(L.total);
    }
    const int cluster = a.r * a.P;
    if (cluster > 8 && (!nonportable_set[slot] || dev >= kMaxDevices)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        nonportable_set[slot] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.Hv * a.P, a.B, 1);
    cfg.blockDim = dim3(warps * 32, 1, 1);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

size_t verify_smem_bytes(int T, int dk, int dv, int P, int act_bytes) {
    const int rows = dv / P;
    return Smem(T, dk, rows, rows / kRowsPerWarp, act_bytes).total;
}

cudaError_t launch_verify(const VerifyArgs &a, gdn_dtype act, cudaStream_t stream) {
    const bool bf = act == GDN_BF16;
    switch (a.dk) {
        case 128: return bf ? launch_t<128, __nv_bfloat16>(a, stream) : launch_t<128, float>(a, stream);
        case 64: return bf ? launch_t<64, __nv_bfloat16>(a, stream) : launch_t<64, float>(a, stream);
        case 32: return bf ? launch_t<32, __nv_bfloat16>(a, stream) : launch_t<32, float>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
