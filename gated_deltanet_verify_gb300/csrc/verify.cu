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
//     Columns j of S (value dims) evolve independently, so a CTA owns a part
//     of them: the head's d_v/8 warps of 8 rows are dealt out in P contiguous
//     parts of floor or ceil(d_v/8 / P) warps (unequal when P does not divide
//     them; the block has the widest part's warps and a narrower part leaves
//     its last warp idle in the recurrence); only the per-head RMSNorm needs
//     all d_v.  Its partial sums are
//     exchanged through distributed shared memory inside the cluster; the
//     q/k conv channels are read by every CTA of the group, and the cluster
//     also orders their in-place conv_state rewrite after all those reads.
//   * Inside a CTA each warp owns 8 value rows j, split into row groups of
//     RPG rows served by LR lanes (LR = 16, RPG = 4 for d_k >= 64; LR = 8,
//     RPG = 2 for d_k = 32).  Lane b of a group holds S[i][j] of its RPG rows
//     for the 16-byte chunks i/4 = b + LR*m.  Per token a lane reads only its
//     own chunks of k and q (each chunk is shared by the 32/LR groups, so
//     shared-memory traffic stays low), the dot products over d_k are FMA
//     chains plus a reduce-scatter over the LR lanes (log2(LR) shuffle
//     levels, 2*RPG values), and one 16-byte store per lane writes LR*16
//     contiguous bytes of a captured row.
//   * Per token both reductions are taken on the state before the update:
//     u = g S^T k, w = beta (v - u), and the read-out S_t^T q = g S^T q +
//     (k.q) w, so a token costs one reduction phase.
//   * Reduction orders depend only on the lane layout, never on P or T: the
//     state after token t is bit-identical whatever the launch shape and
//     however many tokens follow it (the rollback contract relies on this).
//   * Conv + SiLU + L2 norm run before the recurrence with one thread per
//     (token, q|k, 16-channel chunk); a chunk's channels are interleaved
//     (4 channels every 4*chunks) so the vector loads of a warp are
//     conflict-free, and the sums of squares need three shuffle levels.
//   * The RMSNorm partials travel by st.async into the peers' shared memory
//     right after the recurrence (before the conv-window capture is written),
//     completing a transaction-counted mbarrier there; no release fence has
//     to wait behind the capture stores still in flight.  The one cluster
//     barrier arrives right after the loads and completes after the
//     recurrence: it orders every CTA's read of the old conv state before the
//     in-place rewrite, and publishes the initialised mbarriers before any
//     peer writes to them.
//   * Every wait is bounded; a wait that gives up writes GDN_ERR_TIMEOUT to
//     the caller's status word instead of hanging.
//   * The batch's activations arrive as TMA boxes, one per segment (q and k
//     of the key head, this CTA's v and z rows, T tokens each) into their own
//     128-byte aligned areas of shared memory, completing on an mbarrier; the
//     state rows go straight into registers; the pending tokens of a lazy
//     verify and the small parameter / conv-state rows come by 16-byte async
//     copies.
//   * Programmatic dependent launch: the kernel waits on its predecessor only
//     right before its first global read, so its launch overlaps the tail of
//     the previous kernel in the stream; meanwhile it prefetches its state
//     rows and activation segments into L2 (a prefetch returns nothing to the
//     SM, so lines the previous kernel is still writing stay coherent).
//   * A checked build (-DGDN_CHECKED=1) tests every global access against its
//     buffer first (check.cuh); the ordinary build compiles the tests away.
//
// Modes (one template instance each)
//   kChain  the (K+1)-token chain: outputs, optional captures, state and conv
//           state advanced past all T tokens.
//   kTree   a draft tree: each token runs from its parent's state; captures
//           per node, state and conv state left as they were.
//   kLazy   outputs of the batch only, so the state stays the one before it
//           (lazy capture).  With a pending batch (prev buffers and trims) the
//           launch first re-runs that batch's accepted tokens from the stored
//           state, writes the state and conv state after them, and continues
//           from there into the new batch: the commit of one step rides in the
//           verify of the next.
//   kRolled the chain verify started from the state a rollback of the
//           previous batch would leave: per slot, the captured state
//           cap[T-1-trim] and the window rows after that token, read from the
//           previous verify's capture buffers (which this launch then
//           overwrites with its own captures), so a step is one launch.
//   kCommit the lazy counterpart of a rollback: per slot, re-runs the first
//           T - trim[s] tokens from the state before the batch and writes the
//           state and conv state after them; no z, no outputs.  Since the
//           state after token t does not depend on the tokens that follow
//           it, this is bit-identical to a chain verify with capture followed
//           by a rollback with the same trims.
#include "internal.cuh"

#include <cuda_bf16.h>

namespace gdn {
namespace {

constexpr int kRowsPerWarp = 8;
constexpr int kMaxWarps = 8;
constexpr int kMaxThreads = 32 * kMaxWarps;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kSpinLimit = 1 << 22;     // try_wait rounds before a wait gives up

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// four consecutive values as fp32
__device__ __forceinline__ float4 load4(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *p) {
    const uint2 u = *reinterpret_cast<const uint2 *>(p);
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&u.y));
    return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void store4(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16 *p, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    uint2 u;
    u.x = *reinterpret_cast<unsigned *>(&a);
    u.y = *reinterpret_cast<unsigned *>(&b);
    *reinterpret_cast<uint2 *>(p) = u;
}

__device__ __forceinline__ float silu(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

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
    asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};\n" ::"l"(p), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

// The state is rewritten by this kernel, so it is read through the coherent
// path (no .nc), only without allocating in L1.
__device__ __forceinline__ float4 ld_na4(const float *p) {
    float4 v;
    asm volatile("ld.global.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];\n"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

// Warm L2 with the line holding p.  Nothing comes back to the SM, so this may
// run before the grid-dependency wait: a line the previous kernel is still
// writing stays coherent in L2, and the real loads come after the wait.
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p));
}
__device__ __forceinline__ int ld_relaxed_s32(const int32_t *p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n\t}\n" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}\n"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_try_wait_cta(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}\n"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}
// 2-D tile of a tensor map -> own shared memory, completion counted in bytes on an mbarrier
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
// Bounded waits: after kSpinLimit rounds the wait gives up and reports.
__device__ __forceinline__ void report_timeout(int *status) {
    if (status) atomicCAS(status, int(GDN_OK), int(GDN_ERR_TIMEOUT));
}
__device__ __forceinline__ void mbar_wait_cluster(uint32_t bar, uint32_t parity, int *status) {
    for (int i = 0; i < kSpinLimit; ++i)
        if (mbar_try_wait_cluster(bar, parity)) return;
    report_timeout(status);
}
__device__ __forceinline__ void mbar_wait_cta(uint32_t bar, uint32_t parity, int *status) {
    for (int i = 0; i < kSpinLimit; ++i)
        if (mbar_try_wait_cta(bar, parity)) return;
    report_timeout(status);
}
__device__ __forceinline__ void fence_mbarrier_init_cluster() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
// shared::cluster address of `local` in the CTA of cluster rank `rank`
__device__ __forceinline__ uint32_t map_cluster(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
// 4-byte store into a peer CTA's shared memory that completes 4 bytes of its mbarrier's transaction
__device__ __forceinline__ void st_async_f32(uint32_t remote_addr, float v, uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];\n" ::"r"(remote_addr),
                 "r"(__float_as_uint(v)), "r"(remote_bar)
                 : "memory");
}
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

// Shared-memory carve-up; identical on host and device.  The raw q, k and v segments of the window each
// have an area for the batch's Tb tokens, written by one TMA box, and in front of it an area for the
// Tm - Tb pending tokens of a lazy verify (16-byte async copies); TMA destinations start on 128 bytes.
struct Smem {
    int NCH;
    size_t xq_p, xq_c, xk_p, xk_c, xv_p, xv_c, zs, cw, cs, nw, ys, os, gs, bs, kqs, rinv, allp, redbar, loadbar, arow,
        total;
    // rows: the widest part's rows (the stride of the per-CTA row tables, the TMA box width); head_warps: the
    // warps of a whole head (the RMSNorm partials of every part land in every CTA of the head)
    __host__ __device__ Smem(int Tm, int Tb, int dk, int rows, int head_warps, int act_bytes, bool tree)
        : NCH(2 * dk + rows) {
        size_t off = 0;
        auto take = [&](size_t bytes) {
            size_t o = off;
            off += (bytes + 15) & ~size_t(15);
            return o;
        };
        auto take128 = [&](size_t bytes) {
            off = (off + 127) & ~size_t(127);
            return take(bytes);
        };
        const size_t pend = size_t(Tm - Tb), ab = size_t(act_bytes);
        xq_p = take128(pend * dk * ab);             // raw q of the pending tokens
        xq_c = take128(size_t(Tb) * dk * ab);       // raw q of the batch (TMA)
        xk_p = take128(pend * dk * ab);
        xk_c = take128(size_t(Tb) * dk * ab);
        xv_p = take128(pend * rows * ab);           // raw v of own rows
        xv_c = take128(size_t(Tb) * rows * ab);
        zs = take128(size_t(Tb) * rows * ab);       // raw z for own rows (TMA)
        cw = take(size_t(4) * NCH * 4);             // conv weights
        cs = take(size_t(3) * NCH * 4);             // old conv state
        nw = take(size_t(rows) * 4);                // norm weight for own rows
        ys = take(size_t(Tm) * NCH * 4);            // post conv+SiLU (q, k normalised)
        os = take(size_t(Tm) * rows * 4);           // o before the RMSNorm
        gs = take(size_t(Tm) * 4);
        bs = take(size_t(Tm) * 4);
        kqs = take(size_t(Tm) * 4);
        rinv = take(size_t(Tm) * 4);
        allp = take(size_t(Tm) * head_warps * 4);   // per-warp sums of o^2 of the whole head
        redbar = take(8);                           // all RMSNorm partials of the head arrived
        loadbar = take(8);                          // the batch's activation boxes landed
        arow = take(tree ? size_t(Tm) * 5 * 4 : 0); // tree: parent and the window row of each conv tap
        total = off;
    }
};

// MINB: resident CTAs per SM the register budget is sized for.  Two everywhere; three (80 registers, no
// spills) for chain and rolled launches with more CTAs than two per SM, where a third resident CTA keeps
// the SM's stores going while another loads, convolves or normalises (a 48-layer x 8-slot stack layer
// 77.7 -> 75.2 us).  A launch that fits at two per SM keeps the roomier build (one slot: 17.0 us against
// 18.3 us under the tighter budget); so does the lazy mode, slower under it at every size.
template <int DK, typename Act, int MODE, int MINB>
__global__ void __launch_bounds__(kMaxThreads, MINB) verify_kernel(const __grid_constant__ VerifyArgs a) {
    static_assert(DK == 32 || DK == 64 || DK == 128, "d_k must be 32, 64 or 128");
    constexpr bool TREE = MODE == kTree, LAZY = MODE == kLazy, COMMIT = MODE == kCommit, ROLLED = MODE == kRolled;
    constexpr int LR = DK >= 64 ? 16 : 8;          // lanes per row group
    constexpr int NG = 32 / LR;                    // row groups per warp
    constexpr int RPG = kRowsPerWarp / NG;         // rows per group
    constexpr int NV = 2 * RPG;                    // k- and q-dot values per lane (== LR / 2)
    constexpr int NCL = DK / (4 * LR);             // 16-byte chunks per lane per row
    static_assert(NV == LR / 2, "lane layout");

    extern __shared__ __align__(128) unsigned char smem_raw[];   // no static shared memory: the base is aligned

    const int tid = threadIdx.x, nthr = blockDim.x;
    const int lane = tid & 31, wid = tid >> 5;
    const int WARPS = nthr >> 5;                               // warps of the widest part (the block)
    const int ROWS = WARPS * kRowsPerWarp;                     // its rows: the stride of the row tables
    const int T = a.T, Hv = a.Hv, Hk = a.Hk, DV = a.dv, C = a.C, P = a.P;
    const int HW = DV / kRowsPerWarp;                          // warps of a whole head
    const int s = blockIdx.y;
    const int h = blockIdx.x / P, p = blockIdx.x % P;
    const int kh = h / a.r;
    const int w0 = (p * HW) / P;                               // this part: head warps w0 .. w0 + MYW - 1
    const int MYW = ((p + 1) * HW) / P - w0;
    const int MY_ROWS = MYW * kRowsPerWarp;
    const bool active = wid < MYW;                             // warp-uniform: owns rows in the recurrence
    const int j0 = w0 * kRowsPerWarp;                          // first value row of this CTA
    // the q/k conv channels of the key head are read by every CTA of the cluster (its r value heads x P
    // parts); their stores (conv window or per-node capture, conv state) are dealt out in equal runs of
    // 4-channel units, CTA (h mod r, p) taking its run besides its own v channels
    const int crank = (h % a.r) * P + p, csize = a.r * P;
    const int q_u0 = (crank * (DK / 2)) / csize, q_nu = ((crank + 1) * (DK / 2)) / csize - q_u0;

    const Smem L(LAZY ? a.Tm : T, T, DK, ROWS, HW, sizeof(Act), TREE);   // only a lazy launch holds 2T
    Act *zs = reinterpret_cast<Act *>(smem_raw + L.zs);
    float *cw = reinterpret_cast<float *>(smem_raw + L.cw);
    float *cs = reinterpret_cast<float *>(smem_raw + L.cs);
    float *nw = reinterpret_cast<float *>(smem_raw + L.nw);
    float *ys = reinterpret_cast<float *>(smem_raw + L.ys);
    float *os = reinterpret_cast<float *>(smem_raw + L.os);
    float *gs = reinterpret_cast<float *>(smem_raw + L.gs);
    float *bs = reinterpret_cast<float *>(smem_raw + L.bs);
    float *kqs = reinterpret_cast<float *>(smem_raw + L.kqs);
    float *rinv = reinterpret_cast<float *>(smem_raw + L.rinv);
    float *allp = reinterpret_cast<float *>(smem_raw + L.allp);
    const uint32_t redbar = smem_u32(smem_raw + L.redbar);
    const uint32_t loadbar = smem_u32(smem_raw + L.loadbar);
    int *tpar = reinterpret_cast<int *>(smem_raw + L.arow);     // tree: [T] parents, then [T][4] window rows
    int *trow = tpar + T;
    // a checked build tests each global access against its buffer first (compiled away otherwise)
    auto chk = [&](const void *ptr, size_t bytes, const void *base, size_t ext) -> bool {
        return in_bounds(ptr, bytes, base, ext, a.d_status);
    };
    const int NCH = L.NCH;                      // channel stride of the conv tables (widest part)
    const int n_own4 = q_nu + MY_ROWS / 4;      // 4-channel units this CTA stores: its q/k run, its v rows
    auto own_chan = [&](int u) -> int { return u < q_nu ? 4 * (q_u0 + u) : 2 * DK + 4 * (u - q_nu); };

    // local channel c -> global conv channel
    auto gchan = [&](int c) -> int {
        if (c < DK) return kh * DK + c;                                  // q of key head kh
        if (c < 2 * DK) return Hk * DK + kh * DK + (c - DK);            // k of key head kh
        return 2 * Hk * DK + h * DV + j0 + (c - 2 * DK);                 // v rows of this CTA
    };
    int n_prev = 0;                             // lazy: the pending batch's accepted tokens, run first
    // raw input of token t (0..TT-1) at local channel c: the q, k or v area, pending or batch part
    auto xsrc = [&](int t, int c) -> const Act * {
        const bool pend = t < n_prev;
        const size_t r = size_t(pend ? t : t - n_prev);
        if (c < DK) return reinterpret_cast<const Act *>(smem_raw + (pend ? L.xq_p : L.xq_c)) + r * DK + c;
        if (c < 2 * DK) return reinterpret_cast<const Act *>(smem_raw + (pend ? L.xk_p : L.xk_c)) + r * DK + (c - DK);
        return reinterpret_cast<const Act *>(smem_raw + (pend ? L.xv_p : L.xv_c)) + r * ROWS + (c - 2 * DK);
    };
    // window row rho (0..TT+2) of local channel c: old conv state, then the tokens
    auto win = [&](int rho, int c) -> float { return rho < 3 ? cs[rho * NCH + c] : to_f32(*xsrc(rho - 3, c)); };
    auto win4 = [&](int rho, int c) -> float4 {
        return rho < 3 ? load4(cs + rho * NCH + c) : load4(xsrc(rho - 3, c));
    };

    if (smem_u32(smem_raw) & 127u) {            // TMA destinations need 128-byte alignment (uniform: every CTA)
        if (tid == 0 && a.d_status) atomicCAS(a.d_status, int(GDN_OK), int(GDN_ERR_LAUNCH));
        return;
    }
    if (tid == 0) {
        mbar_init(redbar, 1);
        mbar_init(loadbar, 1);
        fence_mbarrier_init_cluster();
        // the single arrival; the phase completes once every partial of the head has landed
        mbar_arrive_expect_tx(redbar, uint32_t(T * HW * 4));
    }
    {
        // while the previous kernel finishes: L2 prefetch of this CTA's state rows (for a rolled verify the
        // captured ones, at a trim read early -- possibly stale, only an address) and of its activation
        // segments (q, k of the key head, its own v and z rows), one 128-byte line per prefetch
        constexpr int kLine = 128;
        const float *st = a.state + ((size_t(s) * Hv + h) * DV + j0) * DK;
        const float *st_base = ROLLED ? a.cap_state : a.state;
        const size_t st_ext = ROLLED ? a.ext_cap_state : a.ext_state;
        if constexpr (ROLLED) {
            int tr = a.trim && chk(a.trim + s, 4, a.trim, a.ext_trim) ? ld_relaxed_s32(a.trim + s) : 0;
            tr = tr < 0 ? 0 : (tr >= T ? T - 1 : tr);
            st = a.cap_state + ((size_t(s) * T + (T - 1 - tr)) * Hv + h) * DV * DK + size_t(j0) * DK;
        }
        const int st_lines = MY_ROWS * DK * 4 / kLine;
        for (int i = tid; i < st_lines; i += nthr) {
            const char *line = reinterpret_cast<const char *>(st) + size_t(i) * kLine;
            if (chk(line, 1, st_base, st_ext)) prefetch_l2(line);
        }
        constexpr int qk_lines = DK * int(sizeof(Act)) / kLine;          // 0 when a segment is below a line
        const int seg = qk_lines > 0 ? 2 * qk_lines + 2 : 4;
        const Act *qkv = static_cast<const Act *>(a.qkv);
        const Act *zp = static_cast<const Act *>(a.z);
        for (int i = tid; i < T * seg; i += nthr) {
            const int t = i / seg, w = i % seg;
            const size_t rw = size_t(s) * a.Ts + t;
            const Act *p;
            bool ok;
            if (w < seg - 2) {
                const int half = qk_lines > 0 ? qk_lines : 1;
                const int part = w / half, l = w % half;
                p = qkv + rw * a.ld_qkv + size_t(part ? Hk + kh : kh) * DK + size_t(l) * (kLine / sizeof(Act));
                ok = chk(p, 1, qkv, a.ext_qkv);
            } else if (w == seg - 2) {
                p = qkv + rw * a.ld_qkv + size_t(2 * Hk) * DK + size_t(h) * DV + j0;
                ok = chk(p, 1, qkv, a.ext_qkv);
            } else {
                if (COMMIT) continue;
                p = zp + rw * a.ld_z + size_t(h) * DV + j0;
                ok = chk(p, 1, zp, a.ext_z);
            }
            if (ok) prefetch_l2(p);
        }
    }
    // everything below may read what the previous kernel in the stream wrote
    grid_dependency_wait();
    int TT = T;                                 // tokens run for this slot
    int src_tok = 0;                            // rolled: the previous batch's accepted token
    if constexpr (COMMIT || LAZY || ROLLED) {
        if (a.trim) {
            // uniform over the cluster: one slot (an unreadable trim counts as out of range)
            const int tr = chk(a.trim + s, 4, a.trim, a.ext_trim) ? a.trim[s] : -1;
            if (tr < 0 || tr >= T) {            // reported; the slot is left untouched
                if (tid == 0 && blockIdx.x == 0 && a.d_status)
                    atomicCAS(a.d_status, int(GDN_OK), int(GDN_ERR_TRIM_RANGE));
                return;
            }
            if constexpr (COMMIT) TT = T - tr;
            else if constexpr (ROLLED) src_tok = T - 1 - tr;
            else {
                n_prev = T - tr;
                TT = n_prev + T;
            }
        }
    }

    // ---------------------------------------------------------------- loads
    // (1) this warp's state rows, straight into registers (recurrence lane layout)
    const int grp = lane / LR, b = lane % LR;
    const int row0 = wid * kRowsPerWarp + grp * RPG;           // first row (within CTA) of this group
    const int my_kind = (b & NV) ? 1 : 0;                       // after the reduce-scatter
    const int my_rho = (b >> 1) & (RPG - 1);
    float S[RPG][NCL][4];
    if (!active) {
#pragma unroll
        for (int rho = 0; rho < RPG; ++rho)
#pragma unroll
            for (int m = 0; m < NCL; ++m) S[rho][m][0] = S[rho][m][1] = S[rho][m][2] = S[rho][m][3] = 0.f;
    } else {
        const float *src = ROLLED ? a.cap_state + ((size_t(s) * T + src_tok) * Hv + h) * DV * DK +
                                        size_t(j0 + row0) * DK + 4 * b
                                  : a.state + ((size_t(s) * Hv + h) * DV + j0 + row0) * DK + 4 * b;
#pragma unroll
        for (int rho = 0; rho < RPG; ++rho)
#pragma unroll
            for (int m = 0; m < NCL; ++m) {
                const float *q = src + size_t(rho) * DK + 4 * LR * m;
                const float4 v = chk(q, 16, ROLLED ? a.cap_state : a.state, ROLLED ? a.ext_cap_state : a.ext_state)
                                     ? ld_na4(q) : make_float4(0.f, 0.f, 0.f, 0.f);
                S[rho][m][0] = v.x; S[rho][m][1] = v.y; S[rho][m][2] = v.z; S[rho][m][3] = v.w;
            }
    }
    // (2) the batch's activations: one TMA box per segment (q and k of the key head, this CTA's v and z
    // rows, T tokens each), completing on loadbar; the pending tokens of a lazy verify, the conv weights /
    // state and the norm weight: 16-byte async copies
    if (tid == 0) {
        const uint32_t seg = uint32_t(T) * sizeof(Act);
        mbar_arrive_expect_tx(loadbar, seg * (2 * DK + ROWS + (COMMIT ? 0 : ROWS)));
        const int y = s * a.Ts;
        tma_load_2d(smem_u32(smem_raw + L.xq_c), &a.qk_map, kh * DK, y, loadbar);
        tma_load_2d(smem_u32(smem_raw + L.xk_c), &a.qk_map, (Hk + kh) * DK, y, loadbar);
        tma_load_2d(smem_u32(smem_raw + L.xv_c), &a.v_map, 2 * Hk * DK + h * DV + j0, y, loadbar);
        if constexpr (!COMMIT) tma_load_2d(smem_u32(smem_raw + L.zs), &a.z_map, h * DV + j0, y, loadbar);
    }
    {
        constexpr int kPer16 = 16 / sizeof(Act);
        const int vq = DK / kPer16, vv = MY_ROWS / kPer16;  // 16-byte vectors per segment
        const int per_t = 2 * vq + vv;                      // q, k, v of a pending token
        const Act *qkv = static_cast<const Act *>(a.qkv_prev);
        for (int i = tid; i < n_prev * per_t; i += nthr) {
            const int t = i / per_t, w = i % per_t;
            const size_t rw = size_t(s) * a.Ts + t;
            const Act *src;
            Act *dst;
            if (w < vq) {
                src = qkv + rw * a.ld_qkv + size_t(kh) * DK + w * kPer16;
                dst = reinterpret_cast<Act *>(smem_raw + L.xq_p) + size_t(t) * DK + w * kPer16;
            } else if (w < 2 * vq) {
                src = qkv + rw * a.ld_qkv + size_t(Hk + kh) * DK + (w - vq) * kPer16;
                dst = reinterpret_cast<Act *>(smem_raw + L.xk_p) + size_t(t) * DK + (w - vq) * kPer16;
            } else {
                src = qkv + rw * a.ld_qkv + size_t(2 * Hk) * DK + size_t(h) * DV + j0 + (w - 2 * vq) * kPer16;
                dst = reinterpret_cast<Act *>(smem_raw + L.xv_p) + size_t(t) * ROWS + (w - 2 * vq) * kPer16;
            }
            if (chk(src, 16, qkv, a.ext_qkv)) cp_async16(dst, src);
        }
        // conv weights (4 rows) and old conv state (3 rows), per segment in float4s
        const int fq = DK / 4, fv = MY_ROWS / 4, per_row = 2 * fq + fv;
        for (int i = tid; i < 7 * per_row; i += nthr) {
            const int rrow = i / per_row, w = i % per_row;
            const int c0 = w < fq ? w * 4 : (w < 2 * fq ? DK + (w - fq) * 4 : 2 * DK + (w - 2 * fq) * 4);
            const int g0 = gchan(c0);
            if (rrow < 4) {
                const float *q = a.conv_w + size_t(rrow) * C + g0;
                if (chk(q, 16, a.conv_w, a.ext_conv_w)) cp_async16(cw + rrow * NCH + c0, q);
            } else if (ROLLED) {    // window rows after the accepted token of the previous batch
                const float *q = a.cap_conv + (size_t(s) * (3 + T) + src_tok + 1 + (rrow - 4)) * C + g0;
                if (chk(q, 16, a.cap_conv, a.ext_cap_conv)) cp_async16(cs + (rrow - 4) * NCH + c0, q);
            } else {
                const float *q = a.conv_state + (size_t(s) * 3 + (rrow - 4)) * C + g0;
                if (chk(q, 16, a.conv_state, a.ext_conv_state)) cp_async16(cs + (rrow - 4) * NCH + c0, q);
            }
        }
        if constexpr (!COMMIT)
            for (int i = tid; i < MY_ROWS / 4; i += nthr)
                if (chk(a.norm_w + j0 + i * 4, 16, a.norm_w, a.ext_norm_w)) cp_async16(nw + i * 4, a.norm_w + j0 + i * 4);
    }
    // (3) gates for this head, one token per thread
    for (int t = tid; t < TT; t += nthr) {
        const bool pend = t < n_prev;
        const size_t idx = (size_t(s) * a.Ts + (pend ? t : t - n_prev)) * a.ld_ab + h;
        const Act *ap = static_cast<const Act *>(pend ? a.alpha_prev : a.alpha) + idx;
        const Act *bp = static_cast<const Act *>(pend ? a.beta_prev : a.beta_raw) + idx;
        const float al = chk(ap, sizeof(Act), ap - idx, a.ext_ab) ? to_f32(*ap) : 0.f;
        const float br = chk(bp, sizeof(Act), bp - idx, a.ext_ab) ? to_f32(*bp) : 0.f;
        const float dtb = chk(a.dt_bias + h, 4, a.dt_bias, a.ext_head) ? __ldg(a.dt_bias + h) : 0.f;
        const float alg = chk(a.A_log + h, 4, a.A_log, a.ext_head) ? __ldg(a.A_log + h) : 0.f;
        const float x = al + dtb;
        const float sp = x > 20.0f ? x : log1pf(expf(x));               // softplus
        gs[t] = expf(-expf(alg) * sp);
        bs[t] = 1.0f / (1.0f + expf(-br));
        if constexpr (TREE) {
            int pt = chk(a.parent + size_t(s) * T + t, 4, a.parent, a.ext_parent) ? __ldg(a.parent + size_t(s) * T + t)
                                                                                  : -1;
            if (pt < -1 || pt >= t) {                   // not a tree in token order: reported, root used
                if (a.d_status) atomicCAS(a.d_status, int(GDN_OK), int(GDN_ERR_TREE));
                pt = -1;
            }
            tpar[t] = pt;
        }
    }
    cp_async_wait_all();
    mbar_wait_cta(loadbar, 0, a.d_status);      // the batch's activation boxes
    __syncthreads();
    if (a.l2_next && tid == 0) {
        // this CTA's share of the region the next launch streams, into L2 while this launch runs (bulk
        // prefetches return nothing to the SM and are not waited for); 16-byte aligned shares of <= 64 KB
        const size_t n_cta = size_t(gridDim.x) * gridDim.y, idx = size_t(blockIdx.y) * gridDim.x + blockIdx.x;
        const size_t share = ((a.l2_next_bytes + n_cta - 1) / n_cta + 15) & ~size_t(15);
        const size_t beg = idx * share, end = beg + share < a.l2_next_bytes ? beg + share : a.l2_next_bytes;
        const char *base = static_cast<const char *>(a.l2_next);
        for (size_t o = beg; o < end; o += 65536) {
            const uint32_t n = uint32_t(end - o < 65536 ? end - o : 65536);
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(base + o), "r"(n) : "memory");
        }
    }
    // cluster phase 1: this CTA has read the old conv state (the copies above have
    // landed) and initialised its mbarrier (published by fence.mbarrier_init)
    cluster_arrive_relaxed();
    if constexpr (TREE) {
        // window row of each conv tap: tap 3 is the token, taps 2, 1, 0 its nearest ancestors; past the
        // root the ancestors continue into the old conv state (node -1 = row 2, -2 = row 1, -3 = row 0)
        for (int t = tid; t < T; t += nthr) {
            int n = t;
            for (int j = 3; j >= 0; --j) {
                trow[t * 4 + j] = 3 + n;
                n = n >= 0 ? tpar[n] : n - 1;
            }
        }
        __syncthreads();
    }
    // window row of conv tap j for token t
    auto tap_row = [&](int t, int j) -> int {
        if constexpr (TREE) return trow[t * 4 + j];
        else return t + j;
    };

    // ------------------------------------ conv + SiLU, q/k L2 norm, k.q per token
    {
        constexpr int QC = DK / 16;                 // 16-channel chunks per q (or k) vector
        constexpr int PER_T = 2 * QC;               // q and k items per token (divides 32)
        const int n_items = TT * PER_T;
        const int n_round = (n_items + 31) & ~31;   // whole warps, so every lane joins the shuffles
        for (int base = wid * 32; base < n_round; base += nthr) {
            const int i = base + lane;
            const bool valid = i < n_items;
            const int t = valid ? i / PER_T : 0, part = (i % PER_T) / QC, c = i % QC;
            float y[4][4];
            float ss = 0.f;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const int ch = part * DK + 4 * (c + QC * m);
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                if (valid) {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float4 w4 = load4(cw + j * NCH + ch), x4 = win4(tap_row(t, j), ch);
                        if (j == 0) acc = make_float4(w4.x * x4.x, w4.y * x4.y, w4.z * x4.z, w4.w * x4.w);
                        else acc = make_float4(fmaf(w4.x, x4.x, acc.x), fmaf(w4.y, x4.y, acc.y),
                                               fmaf(w4.z, x4.z, acc.z), fmaf(w4.w, x4.w, acc.w));
                    }
                }
                y[m][0] = silu(acc.x); y[m][1] = silu(acc.y); y[m][2] = silu(acc.z); y[m][3] = silu(acc.w);
#pragma unroll
                for (int e = 0; e < 4; ++e) ss = fmaf(y[m][e], y[m][e], ss);
            }
#pragma unroll
            for (int msk = 1; msk < QC; msk <<= 1) ss += __shfl_xor_sync(kFull, ss, msk);
            const float inv = 1.0f / sqrtf(ss + a.l2_eps);
            float *yt = ys + size_t(t) * NCH;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
#pragma unroll
                for (int e = 0; e < 4; ++e) y[m][e] *= inv;
                if (valid) store4(yt + part * DK + 4 * (c + QC * m), make_float4(y[m][0], y[m][1], y[m][2], y[m][3]));
            }
            __syncwarp();
            // k.q of the token: the q threads read k^ back for their channels
            float kq = 0.f;
            if (valid && part == 0) {
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    const float4 k4 = load4(yt + DK + 4 * (c + QC * m));
                    kq = fmaf(y[m][0], k4.x, kq); kq = fmaf(y[m][1], k4.y, kq);
                    kq = fmaf(y[m][2], k4.z, kq); kq = fmaf(y[m][3], k4.w, kq);
                }
            }
#pragma unroll
            for (int msk = 1; msk < QC; msk <<= 1) kq += __shfl_xor_sync(kFull, kq, msk);
            if (valid && part == 0 && c == 0) kqs[t] = kq;
            __syncwarp();
        }
    }
    // v: four channels of one token per item
    for (int i = tid; i < TT * (MY_ROWS / 4); i += nthr) {
        const int t = i / (MY_ROWS / 4), c = 2 * DK + 4 * (i % (MY_ROWS / 4));
        float4 acc;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float4 w4 = load4(cw + j * NCH + c), x4 = win4(tap_row(t, j), c);
            if (j == 0) acc = make_float4(w4.x * x4.x, w4.y * x4.y, w4.z * x4.z, w4.w * x4.w);
            else acc = make_float4(fmaf(w4.x, x4.x, acc.x), fmaf(w4.y, x4.y, acc.y), fmaf(w4.z, x4.z, acc.z),
                                   fmaf(w4.w, x4.w, acc.w));
        }
        store4(ys + size_t(t) * NCH + c, make_float4(silu(acc.x), silu(acc.y), silu(acc.z), silu(acc.w)));
    }
    __syncthreads();

    {
        // ------------------------------------------------------------ recurrence
        const bool capture = a.cap_state != nullptr;
        float *cap_row = capture ? a.cap_state + (size_t(h) * DV + j0 + row0) * DK + 4 * b : nullptr;
        const size_t cap_token_stride = size_t(Hv) * DV * DK;
        const float q_scale = a.q_scale;

        // tree: this thread's own rows of a parent's state -- the parent's capture, or the state before
        // the batch -- for a token whose parent is not the token before it
        auto parent_rows = [&](int pt, float (&D)[RPG][NCL][4]) {
            const float *src = pt < 0 ? a.state + ((size_t(s) * Hv + h) * DV + j0 + row0) * DK + 4 * b
                                      : cap_row + (size_t(s) * T + pt) * cap_token_stride;
            const float *sbase = pt < 0 ? a.state : a.cap_state;
            const size_t sext = pt < 0 ? a.ext_state : a.ext_cap_state;
#pragma unroll
            for (int rho = 0; rho < RPG; ++rho)
#pragma unroll
                for (int m = 0; m < NCL; ++m) {
                    const float *q = src + size_t(rho) * DK + 4 * LR * m;
                    const float4 v = chk(q, 16, sbase, sext) ? ld_na4(q) : make_float4(0.f, 0.f, 0.f, 0.f);
                    D[rho][m][0] = v.x; D[rho][m][1] = v.y; D[rho][m][2] = v.z; D[rho][m][3] = v.w;
                }
        };
        // the next token's parent rows, requested one token ahead (the parent is then at most the token
        // before this one, so this thread stored its capture in an earlier iteration; token 0's parent is
        // the state before the batch, already in registers)
        float Sn[TREE ? RPG : 1][TREE ? NCL : 1][4];

        for (int t = 0; t < TT && active; ++t) {
            if constexpr (TREE) {
                // the token runs from its parent's state: already in registers when the parent is t-1,
                // else the rows requested during the previous token
                if (tpar[t] != t - 1) {
#pragma unroll
                    for (int rho = 0; rho < RPG; ++rho)
#pragma unroll
                        for (int m = 0; m < NCL; ++m)
#pragma unroll
                            for (int e = 0; e < 4; ++e) S[rho][m][e] = Sn[rho][m][e];
                }
                if (t + 1 < TT && tpar[t + 1] != t) parent_rows(tpar[t + 1], Sn);
            }
            const float *yt = ys + size_t(t) * NCH;
            const float g = gs[t], beta = bs[t], kq = kqs[t];
            float kk[NCL][4], qq[NCL][4];
#pragma unroll
            for (int m = 0; m < NCL; ++m) {
                const float4 k4 = load4(yt + DK + 4 * (b + LR * m));
                const float4 q4 = load4(yt + 4 * (b + LR * m));
                kk[m][0] = k4.x; kk[m][1] = k4.y; kk[m][2] = k4.z; kk[m][3] = k4.w;
                qq[m][0] = q4.x; qq[m][1] = q4.y; qq[m][2] = q4.z; qq[m][3] = q4.w;
            }
            const float vj = yt[2 * DK + row0 + my_rho];
            // partial dot products of this lane's chunks: vals[kind * RPG + rho]
            float vals[NV];
#pragma unroll
            for (int rho = 0; rho < RPG; ++rho) {
                float dk_ = S[rho][0][0] * kk[0][0], dq_ = S[rho][0][0] * qq[0][0];
#pragma unroll
                for (int m = 0; m < NCL; ++m)
#pragma unroll
                    for (int e = (m == 0 ? 1 : 0); e < 4; ++e) {
                        dk_ = fmaf(S[rho][m][e], kk[m][e], dk_);
                        dq_ = fmaf(S[rho][m][e], qq[m][e], dq_);
                    }
                vals[rho] = dk_;
                vals[RPG + rho] = dq_;
            }
            // reduce-scatter over the LR lanes of the group: masks NV, NV/2, ..., 2 halve
            // the value set; mask 1 completes the sum (lane pairs hold equal values)
#pragma unroll
            for (int half = NV / 2, msk = NV; half >= 1; half >>= 1, msk >>= 1) {
                const bool up = (b & msk) != 0;
#pragma unroll
                for (int i = 0; i < half; ++i) {
                    const float keep = up ? vals[i + half] : vals[i];
                    const float send = up ? vals[i] : vals[i + half];
                    vals[i] = keep + __shfl_xor_sync(kFull, send, msk);
                }
            }
            const float mine = vals[0] + __shfl_xor_sync(kFull, vals[0], 1);
            const float other = __shfl_xor_sync(kFull, mine, NV);
            const float kd = my_kind ? other : mine;       // (S^T k)_j of row my_rho
            const float qd = my_kind ? mine : other;       // (S^T q)_j of row my_rho
            const float w = beta * (vj - g * kd);           // beta (v - (g S)^T k)
            if (!COMMIT && t >= n_prev && my_kind == 0 && (b & 1) == 0)
                os[size_t(t - n_prev) * ROWS + row0 + my_rho] = q_scale * fmaf(g, qd, kq * w);
            // S <- g S + k w^T for the group's rows
#pragma unroll
            for (int rho = 0; rho < RPG; ++rho) {
                const float wr = __shfl_sync(kFull, w, grp * LR + 2 * rho);
#pragma unroll
                for (int m = 0; m < NCL; ++m)
#pragma unroll
                    for (int e = 0; e < 4; ++e) S[rho][m][e] = fmaf(kk[m][e], wr, g * S[rho][m][e]);
            }
            if (LAZY && t + 1 == n_prev) {
                // the pending batch is committed: its state becomes the stored one (own rows only)
                float *dst = a.state + ((size_t(s) * Hv + h) * DV + j0 + row0) * DK + 4 * b;
#pragma unroll
                for (int rho = 0; rho < RPG; ++rho)
#pragma unroll
                    for (int m = 0; m < NCL; ++m) {
                        float *q = dst + size_t(rho) * DK + 4 * LR * m;
                        if (chk(q, 16, a.state, a.ext_state))
                            store4(q, make_float4(S[rho][m][0], S[rho][m][1], S[rho][m][2], S[rho][m][3]));
                    }
            }
            if (capture) {
                float *dst = cap_row + (size_t(s) * T + t) * cap_token_stride;
#pragma unroll
                for (int rho = 0; rho < RPG; ++rho)
#pragma unroll
                    for (int m = 0; m < NCL; ++m) {
                        float *q = dst + size_t(rho) * DK + 4 * LR * m;
                        if (chk(q, 16, a.cap_state, a.ext_cap_state))
                            st_stream4(q, S[rho][m][0], S[rho][m][1], S[rho][m][2], S[rho][m][3]);
                    }
            }
        }
        // the next kernel in the stream may start launching (it waits for this grid's completion itself)
        grid_launch_dependents();
        if constexpr (TREE) {
            // conv state after each node: the window rows of its taps 1, 2, 3, channels this CTA owns (a large
            // store burst, measured to be better issued before the RMSNorm exchange)
            const int n4 = n_own4;
            float *base = a.cap_conv + size_t(s) * T * 3 * C;
            for (int i = tid; i < T * 3 * n4; i += nthr) {
                const int t = i / (3 * n4), rr = (i / n4) % 3, c = own_chan(i % n4);
                float *q = base + (size_t(t) * 3 + rr) * C + gchan(c);
                if (chk(q, 16, a.cap_conv, a.ext_cap_conv)) store4(q, win4(trow[t * 4 + 1 + rr], c));
            }
        }
        __syncwarp();
        cluster_wait_acquire();            // phase 1: every peer's mbarrier is initialised, every old conv row read
        if (!COMMIT && active) {
            // this warp's sums of o^2 per token, sent to the allp table of every CTA of this head
            const int first_rank = (h - kh * a.r) * P;
            const uint32_t allp_local = smem_u32(allp);
            for (int i = lane; i < T * P; i += 32) {
                const int t = i % T, dst_p = i / T;
                const float *o = os + size_t(t) * ROWS + wid * kRowsPerWarp;
                float acc = o[0] * o[0];
#pragma unroll
                for (int r = 1; r < kRowsPerWarp; ++r) acc = fmaf(o[r], o[r], acc);
                const uint32_t rank = uint32_t(first_rank + dst_p);
                const uint32_t off = uint32_t((size_t(t) * HW + w0 + wid) * 4);   // slot: warp of the head
                st_async_f32(map_cluster(allp_local + off, rank), acc, map_cluster(redbar, rank));
            }
        }
        if constexpr (!TREE) if (a.cap_conv) {
            // conv window capture: concat(old conv state, new tokens) of the channels this CTA owns (a rolled
            // verify read its old conv rows from these very rows: after cluster phase 1 like everything here)
            const int n4 = n_own4;
            float *base = a.cap_conv + size_t(s) * (3 + T) * C;
            for (int i = tid; i < (3 + T) * n4; i += nthr) {
                const int rho = i / n4, c = own_chan(i % n4);
                float *q = base + size_t(rho) * C + gchan(c);
                if (chk(q, 16, a.cap_conv, a.ext_cap_conv)) store4(q, win4(rho, c));
            }
        }
        if (!TREE && !LAZY && active) {    // a tree or lazy verify leaves the state as it was
            float *dst = a.state + ((size_t(s) * Hv + h) * DV + j0 + row0) * DK + 4 * b;
#pragma unroll
            for (int rho = 0; rho < RPG; ++rho)
#pragma unroll
                for (int m = 0; m < NCL; ++m) {
                    float *q = dst + size_t(rho) * DK + 4 * LR * m;
                    if (chk(q, 16, a.state, a.ext_state))
                        store4(q, make_float4(S[rho][m][0], S[rho][m][1], S[rho][m][2], S[rho][m][3]));
                }
        }
    }

    // ------------------------------------------------------------- epilogue
    if constexpr (COMMIT) {
        // conv state <- window rows TT .. TT+2 (after cluster phase 1: every reader is done)
        const int n4 = n_own4;
        float *base = a.conv_state + size_t(s) * 3 * C;
        for (int i = tid; i < 3 * n4; i += nthr) {
            const int rr = i / n4, c = own_chan(i % n4);
            float *q = base + size_t(rr) * C + gchan(c);
            if (chk(q, 16, a.conv_state, a.ext_conv_state)) store4(q, win4(TT + rr, c));
        }
        return;
    }
    // one token per thread, in rounds when the block has fewer threads than tokens (one warp of 8 value rows
    // per CTA with T > 32)
    if (tid < T) mbar_wait_cluster(redbar, 0, a.d_status);   // every partial of this head has landed
    for (int t = tid; t < T; t += nthr) {
        const float *ap = allp + size_t(t) * HW;
        float tot = 0.f;
        for (int i = 0; i < HW; ++i) tot += ap[i];                     // head-level warp order: fixed
        rinv[t] = 1.0f / sqrtf(tot / float(DV) + a.rms_eps);
    }
    __syncthreads();
    {
        Act *out = static_cast<Act *>(a.out);
        const int n4 = MY_ROWS / 4;
        for (int i = tid; i < T * n4; i += nthr) {
            const int t = i / n4, c = 4 * (i % n4);
            const float4 zz = load4(zs + size_t(t) * ROWS + c);
            const float4 oo = load4(os + size_t(t) * ROWS + c);
            const float4 ww = load4(nw + c);
            const float ri = rinv[t];
            const float4 y = make_float4(oo.x * ri * ww.x * silu(zz.x), oo.y * ri * ww.y * silu(zz.y),
                                         oo.z * ri * ww.z * silu(zz.z), oo.w * ri * ww.w * silu(zz.w));
            Act *q = out + (size_t(s) * a.Ts + t) * size_t(Hv) * DV + size_t(h) * DV + j0 + c;
            if (chk(q, 4 * sizeof(Act), out, a.ext_out)) store4(q, y);
        }
    }
    if (LAZY && n_prev > 0) {
        // conv state after the committed tokens: window rows n_prev .. n_prev+2 (after cluster phase 1)
        const int n4 = n_own4;
        float *base = a.conv_state + size_t(s) * 3 * C;
        for (int i = tid; i < 3 * n4; i += nthr) {
            const int rr = i / n4, c = own_chan(i % n4);
            float *q = base + size_t(rr) * C + gchan(c);
            if (chk(q, 16, a.conv_state, a.ext_conv_state)) store4(q, win4(n_prev + rr, c));
        }
    }
    if constexpr (MODE == kChain || ROLLED) {
        // conv state <- window rows T .. T+2 (after cluster phase 1: every reader is done)
        const int n4 = n_own4;
        float *base = a.conv_state + size_t(s) * 3 * C;
        for (int i = tid; i < 3 * n4; i += nthr) {
            const int rr = i / n4, c = own_chan(i % n4);
            float *q = base + size_t(rr) * C + gchan(c);
            if (chk(q, 16, a.conv_state, a.ext_conv_state)) store4(q, win4(T + rr, c));
        }
    }
}

template <int DK, typename Act, int MODE, int MINB>
cudaError_t launch_t(const VerifyArgs &a, cudaStream_t stream) {
    const int head_warps = a.dv / kRowsPerWarp;
    const int warps = (head_warps + a.P - 1) / a.P;            // the widest part
    const Smem L(a.Tm, a.T, DK, warps * kRowsPerWarp, head_warps, sizeof(Act), MODE == kTree);
    auto kern = verify_kernel<DK, Act, MODE, MINB>;
    // Function attributes belong to the context: the dynamic shared memory limit set so far (raised
    // when a launch needs more) and the non-portable cluster permission are cached per context id,
    // shared by the host threads under a lock.
    struct Attrs {
        int smem = 0;
        bool nonportable = false;
    };
    static PerContext<Attrs> attrs;
    unsigned long long ctx = 0;
    Attrs have;
    const bool known = current_context_id(&ctx) && attrs.get(ctx, &have);
    const int cluster = a.r * a.P;
    const bool need_np = cluster > 8;
    cudaError_t e = cudaSuccess;
    if (!known || int(L.total) > have.smem || (need_np && !have.nonportable)) {
        Attrs now = have;
        if (int(L.total) > now.smem) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(L.total));
            if (e != cudaSuccess) return e;
            now.smem = int(L.total);
        }
        if (need_np && !now.nonportable) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
            now.nonportable = true;
        }
        if (current_context_id(&ctx)) attrs.put(ctx, now);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.Hv * a.P, a.B, 1);
    cfg.blockDim = dim3(warps * 32, 1, 1);
    cfg.dynamicSmemBytes = L.total;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace

// rows of the widest of the P parts of a head (the last): the block's warps x 8, the TMA box width
int verify_part_rows(int dv, int P) {
    const int head_warps = dv / kRowsPerWarp;
    return ((head_warps + P - 1) / P) * kRowsPerWarp;
}

size_t verify_smem_bytes(int Tm, int T, int dk, int dv, int P, int act_bytes, bool tree) {
    return Smem(Tm, T, dk, verify_part_rows(dv, P), dv / kRowsPerWarp, act_bytes, tree).total;
}

template <int MODE, int MINB>
static cudaError_t launch_mode(const VerifyArgs &a, bool bf, cudaStream_t stream) {
    switch (a.dk) {
        case 128:
            return bf ? launch_t<128, __nv_bfloat16, MODE, MINB>(a, stream) : launch_t<128, float, MODE, MINB>(a, stream);
        case 64:
            return bf ? launch_t<64, __nv_bfloat16, MODE, MINB>(a, stream) : launch_t<64, float, MODE, MINB>(a, stream);
        case 32:
            return bf ? launch_t<32, __nv_bfloat16, MODE, MINB>(a, stream) : launch_t<32, float, MODE, MINB>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_verify(const VerifyArgs &a, gdn_dtype act, int sm_count, cudaStream_t stream) {
    const bool bf = act == GDN_BF16;
    // more CTAs than two per SM: the three-per-SM build of the chain and rolled modes
    const bool dense = (long long)a.Hv * a.P * a.B > 2LL * sm_count;
    switch (a.mode) {
        case kChain: return dense ? launch_mode<kChain, 3>(a, bf, stream) : launch_mode<kChain, 2>(a, bf, stream);
        case kTree: return launch_mode<kTree, 2>(a, bf, stream);
        case kLazy: return launch_mode<kLazy, 2>(a, bf, stream);
        case kCommit: return launch_mode<kCommit, 2>(a, bf, stream);
        case kRolled: return dense ? launch_mode<kRolled, 3>(a, bf, stream) : launch_mode<kRolled, 2>(a, bf, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace gdn
