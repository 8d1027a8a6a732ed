// rollback.cu -- per-slot rollback of the GDN state to the last accepted token.
//
// hf2q qwen35_target.rs, DFlashTarget::rollback_kv: trim 0 is a no-op and
// accepted_idx = n_tokens_max - 1 - trim.  internal.h, DeltaNetCapture: the
// state comes from capture element accepted_idx and the conv state from
// window rows [commit_n .. commit_n + kernel - 2], commit_n = accepted_idx + 1.
//
// After a tree verify the slot moves to its accepted node instead: state and
// conv state come from that node's captures (-1: nothing accepted, no-op).
//
// A pure copy, so HBM-bound: grid (blocks_per_slot, B, layers); every block
// reads the slot's trim (or node) from device memory (the call can live in a
// CUDA graph), and copies its share of the 16-byte vectors with several loads
// in flight per thread.  A slot with an invalid index is left untouched and
// reported through the status word.  The layers of a serving step roll back
// with the same trims once the whole pass has verified, so one launch can take
// them all: the layer's four buffers then come from device pointer tables (an
// entry that is NULL or not 16-byte aligned skips that layer and is reported).
#include "internal.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 8;

__device__ __forceinline__ float4 ld_nc4(const float4 *p) {
    float4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];\n"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

__global__ void __launch_bounds__(kThreads) rollback_kernel(const RollbackArgs a) {
    // while the previous kernel finishes: an L2 prefetch of the line holding this slot's trim (and of the
    // layer's table entries), so that the read after the wait does not go to DRAM; a prefetch returns
    // nothing to the SM, so a trim the previous kernel is still writing is read correctly below
    if (threadIdx.x == 0 && blockIdx.x == 0) {
        asm volatile("prefetch.global.L2 [%0];\n" ::"l"(a.trim + blockIdx.y));
        if (a.tab_state)
            asm volatile("prefetch.global.L2 [%0];\n" ::"l"(a.tab_state + blockIdx.z));
    }
    // programmatic dependent launch: wait for the previous kernel's writes (captures, trims); the next
    // kernel may start launching once every block has issued its copies (signalled at the end, so that
    // its CTAs do not take SM slots from the copy blocks still waiting to run)
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    const int s = blockIdx.y;
    float *state = a.state, *conv_state = a.conv_state;
    const float *cap_state = a.cap_state, *cap_conv = a.cap_conv;
    if (a.tab_state) {
        const int l = blockIdx.z;
        state = a.tab_state[l];
        conv_state = a.tab_conv_state[l];
        cap_state = a.tab_cap_state[l];
        cap_conv = a.tab_cap_conv[l];
        const uintptr_t any = reinterpret_cast<uintptr_t>(state) | reinterpret_cast<uintptr_t>(conv_state) |
                              reinterpret_cast<uintptr_t>(cap_state) | reinterpret_cast<uintptr_t>(cap_conv);
        if (!state || !conv_state || !cap_state || !cap_conv || (any & 15u)) {
            if (blockIdx.x == 0 && s == 0 && threadIdx.x == 0 && a.d_status)
                atomicCAS(a.d_status, int(GDN_OK), int(GDN_ERR_ARG));
            return;
        }
    }
    // a checked build tests each global access against its buffer first (compiled away otherwise)
    auto chk = [&](const void *p, size_t bytes, const void *base, size_t ext) -> bool {
        return in_bounds(p, bytes, base, ext, a.d_status);
    };
    auto launch_next = []() { asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory"); };
    if (!chk(a.trim + s, 4, a.trim, size_t(a.B) * 4)) return;
    const int idx = __ldg(a.trim + s);
    int accepted_idx;
    if (a.tree) {
        if (idx == -1) return;                               // nothing accepted: the state stays
        accepted_idx = idx;
    } else {
        if (idx == 0) return;                                // nothing to discard
        accepted_idx = a.T - 1 - idx;
    }
    if (accepted_idx < 0 || accepted_idx >= a.T) {          // more than was verified
        if (blockIdx.x == 0 && threadIdx.x == 0 && a.d_status)
            atomicCAS(a.d_status, int(GDN_OK), int(GDN_ERR_TRIM_RANGE));
        return;
    }
    const long long n4_state = a.state_elems / 4, n4_conv = a.conv_elems / 4;
    const float4 *src_s = reinterpret_cast<const float4 *>(cap_state + (size_t(s) * a.T + accepted_idx) * a.state_elems);
    float4 *dst_s = reinterpret_cast<float4 *>(state + size_t(s) * a.state_elems);
    // chain: window rows accepted_idx + 1 .. + W-1; tree: the node's own conv state
    const float4 *src_c = reinterpret_cast<const float4 *>(
        a.tree ? cap_conv + (size_t(s) * a.T + accepted_idx) * a.W1 * a.C
               : cap_conv + (size_t(s) * (a.W1 + a.T) + accepted_idx + 1) * a.C);
    float4 *dst_c = reinterpret_cast<float4 *>(conv_state + size_t(s) * a.conv_elems);

    const long long total = n4_state + n4_conv;
    const long long stride = (long long)gridDim.x * kThreads;
    long long i = (long long)blockIdx.x * kThreads + threadIdx.x;
    for (; i + (kUnroll - 1) * stride < n4_state; i += kUnroll * stride) {
        float4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            v[u] = chk(src_s + i + u * stride, 16, cap_state, a.ext_cap_state) ? ld_nc4(src_s + i + u * stride)
                                                                              : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            if (chk(dst_s + i + u * stride, 16, state, a.ext_state)) dst_s[i + u * stride] = v[u];
    }
    for (; i < total; i += stride) {
        if (i < n4_state) {
            if (chk(src_s + i, 16, cap_state, a.ext_cap_state) && chk(dst_s + i, 16, state, a.ext_state))
                dst_s[i] = ld_nc4(src_s + i);
        } else {
            const long long j = i - n4_state;
            if (chk(src_c + j, 16, cap_conv, a.ext_cap_conv) && chk(dst_c + j, 16, conv_state, a.ext_conv_state))
                dst_c[j] = ld_nc4(src_c + j);
        }
    }
    launch_next();
}

}  // namespace

cudaError_t launch_rollback(const RollbackArgs &a, cudaStream_t stream) {
    const long long n4 = (a.state_elems + a.conv_elems) / 4;
    long long per_slot = (n4 + (long long)kThreads * kUnroll - 1) / ((long long)kThreads * kUnroll);
    if (per_slot < 1) per_slot = 1;
    if (per_slot > 65535) per_slot = 65535;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(per_slot), unsigned(a.B), unsigned(a.tab_state ? a.n_layers : 1));
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, rollback_kernel, a);
}

}  // namespace gdn
