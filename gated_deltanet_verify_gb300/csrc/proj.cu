// proj.cu -- the projections either side of the GDN block: the fused input
// projection x -> [qkv | z | alpha | beta_raw] and the output projection
// out -> y, as one hand-written sm_103a GEMM kernel.
//
// Row-major C[M][N] (row stride ldc, bf16) = X[M][K] @ W[N][K]^T, bf16
// operands, fp32 accumulation.  In a verify step M = slots x tokens is small
// (16 rows for one slot) while W holds tens of MB, so the GEMM streams the
// weights: the weight rows are the tensor core's M dimension and the
// activation rows its N.
//
//   * One CTA per 128-row tile of W (and per split of K when the tiles are
//     too few to cover the SMs; a 256-row block of X per grid row).  The tile
//     is D = W_tile X^T (128 x Mt), fp32 in tensor memory (tcgen05.mma
//     kind::f16, bf16 A and B, both K-major from shared memory).
//   * Warp 0 is the TMA producer: each stage holds kKBlk columns of K of the
//     W tile and of X as 64-column (128-byte) TMA boxes in the 128-byte
//     swizzled K-major layout the tensor core reads directly.
//     Two threads issue the MMAs (8 per stage), warp 1 the even stages into
//     one tensor-memory accumulator and warp 2 the odd ones into a second, and
//     free each stage through tcgen05.commit on its "empty" barrier: one
//     thread's MMAs follow each other ~150 cycles apart whatever their size
//     (measured from M = 64, N = 16 to M = 128, N = 256), and two issuing
//     threads on an SM each keep that pace, so a second issuer doubles the
//     rate of these N = 16 MMAs.  The epilogue adds the two accumulators in a
//     fixed order.
//   * Programmatic dependent launch: the weight tiles of the first stages
//     are requested before the grid-dependency wait (the weights do not
//     depend on the previous kernel; X does), so the stream of weights starts
//     while the previous kernel finishes.
//   * Epilogue: thread t of the 128 reads TMEM lane t (weight row n0 + t)
//     and writes column n0 + t of every output row.  With K split S ways the
//     S CTAs of a tile form a thread-block cluster: after a cluster barrier
//     (every split's MMAs are done, so the first split's pipeline buffers are
//     free) the other splits write their fp32 partial tiles into the first
//     split's shared memory (distributed shared memory), and after a second
//     barrier the first split adds them to its own in split order and writes
//     bf16.  No global scratch, and the sum's order is fixed.
//   * Every wait is bounded; a wait that gives up reports GDN_ERR_TIMEOUT on
//     the caller's status word (when one is given) and the tile is skipped.
#include "internal.cuh"

#include <cuda_bf16.h>

namespace gdn {
namespace {

constexpr int kTileN = 128;             // weight rows per CTA (MMA M)
#ifndef GDN_GEMM_KBLK
#define GDN_GEMM_KBLK 128
#endif
constexpr int kKBlk = GDN_GEMM_KBLK;    // K columns per pipeline stage (a multiple of 64: one TMA box per 64)
constexpr int kBoxes = kKBlk / 64;      // 64-column (128-byte) boxes per operand per stage
static_assert(kKBlk % 64 == 0, "whole 128-byte boxes");
constexpr int kMaxMt = 256;             // activation rows per CTA (MMA N)
constexpr int kThreads = 128;
constexpr int kSpin = 1 << 22;          // mbarrier polls before a wait gives up
constexpr int kMaxStages = 16;

struct GemmArgs {
    CUtensorMap w_map, x_map;
    int M, N, K, Mt;                    // Mt: activation rows per CTA (multiple of 16, <= 256)
    int n_kb, kb_per_split, splits, stages;
    long long ldc;
    __nv_bfloat16 *C;
    int *d_status;
};

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n\t}\n" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}\n"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}
// bounded wait; false if it gave up
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (int i = 0; i < kSpin; ++i)
        if (mbar_try(bar, parity)) return true;
    return false;
}
__device__ __forceinline__ void tma_box(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
// shared-memory matrix descriptor of a K-major tile with 128-byte rows in the 128-byte swizzle (the layout a
// SWIZZLE_128B TMA box of 64 bf16 columns leaves): 8-row groups 1024 bytes apart, the leading offset unused
// (one MMA's 16 columns lie inside a row); saddr may point 32 * j bytes into a 1024-aligned tile to select
// columns 16 j .. 16 j + 15
__device__ __forceinline__ uint64_t make_desc_sw128(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)1 << 16;                                    // leading byte offset 16 (unused)
    d |= (uint64_t)(1024 >> 4) << 32;                          // stride byte offset: next 8-row group
    d |= (uint64_t)1 << 46;                                    // descriptor version (sm_100 family)
    d |= (uint64_t)2 << 61;                                    // layout: 128-byte swizzle
    return d;
}
// instruction descriptor: kind::f16 with bf16 A and B, fp32 D, both K-major, M = 128
__host__ __device__ constexpr uint32_t idesc_bf16(int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}
__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
                 "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
                 : "memory");
}
// 16 fp32 columns of this thread's TMEM lane (activation rows come in multiples of 16)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// the same 16 columns summed over the n accumulators (Mt columns apart), in accumulator order
__device__ __forceinline__ void tmem_ld16_sum(uint32_t taddr, int n, int Mt, float *v) {
    tmem_ld16(taddr, v);
    for (int q = 1; q < n; ++q) {
        float w[16];
        tmem_ld16(taddr + (uint32_t)(q * Mt), w);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] += w[i];
    }
}
__device__ __forceinline__ uint32_t map_cluster(uint32_t local, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(local), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;\n" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

// bytes of one pipeline stage: the W tile (128 rows) and the X block (Mt rows), 64 K-columns each
__host__ __device__ constexpr uint32_t w_stage_bytes() { return kTileN * kKBlk * 2; }
__host__ __device__ inline uint32_t x_stage_bytes(int Mt) { return (uint32_t)Mt * kKBlk * 2; }

__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const __grid_constant__ GemmArgs a) {
    extern __shared__ __align__(1024) unsigned char sm[];
    __shared__ __align__(8) uint64_t bars[2 * kMaxStages + 1];   // full[stages], empty[stages], done (2 arrivals)
    __shared__ uint32_t tslot;
    const int tid = threadIdx.x, wid = tid >> 5;
    const int nt = blockIdx.x, mb = blockIdx.y, split = blockIdx.z;   // the splits of a tile: one cluster
    const int n0 = nt * kTileN, m0 = mb * a.Mt;
    const int kb0 = split * a.kb_per_split;
    const int kb1 = min(a.n_kb, kb0 + a.kb_per_split);
    const int S = a.stages;
    const uint32_t wbytes = w_stage_bytes(), xbytes = x_stage_bytes(a.Mt);
    const uint32_t stage_bytes = wbytes + xbytes;
    const uint32_t sbase = (smem_u32(sm) + 1023u) & ~1023u;   // swizzled tiles start on 1024 bytes
    auto full = [&](int s) { return smem_u32(&bars[s]); };
    auto empty = [&](int s) { return smem_u32(&bars[kMaxStages + s]); };
    const uint32_t done = smem_u32(&bars[2 * kMaxStages]);

    if (wid == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(smem_u32(&tslot)),
                     "r"(2 * kMaxMt));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
    }
    if (tid == 32) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), 1);
        }
        mbar_init(done, 2);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tslot;
    bool ok = true;

    if (tid == 0) {
        // ---- producer: the weight boxes of the first stages go out before the dependency wait
        const int pre = min(S, kb1 - kb0);
        const uint32_t xbox = (uint32_t)a.Mt * 128;            // bytes of one X box
        for (int i = 0; i < pre; ++i) {
            const uint32_t st = sbase + (uint32_t)i * stage_bytes;
            mbar_expect_tx(full(i), stage_bytes);
            for (int b = 0; b < kBoxes; ++b) tma_box(st + b * 16384u, &a.w_map, (kb0 + i) * kKBlk + 64 * b, n0, full(i));
        }
        asm volatile("griddepcontrol.wait;\n" ::: "memory");
        for (int i = 0; i < pre; ++i)
            for (int b = 0; b < kBoxes; ++b)
                tma_box(sbase + (uint32_t)i * stage_bytes + wbytes + b * xbox, &a.x_map, (kb0 + i) * kKBlk + 64 * b, m0,
                        full(i));
        for (int i = pre; i < kb1 - kb0 && ok; ++i) {
            const int s = i % S;
            ok = mbar_wait(empty(s), ((i / S) - 1) & 1);       // the MMAs of stage use i - S are done
            const uint32_t st = sbase + (uint32_t)s * stage_bytes;
            mbar_expect_tx(full(s), stage_bytes);
            for (int b = 0; b < kBoxes; ++b) tma_box(st + b * 16384u, &a.w_map, (kb0 + i) * kKBlk + 64 * b, n0, full(s));
            for (int b = 0; b < kBoxes; ++b)
                tma_box(st + wbytes + b * xbox, &a.x_map, (kb0 + i) * kKBlk + 64 * b, m0, full(s));
        }
    } else if (tid == 32 || tid == 64) {
        // ---- MMA issuers: stages e, e + 2, ... into accumulator e (8 MMAs of K = 16 per stage); each stage is
        // freed when its MMAs complete
        const int e = wid - 1;
        const uint32_t acc = tmem + (uint32_t)(e * a.Mt);
        const uint32_t id = idesc_bf16(a.Mt);
        for (int i = e; i < kb1 - kb0 && ok; i += 2) {
            const int s = i % S;
            ok = mbar_wait(full(s), (i / S) & 1);
            fence_after_sync();
            const uint32_t st = sbase + (uint32_t)s * stage_bytes;
#pragma unroll
            for (int j = 0; j < kKBlk / 16; ++j) {          // 16 columns (32 bytes of each row) per MMA
                const uint32_t b = j >> 2, c = 32u * (j & 3);
                mma_bf16(acc, make_desc_sw128(st + b * 16384u + c),
                         make_desc_sw128(st + wbytes + b * (uint32_t)a.Mt * 128u + c), id, (i > e || j > 0) ? 1u : 0u);
            }
            mma_commit(empty(s));
        }
        mma_commit(done);
    }
    __syncwarp();
    // ---- epilogue: the accumulator of weight row n0 + tid, every activation row of the block
    const bool got = mbar_wait(done, 0);
    fence_after_sync();
    // one verdict for the whole CTA (the collective TMEM loads below need every lane of a warp)
    const bool good = __syncthreads_and(got && ok) != 0;
    if (!good && tid == 0 && a.d_status) atomicCAS(a.d_status, int(GDN_OK), int(GDN_ERR_TIMEOUT));
    const int n_acc = kb1 - kb0 > 1 ? 2 : 1;                 // the odd stages' accumulator holds a sum only if used
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const int n = n0 + tid;
    const uint32_t taddr = tmem + ((uint32_t)(32 * wid) << 16);
    if (a.splits == 1) {
        if (good)
            for (int c0 = 0; c0 < a.Mt; c0 += 16) {
                float v[16];
                tmem_ld16_sum(taddr + c0, n_acc, a.Mt, v);
                if (n < a.N)
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int m = m0 + c0 + q;
                        if (m < a.M) a.C[(size_t)m * a.ldc + n] = __float2bfloat16_rn(v[q]);
                    }
            }
    } else {
        // partial tiles of splits 1 .. S-1 -> the first split's shared memory, [split-1][column][row]
        cluster_sync();                            // every split's MMAs are done: split 0's buffers are free
        if (split > 0) {
            const uint32_t dst = map_cluster(sbase, 0) + (uint32_t)((split - 1) * a.Mt * kTileN + tid) * 4u;
            for (int c0 = 0; c0 < a.Mt; c0 += 16) {
                float v[16];
                tmem_ld16_sum(taddr + c0, n_acc, a.Mt, v);
#pragma unroll
                for (int q = 0; q < 16; ++q) st_cluster_f32(dst + (uint32_t)((c0 + q) * kTileN) * 4u, good ? v[q] : 0.f);
            }
        }
        cluster_sync();                            // every partial has landed
        if (split == 0 && good) {
            const float *red = reinterpret_cast<const float *>(sm + (sbase - smem_u32(sm)));
            for (int c0 = 0; c0 < a.Mt; c0 += 16) {
                float v[16];
                tmem_ld16_sum(taddr + c0, n_acc, a.Mt, v);
                if (n < a.N)
#pragma unroll
                    for (int q = 0; q < 16; ++q) {
                        const int m = m0 + c0 + q;
                        float acc = v[q];
                        for (int sp = 1; sp < a.splits; ++sp) acc += red[((sp - 1) * a.Mt + c0 + q) * kTileN + tid];
                        if (m < a.M) a.C[(size_t)m * a.ldc + n] = __float2bfloat16_rn(acc);
                    }
            }
        }
    }
    fence_before_sync();
    __syncthreads();
    if (wid == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "r"(2 * kMaxMt));
}

}  // namespace

// K splits of a tile: enough CTAs to cover the SMs when the output tiles are few, while the other
// splits' partial tiles fit the first split's pipeline buffers (the reduction space)
static int gemm_splits(int n_tiles, int m_blocks, int n_kb, int Mt, size_t smem, int sms) {
    int splits = sms / (n_tiles * m_blocks);
    if (splits > 8) splits = 8;
    if (splits > n_kb) splits = n_kb;
    while (splits > 1 && (size_t)(splits - 1) * Mt * kTileN * 4 > smem) --splits;
    return splits < 1 ? 1 : splits;
}

bool gemm_xwt_bf16(const void *W, const void *X, void *C, int M, int N, int K, long long ldc, int *d_status,
                   cudaStream_t stream, std::string &why) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) {
        why = "the driver's tensor-map encoder is unavailable";
        return false;
    }
    if (K % 8 || K < 8) {
        why = "K must be a positive multiple of 8";
        return false;
    }
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                   cudaSuccess) {
        why = "no usable CUDA device";
        return false;
    }
    GemmArgs a{};
    a.M = M; a.N = N; a.K = K; a.ldc = ldc;
    a.Mt = M >= kMaxMt ? kMaxMt : ((M + 15) / 16) * 16;
    const int m_blocks = (M + a.Mt - 1) / a.Mt;
    const int n_tiles = (N + kTileN - 1) / kTileN;
    a.n_kb = (K + kKBlk - 1) / kKBlk;
    const uint32_t stage = w_stage_bytes() + x_stage_bytes(a.Mt);
    // as many stages as fit in ~216 KB: a stage is held until its MMAs complete, so the bytes in flight per
    // SM set the intake (six 36 KB stages: output projection 14.6 us against 14.9 with five; two CTAs per SM
    // with 100 KB each, the K splits spread over every SM, measured slower: 26 us)
    a.stages = (int)((216u * 1024u) / stage);
    if (a.stages > kMaxStages) a.stages = kMaxStages;
    if (a.stages < 1) {
        why = "pipeline stage larger than shared memory";
        return false;
    }
    const size_t smem = (size_t)a.stages * stage + 1024;          // + room to align the tiles to 1024 bytes
    const int splits = gemm_splits(n_tiles, m_blocks, a.n_kb, a.Mt, smem - 1024, sms);
    a.kb_per_split = (a.n_kb + splits - 1) / splits;
    a.splits = (a.n_kb + a.kb_per_split - 1) / a.kb_per_split;
    a.C = static_cast<__nv_bfloat16 *>(C);
    a.d_status = d_status;
    // tensor maps: 64-column (128-byte) boxes in the 128-byte swizzle
    const cuuint32_t estr[2] = {1, 1};
    {
        const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)N};
        const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
        const cuuint32_t box[2] = {64u, (cuuint32_t)kTileN};
        if (encode(&a.w_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(W), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            why = "weight tensor map";
            return false;
        }
    }
    {
        const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
        const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
        const cuuint32_t box[2] = {64u, (cuuint32_t)a.Mt};
        if (encode(&a.x_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(X), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
            why = "activation tensor map";
            return false;
        }
    }
    cudaError_t e = cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(n_tiles, m_blocks, a.splits);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 1;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = a.splits;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        e = cudaLaunchKernelEx(&cfg, gemm_kernel, a);
    }
    if (e != cudaSuccess) {
        why = std::string("projection GEMM launch: ") + cudaGetErrorString(e);
        return false;
    }
    return true;
}

}  // namespace gdn
