// prefill.cu -- chunkwise (WY / UT-transform) prefill of the Gated DeltaNet
// block on sm_103a tensor cores.
//
// For a chunk of C = 64 tokens with decays accumulated inside the chunk,
// Gamma_r = prod_{u<=r} g_u, and the state S0 at the chunk start, the gated
// delta rule unrolls to (Yang et al., "Parallelizing Linear Transformers with
// the Delta Rule over Sequence Length", 2024; Yang, Kautz & Hatamizadeh,
// "Gated Delta Networks", 2025):
//   A[r][s] = beta_r (Gamma_r / Gamma_s) k_r . k_s   (s < r),   T = (I + A)^-1
//   W = T diag(beta Gamma) K,   U~ = T diag(beta) V,   U = U~ - W S0
//   O = diag(Gamma) Q S0 + (Q K^T (.) M) U,   M[r][s] = Gamma_r / Gamma_s (s <= r)
//   S = Gamma_C S0 + (diag(Gamma_C / Gamma) K)^T U
// Every dense product but G = [K; Q] K^T (fp32 CUDA-core FMA chains, see the
// preparation phase) runs on tcgen05.mma (kind::tf32, fp32 accumulators in
// tensor memory) with 3xTF32 operands: each fp32 operand is split into its
// nearest tf32 value and the nearest tf32 value of the remainder, and A.B is
// taken as hi.hi + hi.lo + lo.hi.  Single-pass tf32 (or bf16) operands are not accurate enough here:
// the delta rule subtracts nearly equal predictions (U~ against W S0) and the
// per-token RMSNorm rescales small outputs, so an operand rounding of 2^-11
// becomes an error of 10-60 % in the outputs; with the split it is ~1e-5.
//
// Work split.  Everything but U, O and S depends only on the chunk itself, so
// one state CTA per (slot, value head) is fed by a shared pool:
//   * preparation CTAs (every SM the state CTAs leave) claim (chunk, key head) work items
//     in chunk order from a counter; per item the q/k work is done once for
//     the r value heads that share the key head (raw window by TMA,
//     conv + SiLU into TMEM, L2 norms, G = [K; Q] K^T in fp32 FMA chains, kept
//     in TMEM), then per
//     value head its gates, v conv (into shared memory), A and the masked,
//     decayed P, T = (I + A)^-1 (16 x 16 blocks), W^T and U~^T; they publish
//     the ready-split operands ([-W; Gamma Q] as one operand, P, Gamma_C/Gamma
//     K planes and U~) to that head's ring of four slots in the caller's
//     workspace (L2-resident) and release a per-slot flag;
//   * the state CTA holds the fp32 state in registers and, chunk by chunk,
//     acquires a slot, pulls it in with bulk copies and runs only the
//     state-dependent products and the epilogue:
//       [X^T | O^T] = S0^T [-W; Gamma Q]^T          (one N 128 product, A from TMEM)
//       U^T = U~^T + X^T,  O^T = (Gamma Q S0)^T + U^T P^T   (N 64)
//       D2  = U^T (diag(Gamma_C / Gamma) K)          (N 128, K 64);  S^T <- Gamma_C S^T + D2
//     then the gated RMSNorm.  It frees the slot once its bulk copies landed.
// The launch is cooperative (every CTA resident at once), so the flag waits
// between the CTAs cannot starve; (slot, head) pairs beyond what fits
// at once go to further launches.  Every wait is bounded and reports
// GDN_ERR_TIMEOUT instead of hanging.  The ring flags are zeroed by a
// stream-ordered memset before each launch.  The conv state (shared by the
// value heads of a key head) is advanced by a second, small kernel.
#include "internal.cuh"

#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <cstdlib>
#include <mutex>
#include <string>

namespace gdn {
namespace {

constexpr int kC = 64;                 // chunk length
constexpr int kD = 128;                // d_k = d_v
constexpr int kCh = 3 * kD;            // conv channels of one value head: q | k | v
constexpr int kThreads = 256;
constexpr int kSpinLimit = 1 << 20;    // try_wait rounds before an mbarrier wait gives up
constexpr int kFlagSpin = 1 << 21;     // polls (with back-off, about a second) before a ring-flag wait gives up
constexpr int kTmemCols = 512;
constexpr int kRing = 4;               // ring slots per (slot, value head)
constexpr int kMaxPrep = 8;            // preparation CTAs per key head, at most (more would only wait)

// dynamic shared memory carve-up (bytes)
constexpr uint32_t kRA = 0;                    // 128 KB: A operand planes; raw chunk inputs at chunk start
constexpr uint32_t kRB = 128 * 1024;           // 64 KB: B operand planes; T and block temporaries
constexpr uint32_t kAM = 192 * 1024;           // 16 KB: A (fp32, 64 x 64, transposed [s][r]); the z tile
constexpr uint32_t kPT = 208 * 1024;           // 16 KB: P (fp32, 64 x 64), stored transposed [s][r]
constexpr uint32_t kMisc = 224 * 1024;
constexpr uint32_t kMbar = kMisc;              // 8 B: tensor-core completion
constexpr uint32_t kRawBar = kMisc + 8;        // 8 B: raw window copies (preparation) / slot copies (state)
constexpr uint32_t kTmemSlot = kMisc + 16;     // 4 B
constexpr uint32_t kFlagOk = kMisc + 20;       // 4 B: result of a ring-flag wait, broadcast to the CTA
constexpr uint32_t kZBar = kMisc + 24;         // 8 B: gate (z) tile copy
constexpr uint32_t kItem = kMisc + 32;         // 4 B: work item claimed by a preparation CTA, broadcast
constexpr uint32_t kMbar2 = kMisc + 40;        // 8 B: tensor-core completion of the second issuing thread
constexpr uint32_t kLogG = kMisc + 48;         // 64 floats each
constexpr uint32_t kBeta = kLogG + 256;
constexpr uint32_t kGam = kBeta + 256;
constexpr uint32_t kRinv = kGam + 256;
constexpr uint32_t kInvQ = kRinv + 256;        // 1 / ||q_t||, 1 / ||k_t||
constexpr uint32_t kInvK = kInvQ + 256;
constexpr uint32_t kRed = kInvK + 256;         // 4 lane quarters x 64 tokens
constexpr uint32_t kLogLo = kRed + 4 * 64 * 4;  // low parts of the cumulative log decays (64 floats)
constexpr uint32_t kSmemBytes = kLogLo + 256;
static_assert(kSmemBytes <= 227 * 1024, "shared memory per CTA");
constexpr int kWin = kC + 3;                   // window rows of a chunk (3 rows of history)
static_assert(kWin * kCh * 4 <= 128 * 1024, "raw chunk window fits the A region");
// RB during the conv phase: the conv state rows (first chunk) and the per-warp sums of squares
constexpr uint32_t kHistOff = 0;               // 3 x 384 floats
constexpr uint32_t kSsqOff = 8 * 1024;         // 8 channel blocks (q, k) x 64 tokens

// TMEM columns of a preparation CTA: G (kept for all value heads of the group), U~^T, W^T and the
// chunk's conv outputs q and k (lane = channel, column = token; not normalised).
constexpr uint32_t kColG = 0, kColUT = 64, kColWT = 128, kColQ = 192, kColK = 256;
static_assert(kColK + 64 <= kTmemCols, "TMEM columns");
// State CTA: (U^T P^T) | X^T (then U^T hi) | (Gamma Q S0)^T | U^T lo | S^T hi (then D2) | S^T lo.  The two
// parts of O^T have accumulators of their own and are added in fp32 on the CUDA cores (a product added
// onto an accumulator that already holds a large value truncates relative to that value)
constexpr uint32_t kSO2 = 0, kSX = 64, kSO = 128, kSUlo = 192, kSShi = 256, kSSlo = 384;
static_assert(kSSlo + 128 <= kTmemCols, "TMEM columns of the state CTA");

// One ring slot: the chunk's operands in the exact shared-memory layout the state CTA uses.
constexpr uint32_t kSlotB = 0;                 // [-W; Gamma Q] planes: one 128 x 128 operand, hi 64 KB + lo 64 KB
constexpr uint32_t kSlotP = 128 * 1024;        // P planes (64 x 64), 32 KB
constexpr uint32_t kSlotKd = 160 * 1024;       // (Gamma_C / Gamma) K planes, as (128 x 64), 64 KB
constexpr uint32_t kSlotU = 224 * 1024;        // U~^T fp32 [128][64], 32 KB
constexpr size_t kSlotBytes = 256 * 1024;
// per (slot, value head): ring flags and the chunk decays (ints: full[4], empty[4], Gamma_C[4] bits)
constexpr size_t kFlagWords = 32;
static_assert(kFlagWords >= 3 * kRing, "flag words");
// v^T of the current value head (128 channels x 64 tokens, rows padded to 68 floats so that a warp's 16-byte
// row accesses fall in distinct banks) lives in the upper half of the A region: free from the end of the G
// product until the A2 operand build, by which time every thread holds its row in registers
constexpr uint32_t kVt = kRA + 64 * 1024;
constexpr int kVtStride = kC + 4;
// fp32 K^ / Q^ rows for the G product (start of the A region), padded so that a warp's 16-byte row reads
// at rows r .. r+7 fall in distinct banks
constexpr int kXStride = kD + 4;
static_assert(2 * kC * kXStride * 4 <= 128 * 1024, "K^ / Q^ rows fit the A region");
static_assert(64 * 1024 + 128 * kVtStride * 4 <= 128 * 1024, "v^T fits the upper half of the A region");

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename Act> __device__ __forceinline__ Act from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}
__device__ __forceinline__ float silu(float x) { return __fdividef(x, 1.0f + __expf(-x)); }

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// (ah + al) + (bh + bl) as a normalised pair of floats (Knuth's two-sum on the high parts): the
// cumulative log decay of a chunk reaches a few hundred in magnitude, and the decay between two nearby
// tokens is exp of the difference of two such sums, so a plain fp32 sum would leave that difference with
// an error of |sum| * 2^-24 (~1e-5 relative in the decay); the pair keeps it to fp32 precision of the
// difference itself
__device__ __forceinline__ void add_pair(float ah, float al, float bh, float bl, float &h, float &l) {
    const float s = ah + bh, bb = s - ah;
    const float e = (ah - (s - bb)) + (bh - bb);
    const float lo = al + bl + e;
    h = s + lo;
    l = lo - (h - s);
}

// ---- 3xTF32 operand planes: canonical K-major, no swizzle -----------------
// 16-byte group (r, k4) of an R x K operand: core matrix (r/8, k4) of 8 rows x 16 B
__device__ __forceinline__ uint32_t plane_off(int r, int k4, int K) {
    return (uint32_t)((((r >> 3) * (K >> 2) + k4) << 7) + ((r & 7) << 4));
}
// x rounded to the nearest tf32 value (ties away from zero; one cvt instruction).
__device__ __forceinline__ float tf32_rn(float x) {
    uint32_t u;
    asm("cvt.rna.tf32.f32 %0, %1;\n" : "=r"(u) : "f"(x));
    return __uint_as_float(u);
}
// x = hi + lo exactly, hi the nearest tf32 value.  A kind::tf32 MMA reads only the upper 19 bits of an fp32
// operand, so it cuts lo's last bits off: an error below 2^-23 |x| whose sign is that of lo, i.e. as often
// toward x as away from it.  (Cutting the bits of x itself to form hi, as a plain mask does, leaves lo with
// x's sign and makes both cuts err toward zero: a one-sided error up to 2^-21 |x|, which the all-heads
// parity test of the 8192-token layer showed in its outputs.)
__device__ __forceinline__ void split_tf32(float x, float &hi, float &lo) {
    hi = tf32_rn(x);
    lo = x - hi;
}
// 4 consecutive k of row r: the tf32 part into the hi plane, the remainder into the lo plane
__device__ __forceinline__ void put4(unsigned char *hi, unsigned char *lo, int r, int k4, int K, float4 v) {
    float4 h, l;
    split_tf32(v.x, h.x, l.x);
    split_tf32(v.y, h.y, l.y);
    split_tf32(v.z, h.z, l.z);
    split_tf32(v.w, h.w, l.w);
    const uint32_t off = plane_off(r, k4, K);
    *reinterpret_cast<float4 *>(hi + off) = h;
    *reinterpret_cast<float4 *>(lo + off) = l;
}
// Lanes 4a .. 4a+3 of a warp hold v[e] = X[row0 + e][4a + (lane & 3)], e = 0..3 (a column each);
// on return lane 4a + c holds X[row0 + c][4a .. 4a+3] (a row each): a 4 x 4 transpose inside each
// lane quad, two butterfly stages of two shuffles.
__device__ __forceinline__ float4 quad_transpose(float v0, float v1, float v2, float v3) {
    const bool b1 = (threadIdx.x & 1) != 0, b2 = (threadIdx.x & 2) != 0;
    float t0 = __shfl_xor_sync(0xffffffffu, b1 ? v0 : v1, 1);
    float t1 = __shfl_xor_sync(0xffffffffu, b1 ? v2 : v3, 1);
    if (b1) { v0 = t0; v2 = t1; } else { v1 = t0; v3 = t1; }
    t0 = __shfl_xor_sync(0xffffffffu, b2 ? v0 : v2, 2);
    t1 = __shfl_xor_sync(0xffffffffu, b2 ? v1 : v3, 2);
    if (b2) { v0 = t0; v1 = t1; } else { v2 = t0; v3 = t1; }
    return make_float4(v0, v1, v2, v3);
}
// Column tl of 32 rows (row0 .. row0+31, values x[0..31]) of a K = 128 operand -> its planes, 16 bytes
// at a time.  Odd lane quads take the row blocks in the order b ^ 1, so the two quads of an 8-lane store
// phase fill all eight 16-byte rows of a core matrix (no bank conflict).
__device__ __forceinline__ void put_col32(unsigned char *hi, unsigned char *lo, int row0, int tl, const float *x) {
    const bool odd = (threadIdx.x & 4) != 0;
#pragma unroll
    for (int b = 0; b < 8; ++b) {
        const int bo = b ^ 1;
        const float4 w = quad_transpose(odd ? x[4 * bo] : x[4 * b], odd ? x[4 * bo + 1] : x[4 * b + 1],
                                        odd ? x[4 * bo + 2] : x[4 * b + 2], odd ? x[4 * bo + 3] : x[4 * b + 3]);
        put4(hi, lo, row0 + 4 * (odd ? bo : b) + (threadIdx.x & 3), tl >> 2, 128, w);
    }
}

// item -> (row, 16-byte group) so that consecutive items fill consecutive 16-byte slots
__device__ __forceinline__ void item_rc(int it, int K, int &r, int &k4) {
    const int cm = it >> 3, groups = K >> 2;
    r = (cm / groups) * 8 + (it & 7);
    k4 = cm % groups;
}

// ---- tcgen05 ---------------------------------------------------------------
__device__ __forceinline__ uint64_t make_desc(uint32_t saddr, int K) {
    uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)(128 >> 4) << 16;                          // LBO: next core matrix along K
    d |= (uint64_t)((((uint32_t)K >> 2) * 128) >> 4) << 32;   // SBO: next 8-row group
    d |= (uint64_t)1 << 46;                                    // descriptor version (sm_100 family)
    return d;                                                  // no swizzle, base offset 0
}
__host__ __device__ constexpr uint32_t idesc_tf32(int N) {
    // D f32, A and B tf32, both K-major, N >> 3, M = 128 >> 4
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
}
__device__ __forceinline__ void mma_tf32(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d),
                 "l"(a), "l"(b), "r"(idesc), "r"(acc));
}
// D (128 x N, fp32 in TMEM) (+)= A (128 x K) . B (N x K)^T with 3xTF32 planes.  The tensor core truncates
// its fp32 accumulator at every step, relative to the accumulator's magnitude, so the small cross terms
// (hi.lo, lo.hi) go in first while the accumulator is still small and the large hi.hi products last:
// measured on the GB300 for K = 128 dot products, this order errs at most ~4 units of 2^-24 of sum |a b|
// (an fp32 FMA chain: ~3.7), against ~18 with the three products interleaved per K step.
__device__ __forceinline__ void mma3(uint32_t d, uint32_t a_hi, uint32_t a_lo, uint32_t b_hi, uint32_t b_lo, int K,
                                     int N, bool accumulate) {
    const uint32_t id = idesc_tf32(N);
    for (int pass = 0; pass < 3; ++pass)
        for (int ks = 0; ks < K / 8; ++ks) {
            const uint32_t o = (uint32_t)ks * 256u;            // 8 tf32 = two core matrices along K
            const uint32_t a = pass == 1 ? a_lo : a_hi, b = pass == 0 ? b_lo : b_hi;
            mma_tf32(d, make_desc(a + o, K), make_desc(b + o, K), id, (pass > 0 || ks > 0 || accumulate) ? 1u : 0u);
        }
}
// D (128 x N) (+)= A (128 x K, tf32 columns of TMEM: lane = row) . B (N x K, smem)^T, 3xTF32
__device__ __forceinline__ void mma_tf32_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d),
                 "r"(a), "l"(b), "r"(idesc), "r"(acc));
}
// (the same pass order as mma3: cross terms first, hi.hi last)
__device__ __forceinline__ void mma3_ts(uint32_t d, uint32_t a_hi, uint32_t a_lo, uint32_t b_hi, uint32_t b_lo, int K,
                                        int N, bool accumulate) {
    const uint32_t id = idesc_tf32(N);
    for (int pass = 0; pass < 3; ++pass)
        for (int ks = 0; ks < K / 8; ++ks) {
            const uint32_t o = (uint32_t)ks * 256u;
            const uint32_t a = pass == 1 ? a_lo : a_hi, b = pass == 0 ? b_lo : b_hi;
            mma_tf32_ts(d, a + 8 * ks, make_desc(b + o, K), id, (pass > 0 || ks > 0 || accumulate) ? 1u : 0u);
        }
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
// 16 fp32 columns of this thread's TMEM lane
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
// 16 fp32 columns into this thread's TMEM lane (completion: tmem_wait_st)
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(
            taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
        "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
        "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])),
        "r"(__float_as_uint(v[11])), "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])),
        "r"(__float_as_uint(v[14])), "r"(__float_as_uint(v[15]))
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory"); }

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}\n"
                 : "=r"(ok)
                 : "r"(bar), "r"(parity)
                 : "memory");
    return ok != 0;
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n\t}\n" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}
// 2-D tile of a tensor map -> own shared memory, completion counted in bytes on an mbarrier
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];\n" ::"r"(
            dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// global -> own shared memory, completion counted in bytes on an mbarrier
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;\n" ::: "memory"); }
__device__ __forceinline__ void st_release(int *p, int v) {
    asm volatile("st.release.gpu.global.s32 [%0], %1;\n" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ int ld_acquire(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];\n" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// one thread polls *p until it reaches target (bounded, with back-off)
__device__ __forceinline__ bool poll_flag(const int *p, int target) {
    for (int it = 0; it < kFlagSpin; ++it) {
        if (ld_acquire(p) >= target) return true;
        __nanosleep(64);
    }
    return false;
}

// Per-CTA views of the ring and flags of one (slot, value head).
struct Ring {
    int *full, *empty;        // [kRing] chunk index + 1 of the last chunk published / consumed per slot
    float *gamma_c;           // [kRing] Gamma_C of the chunk in each slot
    unsigned char *slots;     // [kRing][kSlotBytes]
};

__device__ __forceinline__ Ring ring_of(const PrefillArgs &a, int s, int h) {
    unsigned char *ws = reinterpret_cast<unsigned char *>(a.scratch);
    const size_t pair = (size_t)s * a.Hv + h;
    int *flags = reinterpret_cast<int *>(ws) + pair * kFlagWords;
    Ring r;
    r.full = flags;
    r.empty = flags + kRing;
    r.gamma_c = reinterpret_cast<float *>(flags + 2 * kRing);
    r.slots = ws + a.ring_offset + pair * (kRing * kSlotBytes);
    return r;
}

// Shared context of one CTA.
struct Ctx {
    unsigned char *sm;
    int tid, lane, wid, tl, half;
    uint32_t tmem, tq, mbar, phase, mbar2, phase2;
    bool timed_out;

    __device__ __forceinline__ void commit_wait() {
        if (tid == 0) mma_commit(mbar);
        bool ok = timed_out;           // after one timeout the rest of the launch only drains
        for (int it = 0; it < kSpinLimit && !ok; ++it) ok = mbar_try(mbar, phase & 1u);
        if (!ok) timed_out = true;
        phase ^= 1u;
        fence_after_sync();
    }
    // two independent products issued by two threads (0 and 32): one MMA-issuing thread paces its MMAs
    // ~150-200 cycles apart whatever their size (measured), so two threads finish two products in about
    // the time of one
    __device__ __forceinline__ void commit_wait2() {
        if (tid == 0) mma_commit(mbar);
        if (tid == 32) mma_commit(mbar2);
        bool ok = timed_out, ok2 = timed_out;
        for (int it = 0; it < kSpinLimit && !ok; ++it) ok = mbar_try(mbar, phase & 1u);
        for (int it = 0; it < kSpinLimit && !ok2; ++it) ok2 = mbar_try(mbar2, phase2 & 1u);
        if (!ok || !ok2) timed_out = true;
        phase ^= 1u;
        phase2 ^= 1u;
        fence_after_sync();
    }
    __device__ __forceinline__ void publish() {      // generic smem writes -> visible to the tensor core
        fence_proxy_async();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
    }
    __device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t &ph) {
        bool ok = timed_out;
        for (int it = 0; it < kSpinLimit && !ok; ++it) ok = mbar_try(bar, ph & 1u);
        if (!ok) timed_out = true;
        ph ^= 1u;
        return ok;
    }
    // thread 0 polls a ring flag; the result reaches every thread of the CTA
    __device__ __forceinline__ void wait_flag(const int *p, int target) {
        volatile int *okp = reinterpret_cast<volatile int *>(sm + kFlagOk);
        if (tid == 0) *okp = (timed_out || poll_flag(p, target)) ? 1 : 0;
        __syncthreads();
        if (*okp == 0) timed_out = true;
        __syncthreads();
    }
};

// ---------------------------------------------------------------------------
// preparation CTA: claims (chunk, slot, key head) items; for each, the q/k work
// (conv, norms, G) once, then A, T, W, U~, P for each of the r value heads of
// the group, each published to that head's ring
// ---------------------------------------------------------------------------
template <typename Act>
__device__ __forceinline__ void prepare(const PrefillArgs &a, Ctx &x) {
    unsigned char *sm = x.sm;
    const int tid = x.tid, lane = x.lane, wid = x.wid, tl = x.tl, half = x.half;
    const int Hk = a.Hk, Hv = a.Hv, L = a.L, C = a.C, R = a.r;
    const uint32_t tmem = x.tmem, tq = x.tq;
    const Act *rawA = reinterpret_cast<const Act *>(sm + kRA);        // q|k tiles, later one v tile: [67][128]
    float *hist = reinterpret_cast<float *>(sm + kRB + kHistOff);     // [3][256] q|k, later [3][128] v history
    float *ssq = reinterpret_cast<float *>(sm + kRB + kSsqOff);       // [8][64] partial sums of squares
    float *AMt = reinterpret_cast<float *>(sm + kAM);
    float *Pt = reinterpret_cast<float *>(sm + kPT);
    float *Tm = reinterpret_cast<float *>(sm + kRB + 32 * 1024);      // T (fp32, 64 x 64, row-major)
    float *Xb = reinterpret_cast<float *>(sm + kRB + 48 * 1024);      // block-inversion temporaries
    float *logG = reinterpret_cast<float *>(sm + kLogG);          // cumulative log decays: high parts
    float *logLo = reinterpret_cast<float *>(sm + kLogLo);        // and low parts
    float *betas = reinterpret_cast<float *>(sm + kBeta);
    float *gam = reinterpret_cast<float *>(sm + kGam);
    float *invq = reinterpret_cast<float *>(sm + kInvQ);
    float *invk = reinterpret_cast<float *>(sm + kInvK);
    unsigned char *RA = sm + kRA, *RB = sm + kRB;
    const uint32_t sRA = smem_u32(RA), sRB = smem_u32(RB);
    const uint32_t rawbar = smem_u32(sm + kRawBar);
    uint32_t raw_phase = 0;
    float *vT = reinterpret_cast<float *>(sm + kVt);           // [128 channels][64 tokens, padded]
    constexpr uint32_t kTile = kWin * kD * sizeof(Act);

    // raw window rows t0-3 .. t0+63 of chunk cc: 128-channel tiles of the qkv tensor map, one thread.
    // Rows outside the tensor read as zero; rows of a neighbouring slot and rows past the prompt are never
    // used (the history rows of the first chunk come from the conv state, padded tokens are discarded).
    auto issue_qk = [&](int cc, int s, int kh) {
        const int y = s * L + cc * kC - 3;
        mbar_arrive_expect_tx(rawbar, 2u * kTile);
        tma_load_2d(sRA, &a.qkv_map, kh * kD, y, rawbar);
        tma_load_2d(sRA + kTile, &a.qkv_map, Hk * kD + kh * kD, y, rawbar);
    };
    auto issue_v = [&](int cc, int s, int h) {
        mbar_arrive_expect_tx(rawbar, kTile);
        tma_load_2d(sRA, &a.qkv_map, 2 * Hk * kD + h * kD, s * L + cc * kC - 3, rawbar);
    };
    // gate inputs of (chunk cc, value head h) (threads tid < 64, one token each)
    float g_alpha = 0.f, g_beta = 0.f;
    auto load_gates = [&](int cc, int s, int h) {
        const int t = cc * kC + tid;
        if (tid < kC && t < L) {
            const size_t idx = ((size_t)s * L + t) * Hv + h;
            g_alpha = to_f32(static_cast<const Act *>(a.alpha)[idx]);
            g_beta = to_f32(static_cast<const Act *>(a.beta_raw)[idx]);
        }
    };
    // sliding-window conv + SiLU of 16 tokens of one channel; rows 0-2 of the first chunk from `hist`
    auto conv16 = [&](const Act *src, const float *hrow, int hstride, int g, int tb, int c, int n, float *yv) {
        const float w0 = __ldg(a.conv_w + g), w1 = __ldg(a.conv_w + C + g), w2 = __ldg(a.conv_w + 2 * C + g),
                    w3 = __ldg(a.conv_w + 3 * C + g);
        float x0, x1, x2;
        if (c == 0 && tb == 0) {
            x0 = hrow[0]; x1 = hrow[hstride]; x2 = hrow[2 * hstride];
        } else {
            x0 = to_f32(src[tb * kD]); x1 = to_f32(src[(tb + 1) * kD]); x2 = to_f32(src[(tb + 2) * kD]);
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int t = tb + j;
            const float x3 = to_f32(src[(t + 3) * kD]);
            const float y = silu(fmaf(w3, x3, fmaf(w2, x2, fmaf(w1, x1, w0 * x0))));
            yv[j] = t < n ? y : 0.f;
            x0 = x1; x1 = x2; x2 = x3;
        }
    };

    // A published (chunk, head) is released one phase later (after the next head's v conv, or the next
    // item's q/k conv), so its stores drain while that runs: every thread fences its own stores, the CTA
    // synchronises, thread 0 releases the flag.  pend_* are uniform across the CTA.
    int pend_slot = -1, pend_c = 0, pend_h = 0, pend_s = 0;
    float pend_gamma = 0.f;
    auto fence_pending = [&]() {
        if (pend_slot >= 0) __threadfence();
    };
    auto release_pending = [&]() {            // after a __syncthreads that followed fence_pending()
        if (pend_slot >= 0) {
            if (tid == 0) {
                const Ring rg = ring_of(a, pend_s, pend_h);
                rg.gamma_c[pend_slot] = pend_gamma;
                __threadfence();
                st_release(rg.full + pend_slot, pend_c + 1);
            }
            pend_slot = -1;
        }
    };

    // Work items (chunk, slot, key head) in chunk order, claimed from a counter: a slower SM simply
    // takes fewer.  Every wait of an item refers to a smaller chunk, whose item was claimed earlier.
    const int n_chunks = (L + kC - 1) / kC;
    const int n_items = n_chunks * a.ns * Hk;
    auto claim = [&]() -> int {
        volatile int *ip = reinterpret_cast<volatile int *>(sm + kItem);
        if (tid == 0) *ip = atomicAdd(a.counter, 1);
        __syncthreads();
        const int v = *ip;
        __syncthreads();
        return v;
    };
    auto decode = [&](int item, int &c, int &s, int &kh) {
        c = item / (a.ns * Hk);
        const int r2 = item % (a.ns * Hk);
        s = a.slot0 + r2 / Hk;
        kh = r2 % Hk;
    };
    int item = claim();
    if (item >= n_items) return;
    {
        int c0, s0, kh0;
        decode(item, c0, s0, kh0);
        if (tid == 0) issue_qk(c0, s0, kh0);
        load_gates(c0, s0, kh0 * R);
    }

    while (item < n_items) {
        const int next = claim();
        int c, s, kh;
        decode(item, c, s, kh);
        const int t0 = c * kC, n = min(kC, L - t0);
        const int slot = c % kRing;

        // ---------------- (a) q, k of the key head: conv + SiLU -> TMEM, L2 norms, G = [K; Q] K^T
        if (c == 0) {
            for (int it = tid; it < 3 * (2 * kD / 4); it += kThreads) {   // conv state rows of q, k (fp32)
                const int row = it / (2 * kD / 4), ch = 4 * (it % (2 * kD / 4));
                const int g = ch < kD ? kh * kD + ch : Hk * kD + kh * kD + (ch - kD);
                *reinterpret_cast<float4 *>(hist + row * 2 * kD + ch) =
                    *reinterpret_cast<const float4 *>(a.conv_state + ((size_t)s * 3 + row) * C + g);
            }
        }
        x.wait_bar(rawbar, raw_phase);
        __syncthreads();
        // item = (channel, 16-token segment); the warp's TMEM lane quarter is (ch % 128) / 32 = warp % 4;
        // the warp also sums y^2 over its 32 channels per token (reduce-scatter, fixed order)
#pragma unroll 1
        for (int k = 0; k < 4; ++k) {
            const int it = tid + k * kThreads;
            const int ch = it % (2 * kD), tb = 16 * (it / (2 * kD));
            const int g = ch < kD ? kh * kD + ch : Hk * kD + kh * kD + (ch - kD);
            float yv[16], y2[16];
            conv16(rawA + (ch >> 7) * (kWin * kD) + (ch & (kD - 1)), hist + ch, 2 * kD, g, tb, c, n, yv);
            tmem_st16(tmem + tq + (ch < kD ? kColQ : kColK) + tb, yv);
#pragma unroll
            for (int j = 0; j < 16; ++j) y2[j] = yv[j] * yv[j];
#pragma unroll
            for (int j = 0; j < 16; ++j) y2[j] += __shfl_xor_sync(0xffffffffu, y2[j], 16);
#pragma unroll
            for (int off = 8; off >= 1; off >>= 1) {
                const bool upper = (lane & off) != 0;
#pragma unroll
                for (int i = 0; i < off; ++i) {
                    const float send = upper ? y2[i] : y2[i + off];
                    const float keep = upper ? y2[i + off] : y2[i];
                    y2[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                }
            }
            if (lane < 16) ssq[(ch >> 5) * kC + tb + lane] = y2[0];   // token tb + lane, channel block ch/32
        }
        tmem_wait_st();
        fence_pending();
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
        release_pending();
        // inverse L2 norms of the q and k rows (a zero padded row stays zero)
        if (tid < 2 * kC) {
            const int t = tid & (kC - 1), part = tid >> 6;
            const float *p = ssq + part * 4 * kC + t;
            const float sum = (p[0] + p[kC]) + (p[2 * kC] + p[3 * kC]);
            (part ? invk : invq)[t] = 1.0f / sqrtf(sum + a.l2_eps);
        }
        __syncthreads();
        {
            // K^ and Q^ as fp32 rows of RA (rows 0-63: K^ tokens, rows 64-127: Q^ tokens; the raw window is
            // consumed): this thread holds channel i = tl of 32 tokens and writes column i
            float *Xr = reinterpret_cast<float *>(RA);
            float x32[32];
            tmem_ld16(tmem + tq + kColK + 32 * half, x32);
            tmem_ld16(tmem + tq + kColK + 32 * half + 16, x32 + 16);
#pragma unroll
            for (int q = 0; q < 32; ++q) Xr[(32 * half + q) * kXStride + tl] = x32[q] * invk[32 * half + q];
            tmem_ld16(tmem + tq + kColQ + 32 * half, x32);
            tmem_ld16(tmem + tq + kColQ + 32 * half + 16, x32 + 16);
#pragma unroll
            for (int q = 0; q < 32; ++q) Xr[(kC + 32 * half + q) * kXStride + tl] = x32[q] * invq[32 * half + q];
        }
        __syncthreads();
        {
            // G = [K^; Q^] K^T in fp32 FMA chains, thread (row r = tl, column half) taking G[r][32 half ..
            // 32 half + 31].  These are dot products of unit vectors that nearly cancel (q.k ~ 1e-2 from terms
            // summing to ~1 in magnitude), and the per-token RMSNorm rescales tokens whose output is small:
            // with the tensor core's split operands (error ~2^-22 of the terms) and its truncating
            // accumulation, rare outputs of the 8192-token layer were measured outside the tolerance, so this
            // product is taken at full fp32 precision.  The result goes to TMEM where the value-head phases
            // read it (lane = row r, column = s).
            const float *Xr = reinterpret_cast<const float *>(RA);
            const float4 *xrow = reinterpret_cast<const float4 *>(Xr + tl * kXStride);
            const float *krows = Xr + 32 * half * kXStride;
            float acc[32];
#pragma unroll
            for (int q = 0; q < 32; ++q) acc[q] = 0.f;
#pragma unroll 2
            for (int i4 = 0; i4 < kD / 4; ++i4) {
                const float4 xv = xrow[i4];
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    const float4 kv = *reinterpret_cast<const float4 *>(krows + q * kXStride + 4 * i4);
                    acc[q] = fmaf(xv.x, kv.x, acc[q]);
                    acc[q] = fmaf(xv.y, kv.y, acc[q]);
                    acc[q] = fmaf(xv.z, kv.z, acc[q]);
                    acc[q] = fmaf(xv.w, kv.w, acc[q]);
                }
            }
            tmem_st16(tmem + tq + kColG + 32 * half, acc);
            tmem_st16(tmem + tq + kColG + 32 * half + 16, acc + 16);
            tmem_wait_st();
        }
        x.publish();                                        // G stays in TMEM for every value head
        if (tid == 0) issue_v(c, s, kh * R);

        for (int hi = 0; hi < R; ++hi) {
            const int h = kh * R + hi;
            const Ring ring = ring_of(a, s, h);
            unsigned char *dst_slot = ring.slots + (size_t)slot * kSlotBytes;

            // ---------------- (b) gates of the head; v conv -> v^T scratch
            if (tid < kC) {                    // padded tokens: no decay, no write
                float lg = 0.f, b = 0.f;
                if (tid < n) {
                    const float xx = g_alpha + __ldg(a.dt_bias + h);
                    const float sp = xx > 20.0f ? xx : log1pf(expf(xx));
                    lg = -expf(__ldg(a.A_log + h)) * sp;
                    b = 1.0f / (1.0f + expf(-g_beta));
                }
                logG[tid] = lg;
                betas[tid] = b;
            }
            if (c == 0) {
                for (int it = tid; it < 3 * (kD / 4); it += kThreads) {   // conv state rows of v (fp32)
                    const int row = it / (kD / 4), ch = 4 * (it % (kD / 4));
                    *reinterpret_cast<float4 *>(hist + row * kD + ch) = *reinterpret_cast<const float4 *>(
                        a.conv_state + ((size_t)s * 3 + row) * C + 2 * Hk * kD + h * kD + ch);
                }
            }
            x.wait_bar(rawbar, raw_phase);
            __syncthreads();
            if (wid == 0) {
                // cumulative log decays as (hi, lo) pairs, Gamma = exp(cumsum(log g)): lane l owns tokens
                // 2l, 2l+1; an inclusive scan of the lane totals, then each token from the previous lane's
                const float l0 = logG[2 * lane], l1 = logG[2 * lane + 1];
                float h, lo;
                add_pair(l0, 0.f, l1, 0.f, h, lo);
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float yh = __shfl_up_sync(0xffffffffu, h, off), yl = __shfl_up_sync(0xffffffffu, lo, off);
                    if (lane >= off) add_pair(h, lo, yh, yl, h, lo);
                }
                float ph = __shfl_up_sync(0xffffffffu, h, 1), pl = __shfl_up_sync(0xffffffffu, lo, 1);
                if (lane == 0) ph = pl = 0.f;
                float h0, lo0, h1, lo1;
                add_pair(ph, pl, l0, 0.f, h0, lo0);
                add_pair(h0, lo0, l1, 0.f, h1, lo1);
                logG[2 * lane] = h0;
                logG[2 * lane + 1] = h1;
                logLo[2 * lane] = lo0;
                logLo[2 * lane + 1] = lo1;
                gam[2 * lane] = expf(h0 + lo0);
                gam[2 * lane + 1] = expf(h1 + lo1);
            }
#pragma unroll 1
            for (int k = 0; k < 2; ++k) {
                const int it = tid + k * kThreads;
                const int ch = it % kD, tb = 16 * (it / kD);
                float yv[16];
                conv16(rawA + ch, hist + ch, kD, 2 * Hk * kD + h * kD + ch, tb, c, n, yv);
                float4 *dv = reinterpret_cast<float4 *>(vT + ch * kVtStride + tb);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4)
                    dv[q4] = make_float4(yv[4 * q4], yv[4 * q4 + 1], yv[4 * q4 + 2], yv[4 * q4 + 3]);
            }
            fence_pending();
            __syncthreads();
            release_pending();
            // this thread's row of v^T for the A2 operand below, fetched ahead of the readout
            float4 vpre[8];
            {
                const float4 *vrow = reinterpret_cast<const float4 *>(vT + tl * kVtStride + 32 * half);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) vpre[q4] = vrow[q4];
            }

            // ---------------- (c) A and the masked, decayed P from G
            {
                float g32[32];
                tmem_ld16(tmem + tq + kColG + 32 * half, g32);
                tmem_ld16(tmem + tq + kColG + 32 * half + 16, g32 + 16);
                if (tl < kC) {                 // A[r][s] = beta_r Gamma_r / Gamma_s k_r.k_s for s < r
                    const int r = tl;
                    const float br = betas[r], lr = logG[r], lrl = logLo[r];
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        const int sc = 32 * half + q;
                        AMt[sc * kC + r] = sc < r ? br * __expf((lr - logG[sc]) + (lrl - logLo[sc])) * g32[q] : 0.f;
                    }
                } else {                       // P[r][s] = q_r.k_s Gamma_r / Gamma_s for s <= r
                    const int r = tl - kC;
                    const float lr = logG[r], lrl = logLo[r];
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        const int sc = 32 * half + q;
                        Pt[sc * kC + r] = sc <= r ? __expf((lr - logG[sc]) + (lrl - logLo[sc])) * g32[q] : 0.f;
                    }
                }
            }
            __syncthreads();
            // A1 = (diag(beta Gamma) K^)^T, A2 = (diag(beta) V)^T -> RA: warp (quarter, half) builds rows
            // 32 quarter .. +31 of tokens 32 half .. +31
            auto build_a12 = [&]() {
                float x32[32];
                tmem_ld16(tmem + tq + kColK + 32 * half, x32);
                tmem_ld16(tmem + tq + kColK + 32 * half + 16, x32 + 16);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                    float ka[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int sr = 32 * half + 4 * q4 + e;
                        ka[e] = betas[sr] * gam[sr] * invk[sr] * x32[4 * q4 + e];
                    }
                    put4(RA, RA + 32 * 1024, tl, 8 * half + q4, 64, make_float4(ka[0], ka[1], ka[2], ka[3]));
                }
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                    const float4 v = vpre[q4];
                    const int sr = 32 * half + 4 * q4;
                    put4(RA + 64 * 1024, RA + 96 * 1024, tl, 8 * half + q4, 64,
                         make_float4(betas[sr] * v.x, betas[sr + 1] * v.y, betas[sr + 2] * v.z, betas[sr + 3] * v.w));
                }
            };
            // ---------------- (d) T = (I + A)^-1, 16 x 16 blocks
            // diagonal blocks: forward substitution, one column per thread, in registers, by warps 6-7
            // while warps 0-5 build their rows of the A1 / A2 operands (RA: the v tile is consumed)
            if (wid >= 6) {
                const int b = (tid - 192) >> 4, col = tid & 15, o = 16 * b;
                float tc[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    float acc = r == col ? 1.f : 0.f;
#pragma unroll
                    for (int m = 0; m < r; ++m) acc = fmaf(-AMt[(o + m) * kC + o + r], tc[m], acc);
                    tc[r] = acc;
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) Tm[(o + r) * kC + o + col] = tc[r];
                for (int r = 0; r < 16; ++r)          // the strictly upper blocks of this block column are zero
                    for (int bb = 0; bb < b; ++bb) Tm[(16 * bb + r) * kC + o + col] = 0.f;
            } else {
                build_a12();
            }
            __syncthreads();
            // off-diagonal blocks by distance: T_ij = -T_ii sum_{k=j}^{i-1} A_ik T_kj
            for (int dist = 1; dist < 4; ++dist) {
                const int nb = 4 - dist;               // blocks (j + dist, j), j < nb
                for (int e = tid; e < nb * 256; e += kThreads) {
                    const int j = e >> 8, rr = (e >> 4) & 15, cc = e & 15, i = j + dist;
                    float acc = 0.f;
                    for (int kb = j; kb < i; ++kb)
#pragma unroll
                        for (int m = 0; m < 16; ++m)
                            acc = fmaf(AMt[(16 * kb + m) * kC + 16 * i + rr], Tm[(16 * kb + m) * kC + 16 * j + cc], acc);
                    Xb[e] = acc;
                }
                __syncthreads();
                for (int e = tid; e < nb * 256; e += kThreads) {
                    const int j = e >> 8, rr = (e >> 4) & 15, cc = e & 15, i = j + dist;
                    float acc = 0.f;
#pragma unroll
                    for (int m = 0; m < 16; ++m)
                        acc = fmaf(Tm[(16 * i + rr) * kC + 16 * i + m], Xb[(j << 8) + m * 16 + cc], acc);
                    Tm[(16 * i + rr) * kC + 16 * j + cc] = -acc;
                }
                __syncthreads();
            }
            // B = T (64 x 64) in RB[0, 32K); warps 6-7 build their rows of A1 / A2 now
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                int r, k4;
                item_rc(tid + k * kThreads, 64, r, k4);
                put4(RB, RB + 16 * 1024, r, k4, 64, *reinterpret_cast<const float4 *>(Tm + r * kC + 4 * k4));
            }
            if (wid >= 6) build_a12();
            x.publish();
            if (tid == 0) mma3(tmem + kColWT, sRA, sRA + 32 * 1024, sRB, sRB + 16 * 1024, 64, 64, false);
            else if (tid == 32) mma3(tmem + kColUT, sRA + 64 * 1024, sRA + 96 * 1024, sRB, sRB + 16 * 1024, 64, 64, false);
            x.commit_wait2();

            // the A region is free: fetch the next tile (next head's v, or the next chunk's q, k) and gates
            if (hi + 1 < R) {
                if (tid == 0) issue_v(c, s, h + 1);
                load_gates(c, s, h + 1);
            } else if (next < n_items) {
                int c2, s2, kh2;
                decode(next, c2, s2, kh2);
                if (tid == 0) issue_qk(c2, s2, kh2);
                load_gates(c2, s2, kh2 * R);
            }

            // ---------------- (e) publish (chunk, head) to the head's ring: every operand goes from
            // registers straight to the slot (16-byte stores into L2), in the layout the state CTA copies in
            if (c >= kRing) x.wait_flag(ring.empty + slot, c - kRing + 1);   // the state CTA took c - kRing
            {
                // -W planes, rows 0-63 of the B operand: this thread holds W[r][i = tl] for its 32 values of r
                float x32[32];
                tmem_ld16(tmem + tq + kColWT + 32 * half, x32);
                tmem_ld16(tmem + tq + kColWT + 32 * half + 16, x32 + 16);
#pragma unroll
                for (int q = 0; q < 32; ++q) x32[q] = -x32[q];
                put_col32(dst_slot + kSlotB, dst_slot + kSlotB + 64 * 1024, 32 * half, tl, x32);
                // Gamma Q^ planes, rows 64-127 of the B operand
                tmem_ld16(tmem + tq + kColQ + 32 * half, x32);
                tmem_ld16(tmem + tq + kColQ + 32 * half + 16, x32 + 16);
#pragma unroll
                for (int q = 0; q < 32; ++q) x32[q] *= gam[32 * half + q] * invq[32 * half + q];
                put_col32(dst_slot + kSlotB, dst_slot + kSlotB + 64 * 1024, kC + 32 * half, tl, x32);
                // U~^T fp32 [j = tl][r]
                tmem_ld16(tmem + tq + kColUT + 32 * half, x32);
                tmem_ld16(tmem + tq + kColUT + 32 * half + 16, x32 + 16);
                float4 *urow = reinterpret_cast<float4 *>(dst_slot + kSlotU + (tl * kC + 32 * half) * 4);
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4)
                    urow[q4] = make_float4(x32[4 * q4], x32[4 * q4 + 1], x32[4 * q4 + 2], x32[4 * q4 + 3]);
                // (Gamma_C / Gamma) K^ planes, as (128 x 64): row i = tl, tokens along K
                tmem_ld16(tmem + tq + kColK + 32 * half, x32);
                tmem_ld16(tmem + tq + kColK + 32 * half + 16, x32 + 16);
                const float lc = logG[kC - 1], lcl = logLo[kC - 1];
#pragma unroll
                for (int q4 = 0; q4 < 8; ++q4) {
                    float ka[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int sr = 32 * half + 4 * q4 + e;
                        ka[e] = __expf((lc - logG[sr]) + (lcl - logLo[sr])) * invk[sr] * x32[4 * q4 + e];
                    }
                    put4(dst_slot + kSlotKd, dst_slot + kSlotKd + 32 * 1024, tl, 8 * half + q4, 64,
                         make_float4(ka[0], ka[1], ka[2], ka[3]));
                }
            }
            // P planes (64 x 64)
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                int r, k4;
                item_rc(tid + k * kThreads, 64, r, k4);
                float p[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) p[e] = Pt[(4 * k4 + e) * kC + r];
                put4(dst_slot + kSlotP, dst_slot + kSlotP + 16 * 1024, r, k4, 64, make_float4(p[0], p[1], p[2], p[3]));
            }
            pend_slot = c == a.drop_chunk ? -1 : slot;   // released one phase later (or at the end)
            pend_c = c;
            pend_h = h;
            pend_s = s;
            pend_gamma = gam[kC - 1];
            __syncthreads();
        }
        item = next;
    }
    fence_pending();
    __syncthreads();
    release_pending();
}

// ---------------------------------------------------------------------------
// state CTA: every chunk in order
// ---------------------------------------------------------------------------
template <typename Act>
__device__ __forceinline__ void advance_state(const PrefillArgs &a, Ctx &x, int s, int h) {
    unsigned char *sm = x.sm;
    const int tid = x.tid, lane = x.lane, wid = x.wid, tl = x.tl, half = x.half;
    const int Hv = a.Hv, L = a.L;
    const uint32_t tmem = x.tmem, tq = x.tq;
    float *rinv = reinterpret_cast<float *>(sm + kRinv);
    float *red = reinterpret_cast<float *>(sm + kRed);
    unsigned char *RA = sm + kRA;
    const uint32_t sRA = smem_u32(RA), sRB = smem_u32(sm + kRB);
    const uint32_t ldbar = smem_u32(sm + kRawBar), zbar = smem_u32(sm + kZBar);
    uint32_t ld_phase = 0, z_phase = 0;
    const Ring ring = ring_of(a, s, h);
    Act *out = static_cast<Act *>(a.out);
    const Act *z = static_cast<const Act *>(a.z);

    // thread (j = tl, half) keeps S^T[j][64 half .. 64 half + 63] = S[i][j]
    float St[64];
    {
        const float *src = a.state + (((size_t)s * Hv + h) * kD + tl) * kD + 64 * half;
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const float4 v = *reinterpret_cast<const float4 *>(src + 4 * q);
            St[4 * q] = v.x; St[4 * q + 1] = v.y; St[4 * q + 2] = v.z; St[4 * q + 3] = v.w;
        }
    }

    const int n_chunks = (L + kC - 1) / kC;
    for (int c = 0; c < n_chunks; ++c) {
        const int t0 = c * kC, n = min(kC, L - t0);
        const int slot = c % kRing;
        const unsigned char *src_slot = ring.slots + (size_t)slot * kSlotBytes;

        if constexpr (sizeof(Act) == 2) {       // the gate (z) tile of this chunk -> AMt region
            if (tid == 0) {
                mbar_arrive_expect_tx(zbar, (uint32_t)(kC * kD * sizeof(Act)));
                tma_load_2d(smem_u32(sm + kAM), &a.z_map, h * kD, s * L + t0, zbar);
            }
        }
        x.wait_flag(ring.full + slot, c + 1);
        if (tid == 0) {
            fence_proxy_async_global();
            mbar_arrive_expect_tx(ldbar, 160 * 1024);
            bulk_g2s(sRA, src_slot + kSlotB, 128 * 1024, ldbar);          // [-W; Gamma Q] hi | lo
            bulk_g2s(sRB, src_slot + kSlotP, 32 * 1024, ldbar);           // P hi | lo
        }
        // U~^T row j = tl, tokens 32 half .. 32 half + 31; Gamma_C
        float u32[32];
        {
            const float4 *urow = reinterpret_cast<const float4 *>(src_slot + kSlotU + (tl * kC + 32 * half) * 4);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                const float4 v = urow[q4];
                u32[4 * q4] = v.x; u32[4 * q4 + 1] = v.y; u32[4 * q4 + 2] = v.z; u32[4 * q4 + 3] = v.w;
            }
        }
        const float gc = ring.gamma_c[slot];
        // A = S0^T into TMEM as tf32 hi / lo columns (this thread: row j = tl, columns 64 half .. +63)
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            float hi16[16], lo16[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) split_tf32(St[16 * q4 + e], hi16[e], lo16[e]);
            tmem_st16(tmem + tq + kSShi + 64 * half + 16 * q4, hi16);
            tmem_st16(tmem + tq + kSSlo + 64 * half + 16 * q4, lo16);
        }
        tmem_wait_st();
        x.wait_bar(ldbar, ld_phase);
        x.publish();
        // [X^T | O^T] = S0^T [-W; Gamma Q]^T  (N 128: X^T in the first 64 columns, O^T in the next 64)
        if (tid == 0) mma3_ts(tmem + kSX, tmem + kSShi, tmem + kSSlo, sRA, sRA + 64 * 1024, 128, 128, false);
        x.commit_wait();
        if (tid == 0) {
            mbar_arrive_expect_tx(ldbar, 64 * 1024);
            bulk_g2s(sRA, src_slot + kSlotKd, 64 * 1024, ldbar);          // (Gamma_C/Gamma) K hi | lo
        }
        {
            // U^T = U~^T + X^T, into TMEM as tf32 hi (over X^T) / lo columns
            float x32[32];
            tmem_ld16(tmem + tq + kSX + 32 * half, x32);
            tmem_ld16(tmem + tq + kSX + 32 * half + 16, x32 + 16);
#pragma unroll
            for (int q = 0; q < 32; ++q) u32[q] += x32[q];
#pragma unroll
            for (int q2 = 0; q2 < 2; ++q2) {
                float hi16[16], lo16[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) split_tf32(u32[16 * q2 + e], hi16[e], lo16[e]);
                tmem_st16(tmem + tq + kSX + 32 * half + 16 * q2, hi16);
                tmem_st16(tmem + tq + kSUlo + 32 * half + 16 * q2, lo16);
            }
            tmem_wait_st();
        }
        x.wait_bar(ldbar, ld_phase);
        if (tid == 0) st_release(ring.empty + slot, c + 1);     // the slot's bytes are all on chip
        x.publish();
        // O2^T = U^T P^T (its own accumulator);  D2 = U^T (diag(Gamma_C / Gamma) K)
        if (tid == 0) mma3_ts(tmem + kSO2, tmem + kSX, tmem + kSUlo, sRB, sRB + 16 * 1024, 64, 64, false);
        else if (tid == 32) mma3_ts(tmem + kSShi, tmem + kSX, tmem + kSUlo, sRA, sRA + 32 * 1024, 64, 128, false);
        float zg[32];
        if constexpr (sizeof(Act) == 2) {
            x.wait_bar(zbar, z_phase);
            const Act *zs = reinterpret_cast<const Act *>(sm + kAM);       // [64 tokens][128]
#pragma unroll
            for (int q = 0; q < 32; ++q) zg[q] = to_f32(zs[(32 * half + q) * kD + tl]);
        } else {
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                const int t = 32 * half + q;
                zg[q] = t < n ? to_f32(z[((size_t)s * L + t0 + t) * Hv * kD + (size_t)h * kD + tl]) : 0.f;
            }
        }
        x.commit_wait2();

        // ---------------- outputs (gated RMSNorm) and the state update
        {
            float o32[32], p32[32];
            tmem_ld16(tmem + tq + kSO + 32 * half, o32);
            tmem_ld16(tmem + tq + kSO + 32 * half + 16, o32 + 16);
            tmem_ld16(tmem + tq + kSO2 + 32 * half, p32);
            tmem_ld16(tmem + tq + kSO2 + 32 * half + 16, p32 + 16);
#pragma unroll
            for (int q = 0; q < 32; ++q) o32[q] += p32[q];
            // per-token sums of squares over this warp's 32 columns: reduce-scatter, lane l ends with token l
            float v[32];
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                o32[q] *= a.q_scale;
                v[q] = o32[q] * o32[q];
            }
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                const bool upper = (lane & off) != 0;
#pragma unroll
                for (int i = 0; i < off; ++i) {
                    const float send = upper ? v[i] : v[i + off];
                    const float keep = upper ? v[i + off] : v[i];
                    v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                }
            }
            red[(wid & 3) * 64 + 32 * half + lane] = v[0];                  // lane quarter x token
            __syncthreads();
            if (tid < kC) {
                const float tot = (red[tid] + red[64 + tid]) + (red[128 + tid] + red[192 + tid]);
                rinv[tid] = 1.0f / sqrtf(tot / float(kD) + a.rms_eps);
            }
            __syncthreads();
            const float nw = __ldg(a.norm_w + tl);
#pragma unroll
            for (int q = 0; q < 32; ++q) {
                const int t = 32 * half + q;
                if (t < n) {
                    const size_t o_idx = ((size_t)s * L + t0 + t) * Hv * kD + (size_t)h * kD + tl;
                    out[o_idx] = from_f32<Act>(o32[q] * rinv[t] * nw * silu(zg[q]));
                }
            }
            // S^T <- Gamma_C S^T + D2
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                float d16[16];
                tmem_ld16(tmem + tq + kSShi + 64 * half + 16 * q4, d16);
#pragma unroll
                for (int e = 0; e < 16; ++e) St[16 * q4 + e] = fmaf(gc, St[16 * q4 + e], d16[e]);
            }
        }
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
    }

    float *dst = a.state + (((size_t)s * Hv + h) * kD + tl) * kD + 64 * half;
#pragma unroll
    for (int q = 0; q < 16; ++q)
        *reinterpret_cast<float4 *>(dst + 4 * q) = make_float4(St[4 * q], St[4 * q + 1], St[4 * q + 2], St[4 * q + 3]);
}

// grid: n_prep preparation CTAs (claiming work items), then ns x H_v state CTAs
template <typename Act>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ PrefillArgs a) {
    extern __shared__ __align__(1024) unsigned char sm[];
    Ctx x;
    x.sm = sm;
    x.tid = threadIdx.x; x.lane = x.tid & 31; x.wid = x.tid >> 5;
    x.tl = x.tid & 127; x.half = x.tid >> 7;           // TMEM lane of this thread, column half
    x.phase = 0;
    x.phase2 = 0;
    x.timed_out = false;
    const int n_prep = a.n_prep;
    const bool prep = (int)blockIdx.x < n_prep;
    const int sidx = (int)blockIdx.x - n_prep;

    if (x.wid == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(
                         smem_u32(sm + kTmemSlot)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n");
    }
    x.mbar = smem_u32(sm + kMbar);
    x.mbar2 = smem_u32(sm + kMbar2);
    if (x.tid == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(x.mbar));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(x.mbar2));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(sm + kRawBar)));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(smem_u32(sm + kZBar)));
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    x.tmem = *reinterpret_cast<volatile uint32_t *>(sm + kTmemSlot);
    x.tq = (uint32_t)(32 * (x.wid & 3)) << 16;        // this warp's TMEM lane quarter

    if (prep) prepare<Act>(a, x);
    else advance_state<Act>(a, x, a.slot0 + sidx / a.Hv, sidx % a.Hv);

    if (x.timed_out && x.tid == 0 && a.d_status) atomicCAS(a.d_status, int(GDN_OK), int(GDN_ERR_TIMEOUT));
    fence_before_sync();
    __syncthreads();
    if (x.wid == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(x.tmem), "r"(kTmemCols));
}

// conv state after the prompt: the last three raw inputs (rows before the prompt shift in from the
// old conv state when L < 3).  One thread per (slot, channel), in place.
template <typename Act>
__global__ void __launch_bounds__(256) prefill_conv_state_kernel(const Act *qkv, float *conv_state, int L, int C) {
    const int g = blockIdx.x * blockDim.x + threadIdx.x, s = blockIdx.y;
    if (g >= C) return;
    float *cs = conv_state + (size_t)s * 3 * C + g;
    float nv[3];
#pragma unroll
    for (int rr = 0; rr < 3; ++rr) {
        const int t = L - 3 + rr;
        nv[rr] = t >= 0 ? to_f32(qkv[((size_t)s * L + t) * C + g]) : cs[(size_t)(3 + t) * C];
    }
#pragma unroll
    for (int rr = 0; rr < 3; ++rr) cs[(size_t)rr * C] = nv[rr];
}

}  // namespace

int prefill_check(const gdn_dims &d, std::string &why) {
    if (d.d_k != kD || d.d_v != kD) {
        why = "prefill: d_k and d_v must be 128";
        return GDN_ERR_SHAPE;
    }
    if (d.n_slots > 65535) {
        why = "prefill: n_slots must be <= 65535";
        return GDN_ERR_SHAPE;
    }
    if ((long long)d.n_slots * d.n_tokens >= (1LL << 31)) {
        why = "prefill: n_slots * n_tokens must be below 2^31";
        return GDN_ERR_SHAPE;
    }
    if (d.n_v_heads + d.n_qk_heads > 150) {
        why = "prefill: a slot's CTAs (H_v state + at least H_k preparation) must fit on the device at once";
        return GDN_ERR_SHAPE;
    }
    return GDN_OK;
}

// workspace: ring flags of every (slot, value head), then one work counter per launch
static size_t counters_offset_bytes(const gdn_dims &d) {
    return (size_t)d.n_slots * d.n_v_heads * kFlagWords * sizeof(int);
}
static size_t ring_offset_bytes(const gdn_dims &d) {
    const size_t head = counters_offset_bytes(d) + (size_t)d.n_slots * sizeof(int);
    return (head + 255) & ~(size_t)255;
}

size_t prefill_workspace_bytes(const gdn_dims &d) {
    const size_t pairs = (size_t)d.n_slots * d.n_v_heads;
    return ring_offset_bytes(d) + pairs * kRing * kSlotBytes;
}

cudaError_t launch_prefill(const gdn_dims &d, const gdn_layer_params &p, const void *qkv, const void *z,
                           const void *alpha, const void *beta_raw, float *state, float *conv_state,
                           void *out, void *workspace, int *d_status, cudaStream_t stream) {
    PrefillArgs a{};
    a.B = d.n_slots; a.Hk = d.n_qk_heads; a.Hv = d.n_v_heads; a.L = d.n_tokens;
    a.C = 2 * d.n_qk_heads * kD + d.n_v_heads * kD; a.r = d.n_v_heads / d.n_qk_heads;
    a.rms_eps = d.rms_eps; a.l2_eps = d.l2_eps; a.q_scale = d.q_scale;
    a.conv_w = p.conv_w; a.A_log = p.A_log; a.dt_bias = p.dt_bias; a.norm_w = p.norm_w;
    a.qkv = qkv; a.z = z; a.alpha = alpha; a.beta_raw = beta_raw;
    a.state = state; a.conv_state = conv_state; a.out = out;
    a.scratch = static_cast<float *>(workspace);
    a.ring_offset = ring_offset_bytes(d);
    a.n_prep = 1;
    a.d_status = d_status;
#if GDN_CHECKED
    // Test build only (the ordinary library never reads the environment): fault injection on the host.
    // GDN_FAULT_DROP_CHUNK=<c> makes the preparation CTAs never publish chunk c, so the state CTA's
    // bounded wait runs out and the call reports GDN_ERR_TIMEOUT through d_status (the outputs are then
    // undefined; nothing faults or hangs).
    const char *drop = getenv("GDN_FAULT_DROP_CHUNK");
    a.drop_chunk = drop ? atoi(drop) : -1;
#else
    a.drop_chunk = -1;
#endif
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return cudaErrorNotSupported;
    const bool bf = d.act_dtype == GDN_BF16;
    const CUtensorMapDataType dt = bf ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    const cuuint32_t esz = bf ? 2u : 4u;
    const cuuint32_t estr[2] = {1, 1};
    const cuuint64_t dims[2] = {(cuuint64_t)a.C, (cuuint64_t)a.B * (cuuint64_t)a.L};
    const cuuint64_t strides[1] = {(cuuint64_t)a.C * esz};
    const cuuint32_t box[2] = {(cuuint32_t)kD, (cuuint32_t)kWin};
    if (encode(&a.qkv_map, dt, 2, const_cast<void *>(qkv), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
    const cuuint64_t zdims[2] = {(cuuint64_t)a.Hv * kD, (cuuint64_t)a.B * (cuuint64_t)a.L};
    const cuuint64_t zstrides[1] = {(cuuint64_t)a.Hv * kD * esz};
    const cuuint32_t zbox[2] = {(cuuint32_t)kD, (cuuint32_t)kC};
    if (encode(&a.z_map, dt, 2, const_cast<void *>(z), zdims, zstrides, zbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;

    void (*kern)(PrefillArgs) = bf ? prefill_kernel<__nv_bfloat16> : prefill_kernel<float>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemBytes));
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, kSmemBytes)) != cudaSuccess)
        return e;
    // every CTA of a launch must be resident at once: H_v state CTAs per slot, and the remaining
    // SMs as a pool of preparation CTAs that share all the launch's work items
    const int max_ctas = sms * per_sm;
    if (a.Hv + 1 > max_ctas) return cudaErrorCooperativeLaunchTooLarge;
    int slots_per_launch = max_ctas / (a.Hv + 2 * a.Hk);
    if (slots_per_launch < 1) slots_per_launch = 1;
    // fresh ring flags (and slot decays) for every (slot, head), fresh work counters
    if ((e = cudaMemsetAsync(workspace, 0, a.ring_offset, stream)) != cudaSuccess) return e;
    int *counters = reinterpret_cast<int *>(static_cast<unsigned char *>(workspace) + counters_offset_bytes(d));
    for (int s0 = 0, li = 0; s0 < a.B; s0 += slots_per_launch, ++li) {
        a.slot0 = s0;
        const int ns = a.B - s0 < slots_per_launch ? a.B - s0 : slots_per_launch;
        a.ns = ns;
        a.counter = counters + li;
        int n_prep = max_ctas - ns * a.Hv;
        if (n_prep > ns * a.Hk * kMaxPrep) n_prep = ns * a.Hk * kMaxPrep;
        a.n_prep = n_prep;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(n_prep + ns * a.Hv, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = kSmemBytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if ((e = cudaLaunchKernelEx(&cfg, kern, a)) != cudaSuccess) return e;
    }
    const dim3 cgrid((a.C + 255) / 256, a.B);
    if (bf)
        prefill_conv_state_kernel<__nv_bfloat16><<<cgrid, 256, 0, stream>>>(
            static_cast<const __nv_bfloat16 *>(qkv), conv_state, a.L, a.C);
    else
        prefill_conv_state_kernel<float><<<cgrid, 256, 0, stream>>>(static_cast<const float *>(qkv), conv_state,
                                                                     a.L, a.C);
    return cudaGetLastError();
}

}  // namespace gdn
