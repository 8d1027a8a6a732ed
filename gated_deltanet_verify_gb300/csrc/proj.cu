// proj.cu -- the projections either side of the GDN block as plain bf16 GEMMs
// through cuBLASLt (fp32 accumulation): the fused input projection
// x -> [qkv | z | alpha | beta_raw] and the output projection out -> y.
//
// Row-major C[M][N] (row stride ldc) = X[M][K] @ W[N][K]^T is, in cuBLAS's
// column-major terms, D (N x M, ld ldc) = op_T(A) (N x K) * B (K x M) with A
// the weight stored K x N (ld K) and B the activations stored K x M (ld K):
// the "TN" form, weights K-major.  The matmul descriptor, layouts and the
// algorithm of a shape are chosen once per device and cached.
#include "internal.cuh"

#include <cublasLt.h>

#include <deque>
#include <mutex>

namespace gdn {
namespace {

constexpr int kMaxDevices = 64;

struct Plan {
    int dev, M, N, K;
    long long ldc;
    cublasLtMatmulDesc_t op = nullptr;
    cublasLtMatrixLayout_t a = nullptr, b = nullptr, d = nullptr;
    cublasLtMatmulAlgo_t algo;
    size_t ws_bytes = 0;
};

std::mutex g_mu;
cublasLtHandle_t g_handle[kMaxDevices];
std::deque<Plan> g_plans;           // a deque: references stay valid as plans are added

const char *lt_name(cublasStatus_t s) {
    switch (s) {
        case CUBLAS_STATUS_SUCCESS: return "success";
        case CUBLAS_STATUS_NOT_INITIALIZED: return "not initialised";
        case CUBLAS_STATUS_ALLOC_FAILED: return "allocation failed";
        case CUBLAS_STATUS_INVALID_VALUE: return "invalid value";
        case CUBLAS_STATUS_ARCH_MISMATCH: return "architecture mismatch";
        case CUBLAS_STATUS_EXECUTION_FAILED: return "execution failed";
        case CUBLAS_STATUS_INTERNAL_ERROR: return "internal error";
        case CUBLAS_STATUS_NOT_SUPPORTED: return "not supported";
        default: return "error";
    }
}

#define LT_TRY(call, what)                                                            \
    do {                                                                              \
        cublasStatus_t st_ = (call);                                                  \
        if (st_ != CUBLAS_STATUS_SUCCESS) {                                           \
            why = std::string(what) + ": cuBLASLt " + lt_name(st_);                   \
            return false;                                                             \
        }                                                                             \
    } while (0)

void free_plan(Plan &p) {
    if (p.d) cublasLtMatrixLayoutDestroy(p.d);
    if (p.b) cublasLtMatrixLayoutDestroy(p.b);
    if (p.a) cublasLtMatrixLayoutDestroy(p.a);
    if (p.op) cublasLtMatmulDescDestroy(p.op);
    p.op = nullptr; p.a = p.b = p.d = nullptr;
}

bool make_plan_steps(Plan &p, cublasLtHandle_t h, std::string &why) {
    LT_TRY(cublasLtMatmulDescCreate(&p.op, CUBLAS_COMPUTE_32F, CUDA_R_32F), "matmul descriptor");
    const cublasOperation_t tA = CUBLAS_OP_T, tB = CUBLAS_OP_N;
    LT_TRY(cublasLtMatmulDescSetAttribute(p.op, CUBLASLT_MATMUL_DESC_TRANSA, &tA, sizeof(tA)), "transa");
    LT_TRY(cublasLtMatmulDescSetAttribute(p.op, CUBLASLT_MATMUL_DESC_TRANSB, &tB, sizeof(tB)), "transb");
    LT_TRY(cublasLtMatrixLayoutCreate(&p.a, CUDA_R_16BF, uint64_t(p.K), uint64_t(p.N), int64_t(p.K)), "A layout");
    LT_TRY(cublasLtMatrixLayoutCreate(&p.b, CUDA_R_16BF, uint64_t(p.K), uint64_t(p.M), int64_t(p.K)), "B layout");
    LT_TRY(cublasLtMatrixLayoutCreate(&p.d, CUDA_R_16BF, uint64_t(p.N), uint64_t(p.M), int64_t(p.ldc)), "D layout");
    cublasLtMatmulPreference_t pref = nullptr;
    LT_TRY(cublasLtMatmulPreferenceCreate(&pref), "preference");
    const uint64_t ws = p.ws_bytes;
    cublasStatus_t st = cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws,
                                                             sizeof(ws));
    cublasLtMatmulHeuristicResult_t res = {};
    int n = 0;
    if (st == CUBLAS_STATUS_SUCCESS)
        st = cublasLtMatmulAlgoGetHeuristic(h, p.op, p.a, p.b, p.d, p.d, pref, 1, &res, &n);
    cublasLtMatmulPreferenceDestroy(pref);
    if (st != CUBLAS_STATUS_SUCCESS || n < 1) {
        why = std::string("no cuBLASLt algorithm for the projection GEMM: ") + lt_name(st);
        return false;
    }
    p.algo = res.algo;
    return true;
}

// a plan whose setup failed half way releases what it created
bool make_plan(Plan &p, cublasLtHandle_t h, std::string &why) {
    if (make_plan_steps(p, h, why)) return true;
    free_plan(p);
    return false;
}

}  // namespace

bool gemm_xwt_bf16(const void *W, const void *X, void *C, int M, int N, int K, long long ldc, void *ws,
                   size_t ws_bytes, cudaStream_t stream, std::string &why) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        why = "no usable CUDA device";
        return false;
    }
    const Plan *plan = nullptr;
    cublasLtHandle_t h = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_handle[dev]) LT_TRY(cublasLtCreate(&g_handle[dev]), "handle");
        h = g_handle[dev];
        for (const Plan &p : g_plans)
            if (p.dev == dev && p.M == M && p.N == N && p.K == K && p.ldc == ldc && p.ws_bytes == ws_bytes)
                plan = &p;
        if (!plan) {
            Plan p;
            p.dev = dev; p.M = M; p.N = N; p.K = K; p.ldc = ldc; p.ws_bytes = ws_bytes;
            if (!make_plan(p, h, why)) return false;
            g_plans.push_back(p);
            plan = &g_plans.back();
        }
    }
    const float one = 1.0f, zero = 0.0f;
    LT_TRY(cublasLtMatmul(h, plan->op, &one, W, plan->a, X, plan->b, &zero, C, plan->d, C, plan->d, &plan->algo, ws,
                          ws_bytes, stream),
           "projection GEMM");
    return true;
}

}  // namespace gdn
