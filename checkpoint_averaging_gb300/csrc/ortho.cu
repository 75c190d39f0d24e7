// ortho.cu -- outer orthogonalisation of a plain-mean round: the averaged
// update of every matrix-shaped tensor is replaced by its polar factor
// ("DiffuRefill-1B: Pretraining a Masked Diffusion Language Model on Free,
// Preemptible Notebook GPUs", section 5.3).
//
// Per matrix tensor (row-major m x n):
//   1. Delta = mean_k(x_k) - theta with the plain-mean arithmetic of the fused
//      pass, into a workspace, with |Delta|_F^2 summed in a fixed order;
//   2. X0 = Delta / |Delta|_F, so every singular value lies in (0, 1];
//   3. `iterations` Newton-Schulz steps X <- 1.5 X - 0.5 X (X^T X) (with the
//      smaller Gram matrix), which drive every singular value to 1 and so
//      converge to the polar factor U V^T;
//   4. theta' = theta + s X, s = lr or lr |Delta|_F / sqrt(min(m, n)), then the
//      EMA of the globals.
// The two GEMMs of a step are plain dense contractions and run on the tensor
// cores through cuBLASLt (TF32 inputs with fp32 accumulation, full fp32, or a
// bf16 iterate and Gram matrix with fp32 accumulation),
// loaded with dlopen the first time a context orthogonalises, so the rest of
// the library never depends on it. The element-wise steps are this file's
// kernels.
#include <cublasLt.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <dlfcn.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "cam_internal.h"
#include "side_internal.h"
#include "merge_device.cuh"

namespace cam {
namespace {

// ---- cuBLASLt, resolved at run time ------------------------------------------------

struct LtApi {
    bool ok = false;
    decltype(&cublasLtCreate) create = nullptr;
    decltype(&cublasLtDestroy) destroy = nullptr;
    decltype(&cublasLtMatmulDescCreate) desc_create = nullptr;
    decltype(&cublasLtMatmulDescDestroy) desc_destroy = nullptr;
    decltype(&cublasLtMatmulDescSetAttribute) desc_set = nullptr;
    decltype(&cublasLtMatrixLayoutCreate) layout_create = nullptr;
    decltype(&cublasLtMatrixLayoutDestroy) layout_destroy = nullptr;
    decltype(&cublasLtMatrixLayoutSetAttribute) layout_set = nullptr;
    decltype(&cublasLtMatmulPreferenceCreate) pref_create = nullptr;
    decltype(&cublasLtMatmulPreferenceDestroy) pref_destroy = nullptr;
    decltype(&cublasLtMatmulPreferenceSetAttribute) pref_set = nullptr;
    decltype(&cublasLtMatmulAlgoGetHeuristic) heuristic = nullptr;
    decltype(&cublasLtMatmul) matmul = nullptr;
};

LtApi g_lt;
std::mutex g_lt_mutex;

template <typename F>
bool resolve(void* h, const char* name, F& out) {
    out = reinterpret_cast<F>(dlsym(h, name));
    return out != nullptr;
}

const LtApi* lt_api() {
    std::lock_guard<std::mutex> lock(g_lt_mutex);
    if (g_lt.ok) return &g_lt;
    void* h = dlopen("libcublasLt.so.13", RTLD_NOW | RTLD_GLOBAL);
    if (!h) h = dlopen("/usr/local/cuda/lib64/libcublasLt.so.13", RTLD_NOW | RTLD_GLOBAL);
    if (!h) return nullptr;
    LtApi a;
    bool ok = resolve(h, "cublasLtCreate", a.create) && resolve(h, "cublasLtDestroy", a.destroy) &&
              resolve(h, "cublasLtMatmulDescCreate", a.desc_create) &&
              resolve(h, "cublasLtMatmulDescDestroy", a.desc_destroy) &&
              resolve(h, "cublasLtMatmulDescSetAttribute", a.desc_set) &&
              resolve(h, "cublasLtMatrixLayoutCreate", a.layout_create) &&
              resolve(h, "cublasLtMatrixLayoutDestroy", a.layout_destroy) &&
              resolve(h, "cublasLtMatrixLayoutSetAttribute", a.layout_set) &&
              resolve(h, "cublasLtMatmulPreferenceCreate", a.pref_create) &&
              resolve(h, "cublasLtMatmulPreferenceDestroy", a.pref_destroy) &&
              resolve(h, "cublasLtMatmulPreferenceSetAttribute", a.pref_set) &&
              resolve(h, "cublasLtMatmulAlgoGetHeuristic", a.heuristic) &&
              resolve(h, "cublasLtMatmul", a.matmul);
    if (!ok) return nullptr;
    a.ok = true;
    g_lt = a;
    return &g_lt;
}

constexpr size_t kLtWorkspace = size_t(32) << 20;
constexpr int kOrthoBatchMax = 256;  // matrices orthogonalised together
constexpr int kOrthoBlocksMax = 4096;

// One cached GEMM configuration (column-major D = alpha op(A) op(B) + beta C).
struct GemmPlan {
    int64_t M, N, Kd, lda, ldb, ldc;
    bool ta, tb;
    int precision;
    int32_t batch;                   // matrices per call (strided batch)
    int64_t sa, sb, sc;              // element strides between them
    cublasLtMatmulDesc_t op = nullptr;
    cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
    cublasLtMatmulAlgo_t algo;
};

}  // namespace

// Per-context workspace of the orthogonalisation, made at the first
// orthogonalised commit: two fp32 matrix buffers sized for the context's
// largest matrix, the Gram matrix, reduction partials and a cuBLASLt handle.
struct OrthoWork {
    const LtApi* lt = nullptr;
    cublasLtHandle_t handle = nullptr;
    float* X = nullptr;
    float* Y = nullptr;
    float* G = nullptr;
    double* partials = nullptr;  // [kOrthoBatchMax * kOrthoBlocksMax]
    double* scalars = nullptr;   // [j] = |Delta_j|_F^2
    float* inv_norm = nullptr;   // [j] = 1 / |Delta_j|_F (0 when Delta_j = 0)
    void* lt_ws = nullptr;
    void* block = nullptr;       // one cudaMalloc holding all of the above
    int64_t cap_elems = 0;       // floats in X and in Y
    int64_t cap_gram = 0;        // floats in G
    std::vector<GemmPlan> plans; // cuBLASLt configurations by GEMM shape
};

}  // namespace cam

namespace cam {
namespace {

constexpr int kOrthoThreads = 256;

// Per-group launches: blockIdx.y picks the matrix (slot j of the batch), and
// every matrix keeps the block count its size alone determines, so its
// partials do not depend on the rest of the batch.
struct DeltaArgs {
    const void* x[kOrthoBatchMax][CAM_KMAX];  // [j][k]: worker k's copy of matrix j
    const float* theta[kOrthoBatchMax];
    uint32_t vec[kOrthoBatchMax / 32];        // bit j: matrix j's buffers take 32-byte vectors
    int32_t K;
    float Kf;
    float* X;          // slot j at X + j * n
    int64_t n;         // elements per matrix
    double* partials;  // [j * kOrthoBlocksMax + block]
};

// Delta = (sum_k x_k, arrival order) / K - theta, the plain-mean arithmetic of
// the fused pass, and each block's sum of Delta^2 (fp32 over at most 32
// elements per thread, then fp64, reduced in a fixed order).
template <typename XT>
__global__ void __launch_bounds__(kOrthoThreads) ortho_delta(const __grid_constant__ DeltaArgs a) {
    __shared__ double part[kOrthoThreads / 32];
    const int j = blockIdx.y;
    const void* const* xs = a.x[j];
    const float* theta = a.theta[j];
    float* X = a.X + int64_t(j) * a.n;
    double dacc = 0.0;
    float acc = 0.0f;
    int cnt = 0;
    const int64_t tid = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    int64_t done = 0;
    if ((a.vec[j >> 5] >> (j & 31)) & 1u) {  // 8 elements per step
        const int64_t nv = a.n >> 3;
        for (int64_t v = tid; v < nv; v += stride) {
            dev::XVec<XT> x[CAM_KMAX];
#pragma unroll
            for (int k = 0; k < CAM_KMAX; ++k)
                if (k < a.K) x[k].load(static_cast<const XT*>(xs[k]) + 8 * v);
            float d[8];
            dev::load_s8(theta + 8 * v, d);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float s = 0.0f;
#pragma unroll
                for (int k = 0; k < CAM_KMAX; ++k)
                    if (k < a.K) s = __fadd_rn(s, x[k].get(e));
                d[e] = __fsub_rn(__fdiv_rn(s, a.Kf), d[e]);
                acc = __fmaf_rn(d[e], d[e], acc);
            }
            dev::store_s8(X + 8 * v, d);
            if ((cnt += 8) == 32) {
                dacc += static_cast<double>(acc);
                acc = 0.0f;
                cnt = 0;
            }
        }
        done = 8 * nv;
    }
    for (int64_t i = done + tid; i < a.n; i += stride) {
        float s = 0.0f;
#pragma unroll
        for (int k = 0; k < CAM_KMAX; ++k)
            if (k < a.K) s = __fadd_rn(s, dev::load_x1(static_cast<const XT*>(xs[k]) + i));
        const float d = __fsub_rn(__fdiv_rn(s, a.Kf), theta[i]);
        X[i] = d;
        acc = __fmaf_rn(d, d, acc);
        if (++cnt == 32) {
            dacc += static_cast<double>(acc);
            acc = 0.0f;
            cnt = 0;
        }
    }
    dacc = dev::warp_sum(dacc + static_cast<double>(acc));
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = dacc;
    __syncthreads();
    if (threadIdx.x == 0) {
        double s = 0.0;
        for (int w = 0; w < kOrthoThreads / 32; ++w) s += part[w];
        a.partials[int64_t(j) * kOrthoBlocksMax + blockIdx.x] = s;
    }
}

// |Delta_j|_F^2 in a fixed order, and 1/|Delta_j|_F (0 for a zero update,
// which then stays zero through the iteration and leaves theta unchanged).
// One 32-thread block per matrix.
__global__ void ortho_norm(const double* partials, int nb, double* scalars, float* inv_norm) {
    const int j = blockIdx.x;
    double s = 0.0;
    for (int b = threadIdx.x; b < nb; b += 32) s += partials[int64_t(j) * kOrthoBlocksMax + b];
    s = dev::warp_sum(s);
    if (threadIdx.x == 0) {
        scalars[j] = s;
        inv_norm[j] = s > 0.0 ? static_cast<float>(1.0 / sqrt(s)) : 0.0f;
    }
}

// X_j <- X_j / |Delta_j|_F. Slot j is 32-byte aligned when n is a multiple of 8.
__global__ void ortho_scale(float* X, int64_t n, const float* inv_norm) {
    const int j = blockIdx.y;
    const float f = inv_norm[j];
    float* Xj = X + int64_t(j) * n;
    const int64_t tid = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    int64_t done = 0;
    if ((n & 7) == 0) {
        for (int64_t v = tid; v < (n >> 3); v += stride) {
            float x[8];
            dev::load_s8(Xj + 8 * v, x);
#pragma unroll
            for (int e = 0; e < 8; ++e) x[e] = __fmul_rn(x[e], f);
            dev::store_s8(Xj + 8 * v, x);
        }
        done = n;
    }
    for (int64_t i = done + tid; i < n; i += stride) Xj[i] = __fmul_rn(Xj[i], f);
}

// X_j / |Delta_j|_F (fp32 in X) into the bf16 iterate buffer Y, rounded to
// nearest-even (CAM_ORTHO_BF16).
__global__ void ortho_scale_bf16(const float* X, __nv_bfloat16* Y, int64_t n, const float* inv_norm) {
    const int j = blockIdx.y;
    const float f = inv_norm[j];
    const float* Xj = X + int64_t(j) * n;
    __nv_bfloat16* Yj = Y + int64_t(j) * n;
    const int64_t tid = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    int64_t done = 0;
    if ((n & 7) == 0) {  // 32-byte reads, 16-byte writes (slot bases stay aligned)
        for (int64_t v = tid; v < (n >> 3); v += stride) {
            float x[8];
            dev::load_s8(Xj + 8 * v, x);
            uint4 o;
            uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 b =
                    __floats2bfloat162_rn(__fmul_rn(x[2 * e], f), __fmul_rn(x[2 * e + 1], f));
                ow[e] = *reinterpret_cast<const uint32_t*>(&b);
            }
            *reinterpret_cast<uint4*>(Yj + 8 * v) = o;
        }
        done = n;
    }
    for (int64_t i = done + tid; i < n; i += stride) Yj[i] = __float2bfloat16_rn(__fmul_rn(Xj[i], f));
}

// P_j <- I (r x r) for every slot j; total = slots x r x r.
__global__ void ortho_identity(float* P, int64_t r, int64_t total) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t q = i % (r * r);
        P[i] = (q / r == q % r) ? 1.0f : 0.0f;
    }
}

struct ApplyArgs {
    float* theta[kOrthoBatchMax];
    float* e[kOrthoBatchMax];  // EMA buffers, or null
    uint32_t vec[kOrthoBatchMax / 32];  // bit j: matrix j's buffers take 32-byte vectors
    const void* O;             // the polar factors (fp32, or bf16), slot j at O + j * n
    int64_t n;
    const double* scalars;     // [j] = |Delta_j|_F^2
    float lr;
    int32_t scale_mode;
    int64_t r;                 // min(m, n)
    float beta;
};

// theta' = theta + s O, then e' = beta e + (1 - beta) theta'. OT is the
// polar factor's storage type (float, or bf16 bits widened exactly).
template <typename OT>
__global__ void ortho_apply(const __grid_constant__ ApplyArgs a) {
    const int j = blockIdx.y;
    float* theta = a.theta[j];
    float* e = a.e[j];
    const OT* O = static_cast<const OT*>(a.O) + int64_t(j) * a.n;
    float s = a.lr;
    if (a.scale_mode == CAM_ORTHO_SCALE_MATCH_NORM)
        s = static_cast<float>(static_cast<double>(a.lr) * sqrt(a.scalars[j]) /
                               sqrt(static_cast<double>(a.r)));
    const float omb = __fsub_rn(1.0f, a.beta);
    const int64_t tid = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    int64_t done = 0;
    if ((a.vec[j >> 5] >> (j & 31)) & 1u) {  // 8 elements per step
        const int64_t nv = a.n >> 3;
        for (int64_t v = tid; v < nv; v += stride) {
            float th[8];
            dev::load_s8(theta + 8 * v, th);
            dev::XVec<OT> o;
            o.load(O + 8 * v);
#pragma unroll
            for (int q = 0; q < 8; ++q) th[q] = __fadd_rn(th[q], __fmul_rn(s, o.get(q)));
            dev::store_s8(theta + 8 * v, th);
            if (e) {
                float ev[8];
                dev::load_s8(e + 8 * v, ev);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    ev[q] = __fadd_rn(__fmul_rn(a.beta, ev[q]), __fmul_rn(omb, th[q]));
                dev::store_s8(e + 8 * v, ev);
            }
        }
        done = 8 * nv;
    }
    for (int64_t i = done + tid; i < a.n; i += stride) {
        const float th = __fadd_rn(theta[i], __fmul_rn(s, dev::load_x1(O + i)));
        theta[i] = th;
        if (e) e[i] = __fadd_rn(__fmul_rn(a.beta, e[i]), __fmul_rn(omb, th));
    }
}

}  // namespace
}  // namespace cam

namespace cam {
namespace {

int lt_fail(const char* what, int st) {
    return record_error(CAM_E_CUDA, "orthogonalisation: %s failed (cuBLASLt status %d)", what, st);
}

// Finds or builds the plan for this GEMM shape.
int gemm_plan(OrthoWork* w, int precision, bool ta, bool tb,
              int64_t M, int64_t N, int64_t Kd, int64_t lda, int64_t ldb, int64_t ldc,
              int32_t batch, int64_t sa, int64_t sb, int64_t sc, const GemmPlan** out) {
    std::vector<GemmPlan>& cache = w->plans;
    for (const GemmPlan& p : cache)
        if (p.M == M && p.N == N && p.Kd == Kd && p.lda == lda && p.ldb == ldb && p.ldc == ldc &&
            p.ta == ta && p.tb == tb && p.precision == precision && p.batch == batch &&
            p.sa == sa && p.sb == sb && p.sc == sc) {
            *out = &p;
            return CAM_OK;
        }
    const LtApi& L = *w->lt;
    GemmPlan p{M, N, Kd, lda, ldb, ldc, ta, tb, precision, batch, sa, sb, sc};
    // bf16 operands and results with fp32 accumulation, or fp32 ones in full
    // fp32 or TF32 (inputs rounded to 10-bit mantissas inside the GEMM)
    const cublasComputeType_t ct =
        precision == CAM_ORTHO_TF32 ? CUBLAS_COMPUTE_32F_FAST_TF32 : CUBLAS_COMPUTE_32F;
    const cudaDataType_t dt = precision == CAM_ORTHO_BF16 ? CUDA_R_16BF : CUDA_R_32F;
    int st = L.desc_create(&p.op, ct, CUDA_R_32F);
    if (st != CUBLAS_STATUS_SUCCESS) return lt_fail("matmul descriptor", st);
    const cublasOperation_t oa = ta ? CUBLAS_OP_T : CUBLAS_OP_N, ob = tb ? CUBLAS_OP_T : CUBLAS_OP_N;
    L.desc_set(p.op, CUBLASLT_MATMUL_DESC_TRANSA, &oa, sizeof oa);
    L.desc_set(p.op, CUBLASLT_MATMUL_DESC_TRANSB, &ob, sizeof ob);
    st = L.layout_create(&p.la, dt, ta ? Kd : M, ta ? M : Kd, lda);
    if (st == CUBLAS_STATUS_SUCCESS) st = L.layout_create(&p.lb, dt, tb ? N : Kd, tb ? Kd : N, ldb);
    if (st == CUBLAS_STATUS_SUCCESS) st = L.layout_create(&p.lc, dt, M, N, ldc);
    if (st != CUBLAS_STATUS_SUCCESS) return lt_fail("matrix layout", st);
    if (batch > 1) {
        const cublasLtMatrixLayout_t lays[3] = {p.la, p.lb, p.lc};
        const int64_t strides[3] = {sa, sb, sc};
        for (int i = 0; i < 3 && st == CUBLAS_STATUS_SUCCESS; ++i) {
            st = L.layout_set(lays[i], CUBLASLT_MATRIX_LAYOUT_BATCH_COUNT, &batch, sizeof batch);
            if (st == CUBLAS_STATUS_SUCCESS)
                st = L.layout_set(lays[i], CUBLASLT_MATRIX_LAYOUT_STRIDED_BATCH_OFFSET, &strides[i],
                                  sizeof strides[i]);
        }
        if (st != CUBLAS_STATUS_SUCCESS) return lt_fail("batched layout", st);
    }
    cublasLtMatmulPreference_t pref = nullptr;
    st = L.pref_create(&pref);
    if (st != CUBLAS_STATUS_SUCCESS) return lt_fail("preference", st);
    const uint64_t ws = kLtWorkspace;
    L.pref_set(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws, sizeof ws);
    cublasLtMatmulHeuristicResult_t res;
    int found = 0;
    st = L.heuristic(w->handle, p.op, p.la, p.lb, p.lc, p.lc, pref, 1, &res, &found);
    L.pref_destroy(pref);
    if (st != CUBLAS_STATUS_SUCCESS || found < 1) return lt_fail("algorithm heuristic", st);
    p.algo = res.algo;
    cache.push_back(p);
    *out = &cache.back();
    return CAM_OK;
}

// D = alpha op(A) op(B) + beta C for `batch` matrices at element strides
// sa, sb, sc (column-major; C and D share a layout).
int gemm(OrthoWork* w, int precision, bool ta, bool tb, int64_t M,
         int64_t N, int64_t Kd, float alpha, const void* A, int64_t lda, const void* B,
         int64_t ldb, float beta, const void* C, void* D, int64_t ldc, int32_t batch,
         int64_t sa, int64_t sb, int64_t sc, cudaStream_t s) {
    const GemmPlan* p = nullptr;
    int rc = gemm_plan(w, precision, ta, tb, M, N, Kd, lda, ldb, ldc, batch, sa, sb, sc, &p);
    if (rc != CAM_OK) return rc;
    const int st = w->lt->matmul(w->handle, p->op, &alpha, A, p->la, B, p->lb, &beta, C, p->lc, D,
                                 p->lc, &p->algo, w->lt_ws, kLtWorkspace, s);
    if (st != CUBLAS_STATUS_SUCCESS) return lt_fail("matmul", st);
    return CAM_OK;
}

// The short-side form of the iteration (CAM_ORTHO_SHORT_SIDE) for B
// matrices of m x n with max(m, n) >= 4 r, r = min(m, n). With the iterate
// written X_k = X_0 P_k (tall) or P_k X_0 (wide), a Newton-Schulz step becomes
// P <- 1.5 P - 0.5 P (P^T G P) (tall) or 1.5 P - 0.5 (P G P^T) P (wide) on
// r x r matrices, G the Gram matrix of X_0 on its short side; the polar
// factor is then one product with X_0. The normalised starts are in w->X,
// the factors end in w->Y. Workspace: P in w->G, and G, T, M and P's second
// buffer in w->Y (4 B r^2 <= B m n floats), which the final product then
// overwrites. G and the r x r steps run in fp32; the final product in
// p.precision.
int short_side_iteration(OrthoWork* w, const OrthoParams& p, int64_t m, int64_t n, int B,
                         cudaStream_t s, int64_t* launches) {
    const int64_t r = std::min(m, n), numel = m * n, gram = r * r;
    const bool tall = m >= n;
    const float* A = w->X;  // each X_0 as the column-major n x m matrix X_0^T (ld n)
    float* G = w->Y;
    float* T = G + int64_t(B) * gram;
    float* M = T + int64_t(B) * gram;
    float* Pa = w->G;
    float* Pb = M + int64_t(B) * gram;
    const int fp = CAM_ORTHO_FP32;
    int rc = tall ? gemm(w, fp, false, true, n, n, m, 1.0f, A, n, A, n, 0.0f, G, G, n, B, numel,
                         numel, gram, s)   // G = X_0^T X_0 = A A^T
                  : gemm(w, fp, true, false, m, m, n, 1.0f, A, n, A, n, 0.0f, G, G, m, B, numel,
                         numel, gram, s);  // G = X_0 X_0^T = A^T A
    if (rc != CAM_OK) return rc;
    const int64_t total = int64_t(B) * gram;
    const int blocks =
        static_cast<int>(std::min<int64_t>(4096, (total + kOrthoThreads - 1) / kOrthoThreads));
    ortho_identity<<<blocks, kOrthoThreads, 0, s>>>(Pa, r, total);
    ++*launches;
    cudaError_t ce = cudaGetLastError();
    if (ce != cudaSuccess)
        return record_error(CAM_E_CUDA, "orthogonalisation: launch: %s", cudaGetErrorString(ce));
    float* P = Pa;
    float* Pn = Pb;
    for (int it = 0; it < p.iterations && rc == CAM_OK; ++it) {
        if (tall) {  // T = P^T G; M = T P; P' = 1.5 P - 0.5 P M
            rc = gemm(w, fp, true, false, r, r, r, 1.0f, P, r, G, r, 0.0f, T, T, r, B, gram, gram,
                      gram, s);
            if (rc == CAM_OK)
                rc = gemm(w, fp, false, false, r, r, r, 1.0f, T, r, P, r, 0.0f, M, M, r, B, gram,
                          gram, gram, s);
            if (rc == CAM_OK)
                rc = gemm(w, fp, false, false, r, r, r, -0.5f, P, r, M, r, 1.5f, P, Pn, r, B, gram,
                          gram, gram, s);
        } else {     // T = P G; M = T P^T; P' = 1.5 P - 0.5 M P
            rc = gemm(w, fp, false, false, r, r, r, 1.0f, P, r, G, r, 0.0f, T, T, r, B, gram, gram,
                      gram, s);
            if (rc == CAM_OK)
                rc = gemm(w, fp, false, true, r, r, r, 1.0f, T, r, P, r, 0.0f, M, M, r, B, gram,
                          gram, gram, s);
            if (rc == CAM_OK)
                rc = gemm(w, fp, false, false, r, r, r, -0.5f, M, r, P, r, 1.5f, P, Pn, r, B, gram,
                          gram, gram, s);
        }
        std::swap(P, Pn);
    }
    if (rc != CAM_OK) return rc;
    if (P != Pa) {  // the final product writes over w->Y, where P_b lives
        ce = cudaMemcpyAsync(Pa, P, sizeof(float) * total, cudaMemcpyDeviceToDevice, s);
        if (ce != cudaSuccess)
            return record_error(CAM_E_CUDA, "orthogonalisation: copy: %s", cudaGetErrorString(ce));
        P = Pa;
    }
    // tall: X = X_0 P, column-major P^T A; wide: X = P X_0, column-major A P^T
    return tall ? gemm(w, p.precision, true, false, n, m, n, 1.0f, P, n, A, n, 0.0f, w->Y, w->Y, n,
                       B, gram, numel, numel, s)
                : gemm(w, p.precision, false, true, n, m, m, 1.0f, A, n, P, m, 0.0f, w->Y, w->Y, n,
                       B, numel, gram, numel, s);
}

}  // namespace
}  // namespace cam

namespace cam {

int ortho_create(OrthoWork** out, int64_t cap_elems, int64_t cap_gram) {
    *out = nullptr;
    const LtApi* lt = lt_api();
    if (!lt)
        return record_error(CAM_E_CUDA,
                            "orthogonalisation needs cuBLASLt (libcublasLt.so.13), which could not "
                            "be loaded");
    OrthoWork* w = new (std::nothrow) OrthoWork;
    if (!w) return record_error(CAM_E_NOMEM, "orthogonalisation: out of host memory");
    w->lt = lt;
    w->cap_elems = std::max<int64_t>(cap_elems, 1);
    w->cap_gram = std::max<int64_t>(cap_gram, 1);
    auto up = [](size_t b) { return (b + 255) / 256 * 256; };
    const size_t bx = up(sizeof(float) * size_t(w->cap_elems));
    const size_t bg = up(sizeof(float) * size_t(w->cap_gram));
    const size_t bp = up(sizeof(double) * size_t(kOrthoBatchMax) * kOrthoBlocksMax);
    const size_t bs = up(sizeof(double) * kOrthoBatchMax);
    const size_t bi = up(sizeof(float) * kOrthoBatchMax);
    const size_t total = 2 * bx + bg + bp + bs + bi + kLtWorkspace;
    if (cudaMalloc(&w->block, total) != cudaSuccess) {
        cudaGetLastError();
        delete w;
        return record_error(CAM_E_NOMEM, "orthogonalisation: cudaMalloc(%zu) failed", total);
    }
    char* b = static_cast<char*>(w->block);
    w->X = reinterpret_cast<float*>(b);
    w->Y = reinterpret_cast<float*>(b + bx);
    w->G = reinterpret_cast<float*>(b + 2 * bx);
    w->partials = reinterpret_cast<double*>(b + 2 * bx + bg);
    w->scalars = reinterpret_cast<double*>(b + 2 * bx + bg + bp);
    w->inv_norm = reinterpret_cast<float*>(b + 2 * bx + bg + bp + bs);
    w->lt_ws = b + 2 * bx + bg + bp + bs + bi;
    const int st = lt->create(&w->handle);
    if (st != CUBLAS_STATUS_SUCCESS) {
        cudaFree(w->block);
        delete w;
        return lt_fail("handle", st);
    }
    *out = w;
    return CAM_OK;
}

void ortho_destroy(OrthoWork* w) {
    if (!w) return;
    for (GemmPlan& p : w->plans) {
        w->lt->layout_destroy(p.la);
        w->lt->layout_destroy(p.lb);
        w->lt->layout_destroy(p.lc);
        w->lt->desc_destroy(p.op);
    }
    if (w->handle) w->lt->destroy(w->handle);
    cudaFree(w->block);
    delete w;
}

int ortho_group(OrthoWork* w, const OrthoMatrix* mats, int count, const OrthoParams& p,
                cudaStream_t s, int sm_count, int64_t* launches) {
    if (count <= 0) return CAM_OK;
    const int64_t m = mats[0].rows, n = mats[0].cols, numel = m * n;
    const int64_t r = std::min(m, n), gram = r * r;
    int64_t per = std::min<int64_t>(kOrthoBatchMax, std::min(w->cap_elems / numel, w->cap_gram / gram));
    per = std::max<int64_t>(per, 1);
    for (int first = 0; first < count; first += static_cast<int>(per)) {
        const int B = static_cast<int>(std::min<int64_t>(per, count - first));
        // Blocks per matrix: about 8 per SM over the whole batch, and no more
        // than the matrix has 8-element steps for (small matrices in a big
        // batch would otherwise leave most threads idle).
        const int64_t steps = (numel + 8 * kOrthoThreads - 1) / (8 * kOrthoThreads);
        const int64_t want = (int64_t(sm_count) * 8 + B - 1) / B;
        const int grid = static_cast<int>(
            std::min<int64_t>(kOrthoBlocksMax, std::max<int64_t>(1, std::min(want, steps))));
        // Delta of each matrix into its slot, its norm, and the normalised
        // start: one launch of each kernel for the whole batch.
        // a slot of the workspace is 32-byte aligned when numel is a multiple of 8
        const uintptr_t xa = p.dtype == kDtBF16 ? 16 : 32;
        auto al = [](const void* q, uintptr_t b) { return reinterpret_cast<uintptr_t>(q) % b == 0; };
        DeltaArgs da;
        ApplyArgs aa;
        std::fill(da.vec, da.vec + kOrthoBatchMax / 32, 0u);
        std::fill(aa.vec, aa.vec + kOrthoBatchMax / 32, 0u);
        for (int j = 0; j < B; ++j) {
            const OrthoMatrix& t = mats[first + j];
            bool v = numel % 8 == 0 && al(t.theta, 32);
            for (int k = 0; k < CAM_KMAX; ++k) {
                da.x[j][k] = k < p.K ? t.x[k] : nullptr;
                if (k < p.K) v = v && al(t.x[k], xa);
            }
            da.theta[j] = t.theta;
            if (v) da.vec[j >> 5] |= 1u << (j & 31);
            aa.theta[j] = t.theta;
            aa.e[j] = p.ema ? t.e : nullptr;
            if (numel % 8 == 0 && al(t.theta, 32) && (!p.ema || al(t.e, 32)))
                aa.vec[j >> 5] |= 1u << (j & 31);
        }
        da.K = p.K;
        da.Kf = static_cast<float>(p.K);
        da.X = w->X;
        da.n = numel;
        da.partials = w->partials;
        const dim3 bgrid(grid, B);
        if (p.dtype == kDtBF16) ortho_delta<uint16_t><<<bgrid, kOrthoThreads, 0, s>>>(da);
        else ortho_delta<float><<<bgrid, kOrthoThreads, 0, s>>>(da);
        ortho_norm<<<B, 32, 0, s>>>(w->partials, grid, w->scalars, w->inv_norm);
        const bool bf = p.precision == CAM_ORTHO_BF16;
        if (bf)  // the bf16 iterate starts in Y; X's fp32 Delta is no longer needed
            ortho_scale_bf16<<<bgrid, kOrthoThreads, 0, s>>>(
                w->X, reinterpret_cast<__nv_bfloat16*>(w->Y), numel, w->inv_norm);
        else
            ortho_scale<<<bgrid, kOrthoThreads, 0, s>>>(w->X, numel, w->inv_norm);
        *launches += 3;
        cudaError_t ce = cudaGetLastError();
        if (ce != cudaSuccess)
            return record_error(CAM_E_CUDA, "orthogonalisation: launch: %s", cudaGetErrorString(ce));
        // Newton-Schulz on all B matrices at once. Row-major X (m x n) is the
        // column-major n x m matrix A = X^T (ld n).
        void* cur = bf ? static_cast<void*>(w->Y) : static_cast<void*>(w->X);
        void* nxt = bf ? static_cast<void*>(w->X) : static_cast<void*>(w->Y);
        const bool short_side = p.short_side && std::max(m, n) >= 4 * r;
        if (short_side) {
            const int rc = short_side_iteration(w, p, m, n, B, s, launches);
            if (rc != CAM_OK) return rc;
            cur = w->Y;
        }
        for (int it = 0; !short_side && it < p.iterations; ++it) {
            int rc;
            if (m >= n) {  // G = X^T X = A A^T (n x n); A' = 1.5 A - 0.5 G A
                rc = gemm(w, p.precision, false, true, n, n, m, 1.0f, cur, n, cur, n, 0.0f, w->G, w->G,
                          n, B, numel, numel, gram, s);
                if (rc == CAM_OK)
                    rc = gemm(w, p.precision, false, false, n, m, n, -0.5f, w->G, n, cur, n, 1.5f, cur,
                              nxt, n, B, gram, numel, numel, s);
            } else {       // G = X X^T = A^T A (m x m); A' = 1.5 A - 0.5 A G
                rc = gemm(w, p.precision, true, false, m, m, n, 1.0f, cur, n, cur, n, 0.0f, w->G, w->G,
                          m, B, numel, numel, gram, s);
                if (rc == CAM_OK)
                    rc = gemm(w, p.precision, false, false, n, m, m, -0.5f, cur, n, w->G, m, 1.5f, cur,
                              nxt, n, B, numel, gram, numel, s);
            }
            if (rc != CAM_OK) return rc;
            std::swap(cur, nxt);
        }
        aa.O = cur;
        aa.n = numel;
        aa.scalars = w->scalars;
        aa.lr = p.lr;
        aa.scale_mode = p.scale_mode;
        aa.r = r;
        aa.beta = p.beta;
        if (bf)
            ortho_apply<uint16_t><<<bgrid, kOrthoThreads, 0, s>>>(aa);
        else
            ortho_apply<float><<<bgrid, kOrthoThreads, 0, s>>>(aa);
        *launches += 1;
        ce = cudaGetLastError();
        if (ce != cudaSuccess)
            return record_error(CAM_E_CUDA, "orthogonalisation: launch: %s", cudaGetErrorString(ce));
    }
    return CAM_OK;
}

}  // namespace cam
