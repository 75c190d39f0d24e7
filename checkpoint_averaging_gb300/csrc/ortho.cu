// ortho.cu -- outer orthogonalisation of a plain-mean round: the averaged
// update of every matrix-shaped tensor is replaced by its polar factor
// ("DiffuRefill-1B: Pretraining a Masked Diffusion Language Model on Free,
// Preemptible Notebook GPUs", section 5.3).
//
// Per matrix tensor (row-major m x n; r = min(m, n), L = max(m, n)):
//   1. Delta = mean_k(x_k) - theta with the plain-mean arithmetic of the fused
//      pass, into a workspace, with |Delta|_F^2 summed in a fixed order;
//   2. X0 = Delta / |Delta|_F, so every singular value lies in (0, 1], stored
//      in the wide orientation W (r x L: Delta itself, or its transpose for a
//      tall matrix) and, transposed, as V = W^T, both zero-padded to
//      multiples of 128 (nt_gemm.h);
//   3. `iterations` Newton-Schulz steps W <- 1.5 W - 0.5 (W W^T) W, which
//      drive every singular value to 1 and so converge to the polar factor
//      U V^T. Each step is two NT GEMMs (nt_gemm.cu): H = 1.5 I - 0.5 W W^T
//      (a Gram product with the combination in its epilogue, read with bf16
//      operands from V as V^T V; symmetric, so only its upper triangle is
//      computed and then mirrored), then V' = V H. H is stored in the
//      iterate's type. With TF32 inputs the step stays in the form
//      V' = 1.5 V - 0.5 V G, V read in fp32 by the epilogue. TF32 and the
//      CUDA-core form write W' = V'^T beside V' for their next Gram product;
//   4. theta' = theta + s X, s = lr or lr |Delta|_F / sqrt(min(m, n)), read
//      from V (tall) or W (wide), then the EMA of the globals.
// Equal-shape matrices run as one batch through every kernel.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <vector>

#include "cam_internal.h"
#include "merge_device.cuh"
#include "nt_gemm.h"
#include "side_internal.h"

namespace cam {
namespace {

constexpr int kOrthoBatchMax = 256;  // matrices orthogonalised together
constexpr int kOrthoBlocksMax = 4096;
constexpr int64_t kSplitFloats = int64_t(1) << 25;  // Gram split-K partials (128 MB)
constexpr int kOrthoPassChunks = 8;  // chunks iterated together (problems of one GEMM launch)

int64_t pad128(int64_t v) { return (v + 127) / 128 * 128; }

}  // namespace

// Per-context workspace of the orthogonalisation, made at the first
// orthogonalised commit: Delta (dense fp32), two iterates W and two
// transposes V in the padded layout (up to 4 bytes an element), the Gram
// matrices, the short-side form's six r x r matrices per batch slot, the
// Gram split partials and the norm reduction.
struct OrthoWork {
    float* X = nullptr;          // Delta, matrix j dense at X + j m n
    void* W[2] = {nullptr, nullptr};
    void* V[2] = {nullptr, nullptr};
    void* G = nullptr;
    float* Sq = nullptr;         // short side: G0, P, Pt, P', Pt', T, M per slot
    float* split = nullptr;      // Gram split-K partials
    double* partials = nullptr;  // [kOrthoBatchMax * kOrthoBlocksMax]
    double* scalars = nullptr;   // [j] = |Delta_j|_F^2
    float* inv_norm = nullptr;   // [j] = 1 / |Delta_j|_F (0 when Delta_j = 0)
    int32_t* sched = nullptr;    // the Gram launches' unit counters (0 between launches)
    void* block = nullptr;       // one cudaMalloc holding all of the above
    int64_t cap_pad = 0;         // elements in each W / V buffer and floats in X
    int64_t cap_gram = 0;        // elements in G
    int64_t cap_sq = 0;          // floats in Sq (7 squares of the largest matrix)
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

__device__ __forceinline__ void put(float* p, float v) { *p = v; }
__device__ __forceinline__ void put(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// X0_j = Delta_j / |Delta_j|_F into W_j (rp x Lp, the wide orientation) and
// V_j = W_j^T (Lp x rp), rounded once to the iterate's storage type, zero
// outside the matrix. Blocks of 32 x 8 threads move 32 x 32 tiles of the
// (L, r) index space through shared memory, so that reads of Delta and
// writes of both copies are coalesced. grid: (Lp / 32, rp / 32, batch).
template <typename T>
__global__ void ortho_pack(const float* X, int64_t m, int64_t n, const float* inv_norm, T* W, T* V,
                           int64_t rp, int64_t Lp) {
    __shared__ float tile[32][33];  // [L index][r index]
    const int j = blockIdx.z;
    const int64_t i0 = int64_t(blockIdx.x) * 32, a0 = int64_t(blockIdx.y) * 32;
    const int tx = threadIdx.x, ty = threadIdx.y;
    const bool tall = m >= n;
    const int64_t r = tall ? n : m, L = tall ? m : n;
    const float f = inv_norm[j];
    const float* Xj = X + int64_t(j) * m * n;
    for (int q = ty; q < 32; q += 8) {
        if (tall) {  // Delta[i][a]: a along the row
            const int64_t i = i0 + q, a = a0 + tx;
            tile[q][tx] = (i < L && a < r) ? __fmul_rn(Xj[i * n + a], f) : 0.0f;
        } else {     // Delta[a][i]: i along the row
            const int64_t a = a0 + q, i = i0 + tx;
            tile[tx][q] = (i < L && a < r) ? __fmul_rn(Xj[a * n + i], f) : 0.0f;
        }
    }
    __syncthreads();
    T* Wj = W + int64_t(j) * rp * Lp;
    T* Vj = V + int64_t(j) * Lp * rp;
    for (int q = ty; q < 32; q += 8) {
        put(Vj + (i0 + q) * rp + a0 + tx, tile[q][tx]);  // V[i][a]
        put(Wj + (a0 + q) * Lp + i0 + tx, tile[tx][q]);  // W[a][i]
    }
}

// P_j <- the r x r identity inside its rp x rp square (zero elsewhere, so the
// padding stays zero through the short-side steps); total = slots x rp x rp.
__global__ void ortho_identity(float* P, int64_t r, int64_t rp, int64_t total) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t q = i % (rp * rp), row = q / rp, col = q % rp;
        P[i] = (row == col && row < r) ? 1.0f : 0.0f;
    }
}

struct ApplyArgs {
    float* theta[kOrthoBatchMax];
    float* e[kOrthoBatchMax];  // EMA buffers, or null
    uint32_t vec[kOrthoBatchMax / 32];  // bit j: matrix j's buffers take 32-byte vectors
    const void* O;             // the polar factors (fp32, or bf16) in the matrices' own
                               // orientation: row i of slot j at O + j * so + i * ld
    int64_t ld, so;
    int64_t n, cols;           // elements and columns per matrix
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
    const OT* O = static_cast<const OT*>(a.O) + int64_t(j) * a.so;
    float s = a.lr;
    if (a.scale_mode == CAM_ORTHO_SCALE_MATCH_NORM)
        s = static_cast<float>(static_cast<double>(a.lr) * sqrt(a.scalars[j]) /
                               sqrt(static_cast<double>(a.r)));
    const float omb = __fsub_rn(1.0f, a.beta);
    const int64_t tid = blockIdx.x * int64_t(blockDim.x) + threadIdx.x;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    int64_t done = 0;
    if ((a.vec[j >> 5] >> (j & 31)) & 1u) {  // 8 elements per step, never across a row
        const int64_t nv = a.n >> 3;
        for (int64_t v = tid; v < nv; v += stride) {
            const int64_t i = 8 * v, row = i / a.cols, col = i - row * a.cols;
            float th[8];
            dev::load_s8(theta + i, th);
            dev::XVec<OT> o;
            o.load(O + row * a.ld + col);
#pragma unroll
            for (int q = 0; q < 8; ++q) th[q] = __fadd_rn(th[q], __fmul_rn(s, o.get(q)));
            dev::store_s8(theta + i, th);
            if (e) {
                float ev[8];
                dev::load_s8(e + i, ev);
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    ev[q] = __fadd_rn(__fmul_rn(a.beta, ev[q]), __fmul_rn(omb, th[q]));
                dev::store_s8(e + i, ev);
            }
        }
        done = 8 * nv;
    }
    for (int64_t i = done + tid; i < a.n; i += stride) {
        const int64_t row = i / a.cols, col = i - row * a.cols;
        const float th = __fadd_rn(theta[i], __fmul_rn(s, dev::load_x1(O + row * a.ld + col)));
        theta[i] = th;
        if (e) e[i] = __fadd_rn(__fmul_rn(a.beta, e[i]), __fmul_rn(omb, th));
    }
}

int launch_error(const char* what) {
    const cudaError_t ce = cudaGetLastError();
    if (ce == cudaSuccess) return CAM_OK;
    return record_error(CAM_E_CUDA, "orthogonalisation: %s: %s", what, cudaGetErrorString(ce));
}

// Shape of one batch in the padded layout.
struct Shape {
    int64_t m, n, r, L, rp, Lp;
    bool tall;
};

// One NT GEMM over `B` slots; strides in elements.
NtGemm nt(int precision, int epi, int B, int64_t M, int64_t N, int64_t K, const void* A,
          int64_t lda, int64_t sA, const void* Bm, int64_t ldb, int64_t sB) {
    NtGemm g;
    std::memset(&g, 0, sizeof g);
    g.precision = precision;
    g.epilogue = epi;
    g.batch = B;
    g.M = M;
    g.N = N;
    g.K = K;
    g.A = A;
    g.lda = lda;
    g.sA = sA;
    g.B = Bm;
    g.ldb = ldb;
    g.sB = sB;
    g.alpha = 1.0f;
    g.beta = 0.0f;
    g.diag = 0.0f;
    return g;
}

// One batch of equal-shape matrices inside a pass: its slots in the scalar
// arrays and its offsets (in elements) in the workspace buffers.
struct Chunk {
    const OrthoMatrix* mats;
    int count;
    Shape sh;
    int slot0;          // first slot: partials, scalars and inv_norm
    int64_t off_x;      // Delta (floats)
    int64_t off_pad;    // W and V (elements of the iterate's type)
    int64_t off_gram;   // G (elements of the iterate's type)
    int64_t padded() const { return sh.rp * sh.Lp; }
    int64_t sq() const { return sh.rp * sh.rp; }
};

void* at(void* base, int64_t elems, int64_t eb) { return static_cast<char*>(base) + elems * eb; }

// The short-side form of the iteration (CAM_ORTHO_SHORT_SIDE), for matrices
// with L >= 4 r: with W_k = P_k W_0, a Newton-Schulz step becomes
// P <- 1.5 P - 0.5 (P G0 P^T) P on r x r matrices, G0 = W_0 W_0^T; the polar
// factor is then one product with W_0. G0 and the r x r steps run in fp32 on
// the CUDA cores; the final product in p.precision. Per slot, Sq holds G0, P,
// P^T, their next values, T = P G0 and M = T P^T. The chunk runs alone in its
// pass (offsets 0); the factor ends in W[1] (and V[1] = its transpose).
int short_side_iteration(OrthoWork* w, const OrthoParams& p, const Shape& sh, int B, cudaStream_t s,
                         int sm_count, int64_t* launches) {
    const int64_t rp = sh.rp, Lp = sh.Lp, sq = rp * rp;
    const int fp = CAM_ORTHO_FP32;
    float* G0 = w->Sq;
    float* P = G0 + B * sq;
    float* Pt = P + B * sq;
    float* Pn = Pt + B * sq;
    float* Ptn = Pn + B * sq;
    float* T = Ptn + B * sq;
    float* M = T + B * sq;
    // G0 = W0 W0^T
    NtGemm g = nt(fp, kNtAxpby, B, rp, rp, Lp, w->W[0], Lp, rp * Lp, w->W[0], Lp, rp * Lp);
    g.Y = G0;
    g.ldy = rp;
    g.sY = sq;
    g.partials = w->split;  // the CUDA-core kernel splits long K ranges
    g.partial_floats = kSplitFloats;
    int rc = nt_gemm(&g, 1, sm_count, p.status, s, launches);
    if (rc != CAM_OK) return rc;
    const int64_t total = int64_t(B) * sq;
    const int blocks =
        static_cast<int>(std::min<int64_t>(4096, (total + kOrthoThreads - 1) / kOrthoThreads));
    ortho_identity<<<blocks, kOrthoThreads, 0, s>>>(P, sh.r, rp, total);
    ortho_identity<<<blocks, kOrthoThreads, 0, s>>>(Pt, sh.r, rp, total);
    *launches += 2;
    if ((rc = launch_error("launch")) != CAM_OK) return rc;
    for (int it = 0; it < p.iterations; ++it) {
        g = nt(fp, kNtAxpby, B, rp, rp, rp, P, rp, sq, G0, rp, sq);  // T = P G0 (G0 symmetric)
        g.Y = T;
        g.ldy = rp;
        g.sY = sq;
        g.partials = w->split;
        g.partial_floats = kSplitFloats;
        if ((rc = nt_gemm(&g, 1, sm_count, p.status, s, launches)) != CAM_OK) return rc;
        g = nt(fp, kNtAxpby, B, rp, rp, rp, T, rp, sq, P, rp, sq);  // M = T P^T
        g.Y = M;
        g.ldy = rp;
        g.sY = sq;
        g.partials = w->split;
        g.partial_floats = kSplitFloats;
        if ((rc = nt_gemm(&g, 1, sm_count, p.status, s, launches)) != CAM_OK) return rc;
        // P'^T = 1.5 P^T - 0.5 P^T M (M symmetric), and P' beside it
        g = nt(fp, kNtAxpby, B, rp, rp, rp, Pt, rp, sq, M, rp, sq);
        g.alpha = -0.5f;
        g.beta = 1.5f;
        g.C = Pt;
        g.ldc = rp;
        g.sC = sq;
        g.Y = Ptn;
        g.ldy = rp;
        g.sY = sq;
        g.Yt = Pn;
        g.ldyt = rp;
        g.sYt = sq;
        if ((rc = nt_gemm(&g, 1, sm_count, p.status, s, launches)) != CAM_OK) return rc;
        std::swap(P, Pn);
        std::swap(Pt, Ptn);
    }
    // W = P W0 = NT(P, V0), V = W^T
    g = nt(p.precision, kNtAxpby, B, rp, Lp, rp, P, rp, sq, w->V[0], rp, Lp * rp);
    g.Y = w->W[1];
    g.ldy = Lp;
    g.sY = rp * Lp;
    g.Yt = w->V[1];
    g.ldyt = rp;
    g.sYt = Lp * rp;
    return nt_gemm(&g, 1, sm_count, p.status, s, launches);
}

// Delta, its norm and the normalised start (both orientations) of one chunk:
// one launch of each kernel for its matrices.
int prepare_chunk(OrthoWork* w, const Chunk& ch, const OrthoParams& p, cudaStream_t s,
                  int sm_count, int64_t* launches, int* grid_out) {
    const Shape& sh = ch.sh;
    const int B = ch.count;
    const int64_t numel = sh.m * sh.n;
    const int64_t eb = nt_elem_bytes(p.precision);
    // Blocks per matrix: about 8 per SM over the whole chunk, and no more than
    // the matrix has 8-element steps for (small matrices in a big batch would
    // otherwise leave most threads idle).
    const int64_t steps = (numel + 8 * kOrthoThreads - 1) / (8 * kOrthoThreads);
    const int64_t want = (int64_t(sm_count) * 8 + B - 1) / B;
    const int grid = static_cast<int>(
        std::min<int64_t>(kOrthoBlocksMax, std::max<int64_t>(1, std::min(want, steps))));
    *grid_out = grid;
    // a slot of Delta is 32-byte aligned when numel is a multiple of 8
    const uintptr_t xa = p.dtype == kDtBF16 ? 16 : 32;
    auto al = [](const void* q, uintptr_t b) { return reinterpret_cast<uintptr_t>(q) % b == 0; };
    DeltaArgs da;
    std::fill(da.vec, da.vec + kOrthoBatchMax / 32, 0u);
    for (int j = 0; j < B; ++j) {
        const OrthoMatrix& t = ch.mats[j];
        bool v = numel % 8 == 0 && ch.off_x % 8 == 0 && al(t.theta, 32);
        for (int k = 0; k < CAM_KMAX; ++k) {
            da.x[j][k] = k < p.K ? t.x[k] : nullptr;
            if (k < p.K) v = v && al(t.x[k], xa);
        }
        da.theta[j] = t.theta;
        if (v) da.vec[j >> 5] |= 1u << (j & 31);
    }
    da.K = p.K;
    da.Kf = static_cast<float>(p.K);
    da.X = w->X + ch.off_x;
    da.n = numel;
    da.partials = w->partials + int64_t(ch.slot0) * kOrthoBlocksMax;
    const dim3 bgrid(grid, B);
    if (p.dtype == kDtBF16) ortho_delta<uint16_t><<<bgrid, kOrthoThreads, 0, s>>>(da);
    else ortho_delta<float><<<bgrid, kOrthoThreads, 0, s>>>(da);
    ortho_norm<<<B, 32, 0, s>>>(da.partials, grid, w->scalars + ch.slot0, w->inv_norm + ch.slot0);
    const dim3 pgrid(static_cast<unsigned>(sh.Lp / 32), static_cast<unsigned>(sh.rp / 32), B);
    if (p.precision == CAM_ORTHO_BF16)
        ortho_pack<__nv_bfloat16><<<pgrid, dim3(32, 8), 0, s>>>(
            da.X, sh.m, sh.n, w->inv_norm + ch.slot0,
            static_cast<__nv_bfloat16*>(at(w->W[0], ch.off_pad, eb)),
            static_cast<__nv_bfloat16*>(at(w->V[0], ch.off_pad, eb)), sh.rp, sh.Lp);
    else
        ortho_pack<float><<<pgrid, dim3(32, 8), 0, s>>>(
            da.X, sh.m, sh.n, w->inv_norm + ch.slot0, static_cast<float*>(at(w->W[0], ch.off_pad, eb)),
            static_cast<float*>(at(w->V[0], ch.off_pad, eb)), sh.rp, sh.Lp);
    *launches += 3;
    return launch_error("launch");
}

// theta' = theta + s X and the EMA for one chunk, X read from V (tall) or W
// (wide) of iterate buffer `cur`.
int apply_chunk(OrthoWork* w, const Chunk& ch, const OrthoParams& p, int cur, int grid,
                cudaStream_t s, int64_t* launches) {
    const Shape& sh = ch.sh;
    const int B = ch.count;
    const int64_t eb = nt_elem_bytes(p.precision);
    auto al = [](const void* q, uintptr_t b) { return reinterpret_cast<uintptr_t>(q) % b == 0; };
    ApplyArgs aa;
    std::fill(aa.vec, aa.vec + kOrthoBatchMax / 32, 0u);
    for (int j = 0; j < B; ++j) {
        const OrthoMatrix& t = ch.mats[j];
        aa.theta[j] = t.theta;
        aa.e[j] = p.ema ? t.e : nullptr;
        if (sh.n % 8 == 0 && al(t.theta, 32) && (!p.ema || al(t.e, 32)))
            aa.vec[j >> 5] |= 1u << (j & 31);
    }
    aa.O = at(sh.tall ? w->V[cur] : w->W[cur], ch.off_pad, eb);
    aa.ld = sh.tall ? sh.rp : sh.Lp;
    aa.so = ch.padded();
    aa.n = sh.m * sh.n;
    aa.cols = sh.n;
    aa.scalars = w->scalars + ch.slot0;
    aa.lr = p.lr;
    aa.scale_mode = p.scale_mode;
    aa.r = sh.r;
    aa.beta = p.beta;
    const dim3 bgrid(grid, B);
    if (p.precision == CAM_ORTHO_BF16)
        ortho_apply<uint16_t><<<bgrid, kOrthoThreads, 0, s>>>(aa);
    else
        ortho_apply<float><<<bgrid, kOrthoThreads, 0, s>>>(aa);
    *launches += 1;
    return launch_error("launch");
}

// One pass: chunks that share the workspace, iterated together: each
// Newton-Schulz step is one Gram launch and one update launch over all of
// them (nt_gemm's problems).
int run_pass(OrthoWork* w, const std::vector<Chunk>& pass, const OrthoParams& p, cudaStream_t s,
             int sm_count, int64_t* launches) {
    std::vector<int> grids(pass.size());
    for (size_t i = 0; i < pass.size(); ++i) {
        const int rc = prepare_chunk(w, pass[i], p, s, sm_count, launches, &grids[i]);
        if (rc != CAM_OK) return rc;
    }
    const int64_t eb = nt_elem_bytes(p.precision);
    int cur = 0;
    const bool short_side = pass.size() == 1 && p.short_side && pass[0].sh.L >= 4 * pass[0].sh.r;
    if (short_side) {
        const int rc = short_side_iteration(w, p, pass[0].sh, pass[0].count, s, sm_count, launches);
        if (rc != CAM_OK) return rc;
        cur = 1;
    }
    // bf16 and fp32: H = 1.5 I - 0.5 W W^T (upper triangle, mirrored), then
    // V' = V H. TF32: G = W W^T, then V' = 1.5 V - 0.5 V G with V read in
    // fp32 in the epilogue, so that only the correction passes through TF32
    // inputs (V H would round the whole iterate to TF32 on every step).
    const bool cform = p.precision == CAM_ORTHO_TF32;
    // With bf16 operands the Gram product reads V itself (MN-major operands:
    // G = V^T V), so W = V^T is written only where the applied step reads it,
    // on the last step of a wide matrix. TF32 (whose MMA is given K-major
    // operands only) and the CUDA-core form keep both orientations.
    const bool mn = p.precision == CAM_ORTHO_BF16;
    NtGemm gram[kOrthoPassChunks], upd[kOrthoPassChunks];
    const int n = static_cast<int>(pass.size());
    for (int it = 0; !short_side && it < p.iterations; ++it) {
        const bool last = it + 1 == p.iterations;
        for (int i = 0; i < n; ++i) {
            const Chunk& ch = pass[i];
            const Shape& sh = ch.sh;
            const int64_t padded = ch.padded(), sq = ch.sq();
            void* Wc = at(w->W[cur], ch.off_pad, eb);
            void* Vc = at(w->V[cur], ch.off_pad, eb);
            void* G = at(w->G, ch.off_gram, eb);
            NtGemm& g = gram[i];
            if (mn) {
                g = nt(p.precision, kNtGram, ch.count, sh.rp, sh.rp, sh.Lp, Vc, sh.rp, padded, Vc,
                       sh.rp, padded);
                g.mn_major = true;
            } else {
                g = nt(p.precision, kNtGram, ch.count, sh.rp, sh.rp, sh.Lp, Wc, sh.Lp, padded, Wc,
                       sh.Lp, padded);
            }
            g.alpha = cform ? 1.0f : -0.5f;
            g.diag = cform ? 0.0f : 1.5f;
            g.Y = G;
            g.ldy = sh.rp;
            g.sY = sq;
            g.partials = w->split;
            g.partial_floats = kSplitFloats;
            g.sched = w->sched;
            // V' = V H (or 1.5 V - 0.5 V G), W' = V'^T
            NtGemm& u = upd[i];
            u = nt(p.precision, kNtAxpby, ch.count, sh.Lp, sh.rp, sh.rp, Vc, sh.rp, padded, G, sh.rp,
                   sq);
            if (cform) {
                u.alpha = -0.5f;
                u.beta = 1.5f;
                u.C = Vc;
                u.ldc = sh.rp;
                u.sC = padded;
            }
            u.Y = at(w->V[1 - cur], ch.off_pad, eb);
            u.ldy = sh.rp;
            u.sY = padded;
            if (!mn || (last && !sh.tall)) {
                u.Yt = at(w->W[1 - cur], ch.off_pad, eb);
                u.ldyt = sh.Lp;
                u.sYt = padded;
            }
        }
        int rc = nt_gemm(gram, n, sm_count, p.status, s, launches);
        if (rc == CAM_OK) rc = nt_gemm(upd, n, sm_count, p.status, s, launches);
        if (rc != CAM_OK) return rc;
        cur ^= 1;
    }
    for (size_t i = 0; i < pass.size(); ++i) {
        const int rc = apply_chunk(w, pass[i], p, cur, grids[i], s, launches);
        if (rc != CAM_OK) return rc;
    }
    return CAM_OK;
}

}  // namespace
}  // namespace cam

namespace cam {

int ortho_create(OrthoWork** out, int64_t cap_pad, int64_t cap_gram, int64_t big_gram) {
    *out = nullptr;
    OrthoWork* w = new (std::nothrow) OrthoWork;
    if (!w) return record_error(CAM_E_NOMEM, "orthogonalisation: out of host memory");
    w->cap_pad = std::max<int64_t>(cap_pad, 128 * 128);
    w->cap_gram = std::max<int64_t>(cap_gram, 128 * 128);
    w->cap_sq = 7 * std::max<int64_t>(big_gram, 128 * 128);
    auto up = [](size_t b) { return (b + 255) / 256 * 256; };
    const size_t bx = up(sizeof(float) * size_t(w->cap_pad));
    const size_t bg = up(sizeof(float) * size_t(w->cap_gram));
    const size_t bq = up(sizeof(float) * size_t(w->cap_sq));
    const size_t bk = up(sizeof(float) * size_t(kSplitFloats));
    const size_t bp = up(sizeof(double) * size_t(kOrthoBatchMax) * kOrthoBlocksMax);
    const size_t bs = up(sizeof(double) * kOrthoBatchMax);
    const size_t bi = up(sizeof(float) * kOrthoBatchMax);
    const size_t bc = 256;  // the unit counters
    const size_t total = 5 * bx + bg + bq + bk + bp + bs + bi + bc;
    if (cudaMalloc(&w->block, total) != cudaSuccess) {
        cudaGetLastError();
        delete w;
        return record_error(CAM_E_NOMEM, "orthogonalisation: cudaMalloc(%zu) failed", total);
    }
    char* b = static_cast<char*>(w->block);
    w->X = reinterpret_cast<float*>(b);
    w->W[0] = b + bx;
    w->W[1] = b + 2 * bx;
    w->V[0] = b + 3 * bx;
    w->V[1] = b + 4 * bx;
    b += 5 * bx;
    w->G = b;
    w->Sq = reinterpret_cast<float*>(b + bg);
    w->split = reinterpret_cast<float*>(b + bg + bq);
    w->partials = reinterpret_cast<double*>(b + bg + bq + bk);
    w->scalars = reinterpret_cast<double*>(b + bg + bq + bk + bp);
    w->inv_norm = reinterpret_cast<float*>(b + bg + bq + bk + bp + bs);
    w->sched = reinterpret_cast<int32_t*>(b + bg + bq + bk + bp + bs + bi);
    // (once per context: finished before any stream's GEMM can read them)
    if (cudaMemset(w->sched, 0, bc) != cudaSuccess || cudaStreamSynchronize(nullptr) != cudaSuccess) {
        cudaGetLastError();
        cudaFree(w->block);
        delete w;
        return record_error(CAM_E_CUDA, "orthogonalisation: clearing the unit counters failed");
    }
    *out = w;
    return CAM_OK;
}

void ortho_destroy(OrthoWork* w) {
    if (!w) return;
    cudaFree(w->block);
    delete w;
}

int ortho_round(OrthoWork* w, const std::vector<std::vector<OrthoMatrix>>& groups,
                const OrthoParams& p, cudaStream_t s, int sm_count, int64_t* launches) {
    // Chunks: each shape group cut into batches the workspace holds.
    std::vector<Chunk> chunks;
    for (const auto& grp : groups) {
        if (grp.empty()) continue;
        Shape sh;
        sh.m = grp[0].rows;
        sh.n = grp[0].cols;
        sh.tall = sh.m >= sh.n;
        sh.r = std::min(sh.m, sh.n);
        sh.L = std::max(sh.m, sh.n);
        sh.rp = pad128(sh.r);
        sh.Lp = pad128(sh.L);
        const int64_t padded = sh.rp * sh.Lp, sq = sh.rp * sh.rp;
        const bool short_side = p.short_side && sh.L >= 4 * sh.r;
        int64_t per = std::min<int64_t>(kOrthoBatchMax, std::min(w->cap_pad / padded, w->cap_gram / sq));
        if (short_side) per = std::min<int64_t>(per, w->cap_sq / (7 * sq));
        per = std::max<int64_t>(per, 1);
        for (size_t first = 0; first < grp.size(); first += per) {
            Chunk ch{};
            ch.mats = grp.data() + first;
            ch.count = static_cast<int>(std::min<int64_t>(per, int64_t(grp.size() - first)));
            ch.sh = sh;
            chunks.push_back(ch);
        }
    }
    // Passes: consecutive chunks of one tile width that fit the workspace
    // together; a short-side chunk runs alone.
    size_t i = 0;
    while (i < chunks.size()) {
        std::vector<Chunk> pass;
        int64_t pad = 0, gram = 0;
        int slots = 0;
        const bool wide256 = chunks[i].sh.rp % 256 == 0;
        while (i < chunks.size()) {
            Chunk ch = chunks[i];
            const bool ss = p.short_side && ch.sh.L >= 4 * ch.sh.r;
            const int64_t need_pad = ch.padded() * ch.count, need_gram = ch.sq() * ch.count;
            const bool fits = pad + need_pad <= w->cap_pad && gram + need_gram <= w->cap_gram &&
                              slots + ch.count <= kOrthoBatchMax &&
                              int(pass.size()) < kOrthoPassChunks &&
                              (ch.sh.rp % 256 == 0) == wide256;
            if (!pass.empty() && (ss || !fits)) break;
            ch.slot0 = slots;
            ch.off_x = pad;  // Delta holds m n <= padded floats per matrix
            ch.off_pad = pad;
            ch.off_gram = gram;
            pass.push_back(ch);
            pad += need_pad;
            gram += need_gram;
            slots += ch.count;
            ++i;
            if (ss) break;
        }
        const int rc = run_pass(w, pass, p, s, sm_count, launches);
        if (rc != CAM_OK) return rc;
    }
    return CAM_OK;
}

}  // namespace cam
