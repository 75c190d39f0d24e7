// nt_gemm.h -- the dense contractions of the outer orthogonalisation
// (Newton-Schulz steps toward the polar factor, "DiffuRefill-1B" technical
// report, section 5.3), as batched "NT" GEMMs over this library's padded
// operand layout:
//
//     D[b][i][j] = sum_k A[b][i][k] * B[b][j][k]      (A: M x K, B: N x K)
//
// Both operands are row-major with K contiguous ("K-major" for the tensor
// cores), so every product the iteration needs is one of these: the matrix
// H = 1.5 I - 0.5 W W^T of an iterate W (a Gram product, A = B = W, with the
// step's combination in its epilogue), and the update V' = V H of its
// transpose V = W^T (A = V, B = H, which is symmetric), whose epilogue also
// writes W' = V'^T for the next Gram product.
//
// M, N and K are multiples of 128, with zero padding outside the matrices'
// own extent (zero rows and columns stay zero through the iteration), so no
// kernel handles a ragged edge.
//
// Precisions: CAM_ORTHO_BF16 (bf16 operands and results, fp32 accumulation)
// and CAM_ORTHO_TF32 (fp32 storage read as TF32, fp32 accumulation) run on the
// tensor cores (tcgen05.mma with TMEM accumulators, operands staged by TMA,
// results written back by TMA); CAM_ORTHO_FP32 runs a CUDA-core fp32 kernel.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace cam {

// What the epilogue does with the accumulated tile D.
enum NtEpilogue : int {
    // Y = alpha D + beta C + diag I (C optional: CUDA-core kernel only),
    // stored to Y (optional) and, transposed, to Yt (optional).
    kNtAxpby = 0,
    // Y = alpha D + diag I with D the Gram matrix of A (B must be A, M = N):
    // only tiles that reach the upper triangle are computed; each stores its
    // 32 x 32 boxes on and above the diagonal and mirrors those above it, so
    // Y is the whole symmetric matrix, every element written once.
    kNtGram = 1,
};

struct NtGemm {
    int precision;          // CAM_ORTHO_BF16, CAM_ORTHO_TF32 or CAM_ORTHO_FP32
    int epilogue;           // NtEpilogue
    int32_t batch;          // matrices, each at its own batch stride
    int64_t M, N, K;        // multiples of 128
    const void* A; int64_t lda, sA;   // row stride and batch stride, in elements
    const void* B; int64_t ldb, sB;
    // A stored transposed (K x M, row stride lda) and B likewise (K x N):
    // "MN-major" operands, for the Gram product V^T V of a tall iterate V
    // without its transpose (bf16 Gram products only)
    bool mn_major;
    float alpha, beta, diag;
    const void* C; int64_t ldc, sC;   // CAM_ORTHO_FP32 only: read when beta != 0
    void* Y; int64_t ldy, sY;
    void* Yt; int64_t ldyt, sYt;      // kNtAxpby: transposed copy, or null
    // Gram matrices of long operands split their K range over several blocks
    // into fp32 partial tiles here (summed in a fixed order by a second
    // kernel); null or too small: no split.
    float* partials; int64_t partial_floats;
    // Gram products on the tensor cores: two int32 counters in device memory,
    // 0 before the first launch, through which the launch hands out its tiles
    // (and which it leaves at 0); launches that share them run one at a time
    int32_t* sched;
};

// Enqueues n products (1 <= n <= 8) on `s` as one launch of the tensor-core
// kernel: every problem of a launch has the same precision, epilogue, alpha,
// beta and diag; their tiles are numbered one problem after another and the
// persistent grid takes them in turn, so small products share the GPU
// instead of each leaving most of it idle. Gram products whose tiles are long
// split their K range (partials summed afterwards, one launch per such
// problem). The launch is a programmatic dependent of the previous kernel on
// the stream: its set-up overlaps that kernel's tail, and it reads and writes
// global memory only once that kernel has completed. (CAM_ORTHO_FP32: one
// CUDA-core launch per problem.) `status` is the context's device status
// word: a tensor-core kernel whose barrier wait runs out (a fault of this
// library, never expected) sets CAM_STATUS_GEMM_TIMEOUT there and returns.
// Counts the kernels launched in *launches.
int nt_gemm(const NtGemm* g, int n, int sm_count, int32_t* status, cudaStream_t s,
            int64_t* launches);

// Bytes of one stored element: bf16 for CAM_ORTHO_BF16, fp32 otherwise.
inline int64_t nt_elem_bytes(int precision) { return precision == 2 /* CAM_ORTHO_BF16 */ ? 2 : 4; }

}  // namespace cam
