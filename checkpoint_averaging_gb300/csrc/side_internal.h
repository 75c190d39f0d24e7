// side_internal.h -- structures of the paths beside the merge pass: eager
// folds (eager.cu) and the outer orthogonalisation (ortho.cu), shared with the
// host runtime. Kept apart from cam_internal.h, which the merge pass is built
// from, so that these paths change without touching it.
#pragma once

#include <vector>

#include "cam_internal.h"

namespace cam {

// Eagerly folded rounds (cam_merge_fold, eager.cu). One launch covers up to
// kEagerTensors of the fragment's local tensors [local0, local0 + n_local).
constexpr int kEagerTensors = 1024;

// Folds one arriving worker into the round's fp32 running sum.
struct FoldArgs {
    const ChunkDesc* chunks;   // first chunk of this launch (device)
    const TensorSlot* slots;   // the fragment's tensors, by local index (device)
    double* worker_partials;   // [chunk * CAM_KMAX + k]: this worker's drift partials, or null
    int32_t* status;           // device status word (kStatus* bits)
    int32_t n_chunks;
    int32_t local0;
    int32_t n_local;
    int32_t k;                 // the worker's arrival index
    int32_t first;             // 1: the sum starts at +0 (first arrival)
    float w;                   // (float)tokens, token-weighted delta mode
    uint32_t vec[kEagerTensors / 32];  // bit l: tensor local0+l takes the vector path
    const void* x[kEagerTensors];      // the worker's copy of tensor local0+l
    float* sum[kEagerTensors];         // the running sum of tensor local0+l
};
static_assert(sizeof(FoldArgs) <= 32000, "kernel parameter block too large");

// The final pass of an eagerly folded round: fold the workers accumulated
// after the round's folds (P of them, arrival order; often just the last
// arrival), then finalize from the running sum: outer step, EMA, running
// average, drift partials and published copies.
constexpr int kFinalPtrs = 3 * kEagerTensors;
struct FinalArgs {
    const ChunkDesc* chunks;
    const TensorSlot* slots;
    double* partials;          // drift partial per chunk of this launch, or null
    int32_t* status;           // device status word (kStatus* bits)
    int32_t n_chunks;
    int32_t local0;
    int32_t n_local;
    int32_t K;
    float Kf;                  // (float)K
    float W;                   // (float)sum tokens
    float lr, mu, beta;
    float swa_n;               // globals in the running average after this round
    DivPlan div;               // the division: by Kf (plain mean) or W (delta)
    DivPlan swa_div;           // the running average's division, by swa_n
    int32_t stride;            // pointers per tensor in ptr[]: 3 + P
    int32_t P;                 // workers folded by this pass
    int32_t first_k;           // arrival index of the first of them (the folds before)
    float wp[CAM_KMAX];        // (float)tokens of those workers
    double* worker_partials;   // [chunk * CAM_KMAX + k]: their drift partials, or null
    uint32_t vec[kEagerTensors / 32];
    // per local tensor l, at ptr[l * stride]: the running sum, then the copy
    // of the new theta and of the EMA (or null), then the P workers' copies
    const void* ptr[kFinalPtrs];
};
static_assert(sizeof(FinalArgs) <= 32000, "kernel parameter block too large");

cudaError_t launch_fold(const FoldArgs& a, int dtype, int mode, bool worker_drift, int grid,
                        cudaStream_t s);
cudaError_t launch_final(const FinalArgs& a, int dtype, int mode, bool ema, bool norm, bool pub,
                         bool swa, bool worker_drift, int grid, cudaStream_t s);

// Outer orthogonalisation (ortho.cu): a per-context workspace, made at the
// first orthogonalised commit, and the per-matrix pipeline.
struct OrthoWork;
struct OrthoMatrix {
    float* theta;
    float* e;                    // EMA buffer or null
    int64_t rows, cols;          // row-major
    const void* x[CAM_KMAX];     // the included workers' copies, arrival order
};
struct OrthoParams {
    int K, dtype;
    float lr;
    int scale_mode, precision, iterations;
    bool ema;
    float beta;
    bool short_side;  // iterate in the short side's space (CAM_ORTHO_SHORT_SIDE)
    int32_t* status;  // the context's device status word
};
// cap_pad / cap_gram: elements in each iterate buffer and in the Gram buffer,
// in the GEMMs' layout (r x L and r x r, each side padded to a multiple of
// 128; at least one matrix's worth, batches of equal-shape matrices share
// them); big_gram: the largest padded r x r (the short-side form's squares).
int ortho_create(OrthoWork** out, int64_t cap_pad, int64_t cap_gram, int64_t big_gram);
void ortho_destroy(OrthoWork* w);
// Orthogonalises a round's matrices, given as groups of equal shape: each
// group in batches the workspace holds, and batches of one tile width that
// fit the workspace together iterated in step (one Gram and one update GEMM
// launch per Newton-Schulz step for all of them).
int ortho_round(OrthoWork* w, const std::vector<std::vector<OrthoMatrix>>& groups,
                const OrthoParams& p, cudaStream_t s, int sm_count, int64_t* launches);

}  // namespace cam
