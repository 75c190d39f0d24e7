// cam_internal.h -- structures shared by the host runtime and the CUDA kernels
// of libcam. Not part of the C ABI (include/cam.h is).
#pragma once

#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>

#include "cam.h"

namespace cam {

// Threads per block of the fused merge pass, and elements one thread handles
// per step of its chunk loop (one 32-byte fp32 vector / one 16-byte bf16 one).
constexpr int kThreads = 256;
constexpr int kVec = 8;
// Chunks are multiples of one block-step so that every chunk start keeps the
// tensor's vector alignment.
constexpr int kChunkQuantum = kThreads * kVec;  // 2048 elements
constexpr int kMaxChunkElems = 8 * kChunkQuantum;
// Worker pointers carried in one launch's parameter block. Kernel parameters
// may take up to 32,764 bytes; this keeps MergeArgs under that.
constexpr int kXCap = 3520;

// The staged form of the fused pass (merge_staged.cuh): one block per SM of
// 16 consumer warps, one producer warp that streams tiles of kStTile elements
// of every input array into a ring of shared-memory stages with bulk copies,
// and one warp that reduces the drift partials.
constexpr int kStConsumerWarps = 16;
constexpr int kStConsumers = kStConsumerWarps * 32;
constexpr int kStThreads = kStConsumers + 64;
constexpr int kStTile = kStConsumers * 4;      // 2048 elements: 4 per consumer
constexpr int kStMaxStages = 16;
constexpr int kStRedSlots = 2;                 // drift hand-over buffers (double buffering)
constexpr int kStSmemBytes = 224 * 1024;       // dynamic shared memory: ring + hand-over
static_assert(kChunkQuantum % kStTile == 0, "tiles must not straddle chunks");

// Fragments of at most this many chunks (with the round's drift norms asked
// for) take the register form with the norm finish fused into its last block.
constexpr int kFuseMaxChunks = 4096;

// Bits of the context's device status word (cam_ctx_status).
constexpr int32_t kStatusWaitTimeout = 1;  // a staged pass gave up waiting on a barrier
constexpr int32_t kStatusBadChunk = 4;     // a merge pass met a chunk outside its tensor
constexpr int32_t kStatusProtocol = 8;     // a staged pass found a stage out of sequence

// One chunk of the fragment's element space: elements [start, start+len) of
// the fragment's local tensor `local`. Chunks never straddle tensors.
struct ChunkDesc {
    int64_t start;
    int32_t local;
    int32_t len;
};
static_assert(sizeof(ChunkDesc) == 16, "ChunkDesc is one 16-byte load");

// A fragment tensor's caller-owned state buffers.
struct TensorSlot {
    float* theta;
    float* m;
    float* e;
    float* swa;  // uniform running average of the globals, or null
    int64_t numel;
};

// Parameter block of the deterministic norm finish.
struct NormArgs {
    const double* partials;     // [n_chunks of the fragment]
    const int32_t* first_chunk; // [n_tensors + 1]: tensor t owns chunks [first[t], first[t+1])
    int32_t n_tensors;
    double* tsq;                // scratch [n_tensors]: squared norms
    double* per_tensor;         // output or null
    double* per_fragment;       // output or null
    // per-worker drift (K > 0 when asked for)
    int32_t K;
    const double* worker_partials;  // [n_chunks * CAM_KMAX]
    double* worker_tsq;             // scratch [n_tensors * CAM_KMAX]
    double* per_worker_tensor;      // output [K * n_tensors] or null
    double* per_worker;             // output [K] or null
    // the fused finish (K = 0 only): the fragment's chunk count, and 1 when
    // the launch gives every block finish_smem_bytes() of dynamic shared
    // memory, into which the finishing block copies the partials first
    int32_t n_chunks;
    int32_t shared;
};

// The divisor of a round's division (the worker count in plain-mean mode,
// the token total in delta mode) and what its reciprocal form needs: the
// reciprocal as two terms, y = RN(1/d) and y_lo = RN(1/d - y), and the
// dividends s that take that form, |s| in [2^lo_e, 2^hi_e) -- as floats lo_f
// and hi_f, and as the bit patterns [lo, lo + span) of |s|. For those no
// intermediate of the form leaves the normal range (the derivation is at
// div_fast in merge_device.cuh). A zero dividend gives itself; every other
// dividend, and every dividend of a divisor outside [2^-100, 2^100]
// (active 0: span 0, lo_f = inf, hi_f = 0), takes the division instruction
// sequence.
struct DivPlan {
    float d;
    float y;
    float y_lo;
    float lo_f;
    float hi_f;
    uint32_t lo;
    uint32_t span;
    uint32_t active;
};

inline DivPlan div_plan(float d) {
    // (host binary32 division: correctly rounded; 1/d - y is exact in binary64
    // up to the binary64 quotient's rounding, 2^-53 of 1/d)
    const float y = 1.0f / d;
    DivPlan p{d, y, static_cast<float>(1.0 / static_cast<double>(d) - static_cast<double>(y)),
              HUGE_VALF, 0.0f, 0u, 0u, 0u};
    if (d >= 0x1p-100f && d <= 0x1p100f) {
        int e = 0;
        std::frexp(d, &e);  // d in [2^(e-1), 2^e)
        const int lo_e = e - 124 > -100 ? e - 124 : -100;
        const int hi_e = e + 124 < 126 ? e + 124 : 126;
        p.lo_f = std::ldexp(1.0f, lo_e);
        p.hi_f = std::ldexp(1.0f, hi_e);
        p.lo = static_cast<uint32_t>(lo_e + 127) << 23;
        p.span = (static_cast<uint32_t>(hi_e + 127) << 23) - p.lo;
        p.active = 1u;
    }
    return p;
}

// Dynamic shared memory of a fused finish that stages the partials, the
// squared norms and the chunk index of a fragment of n_tensors tensors and
// n_chunks chunks; launches give it when it is at most kFinishSmemMax.
inline size_t finish_smem_bytes(int64_t n_tensors, int64_t n_chunks) {
    return size_t(8 * n_chunks + 8 * n_tensors + 4 * (n_tensors + 1));
}
constexpr size_t kFinishSmemMax = 40 * 1024;  // (with the static shared memory, within the default 48 KB)

// Parameter block of one launch of the fused merge pass. The launch covers
// the fragment's local tensors [local0, local0 + n_local) and their chunks.
struct MergeArgs {
    const ChunkDesc* chunks;  // first chunk of this launch (device)
    const TensorSlot* slots;  // the fragment's tensors, by local index (device)
    double* partials;         // drift partial per chunk of this launch (device) or null
    double* worker_partials;  // [chunk * CAM_KMAX + k]: worker k's drift partials, or null
    int32_t n_chunks;
    int32_t local0;
    int32_t n_local;
    int32_t K;
    int32_t stride;           // pointers per tensor in x: K, or K + 2 when publishing
    float Kf;                 // (float)K
    float w[CAM_KMAX];        // (float)tokens_k
    float W;                  // (float)sum tokens
    float lr, mu, beta;
    float swa_n;              // globals in the running average after this round
    DivPlan div;              // the division: by Kf (plain mean) or W (delta)
    DivPlan swa_div;          // the running average's division, by swa_n
    int32_t* status;          // device status word (kStatus* bits)
    int32_t st_stages;        // staged pass: stages in the shared-memory ring
    int32_t st_stage_bytes;   // staged pass: bytes of one stage
    int32_t test_stall;       // staged pass, CAM_TEST_STALL_STAGED: withhold the first tile,
                              // give up waiting after kTestWaitLimitNs
    int32_t test_tag;         // staged pass, CAM_TEST_BAD_TAG: give the end marker a wrong
                              // fill number, give up waiting after kTestWaitLimitNs
    // Register pass with the norm finish fused (MergeVariant::fin): the last
    // block to finish its chunks (counted on *fin_counter, which it resets to
    // 0) finishes the norms as the norm pass would, so that pass is not
    // launched.
    unsigned int* fin_counter;
    NormArgs fin;
    uint32_t vec[(kXCap + 31) / 32];  // bit l: tensor local0+l takes the vector path
    // x[l*stride + k]: worker k's copy of tensor local0+l; when publishing,
    // x[l*stride + K] and x[l*stride + K + 1] take the new theta and EMA. The
    // spare slots keep every x[l*stride + k] with k < CAM_KMAX + 2 inside.
    const void* x[kXCap + CAM_KMAX + 2];
};
static_assert(sizeof(MergeArgs) <= 32000, "kernel parameter block too large");


enum Variant : int { kDtF32 = 0, kDtBF16 = 1 };

// Records a message for the calling thread (returned by cam_last_error) and
// returns `code`.
int record_error(int code, const char* fmt, ...);

// Launches one fused merge pass with `grid` blocks.
// Variant selection of the fused pass. norm_level: 0 none, 1 round drift,
// 2 round drift and per-worker drift.
struct MergeVariant {
    int dtype, mode;
    bool ema;
    int norm_level;
    bool pub, swa;
    bool fin = false;  // register form: finish the norms in the pass's last block
};
using MergeFn = void (*)(MergeArgs);
MergeFn pick_merge_f32(const MergeVariant& v);
MergeFn pick_merge_bf16(const MergeVariant& v);
cudaError_t launch_merge(const MergeArgs& a, const MergeVariant& v, int grid, cudaStream_t s);
// The staged pass: one block of kStThreads per SM, a ring of st_stages stages.
MergeFn pick_staged_f32(const MergeVariant& v);
MergeFn pick_staged_bf16(const MergeVariant& v);
// State arrays a variant streams besides the workers (theta, m, e, swa).
int staged_state_arrays(const MergeVariant& v);
// Bytes of one stage for K workers of that variant.
int64_t staged_stage_bytes(const MergeVariant& v, int K);
// Bytes of the drift hand-over buffers after the ring (0 without norms).
int64_t staged_red_bytes(const MergeVariant& v, int K);
// Lets every staged variant use kStSmemBytes of dynamic shared memory.
cudaError_t staged_prepare();
cudaError_t launch_merge_staged(const MergeArgs& a, const MergeVariant& v, int grid,
                                cudaStream_t s);
// Resident blocks per SM of that variant (0 on error).
int merge_blocks_per_sm(const MergeVariant& v);

// ---- several rounds in one register-form pass (cam_merge_commit_many) -------

constexpr int kMultiMax = CAM_MAX_OPEN_ROUNDS;  // rounds per pass
constexpr int kMultiXCap = 3584;                // worker and copy pointers per pass

// One round of a multi-round pass: its fragment's tables, its finish, the
// place of its chunks among the pass's and of its pointers in x[], and the
// scalars the per-element arithmetic reads (merge_elem's K, Kf, w, W, lr, mu,
// beta, div).
struct MultiRound {
    const ChunkDesc* chunks;   // the fragment's chunk table (device)
    const TensorSlot* slots;   // the fragment's tensors, by local index (device)
    double* partials;          // the fragment's drift partials (norms only)
    unsigned int* fin_counter; // blocks done with this round's chunks (norms only)
    NormArgs fin;              // the finish of this round's norms (norms only)
    int32_t c_begin;           // the round's chunks are the pass's [c_begin, c_begin + n_chunks)
    int32_t n_chunks;
    int32_t x0;                // x[x0 + l * stride + k]: worker k's copy of local tensor l
    int32_t vec0;              // bit vec0 + l of vec[]: tensor l takes the vector path
    int32_t n_local;           // the fragment's tensors
    int32_t stride;            // K, or K + 2 when publishing
    int32_t K;
    float Kf;
    float w[CAM_KMAX];
    float W, lr, mu, beta;
    DivPlan div;               // the division: by Kf (plain mean) or W (delta)
};

struct MultiArgs {
    int32_t n_rounds;
    int32_t n_chunks;          // all rounds' chunks
    int32_t* status;           // device status word (kStatus* bits)
    int32_t pad;
    MultiRound r[kMultiMax];
    uint32_t vec[kMultiXCap / 32];
    const void* x[kMultiXCap + CAM_KMAX + 2];
};
static_assert(sizeof(MultiArgs) <= 32000, "kernel parameter block too large");

// The multi-round pass of a variant (no running average, norm level 0 or 1,
// the norms finished in the pass), with `smem` bytes of dynamic shared
// memory for the finishes.
cudaError_t launch_merge_multi(const MultiArgs& a, const MergeVariant& v, int grid, size_t smem,
                               cudaStream_t s);
int multi_blocks_per_sm(const MergeVariant& v);
cudaError_t launch_norm_finish(const NormArgs& a, cudaStream_t s);
cudaError_t launch_fill(float* dst, int64_t n, float v, cudaStream_t s);
cudaError_t launch_copy(float* dst, const float* src, int64_t n, cudaStream_t s);

}  // namespace cam
