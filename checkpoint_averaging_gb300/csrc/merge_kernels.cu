// merge_kernels.cu -- the device side of the DiLoCo outer merge for sm_103a.
//
// merge_fused: one pass over a fragment's ragged tensor list that, per
// element, widens the K workers' values to fp32, folds them in arrival order
// (plain mean, or token-weighted mean of the deltas), applies the outer step
// (plain replacement, or outer Nesterov), updates the EMA of the globals and
// accumulates the squared drift. Every state element (theta, m, e) is read at
// most once and written once, every worker element is read once.
//   Plain mean in a running fp32 sum as checkpoints arrive: "DiffuRefill-1B"
//   model card, "How it is trained", Merging. Plain replacement and the EMA of
//   globals (beta 0.9): "DiffuRefill-1B: Pretraining a Masked Diffusion
//   Language Model on Free, Preemptible Notebook GPUs", section 3, Table 2.
//   Token-weighted delta mean and outer Nesterov (lr 0.7, momentum 0.9):
//   "Pythia-14M on four rented GPUs and a bucket", "Getting updates through
//   the bucket".
//
// The pass is HBM-bound (a handful of flops per 20-40 bytes), so the design is
// about bytes in flight: 32-byte fp32 / 16-byte bf16 vector loads per thread,
// read-once worker data loaded through the non-coherent path without L1
// allocation and marked evict-first in L2, and a persistent grid striding over
// fixed-size chunks of the fragment. Arithmetic uses explicit round-to-nearest
// intrinsics, so no multiply-add is contracted and every result is the fixed
// sequence of binary32 operations the C ABI documents.
//
// norm_finish: sums the per-chunk drift partials per tensor and per fragment
// in a fixed order, so norms are bitwise reproducible.
#include <cuda_runtime.h>

#include "cam_internal.h"
#include "merge_device.cuh"

namespace cam {
namespace {

using namespace cam::dev;

// ---- the fused pass ------------------------------------------------------------

template <typename XT, int MODE, bool EMA, bool NORM, bool PUB, bool SWA>
__global__ void __launch_bounds__(kThreads, 2)
    merge_fused(const __grid_constant__ MergeArgs a) {
    __shared__ double warp_part[kThreads / 32];
    for (int c = blockIdx.x; c < a.n_chunks; c += gridDim.x) {
        const ChunkDesc ch = a.chunks[c];
        const int l = ch.local - a.local0;
        const TensorSlot ts = a.slots[ch.local];
        const void* const* xs = a.x + static_cast<int64_t>(l) * a.stride;
        const bool vec = (a.vec[l >> 5] >> (l & 31)) & 1u;
        float acc = 0.0f;
        if (vec) {
            const int nv = ch.len >> 3;
            for (int v = threadIdx.x; v < nv; v += kThreads)
                merge_vec8<XT, MODE, EMA, NORM, PUB, SWA>(a, xs, ts, ch.start + 8 * int64_t(v), acc);
            const int tail = ch.len & 7;
            if (static_cast<int>(threadIdx.x) < tail)
                merge_one<XT, MODE, EMA, NORM, PUB, SWA>(a, xs, ts,
                                                    ch.start + 8 * int64_t(nv) + threadIdx.x, acc);
        } else {
            for (int j = threadIdx.x; j < ch.len; j += kThreads)
                merge_one<XT, MODE, EMA, NORM, PUB, SWA>(a, xs, ts, ch.start + j, acc);
        }
        if (NORM) {
            // fp32 within a thread (at most a few dozen squares), fp64 above.
            const double d = warp_sum(static_cast<double>(acc));
            if ((threadIdx.x & 31) == 0) warp_part[threadIdx.x >> 5] = d;
            __syncthreads();
            if (threadIdx.x == 0) {
                double s = 0.0;
#pragma unroll
                for (int w = 0; w < kThreads / 32; ++w) s += warp_part[w];
                a.partials[c] = s;
            }
            __syncthreads();
        }
    }
}

__global__ void __launch_bounds__(1024) norm_finish(const NormArgs a) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int n_warps = blockDim.x >> 5;
    for (int t = warp; t < a.n_tensors; t += n_warps) {
        double s = 0.0;
        for (int c = a.first_chunk[t] + lane; c < a.first_chunk[t + 1]; c += 32)
            s += a.partials[c];
        s = warp_sum(s);
        if (lane == 0) a.tsq[t] = s;
    }
    __syncthreads();
    if (warp == 0) {
        double s = 0.0;
        for (int t = lane; t < a.n_tensors; t += 32) s += a.tsq[t];
        s = warp_sum(s);
        if (lane == 0 && a.per_fragment) *a.per_fragment = sqrt(s);
    }
    if (a.per_tensor)
        for (int t = threadIdx.x; t < a.n_tensors; t += blockDim.x)
            a.per_tensor[t] = sqrt(a.tsq[t]);
}

__global__ void fill_kernel(float* dst, int64_t n, float v) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
         i += int64_t(gridDim.x) * blockDim.x)
        dst[i] = v;
}

__global__ void copy_kernel(float* dst, const float* src, int64_t n) {
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n;
         i += int64_t(gridDim.x) * blockDim.x)
        dst[i] = src[i];
}

// ---- variant dispatch ------------------------------------------------------------

using MergeFn = void (*)(MergeArgs);

template <typename XT, int MODE, bool PUB, bool SWA>
MergeFn pick_en(bool ema, bool norm) {
    if (ema)
        return norm ? merge_fused<XT, MODE, true, true, PUB, SWA>
                    : merge_fused<XT, MODE, true, false, PUB, SWA>;
    return norm ? merge_fused<XT, MODE, false, true, PUB, SWA>
                : merge_fused<XT, MODE, false, false, PUB, SWA>;
}

template <bool PUB, bool SWA>
MergeFn pick_dm(const MergeVariant& v) {
    if (v.dtype == kDtBF16)
        return v.mode == kDelta ? pick_en<uint16_t, kDelta, PUB, SWA>(v.ema, v.norm)
                                : pick_en<uint16_t, kMean, PUB, SWA>(v.ema, v.norm);
    return v.mode == kDelta ? pick_en<float, kDelta, PUB, SWA>(v.ema, v.norm)
                            : pick_en<float, kMean, PUB, SWA>(v.ema, v.norm);
}

MergeFn pick(const MergeVariant& v) {
    if (v.pub) return v.swa ? pick_dm<true, true>(v) : pick_dm<true, false>(v);
    return v.swa ? pick_dm<false, true>(v) : pick_dm<false, false>(v);
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, const MergeVariant& v, int grid, cudaStream_t s) {
    MergeFn fn = pick(v);
    void* args[] = {const_cast<MergeArgs*>(&a)};
    return cudaLaunchKernel(reinterpret_cast<const void*>(fn), dim3(grid), dim3(kThreads),
                            args, 0, s);
}

int merge_blocks_per_sm(const MergeVariant& v) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &n, reinterpret_cast<const void*>(pick(v)), kThreads, 0) !=
        cudaSuccess)
        return 0;
    return n;
}

cudaError_t launch_norm_finish(const NormArgs& a, cudaStream_t s) {
    norm_finish<<<1, 1024, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_fill(float* dst, int64_t n, float v, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const int64_t blocks = (n + 255) / 256;
    fill_kernel<<<static_cast<int>(blocks < 4096 ? blocks : 4096), 256, 0, s>>>(dst, n, v);
    return cudaGetLastError();
}

cudaError_t launch_copy(float* dst, const float* src, int64_t n, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    const int64_t blocks = (n + 255) / 256;
    copy_kernel<<<static_cast<int>(blocks < 4096 ? blocks : 4096), 256, 0, s>>>(dst, src, n);
    return cudaGetLastError();
}

}  // namespace cam
