// merge_fused.cuh -- the fused merge pass of the context path, as a template,
// and its variant dispatch. Each worker dtype instantiates it in its own
// translation unit (merge_fused_f32.cu, merge_fused_bf16.cu) so the variants
// compile in parallel.
//
// One launch covers the chunks of a fragment's tensors [local0, local0 +
// n_local). A persistent grid strides over the chunks; per chunk every thread
// takes 8 consecutive elements per step (merge_device.cuh). The norm level NL
// selects the drift diagnostics accumulated on the way:
//   0  none;
//   1  the mean worker displacement (the round's drift), one fp64 partial per
//      chunk;
//   2  as 1, plus each worker's own displacement x_k - theta_old, K partials
//      per chunk.
// Squares are summed in fp32 within a thread (at most 64 elements of one
// chunk), then in fp64 across the warp and the block in a fixed order, so the
// partials are reproducible bit for bit.
#pragma once

#include <cuda_runtime.h>

#include "cam_internal.h"
#include "merge_device.cuh"

namespace cam {
namespace dev {

template <typename XT, int MODE, bool EMA, int NL, bool PUB, bool SWA>
__global__ void __launch_bounds__(kThreads, 2)
    merge_fused(const __grid_constant__ MergeArgs a) {
    constexpr bool NORM = NL >= 1;
    constexpr bool WD = NL >= 2;
    constexpr int kWarps = kThreads / 32;
    // Two slots, alternating by chunk, so one barrier per chunk suffices: a
    // slot is written again only after the next chunk's barrier, which thread
    // 0 reaches only once it has read the slot.
    __shared__ double warp_part[2][kWarps];
    __shared__ double worker_part[2][WD ? kWarps * CAM_KMAX : 1];
    int parity = 0;
    for (int c = blockIdx.x; c < a.n_chunks; c += gridDim.x, parity ^= 1) {
        const ChunkDesc ch = a.chunks[c];
        const int l = ch.local - a.local0;
        const TensorSlot ts = a.slots[ch.local];
        const void* const* xs = a.x + static_cast<int64_t>(l) * a.stride;
        const bool vec = (a.vec[l >> 5] >> (l & 31)) & 1u;
        float acc = 0.0f;
        float accw[CAM_KMAX];
#pragma unroll
        for (int k = 0; k < CAM_KMAX; ++k) accw[k] = 0.0f;
        if (vec) {
            const int nv = ch.len >> 3;
            for (int v = threadIdx.x; v < nv; v += kThreads)
                merge_vec8<XT, MODE, EMA, NORM, PUB, SWA, WD>(a, xs, ts, ch.start + 8 * int64_t(v),
                                                              acc, accw);
            const int tail = ch.len & 7;
            if (static_cast<int>(threadIdx.x) < tail)
                merge_one<XT, MODE, EMA, NORM, PUB, SWA, WD>(
                    a, xs, ts, ch.start + 8 * int64_t(nv) + threadIdx.x, acc, accw);
        } else {
            for (int j = threadIdx.x; j < ch.len; j += kThreads)
                merge_one<XT, MODE, EMA, NORM, PUB, SWA, WD>(a, xs, ts, ch.start + j, acc, accw);
        }
        if constexpr (NORM) {
            const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
            const double d = warp_sum(static_cast<double>(acc));
            if (lane == 0) warp_part[parity][warp] = d;
            if constexpr (WD) {
#pragma unroll
                for (int k = 0; k < CAM_KMAX; ++k)
                    if (k < a.K) {  // K is the same for the whole block
                        const double dk = warp_sum(static_cast<double>(accw[k]));
                        if (lane == 0) worker_part[parity][warp * CAM_KMAX + k] = dk;
                    }
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                double s = 0.0;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) s += warp_part[parity][w];
                a.partials[c] = s;
            }
            if constexpr (WD) {
                if (static_cast<int>(threadIdx.x) < a.K) {
                    const int k = threadIdx.x;
                    double s = 0.0;
#pragma unroll
                    for (int w = 0; w < kWarps; ++w) s += worker_part[parity][w * CAM_KMAX + k];
                    a.worker_partials[static_cast<int64_t>(c) * CAM_KMAX + k] = s;
                }
            }
        }
    }
}

template <typename XT, int MODE, bool PUB, bool SWA>
MergeFn pick_level(bool ema, int nl) {
    if (ema) {
        if (nl == 0) return merge_fused<XT, MODE, true, 0, PUB, SWA>;
        if (nl == 1) return merge_fused<XT, MODE, true, 1, PUB, SWA>;
        return merge_fused<XT, MODE, true, 2, PUB, SWA>;
    }
    if (nl == 0) return merge_fused<XT, MODE, false, 0, PUB, SWA>;
    if (nl == 1) return merge_fused<XT, MODE, false, 1, PUB, SWA>;
    return merge_fused<XT, MODE, false, 2, PUB, SWA>;
}

template <typename XT, bool PUB, bool SWA>
MergeFn pick_mode(const MergeVariant& v) {
    return v.mode == kDelta ? pick_level<XT, kDelta, PUB, SWA>(v.ema, v.norm_level)
                            : pick_level<XT, kMean, PUB, SWA>(v.ema, v.norm_level);
}

template <typename XT>
MergeFn pick_for_dtype(const MergeVariant& v) {
    if (v.pub) return v.swa ? pick_mode<XT, true, true>(v) : pick_mode<XT, true, false>(v);
    return v.swa ? pick_mode<XT, false, true>(v) : pick_mode<XT, false, false>(v);
}

}  // namespace dev
}  // namespace cam
