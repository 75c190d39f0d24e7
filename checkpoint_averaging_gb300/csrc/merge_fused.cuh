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
// partials are reproducible bit for bit. With fuse_finish the launch also
// finishes the norms from those partials in its last block (norm_device.cuh's
// finish_norms, the same sums as the separate norm pass).
#pragma once

#include <cuda_runtime.h>

#include "cam_internal.h"
#include "merge_device.cuh"
#include "norm_device.cuh"

namespace cam {
namespace dev {

template <typename XT, int MODE, bool EMA, int NL, bool PUB, bool SWA, bool FIN = false>
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
        // (a chunk that fails the device-side checks is skipped, its partials 0;
        // its slot is loaded once, before the check, which measured 17 %
        // faster on the running-average round than a separate size load)
        const ChunkDesc ch = a.chunks[c];
        const bool in_launch = chunk_in_launch(ch, a.local0, a.n_local);
        const TensorSlot ts = a.slots[in_launch ? ch.local : a.local0];
        if (!in_launch || !chunk_in_tensor(ch, ts)) {
            if (threadIdx.x == 0) {
                atomicOr(a.status, kStatusBadChunk);
                if (NORM) a.partials[c] = 0.0;
                if constexpr (WD) {
#pragma unroll
                    for (int k = 0; k < CAM_KMAX; ++k)
                        if (k < a.K) a.worker_partials[static_cast<int64_t>(c) * CAM_KMAX + k] = 0.0;
                }
            }
            parity ^= 1;  // the slots stay as they were: no barrier for this chunk
            continue;
        }
        const int l = ch.local - a.local0;
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
    if constexpr (NORM && FIN) {
        // Every block passes here once, after its last chunk. The partial
        // writes are fenced before the count; the block that brings the count
        // to gridDim.x sees every block's partials (read through L2), finishes
        // the norms and resets the count for the next launch.
        __shared__ int last;
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) last = atomicAdd(a.fin_counter, 1u) == gridDim.x - 1;
        __syncthreads();
        if (last) {
            __threadfence();
            finish_norms_tail(a.fin);
            if (threadIdx.x == 0) *a.fin_counter = 0u;
        }
    }
}

// The fused finish exists for norm level 1 (the round's drift): with
// per-worker drift as well, the finish's registers would push the fp32
// variants' main loop into spilling.
template <typename XT, int MODE, bool EMA, bool PUB, bool SWA>
MergeFn pick_fin(int nl, bool fin) {
    if (nl == 0) return merge_fused<XT, MODE, EMA, 0, PUB, SWA>;
    if (nl == 1)
        return fin ? merge_fused<XT, MODE, EMA, 1, PUB, SWA, true> : merge_fused<XT, MODE, EMA, 1, PUB, SWA>;
    return merge_fused<XT, MODE, EMA, 2, PUB, SWA>;
}

template <typename XT, int MODE, bool PUB, bool SWA>
MergeFn pick_level(bool ema, int nl, bool fin) {
    return ema ? pick_fin<XT, MODE, true, PUB, SWA>(nl, fin) : pick_fin<XT, MODE, false, PUB, SWA>(nl, fin);
}

template <typename XT, bool PUB, bool SWA>
MergeFn pick_mode(const MergeVariant& v) {
    return v.mode == kDelta ? pick_level<XT, kDelta, PUB, SWA>(v.ema, v.norm_level, v.fin)
                            : pick_level<XT, kMean, PUB, SWA>(v.ema, v.norm_level, v.fin);
}

template <typename XT>
MergeFn pick_for_dtype(const MergeVariant& v) {
    if (v.pub) return v.swa ? pick_mode<XT, true, true>(v) : pick_mode<XT, true, false>(v);
    return v.swa ? pick_mode<XT, false, true>(v) : pick_mode<XT, false, false>(v);
}

}  // namespace dev
}  // namespace cam
