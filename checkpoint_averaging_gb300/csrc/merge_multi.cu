// merge_multi.cu -- several rounds on disjoint fragments in one register-form
// merge pass (cam_merge_commit_many, declared in include/cam.h).
//
// "Pythia-14M on four rented GPUs and a bucket", "Getting updates through the
// bucket": parameters split into fragments, rounds per fragment, two of them
// in flight at once. Rounds that close together are merged here in one
// launch: the pass numbers every round's chunks one round after another and
// a persistent grid strides over all of them, so a short round's chunks and
// its norm finish run while the other blocks still stream a long round,
// instead of each round paying a launch, a ramp and a finish of its own.
//
// Per chunk the arithmetic is merge_fused's (merge_device.cuh's merge_vec8 /
// merge_one with the chunk's round as the source of K, w, W, lr, mu, beta),
// and the drift partials are summed in the same fixed order, so every round
// ends with the bits a commit of its own gives. The block that finishes the
// last of a round's chunks among those the round's blocks took (counted on
// that round's fin_counter, which it resets) finishes that round's norms
// (finish_norms_tail, the norm pass's sums).
#include <cuda_runtime.h>

#include "cam_internal.h"
#include "merge_device.cuh"
#include "norm_device.cuh"

namespace cam {
namespace {

using namespace cam::dev;

template <typename XT, int MODE, bool EMA, bool NORM, bool PUB>
__global__ void __launch_bounds__(kThreads, 2) merge_multi(const __grid_constant__ MultiArgs a) {
    constexpr int kWarps = kThreads / 32;
    // two slots alternating by chunk, one barrier per chunk (as merge_fused)
    __shared__ double warp_part[2][kWarps];
    __shared__ int last;
    int parity = 0;
    for (int c = blockIdx.x; c < a.n_chunks; c += gridDim.x, parity ^= 1) {
        int r = 0;  // the chunk's round (block-uniform)
#pragma unroll
        for (int q = 1; q < kMultiMax; ++q)
            if (q < a.n_rounds && c >= a.r[q].c_begin) r = q;
        const MultiRound& R = a.r[r];
        const int cl = c - R.c_begin;
        const ChunkDesc ch = R.chunks[cl];
        // the device-side check: a chunk outside its round's tensors is
        // taken as an empty chunk (nothing read or written, partial 0)
        const bool in_launch = static_cast<uint32_t>(ch.local) < static_cast<uint32_t>(R.n_local);
        const TensorSlot ts = R.slots[in_launch ? ch.local : 0];
        const bool ok = in_launch && chunk_in_tensor(ch, ts);
        if (!ok && threadIdx.x == 0) atomicOr(a.status, kStatusBadChunk);
        const int l = ok ? ch.local : 0;
        const int len = ok ? ch.len : 0;
        const void* const* xs = a.x + R.x0 + static_cast<int64_t>(l) * R.stride;
        const int vb = R.vec0 + l;
        float acc = 0.0f;
        if ((a.vec[vb >> 5] >> (vb & 31)) & 1u) {
            const int nv = len >> 3;
            for (int v = threadIdx.x; v < nv; v += kThreads) {
                const int64_t i = ch.start + 8 * int64_t(v);
                if constexpr (sizeof(XT) == 4) {
                    // fp32 workers in two steps of four: the round's scalars,
                    // held in registers here, leave no room for eight elements
                    // of every worker (eight measured 9 % slower with spills,
                    // two 27 % slower)
                    constexpr int N = 4;
#pragma unroll
                    for (int h = 0; h < 8; h += N)
                        merge_vecn_f32<N, MODE, EMA, NORM, PUB, false, false>(R, xs, ts, i + h, acc,
                                                                              nullptr);
                } else {
                    merge_vec8<XT, MODE, EMA, NORM, PUB>(R, xs, ts, i, acc);
                }
            }
            const int tail = len & 7;
            if (static_cast<int>(threadIdx.x) < tail)
                merge_one<XT, MODE, EMA, NORM, PUB>(R, xs, ts, ch.start + 8 * int64_t(nv) + threadIdx.x,
                                                    acc);
        } else {
            for (int j = threadIdx.x; j < len; j += kThreads)
                merge_one<XT, MODE, EMA, NORM, PUB>(R, xs, ts, ch.start + j, acc);
        }
        if constexpr (NORM) {
            const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
            const double d = warp_sum(static_cast<double>(acc));
            if (lane == 0) warp_part[parity][warp] = d;
            __syncthreads();
            if (threadIdx.x == 0) {
                double s = 0.0;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) s += warp_part[parity][w];
                R.partials[cl] = s;
            }
            // The block's last chunk of round r: the partial writes are
            // fenced before the count; the block that brings the count to the
            // round's number of blocks (min(grid, its chunks)) sees every
            // partial of the round, finishes its norms and resets the count.
            if (c + static_cast<int>(gridDim.x) >= R.c_begin + R.n_chunks) {
                __threadfence();
                __syncthreads();
                if (threadIdx.x == 0) {
                    const unsigned int blocks =
                        min(gridDim.x, static_cast<unsigned int>(R.n_chunks));
                    last = atomicAdd(R.fin_counter, 1u) == blocks - 1;
                }
                __syncthreads();
                if (last) {
                    __threadfence();
                    finish_norms_tail(R.fin);
                    if (threadIdx.x == 0) *R.fin_counter = 0u;
                }
            }
        }
    }
}

using MultiFn = void (*)(MultiArgs);

template <typename XT, int MODE, bool EMA>
MultiFn pick_norm_pub(const MergeVariant& v) {
    if (v.norm_level >= 1)
        return v.pub ? merge_multi<XT, MODE, EMA, true, true> : merge_multi<XT, MODE, EMA, true, false>;
    return v.pub ? merge_multi<XT, MODE, EMA, false, true> : merge_multi<XT, MODE, EMA, false, false>;
}

template <typename XT>
MultiFn pick_dtype(const MergeVariant& v) {
    if (v.mode == CAM_MODE_DELTA_NESTEROV)
        return v.ema ? pick_norm_pub<XT, CAM_MODE_DELTA_NESTEROV, true>(v)
                     : pick_norm_pub<XT, CAM_MODE_DELTA_NESTEROV, false>(v);
    return v.ema ? pick_norm_pub<XT, CAM_MODE_MEAN_REPLACE, true>(v)
                 : pick_norm_pub<XT, CAM_MODE_MEAN_REPLACE, false>(v);
}

MultiFn pick_multi(const MergeVariant& v) {
    return v.dtype == kDtBF16 ? pick_dtype<uint16_t>(v) : pick_dtype<float>(v);
}

}  // namespace

cudaError_t launch_merge_multi(const MultiArgs& a, const MergeVariant& v, int grid, size_t smem,
                               cudaStream_t s) {
    if (v.swa || v.norm_level > 1 || smem > kFinishSmemMax || a.n_rounds < 1 ||
        a.n_rounds > kMultiMax || a.status == nullptr)
        return cudaErrorInvalidValue;
    void* args[] = {const_cast<MultiArgs*>(&a)};
    return cudaLaunchKernel(reinterpret_cast<const void*>(pick_multi(v)), dim3(grid),
                            dim3(kThreads), args, smem, s);
}

int multi_blocks_per_sm(const MergeVariant& v) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
            &n, reinterpret_cast<const void*>(pick_multi(v)), kThreads, kFinishSmemMax) !=
        cudaSuccess)
        return 0;
    return n;
}

}  // namespace cam
