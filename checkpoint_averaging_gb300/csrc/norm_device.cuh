// norm_device.cuh -- the fixed-order sums that finish the drift norms: the
// separate norm pass (merge_kernels.cu, noalloc.cu) and the tail of a
// register-form merge pass that finishes them itself (merge_fused.cuh).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "cam_internal.h"
#include "merge_device.cuh"

namespace cam {
namespace dev {

// The fixed order every drift norm is summed in, per tensor t with chunks
// [c0, c1): lane l of a warp adds the partials c0 + l, c0 + l + 32, ... in
// that order (starting from +0.0), then the warp adds its lanes in an xor
// butterfly (offsets 16, 8, 4, 2, 1); lane 0 holds the result. The same
// order makes the fragment total from the tensors' squared norms.
//
// fp64 additions are slow on this GPU (a warp's add takes tens of cycles of
// the SM's fp64 pipe), so the code below skips every addition whose operand
// is the +0.0 a lane without a partial holds: a lane starts from its first
// partial (+0.0 + x is x), and the butterfly stops at the smallest power of
// two g >= min(n, 32) lanes, n = c1 - c0 (the lanes from g on hold +0.0, and
// no lane below g reads one of them in the steps with offsets below g, while
// the larger offsets add +0.0 to the lanes below g). Adding +0.0 to a sum of
// squares (never -0.0) leaves its bits unchanged, so the result is that of
// the full order, bit for bit, with no fp64 addition for a tensor of one
// chunk and ceil(log2 n) for one of n <= 32.

// Lanes of the butterfly a sum over n partials needs.
__device__ __forceinline__ int sum_lanes(int n) {
    return n >= 32 ? 32 : n <= 1 ? 1 : 1 << (32 - __clz(n - 1));
}

// The butterfly over the first g lanes (every lane of the warp calls it).
__device__ __forceinline__ double group_sum(double v, int g) {
    for (int o = g >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// Lane `lane`'s sum of v[c * stride] for c = c0 + lane, c0 + lane + 32, ...
// below c1, added in that order (+0.0 when it has none). Eight loads are in
// flight before their adds, so a long tensor costs a few memory latencies
// instead of one per chunk. COHERENT reads through L2 only (ld.global.cg): for
// partials written by other blocks of the same launch; otherwise the
// read-only path.
template <bool COHERENT = false>
__device__ __forceinline__ double lane_sum(const double* v, int64_t stride, int c0, int c1,
                                           int lane) {
    auto ld = [&](int c) { return COHERENT ? __ldcg(v + c * stride) : __ldg(v + c * stride); };
    double s = 0.0;
    for (int k = 0; k < c1 - c0; k += 32 * 8) {  // k: the batch's offset for lane 0
        double x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int c = c0 + k + 32 * j + lane;
            x[j] = c < c1 ? ld(c) : 0.0;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (k + 32 * j < c1 - c0) s = (k + j == 0) ? x[0] : s + x[j];  // (warp-uniform)
    }
    return s;
}

// The warp's total of v[c * stride] over [c0, c1) in the fixed order, valid
// in lane 0.
template <bool COHERENT = false>
__device__ __forceinline__ double chunk_sum(const double* v, int64_t stride, int c0, int c1,
                                            int lane) {
    return group_sum(lane_sum<COHERENT>(v, stride, c0, c1, lane), sum_lanes(c1 - c0));
}

// The squared norms of tensors t0 .. t0 + U - 1 (those below n_tensors), by
// one warp, in the fixed order; lane 0 stores each to out[t * ostride]. The U
// tensors' bounds, then their first kFirst partials per lane, are loaded
// together, and a long tensor's remaining partials kNext per lane at a time,
// so a fragment of many short tensors, or one long one, costs a few memory
// latencies per warp instead of two per tensor.
template <bool COHERENT, int U, int kFirst, int kNext>
__device__ __forceinline__ void tensor_sums(const double* v, int64_t stride, const int32_t* first,
                                            int t0, int n_tensors, int lane, double* out,
                                            int64_t ostride) {
    auto ld = [&](int c) { return COHERENT ? __ldcg(v + c * stride) : __ldg(v + c * stride); };
    int c0[U], c1[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const bool in = t0 + u < n_tensors;
        c0[u] = in ? first[t0 + u] : 0;
        c1[u] = in ? first[t0 + u + 1] : 0;
    }
    double s[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
        double x[kFirst];
#pragma unroll
        for (int j = 0; j < kFirst; ++j) {
            const int c = c0[u] + lane + 32 * j;
            x[j] = c < c1[u] ? ld(c) : 0.0;
        }
        s[u] = x[0];
#pragma unroll
        for (int j = 1; j < kFirst; ++j)
            if (c0[u] + 32 * j < c1[u]) s[u] += x[j];
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        for (int c = c0[u] + lane + 32 * kFirst, b = kFirst; c0[u] + 32 * b < c1[u];
             c += 32 * kNext, b += kNext) {
            double x[kNext];
#pragma unroll
            for (int j = 0; j < kNext; ++j) x[j] = c + 32 * j < c1[u] ? ld(c + 32 * j) : 0.0;
#pragma unroll
            for (int j = 0; j < kNext; ++j)
                if (c0[u] + 32 * (b + j) < c1[u]) s[u] += x[j];
        }
        const double w = group_sum(s[u], sum_lanes(c1[u] - c0[u]));
        if (lane == 0 && t0 + u < n_tensors) out[(t0 + u) * ostride] = w;
    }
}

// Finishes the norms from the per-chunk partials with one whole block (any
// multiple of 32 threads; every thread must call it): per tensor a warp's
// fixed-order sum (tensor_sums, four tensors per warp at a time); per
// (tensor, worker) the same; then warp 0 the fragment total and one warp per
// worker that worker's total, over the tensors in the same order. The sums do
// not depend on the block size, so every caller gets the same bits.
template <bool COHERENT>
__device__ __forceinline__ void finish_norms(const NormArgs& a) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int n_warps = blockDim.x >> 5;
    constexpr int U = 4, FIRST = 4, NEXT = 16;  // (larger batches raise the fused pass's registers)
    for (int t0 = warp * U; t0 < a.n_tensors; t0 += n_warps * U)
        tensor_sums<COHERENT, U, FIRST, NEXT>(a.partials, 1, a.first_chunk, t0, a.n_tensors, lane, a.tsq, 1);
    // per worker and tensor: one warp per (tensor, worker) pair
    for (int p = warp; p < a.n_tensors * a.K; p += n_warps) {
        const int t = p / a.K, k = p % a.K;
        const double s = chunk_sum<COHERENT>(a.worker_partials + k, CAM_KMAX, a.first_chunk[t],
                                             a.first_chunk[t + 1], lane);
        if (lane == 0) a.worker_tsq[static_cast<int64_t>(t) * CAM_KMAX + k] = s;
    }
    __syncthreads();
    if (warp == 0) {
        const double s = chunk_sum<COHERENT>(a.tsq, 1, 0, a.n_tensors, lane);
        if (lane == 0 && a.per_fragment) *a.per_fragment = sqrt(s);
    }
    for (int k = warp; k < a.K; k += n_warps) {  // one warp per worker's total
        const double s = chunk_sum<COHERENT>(a.worker_tsq + k, CAM_KMAX, 0, a.n_tensors, lane);
        if (lane == 0 && a.per_worker) a.per_worker[k] = sqrt(s);
    }
    if (a.per_tensor)
        for (int t = threadIdx.x; t < a.n_tensors; t += blockDim.x)
            a.per_tensor[t] = sqrt(a.tsq[t]);
    if (a.per_worker_tensor)
        for (int p = threadIdx.x; p < a.n_tensors * a.K; p += blockDim.x) {
            const int k = p / a.n_tensors, t = p % a.n_tensors;
            a.per_worker_tensor[p] = sqrt(a.worker_tsq[static_cast<int64_t>(t) * CAM_KMAX + k]);
        }
}

// finish_norms (K = 0) with the fragment's partials and chunk index first
// copied into shared memory sm (finish_smem_bytes of it), all the block's
// loads in flight at once: the same sums in the same order, so the same bits,
// with one memory latency before them instead of two per warp's batch of
// tensors and one more for the squared norms.
__device__ __forceinline__ void finish_norms_shared(const NormArgs& a, unsigned char* sm) {
    const int n = a.n_chunks, T = a.n_tensors;
    double* part = reinterpret_cast<double*>(sm);
    double* tsq = part + n;
    int32_t* first = reinterpret_cast<int32_t*>(tsq + T);
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int n_warps = blockDim.x >> 5;
    // the partials were written by other blocks of this launch: read through L2
    for (int i0 = threadIdx.x; i0 < n; i0 += 8 * blockDim.x) {
        double x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int i = i0 + j * blockDim.x;
            x[j] = i < n ? __ldcg(a.partials + i) : 0.0;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (i0 + j * blockDim.x < n) part[i0 + j * blockDim.x] = x[j];
    }
    for (int i = threadIdx.x; i <= T; i += blockDim.x) first[i] = a.first_chunk[i];
    __syncthreads();
    for (int t = warp; t < T; t += n_warps) {
        const int c0 = first[t], n_t = first[t + 1] - c0;
        double s = lane < n_t ? part[c0 + lane] : 0.0;
        for (int k = 32; k < n_t; k += 32)
            if (k + lane < n_t) s += part[c0 + k + lane];
        s = group_sum(s, sum_lanes(n_t));
        if (lane == 0) tsq[t] = s;
    }
    __syncthreads();
    if (warp == 0) {
        double s = lane < T ? tsq[lane] : 0.0;
        for (int k = 32; k < T; k += 32)
            if (k + lane < T) s += tsq[k + lane];
        s = group_sum(s, sum_lanes(T));
        if (lane == 0 && a.per_fragment) *a.per_fragment = sqrt(s);
    }
    if (a.per_tensor)
        for (int t = threadIdx.x; t < T; t += blockDim.x) a.per_tensor[t] = sqrt(tsq[t]);
}

// finish_norms over partials written by other blocks of the calling launch,
// out of line: inlined into the merge pass's tail it would crowd the
// registers of that pass's main loop. With shared set (K = 0), through the
// launch's dynamic shared memory.
static __device__ __noinline__ void finish_norms_tail(const NormArgs& a) {
    extern __shared__ __align__(16) unsigned char fin_smem[];
    if (a.shared && a.K == 0)
        finish_norms_shared(a, fin_smem);
    else
        finish_norms<true>(a);
}

}  // namespace dev
}  // namespace cam
