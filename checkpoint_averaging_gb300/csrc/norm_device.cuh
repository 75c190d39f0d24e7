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

// Lane `lane`'s sum of v[c * stride] for c = c0 + lane, c0 + lane + 32, ...
// below c1, added in that order. Eight loads are in flight before their
// adds, so a long tensor costs a few memory latencies instead of one per
// chunk; slots past the end add +0.0, which leaves the (non-negative) sum's
// bits unchanged. COHERENT reads through L2 only (ld.global.cg): for partials
// written by other blocks of the same launch; otherwise the read-only path.
template <bool COHERENT = false>
__device__ __forceinline__ double lane_sum(const double* v, int64_t stride, int c0, int c1,
                                           int lane) {
    double s = 0.0;
    for (int c = c0 + lane; c < c1; c += 32 * 8) {
        double x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const double* q = v + (c + 32 * j) * stride;
            x[j] = c + 32 * j < c1 ? (COHERENT ? __ldcg(q) : __ldg(q)) : 0.0;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) s += x[j];
    }
    return s;
}

// The squared norms of tensors t0 .. t0 + U - 1 (those below n_tensors), by
// one warp: per tensor the same fixed-order sum as lane_sum (lane l adds the
// partials c = first[t] + l, + 32, ... below first[t + 1], in that order)
// followed by warp_sum; lane 0 stores it to out[t * ostride]. The U tensors'
// bounds, then their first kFirst partials per lane, are loaded together, and
// a long tensor's remaining partials kNext per lane at a time (adding the +0.0
// that fills a batch past the end leaves a non-negative sum's bits as they
// are), so a fragment of many short tensors, or one long one, costs a few
// memory latencies per warp instead of two per tensor.
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
        s[u] = 0.0;
#pragma unroll
        for (int j = 0; j < kFirst; ++j) s[u] += x[j];
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
        for (int c = c0[u] + lane + 32 * kFirst; c < c1[u]; c += 32 * kNext) {
            double x[kNext];
#pragma unroll
            for (int j = 0; j < kNext; ++j) x[j] = c + 32 * j < c1[u] ? ld(c + 32 * j) : 0.0;
#pragma unroll
            for (int j = 0; j < kNext; ++j) s[u] += x[j];
        }
        const double w = warp_sum(s[u]);
        if (lane == 0 && t0 + u < n_tensors) out[(t0 + u) * ostride] = w;
    }
}

// Finishes the norms from the per-chunk partials with one whole block (any
// multiple of 32 threads; every thread must call it): per tensor, a warp's
// fixed-order lane sums and xor butterfly (tensor_sums, four tensors per warp
// at a time); per (tensor, worker) the same; then warp 0 the fragment total
// and one warp per worker that worker's total, each over the tensors in the
// same lane-strided order. The sums do not depend on the block size, so every
// caller gets the same bits.
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
        double s = lane_sum<COHERENT>(a.worker_partials + k, CAM_KMAX, a.first_chunk[t],
                                      a.first_chunk[t + 1], lane);
        s = warp_sum(s);
        if (lane == 0) a.worker_tsq[static_cast<int64_t>(t) * CAM_KMAX + k] = s;
    }
    __syncthreads();
    if (warp == 0) {
        double s = 0.0;
        for (int t = lane; t < a.n_tensors; t += 32) s += a.tsq[t];
        s = warp_sum(s);
        if (lane == 0 && a.per_fragment) *a.per_fragment = sqrt(s);
    }
    for (int k = warp; k < a.K; k += n_warps) {  // one warp per worker's total
        double s = 0.0;
        for (int t = lane; t < a.n_tensors; t += 32)
            s += a.worker_tsq[static_cast<int64_t>(t) * CAM_KMAX + k];
        s = warp_sum(s);
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

// finish_norms over partials written by other blocks of the calling launch,
// out of line: inlined into the merge pass's tail it would crowd the
// registers of that pass's main loop.
static __device__ __noinline__ void finish_norms_tail(const NormArgs& a) {
    finish_norms<true>(a);
}

}  // namespace dev
}  // namespace cam
