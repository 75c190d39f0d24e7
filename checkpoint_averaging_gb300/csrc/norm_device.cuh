// norm_device.cuh -- the fixed-order partial sums of the norm finishing
// kernels (merge_kernels.cu, noalloc.cu).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace cam {
namespace dev {

// Lane `lane`'s sum of v[c * stride] for c = c0 + lane, c0 + lane + 32, ...
// below c1, added in that order. Eight loads are in flight before their
// adds, so a long tensor costs a few memory latencies instead of one per
// chunk; slots past the end add +0.0, which leaves the (non-negative) sum's
// bits unchanged.
__device__ __forceinline__ double lane_sum(const double* v, int64_t stride, int c0, int c1,
                                           int lane) {
    double s = 0.0;
    for (int c = c0 + lane; c < c1; c += 32 * 8) {
        double x[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = c + 32 * j < c1 ? __ldg(v + (c + 32 * j) * stride) : 0.0;
#pragma unroll
        for (int j = 0; j < 8; ++j) s += x[j];
    }
    return s;
}

}  // namespace dev
}  // namespace cam
