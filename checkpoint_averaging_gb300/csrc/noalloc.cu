// noalloc.cu -- cam_merge_round_noalloc: one merge round in a single call that
// allocates no memory (declaration and contract in include/cam.h).
//
// Callers that may not allocate device memory use this call. Examples are code
// running inside a framework whose pool has already reserved the GPU's memory,
// and paths where the device-wide synchronisation of cudaMalloc/cudaFree is not
// acceptable. It runs the same per-element arithmetic as the context path
// (merge_device.cuh), with two differences:
//   - the chunk -> tensor map travels in the kernel's parameter block instead of
//     a device table;
//   - the drift partials go to one fixed array in the library's device memory,
//     whose address is looked up once per device.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "cam_internal.h"
#include "merge_device.cuh"
#include "norm_device.cuh"

#define CAM_API extern "C" __attribute__((visibility("default")))

namespace {

constexpr int kScratchDoubles = CAM_NOALLOC_MAX_CHUNKS + CAM_NOALLOC_MAX_TENSORS;

}  // namespace

// Drift partials of every chunk of a call, then the squared norm of every
// tensor. Shared by all calls on a device; see include/cam.h.
static __device__ __align__(256) double g_noalloc_scratch[kScratchDoubles];

namespace cam {
namespace {

using namespace cam::dev;

constexpr int kNaTensors = 256;  // tensors per launch of the no-allocation pass
constexpr int kMaxDevices = 64;

// Parameter block of one launch: tensors [first, first + n_local) of the call.
// The scalar names match what merge_elem reads.
struct NoAllocArgs {
    int32_t K;
    float Kf;
    float w[CAM_KMAX];
    float W;
    float lr, mu, beta;
    DivPlan div;       // the division: by Kf (plain mean) or W (delta)
    double* partials;  // scratch entry of this launch's first chunk
    int32_t n_chunks;
    int32_t n_local;
    int32_t chunk_elems;
    uint32_t vec[kNaTensors / 32];
    int32_t first_chunk[kNaTensors + 1];  // launch-relative; [n_local] == n_chunks
    TensorSlot slots[kNaTensors];
    const void* x[kNaTensors * CAM_KMAX];  // x[l*K + k]
};
static_assert(sizeof(NoAllocArgs) <= 32000, "kernel parameter block too large");

struct NoAllocNormArgs {
    const double* partials;
    double* tsq;
    double* per_tensor;
    double* per_round;
    int32_t n_tensors;
    int32_t first_chunk[CAM_NOALLOC_MAX_TENSORS + 1];
};
static_assert(sizeof(NoAllocNormArgs) <= 32000, "kernel parameter block too large");

template <typename XT, int MODE, bool EMA, bool NORM>
__global__ void __launch_bounds__(kThreads, 2)
    merge_fused_noalloc(const __grid_constant__ NoAllocArgs a) {
    __shared__ double warp_part[kThreads / 32];
    for (int c = blockIdx.x; c < a.n_chunks; c += gridDim.x) {
        // the chunk's tensor: the last l with first_chunk[l] <= c (tensors with
        // no elements share their start with the next tensor and are skipped)
        int lo = 0, hi = a.n_local - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.first_chunk[mid] <= c) lo = mid;
            else hi = mid - 1;
        }
        const int l = lo;
        const TensorSlot ts = a.slots[l];
        const int64_t start = int64_t(c - a.first_chunk[l]) * a.chunk_elems;
        const int len = static_cast<int>(min(int64_t(a.chunk_elems), ts.numel - start));
        const void* const* xs = a.x + static_cast<int64_t>(l) * a.K;
        const bool vec = (a.vec[l >> 5] >> (l & 31)) & 1u;
        float acc = 0.0f;
        if (vec) {
            const int nv = len >> 3;
            for (int v = threadIdx.x; v < nv; v += kThreads)
                merge_vec8<XT, MODE, EMA, NORM>(a, xs, ts, start + 8 * int64_t(v), acc);
            const int tail = len & 7;
            if (static_cast<int>(threadIdx.x) < tail)
                merge_one<XT, MODE, EMA, NORM>(a, xs, ts, start + 8 * int64_t(nv) + threadIdx.x,
                                               acc);
        } else {
            for (int j = threadIdx.x; j < len; j += kThreads)
                merge_one<XT, MODE, EMA, NORM>(a, xs, ts, start + j, acc);
        }
        if (NORM) {
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

__global__ void __launch_bounds__(1024) norm_finish_noalloc(const __grid_constant__ NoAllocNormArgs a) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int n_warps = blockDim.x >> 5;
    for (int t = warp; t < a.n_tensors; t += n_warps) {
        double s = lane_sum(a.partials, 1, a.first_chunk[t], a.first_chunk[t + 1], lane);
        s = warp_sum(s);
        if (lane == 0) a.tsq[t] = s;
    }
    __syncthreads();
    if (warp == 0) {
        double s = 0.0;
        for (int t = lane; t < a.n_tensors; t += 32) s += a.tsq[t];
        s = warp_sum(s);
        if (lane == 0 && a.per_round) *a.per_round = sqrt(s);
    }
    if (a.per_tensor)
        for (int t = threadIdx.x; t < a.n_tensors; t += blockDim.x) a.per_tensor[t] = sqrt(a.tsq[t]);
}

using NaFn = void (*)(NoAllocArgs);

template <typename XT, int MODE>
NaFn pick3(bool ema, bool norm) {
    if (ema)
        return norm ? merge_fused_noalloc<XT, MODE, true, true>
                    : merge_fused_noalloc<XT, MODE, true, false>;
    return norm ? merge_fused_noalloc<XT, MODE, false, true>
                : merge_fused_noalloc<XT, MODE, false, false>;
}

NaFn pick(int dtype, int mode, bool ema, bool norm) {
    if (dtype == kDtBF16)
        return mode == kDelta ? pick3<uint16_t, kDelta>(ema, norm) : pick3<uint16_t, kMean>(ema, norm);
    return mode == kDelta ? pick3<float, kDelta>(ema, norm) : pick3<float, kMean>(ema, norm);
}

// Per-device set-up, done by the first call on each device.
struct DeviceSetup {
    bool ready = false;
    double* scratch = nullptr;
    int sm_count = 0;
    int bps[2][2][2][2] = {};
};
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mutex;

int setup_device(int dev, const DeviceSetup** out) {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    DeviceSetup& s = g_setup[dev];
    if (!s.ready) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess)
            return record_error(CAM_E_CUDA, "cam_merge_round_noalloc: scratch address on device %d: %s",
                                dev, cudaGetErrorString(e));
        e = cudaDeviceGetAttribute(&s.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return record_error(CAM_E_CUDA, "cam_merge_round_noalloc: SM count: %s", cudaGetErrorString(e));
        for (int dt = 0; dt < 2; ++dt)
            for (int md = 0; md < 2; ++md)
                for (int em = 0; em < 2; ++em)
                    for (int nm = 0; nm < 2; ++nm) {
                        int n = 0;
                        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                            &n, reinterpret_cast<const void*>(pick(dt, md, em, nm)), kThreads, 0);
                        if (e != cudaSuccess)
                            return record_error(CAM_E_CUDA, "cam_merge_round_noalloc: occupancy: %s",
                                                cudaGetErrorString(e));
                        s.bps[dt][md][em][nm] = std::max(1, n);
                    }
        s.scratch = static_cast<double*>(p);
        s.ready = true;
    }
    *out = &s;
    return CAM_OK;
}

// Elements per chunk: the context path's policy (>= 8 chunks per SM, whole
// block-steps, at most kMaxChunkElems).
int32_t chunk_elems_for(int64_t n, int sm_count) {
    const int64_t q = kChunkQuantum;
    const int64_t target = std::max<int64_t>(1, int64_t(sm_count) * 8);
    int64_t c = (n + target - 1) / target;
    c = ((c + q - 1) / q) * q;
    return static_cast<int32_t>(std::min<int64_t>(std::max<int64_t>(c, q), kMaxChunkElems));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace cam

using cam::record_error;

CAM_API int cam_merge_round_noalloc(int32_t n_tensors, const int64_t* numel, float* const* master,
                                    float* const* momentum, float* const* ema, int32_t n_workers,
                                    const void* const* ckpt, cam_dtype dtype, const int64_t* tokens,
                                    cam_mode mode, float lr, float mu, int32_t ema_update,
                                    float beta, double* per_tensor, double* per_round,
                                    void* stream) {
    const char* fn = "cam_merge_round_noalloc";
    if (n_tensors < 0 || n_tensors > CAM_NOALLOC_MAX_TENSORS)
        return record_error(CAM_E_ARG, "%s: n_tensors %d outside [0, %d]", fn, n_tensors,
                            CAM_NOALLOC_MAX_TENSORS);
    if (n_workers < 1 || n_workers > CAM_KMAX)
        return record_error(CAM_E_ARG, "%s: n_workers %d outside [1, %d]", fn, n_workers, CAM_KMAX);
    if (dtype != CAM_F32 && dtype != CAM_BF16)
        return record_error(CAM_E_ARG, "%s: unknown dtype %d", fn, static_cast<int>(dtype));
    if (mode != CAM_MODE_MEAN_REPLACE && mode != CAM_MODE_DELTA_NESTEROV)
        return record_error(CAM_E_ARG, "%s: unknown mode %d", fn, static_cast<int>(mode));
    const bool delta = mode == CAM_MODE_DELTA_NESTEROV;
    const bool do_ema = ema_update != 0;
    const bool norms = per_tensor != nullptr || per_round != nullptr;
    if (!std::isfinite(lr) || !std::isfinite(mu) || !std::isfinite(beta))
        return record_error(CAM_E_ARG, "%s: lr, mu and beta must be finite", fn);
    if (n_tensors > 0 && (!numel || !master || !ckpt))
        return record_error(CAM_E_ARG, "%s: numel, master and ckpt are required", fn);
    if (delta && n_tensors > 0 && !momentum)
        return record_error(CAM_E_ARG, "%s: Nesterov needs momentum buffers", fn);
    if (do_ema && n_tensors > 0 && !ema)
        return record_error(CAM_E_ARG, "%s: ema_update needs EMA buffers", fn);
    int64_t W = 0;
    if (delta) {
        if (!tokens) return record_error(CAM_E_ARG, "%s: tokens are required", fn);
        for (int k = 0; k < n_workers; ++k) {
            if (tokens[k] < 0 || tokens[k] > (int64_t(1) << 56))
                return record_error(CAM_E_ARG, "%s: tokens[%d] out of range", fn, k);
            W += tokens[k];
        }
        if (W <= 0) return record_error(CAM_E_ARG, "%s: total token count must be > 0", fn);
    }
    int64_t n_elems = 0, min_chunks = 0;
    for (int32_t t = 0; t < n_tensors; ++t) {
        if (numel[t] < 0 || numel[t] > (int64_t(1) << 40))
            return record_error(CAM_E_ARG, "%s: numel[%d] out of range", fn, t);
        if (numel[t] == 0) continue;
        if (!master[t] || (delta && !momentum[t]) || (do_ema && !ema[t]))
            return record_error(CAM_E_ARG, "%s: state pointer of tensor %d is NULL", fn, t);
        for (int k = 0; k < n_workers; ++k)
            if (!ckpt[size_t(k) * n_tensors + t])
                return record_error(CAM_E_ARG, "%s: ckpt[%d][%d] is NULL", fn, k, t);
        n_elems += numel[t];
        min_chunks += (numel[t] + cam::kMaxChunkElems - 1) / cam::kMaxChunkElems;
    }
    // Chunks are at most kMaxChunkElems long, so this many at least: a round
    // beyond the scratch is refused here, before any CUDA call.
    if (min_chunks > CAM_NOALLOC_MAX_CHUNKS)
        return record_error(CAM_E_ARG,
                            "%s: round too large for the fixed scratch: more than %d chunks of "
                            "%d elements",
                            fn, CAM_NOALLOC_MAX_CHUNKS, cam::kMaxChunkElems);

    int dev = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess)
        return record_error(CAM_E_CUDA, "%s: no usable CUDA device: %s", fn, cudaGetErrorString(ce));
    if (dev < 0 || dev >= cam::kMaxDevices)
        return record_error(CAM_E_CUDA, "%s: device %d beyond the supported %d", fn, dev, cam::kMaxDevices);
    const cam::DeviceSetup* setup = nullptr;
    int rc = cam::setup_device(dev, &setup);
    if (rc != CAM_OK) return rc;

    const int32_t chunk = cam::chunk_elems_for(n_elems, setup->sm_count);
    cam::NoAllocNormArgs na;
    na.first_chunk[0] = 0;
    int64_t n_chunks = 0;
    for (int32_t t = 0; t < n_tensors; ++t) {
        n_chunks += (numel[t] + chunk - 1) / chunk;
        if (n_chunks > CAM_NOALLOC_MAX_CHUNKS)
            return record_error(CAM_E_ARG,
                                "%s: round too large for the fixed scratch: more than %d chunks of "
                                "%d elements",
                                fn, CAM_NOALLOC_MAX_CHUNKS, chunk);
        na.first_chunk[t + 1] = static_cast<int32_t>(n_chunks);
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uintptr_t xa = dtype == CAM_F32 ? 32 : 16;
    cam::NoAllocArgs a;
    a.K = n_workers;
    a.Kf = static_cast<float>(n_workers);
    for (int k = 0; k < CAM_KMAX; ++k)
        a.w[k] = (delta && k < n_workers) ? static_cast<float>(tokens[k]) : 0.0f;
    a.W = static_cast<float>(W);
    a.div = cam::div_plan(delta ? a.W : a.Kf);
    a.lr = lr;
    a.mu = mu;
    a.beta = beta;
    a.chunk_elems = chunk;
    const int bps = setup->bps[dtype][mode][do_ema][norms];
    for (int32_t t0 = 0; t0 < n_tensors; t0 += cam::kNaTensors) {
        const int n = std::min(cam::kNaTensors, n_tensors - t0);
        const int32_t c0 = na.first_chunk[t0];
        a.n_local = n;
        a.n_chunks = na.first_chunk[t0 + n] - c0;
        if (a.n_chunks == 0) continue;
        a.partials = setup->scratch + c0;
        std::fill(a.vec, a.vec + cam::kNaTensors / 32, 0u);
        for (int l = 0; l <= n; ++l) a.first_chunk[l] = na.first_chunk[t0 + l] - c0;
        for (int l = 0; l < n; ++l) {
            const int32_t t = t0 + l;
            float* th = master[t];
            float* m = delta ? momentum[t] : nullptr;
            float* e = do_ema ? ema[t] : nullptr;
            a.slots[l] = cam::TensorSlot{th, m, e, nullptr, numel[t]};
            bool v = cam::aligned(th, 32) && (!delta || cam::aligned(m, 32)) &&
                     (!do_ema || cam::aligned(e, 32));
            for (int k = 0; k < n_workers; ++k) {
                const void* xp = ckpt[size_t(k) * n_tensors + t];
                a.x[size_t(l) * n_workers + k] = xp;
                v = v && cam::aligned(xp, xa);
            }
            if (v) a.vec[l >> 5] |= 1u << (l & 31);
        }
        const int grid = static_cast<int>(std::min<int64_t>(a.n_chunks, int64_t(setup->sm_count) * bps));
        void* args[] = {&a};
        ce = cudaLaunchKernel(reinterpret_cast<const void*>(cam::pick(dtype, mode, do_ema, norms)),
                              dim3(grid), dim3(cam::kThreads), args, 0, s);
        if (ce != cudaSuccess)
            return record_error(CAM_E_CUDA, "%s: launch: %s", fn, cudaGetErrorString(ce));
    }
    if (norms) {
        na.partials = setup->scratch;
        na.tsq = setup->scratch + CAM_NOALLOC_MAX_CHUNKS;
        na.per_tensor = per_tensor;
        na.per_round = per_round;
        na.n_tensors = n_tensors;
        void* args[] = {&na};
        ce = cudaLaunchKernel(reinterpret_cast<const void*>(cam::norm_finish_noalloc), dim3(1),
                              dim3(1024), args, 0, s);
        if (ce != cudaSuccess)
            return record_error(CAM_E_CUDA, "%s: norm launch: %s", fn, cudaGetErrorString(ce));
    }
    return CAM_OK;
}
