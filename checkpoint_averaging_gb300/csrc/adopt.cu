// adopt.cu -- cam_adopt_keep_drift: a worker adopting the new global while
// keeping the progress it made since its last push (declaration in
// include/cam.h).
//
// "DiffuRefill-1B: Pretraining a Masked Diffusion Language Model on Free,
// Preemptible Notebook GPUs", section 5.1: adopting the global as
// theta <- theta + (g - theta_pushed) keeps each worker's progress since its
// last push; the run measured it worse than plain replacement and used
// replacement. Per element: d = g - theta_pushed, theta' = theta + d, each a
// binary32 operation rounded to nearest-even. Streaming, HBM-bound (16 B per
// element with fp32 pushed copies, 14 B with bf16), no scratch and no
// allocation: the chunk map travels in the kernel parameter block.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>

#include "cam_internal.h"
#include "merge_device.cuh"

#define CAM_API extern "C" __attribute__((visibility("default")))

namespace cam {
namespace {

using namespace cam::dev;

constexpr int kAdTensors = 512;  // tensors per launch

struct AdoptArgs {
    int32_t n_chunks;
    int32_t n_local;
    int32_t chunk_elems;
    uint32_t vec[kAdTensors / 32];
    int32_t first_chunk[kAdTensors + 1];  // launch-relative; [n_local] == n_chunks
    float* theta[kAdTensors];
    const float* global[kAdTensors];
    const void* pushed[kAdTensors];
    int64_t numel[kAdTensors];
};
static_assert(sizeof(AdoptArgs) <= 32000, "kernel parameter block too large");

template <typename XT>
__global__ void __launch_bounds__(kThreads) adopt_keep_drift(const __grid_constant__ AdoptArgs a) {
    for (int c = blockIdx.x; c < a.n_chunks; c += gridDim.x) {
        int lo = 0, hi = a.n_local - 1;  // the last tensor whose first chunk is <= c
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (a.first_chunk[mid] <= c) lo = mid;
            else hi = mid - 1;
        }
        const int l = lo;
        const int64_t start = int64_t(c - a.first_chunk[l]) * a.chunk_elems;
        const int len = static_cast<int>(min(int64_t(a.chunk_elems), a.numel[l] - start));
        float* th = a.theta[l] + start;
        const float* g = a.global[l] + start;
        const XT* p = static_cast<const XT*>(a.pushed[l]) + start;
        int done = 0;
        if ((a.vec[l >> 5] >> (l & 31)) & 1u) {
            const int nv = len >> 3;
            for (int v = threadIdx.x; v < nv; v += kThreads) {
                XVec<float> gv;
                XVec<XT> pv;
                float t[8];
                gv.load(g + 8 * v);
                pv.load(p + 8 * v);
                load_s8(th + 8 * v, t);
#pragma unroll
                for (int j = 0; j < 8; ++j) t[j] = __fadd_rn(t[j], __fsub_rn(gv.get(j), pv.get(j)));
                store_s8(th + 8 * v, t);
            }
            done = 8 * nv;
        }
        for (int j = done + threadIdx.x; j < len; j += kThreads)
            th[j] = __fadd_rn(th[j], __fsub_rn(g[j], load_x1(p + j)));
    }
}

bool aligned(const void* q, uintptr_t n) { return (reinterpret_cast<uintptr_t>(q) % n) == 0; }

}  // namespace
}  // namespace cam

using cam::record_error;

CAM_API int cam_adopt_keep_drift(int32_t n_tensors, const int64_t* numel, float* const* theta_w,
                                 const float* const* global, const void* const* pushed,
                                 cam_dtype pushed_dtype, void* stream) {
    const char* fn = "cam_adopt_keep_drift";
    if (n_tensors < 0) return record_error(CAM_E_ARG, "%s: n_tensors < 0", fn);
    if (pushed_dtype != CAM_F32 && pushed_dtype != CAM_BF16)
        return record_error(CAM_E_ARG, "%s: unknown dtype %d", fn, static_cast<int>(pushed_dtype));
    if (n_tensors > 0 && (!numel || !theta_w || !global || !pushed))
        return record_error(CAM_E_ARG, "%s: numel, theta_w, global and pushed are required", fn);
    int64_t n_elems = 0;
    for (int32_t t = 0; t < n_tensors; ++t) {
        if (numel[t] < 0 || numel[t] > (int64_t(1) << 40))
            return record_error(CAM_E_ARG, "%s: numel[%d] out of range", fn, t);
        if (numel[t] > 0 && (!theta_w[t] || !global[t] || !pushed[t]))
            return record_error(CAM_E_ARG, "%s: a pointer of tensor %d is NULL", fn, t);
        n_elems += numel[t];
    }
    int dev = 0, sms = 0;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce == cudaSuccess) ce = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (ce != cudaSuccess)
        return record_error(CAM_E_CUDA, "%s: no usable CUDA device: %s", fn, cudaGetErrorString(ce));
    // chunking: >= 8 chunks per SM, whole block-steps, at most kMaxChunkElems
    const int64_t q = cam::kChunkQuantum;
    int64_t chunk = (n_elems + int64_t(sms) * 8 - 1) / (int64_t(sms) * 8);
    chunk = std::min<int64_t>(std::max<int64_t>((chunk + q - 1) / q * q, q), cam::kMaxChunkElems);
    const uintptr_t pa = pushed_dtype == CAM_F32 ? 32 : 16;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cam::AdoptArgs a;
    a.chunk_elems = static_cast<int32_t>(chunk);
    for (int32_t t0 = 0; t0 < n_tensors; t0 += cam::kAdTensors) {
        const int n = std::min(cam::kAdTensors, n_tensors - t0);
        std::fill(a.vec, a.vec + cam::kAdTensors / 32, 0u);
        int64_t nc = 0;
        a.first_chunk[0] = 0;
        for (int l = 0; l < n; ++l) {
            const int32_t t = t0 + l;
            a.theta[l] = theta_w[t];
            a.global[l] = global[t];
            a.pushed[l] = pushed[t];
            a.numel[l] = numel[t];
            nc += (numel[t] + chunk - 1) / chunk;
            if (nc > INT32_MAX) return record_error(CAM_E_ARG, "%s: too many elements in one call", fn);
            a.first_chunk[l + 1] = static_cast<int32_t>(nc);
            if (cam::aligned(theta_w[t], 32) && cam::aligned(global[t], 32) &&
                cam::aligned(pushed[t], pa))
                a.vec[l >> 5] |= 1u << (l & 31);
        }
        if (nc == 0) continue;
        a.n_chunks = static_cast<int32_t>(nc);
        a.n_local = n;
        const int grid = static_cast<int>(std::min<int64_t>(nc, int64_t(sms) * 4));
        void* args[] = {&a};
        const void* kern = pushed_dtype == CAM_BF16
                               ? reinterpret_cast<const void*>(cam::adopt_keep_drift<uint16_t>)
                               : reinterpret_cast<const void*>(cam::adopt_keep_drift<float>);
        ce = cudaLaunchKernel(kern, dim3(grid), dim3(cam::kThreads), args, 0, s);
        if (ce != cudaSuccess)
            return record_error(CAM_E_CUDA, "%s: launch: %s", fn, cudaGetErrorString(ce));
    }
    return CAM_OK;
}
