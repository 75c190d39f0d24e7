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
// (and per worker, when asked) in a fixed order, so norms are bitwise
// reproducible. The fused pass itself is in merge_fused.cuh.
#include <cuda_runtime.h>

#include "cam_internal.h"
#include "merge_device.cuh"
#include "norm_device.cuh"

namespace cam {
namespace {

using namespace cam::dev;

__global__ void __launch_bounds__(256, 1) norm_finish(const NormArgs a) {
    finish_norms<false>(a);
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

MergeFn pick(const MergeVariant& v) {
    return v.dtype == kDtBF16 ? pick_merge_bf16(v) : pick_merge_f32(v);
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, const MergeVariant& v, int grid, cudaStream_t s) {
    MergeFn fn = pick(v);
    void* args[] = {const_cast<MergeArgs*>(&a)};
    // a fused finish that stages its partials in shared memory gets it here
    const size_t smem = v.fin && a.fin.shared ? finish_smem_bytes(a.fin.n_tensors, a.fin.n_chunks) : 0;
    if (smem > kFinishSmemMax) return cudaErrorInvalidValue;
    return cudaLaunchKernel(reinterpret_cast<const void*>(fn), dim3(grid), dim3(kThreads),
                            args, smem, s);
}

int staged_state_arrays(const MergeVariant& v) {
    const bool delta = v.mode == CAM_MODE_DELTA_NESTEROV;
    return int(delta || v.norm_level >= 1) + int(delta) + int(v.ema) + int(v.swa);
}

int64_t staged_stage_bytes(const MergeVariant& v, int K) {
    const int64_t xb = v.dtype == kDtBF16 ? 2 : 4;
    return int64_t(kStTile) * (K * xb + 4 * staged_state_arrays(v));
}

int64_t staged_red_bytes(const MergeVariant& v, int K) {
    if (v.norm_level < 1) return 0;
    const int quantities = 1 + (v.norm_level >= 2 ? K : 0);
    return int64_t(kStRedSlots) * quantities * kStConsumers * 4;
}

namespace {

MergeFn pick_staged(const MergeVariant& v) {
    return v.dtype == kDtBF16 ? pick_staged_bf16(v) : pick_staged_f32(v);
}

}  // namespace

cudaError_t staged_prepare() {
    for (int dt = 0; dt < 2; ++dt)
        for (int md = 0; md < 2; ++md)
            for (int em = 0; em < 2; ++em)
                for (int nl = 0; nl < 3; ++nl)
                    for (int pb = 0; pb < 2; ++pb)
                        for (int sw = 0; sw < 2; ++sw) {
                            const MergeVariant v{dt, md, em != 0, nl, pb != 0, sw != 0};
                            const cudaError_t ce = cudaFuncSetAttribute(
                                reinterpret_cast<const void*>(pick_staged(v)),
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kStSmemBytes);
                            if (ce != cudaSuccess) return ce;
                        }
    return cudaSuccess;
}

cudaError_t launch_merge_staged(const MergeArgs& a, const MergeVariant& v, int grid,
                                cudaStream_t s) {
    const size_t smem = size_t(a.st_stages) * size_t(a.st_stage_bytes) +
                        size_t(staged_red_bytes(v, a.K));
    if (a.st_stages < 2 || a.st_stages > kStMaxStages || smem > size_t(kStSmemBytes) ||
        a.st_stage_bytes != staged_stage_bytes(v, a.K) || a.status == nullptr)
        return cudaErrorInvalidValue;
    void* args[] = {const_cast<MergeArgs*>(&a)};
    return cudaLaunchKernel(reinterpret_cast<const void*>(pick_staged(v)), dim3(grid),
                            dim3(kStThreads), args, smem, s);
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
    norm_finish<<<1, 256, 0, s>>>(a);
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
