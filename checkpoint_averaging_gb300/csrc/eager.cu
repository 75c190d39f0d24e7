// eager.cu -- rounds whose checkpoints are folded as they arrive
// (cam_merge_fold, declared in include/cam.h).
//
// "DiffuRefill-1B" model card, "How it is trained", Merging: the merger keeps
// a running fp32 sum and adds each downloaded checkpoint to it on arrival, so
// only the last arrival's fold remains once the quorum is in. Here:
//
//   fold_worker   s <- s + x_k (plain mean) or s + w_k (x_k - theta)
//                 (token-weighted delta mean), s starting at +0 with the
//                 first arrival; optionally worker k's squared drift
//                 (x_k - theta)^2 per chunk. Reads the worker (device or
//                 host memory) and s, writes s: the worker is no longer needed
//                 once this launch has run.
//   final_pass    at commit: folds the workers accumulated after the folds
//                 (typically the last arrival, read once, here), then from s:
//                 finalize, outer step, EMA, running average, drift partials
//                 and published copies, through the same merge_finish as the
//                 fused pass. Folding the last arrival here overlaps its
//                 host-to-device stream with the published copies'
//                 device-to-host stream.
//
// Per element the operations are those of the fused pass in the same order,
// so an eagerly folded round ends with the same bits as a round whose
// workers are all read at commit. Both kernels are HBM-bound streaming passes
// in the register form: persistent grid, 8 elements per thread per step,
// 256-bit loads and stores where aligned.
#include <cuda_runtime.h>

#include "cam_internal.h"
#include "side_internal.h"
#include "merge_device.cuh"

namespace cam {
namespace {

using namespace cam::dev;

template <typename XT, int MODE, bool WD>
__global__ void __launch_bounds__(kThreads, 2) fold_worker(const __grid_constant__ FoldArgs a) {
    constexpr int kWarps = kThreads / 32;
    __shared__ double part[2][kWarps];
    int parity = 0;
    for (int c = blockIdx.x; c < a.n_chunks; c += gridDim.x, parity ^= 1) {
        const ChunkDesc ch = a.chunks[c];
        const bool in_launch = chunk_in_launch(ch, a.local0, a.n_local);
        const TensorSlot ts = a.slots[in_launch ? ch.local : a.local0];
        if (!in_launch || !chunk_in_tensor(ch, ts)) {  // skipped, its partial 0
            if (threadIdx.x == 0) {
                atomicOr(a.status, kStatusBadChunk);
                if (WD) a.worker_partials[static_cast<int64_t>(c) * CAM_KMAX + a.k] = 0.0;
            }
            parity ^= 1;  // the slots stay as they were: no barrier for this chunk
            continue;
        }
        const int l = ch.local - a.local0;
        const XT* x = static_cast<const XT*>(a.x[l]) + ch.start;
        float* s = a.sum[l] + ch.start;
        const float* th = ts.theta + ch.start;
        float accw = 0.0f;
        int done = 0;
        if ((a.vec[l >> 5] >> (l & 31)) & 1u) {
            const int nv = ch.len >> 3;
            for (int v = threadIdx.x; v < nv; v += kThreads) {
                XVec<XT> xv;
                xv.load(x + 8 * v);
                float sv[8], t[8];
                if (a.first) {
#pragma unroll
                    for (int j = 0; j < 8; ++j) sv[j] = 0.0f;
                } else {
                    load_s8(s + 8 * v, sv);
                }
                if (MODE == kDelta || WD) load_s8(th + 8 * v, t);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float xj = xv.get(j);
                    if constexpr (WD) {
                        const float d = __fsub_rn(xj, t[j]);
                        accw = __fmaf_rn(d, d, accw);
                    }
                    sv[j] = fold_term<MODE>(sv[j], xj, a.w, (MODE == kDelta) ? t[j] : 0.0f);
                }
                store_s8(s + 8 * v, sv);
            }
            done = 8 * nv;
        }
        for (int j = done + threadIdx.x; j < ch.len; j += kThreads) {
            const float xj = load_x1(x + j);
            const float t = (MODE == kDelta || WD) ? th[j] : 0.0f;
            if constexpr (WD) {
                const float d = __fsub_rn(xj, t);
                accw = __fmaf_rn(d, d, accw);
            }
            s[j] = fold_term<MODE>(a.first ? 0.0f : s[j], xj, a.w, t);
        }
        if constexpr (WD) {
            const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
            const double d = warp_sum(static_cast<double>(accw));
            if (lane == 0) part[parity][warp] = d;
            __syncthreads();  // the slot is rewritten only two chunks later
            if (threadIdx.x == 0) {
                double sum = 0.0;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) sum += part[parity][w];
                a.worker_partials[static_cast<int64_t>(c) * CAM_KMAX + a.k] = sum;
            }
        }
    }
}

template <typename XT, int MODE, bool EMA, bool NORM, bool PUB, bool SWA, bool PEND, bool WD>
__global__ void __launch_bounds__(kThreads, 2) final_pass(const __grid_constant__ FinalArgs a) {
    constexpr int kWarps = kThreads / 32;
    __shared__ double part[2][kWarps];
    __shared__ double part_w[WD ? 2 : 1][WD ? CAM_KMAX : 1][kWarps];
    int parity = 0;
    for (int c = blockIdx.x; c < a.n_chunks; c += gridDim.x, parity ^= 1) {
        const ChunkDesc ch = a.chunks[c];
        const bool in_launch = chunk_in_launch(ch, a.local0, a.n_local);
        const TensorSlot ts = a.slots[in_launch ? ch.local : a.local0];
        if (!in_launch || !chunk_in_tensor(ch, ts)) {  // skipped, its partials 0
            if (threadIdx.x == 0) {
                atomicOr(a.status, kStatusBadChunk);
                if (NORM) a.partials[c] = 0.0;
                for (int p = 0; WD && p < a.P; ++p)
                    a.worker_partials[static_cast<int64_t>(c) * CAM_KMAX + a.first_k + p] = 0.0;
            }
            parity ^= 1;  // the slots stay as they were: no barrier for this chunk
            continue;
        }
        const int l = ch.local - a.local0;
        const void* const* tp = a.ptr + static_cast<int64_t>(l) * a.stride;
        const float* sum = static_cast<const float*>(tp[0]) + ch.start;
        const void* const* xs = tp + 3;  // the workers folded here
        float* th_p = ts.theta + ch.start;
        float* m_p = ts.m + ch.start;
        float* e_p = ts.e + ch.start;
        float* sw_p = ts.swa + ch.start;
        float* pt = PUB ? static_cast<float*>(const_cast<void*>(tp[1])) + ch.start : nullptr;
        float* pe = (PUB && EMA && tp[2]) ? static_cast<float*>(const_cast<void*>(tp[2])) + ch.start
                                          : nullptr;
        float acc = 0.0f;
        float accw[WD ? CAM_KMAX : 1];  // each folded worker's squared drift, as fold_worker sums it
#pragma unroll
        for (int p = 0; p < (WD ? CAM_KMAX : 1); ++p) accw[p] = 0.0f;
        int done = 0;
        if ((a.vec[l >> 5] >> (l & 31)) & 1u) {
            const int nv = ch.len >> 3;
            for (int v = threadIdx.x; v < nv; v += kThreads) {
                float sv[8], th[8], m[8], e[8], sw[8];
                load_s8(sum + 8 * v, sv);
                if (MODE == kDelta || NORM || WD) load_s8(th_p + 8 * v, th);
                if (MODE == kDelta) load_s8(m_p + 8 * v, m);
                if (EMA) load_s8(e_p + 8 * v, e);
                if constexpr (SWA) load_s8(sw_p + 8 * v, sw);
                if constexpr (PEND) {
                    // worker by worker (one vector live), each element's
                    // folds still in arrival order
#pragma unroll
                    for (int p = 0; p < CAM_KMAX; ++p) {
                        if (p >= a.P) break;
                        XVec<XT> xv;
                        xv.load(static_cast<const XT*>(xs[p]) + ch.start + 8 * v);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            if constexpr (WD) {
                                const float d = __fsub_rn(xv.get(j), th[j]);
                                accw[p] = __fmaf_rn(d, d, accw[p]);
                            }
                            sv[j] = fold_term<MODE>(sv[j], xv.get(j), a.wp[p],
                                                    (MODE == kDelta) ? th[j] : 0.0f);
                        }
                    }
                }
                merge_finish_n<8, MODE, EMA, NORM, SWA>(a, sv, th, m, e, sw, acc);
                store_s8(th_p + 8 * v, th);
                if (MODE == kDelta) store_s8(m_p + 8 * v, m);
                if (EMA) store_s8(e_p + 8 * v, e);
                if constexpr (SWA) store_s8(sw_p + 8 * v, sw);
                if (PUB) {
                    store_s8(pt + 8 * v, th);
                    if (pe) store_s8(pe + 8 * v, e);
                }
            }
            done = 8 * nv;
        }
        for (int j = done + threadIdx.x; j < ch.len; j += kThreads) {
            float th = (MODE == kDelta || NORM || WD) ? th_p[j] : 0.0f;
            float m = (MODE == kDelta) ? m_p[j] : 0.0f;
            float e = EMA ? e_p[j] : 0.0f;
            float s = sum[j];
            if constexpr (PEND) {
#pragma unroll
                for (int p = 0; p < CAM_KMAX; ++p) {
                    if (p >= a.P) break;
                    const float x = load_x1(static_cast<const XT*>(xs[p]) + ch.start + j);
                    if constexpr (WD) {
                        const float d = __fsub_rn(x, th);
                        accw[p] = __fmaf_rn(d, d, accw[p]);
                    }
                    s = fold_term<MODE>(s, x, a.wp[p], th);
                }
            }
            merge_finish<MODE, EMA, NORM>(a, s, th, m, e, acc);
            th_p[j] = th;
            if (MODE == kDelta) m_p[j] = m;
            if (EMA) e_p[j] = e;
            if constexpr (SWA) sw_p[j] = swa_fold(a, sw_p[j], th);
            if (PUB) {
                pt[j] = th;
                if (pe) pe[j] = e;
            }
        }
        if constexpr (NORM) {
            const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
            const double d = warp_sum(static_cast<double>(acc));
            if (lane == 0) part[parity][warp] = d;
            if constexpr (WD) {
#pragma unroll
                for (int p = 0; p < CAM_KMAX; ++p) {
                    if (p >= a.P) break;
                    const double dw = warp_sum(static_cast<double>(accw[p]));
                    if (lane == 0) part_w[parity][p][warp] = dw;
                }
            }
            __syncthreads();
            if (threadIdx.x == 0) {
                double s = 0.0;
#pragma unroll
                for (int w = 0; w < kWarps; ++w) s += part[parity][w];
                a.partials[c] = s;
                if constexpr (WD) {
                    for (int p = 0; p < a.P; ++p) {
                        double sw = 0.0;
#pragma unroll
                        for (int w = 0; w < kWarps; ++w) sw += part_w[parity][p][w];
                        a.worker_partials[static_cast<int64_t>(c) * CAM_KMAX + a.first_k + p] = sw;
                    }
                }
            }
        }
    }
}

using FoldFn = void (*)(FoldArgs);
using FinalFn = void (*)(FinalArgs);

template <typename XT>
FoldFn pick_fold(int mode, bool wd) {
    if (mode == kDelta) return wd ? fold_worker<XT, kDelta, true> : fold_worker<XT, kDelta, false>;
    return wd ? fold_worker<XT, kMean, true> : fold_worker<XT, kMean, false>;
}

template <typename XT, int MODE, bool EMA, bool NORM, bool PEND, bool WD>
FinalFn pick_final_ps(bool pub, bool swa) {
    if (pub)
        return swa ? final_pass<XT, MODE, EMA, NORM, true, true, PEND, WD>
                   : final_pass<XT, MODE, EMA, NORM, true, false, PEND, WD>;
    return swa ? final_pass<XT, MODE, EMA, NORM, false, true, PEND, WD>
               : final_pass<XT, MODE, EMA, NORM, false, false, PEND, WD>;
}

// norm: 0 none, 1 round drift, 2 round drift and the folded workers' drift
template <typename XT, int MODE, bool PEND>
FinalFn pick_final_mode(bool ema, int norm, bool pub, bool swa) {
    if (ema)
        return norm == 2 ? pick_final_ps<XT, MODE, true, true, PEND, PEND>(pub, swa)
             : norm == 1 ? pick_final_ps<XT, MODE, true, true, PEND, false>(pub, swa)
                         : pick_final_ps<XT, MODE, true, false, PEND, false>(pub, swa);
    return norm == 2 ? pick_final_ps<XT, MODE, false, true, PEND, PEND>(pub, swa)
         : norm == 1 ? pick_final_ps<XT, MODE, false, true, PEND, false>(pub, swa)
                     : pick_final_ps<XT, MODE, false, false, PEND, false>(pub, swa);
}

template <typename XT, bool PEND>
FinalFn pick_final_xt(int mode, bool ema, int norm, bool pub, bool swa) {
    return mode == kDelta ? pick_final_mode<XT, kDelta, PEND>(ema, norm, pub, swa)
                          : pick_final_mode<XT, kMean, PEND>(ema, norm, pub, swa);
}

}  // namespace

cudaError_t launch_fold(const FoldArgs& a, int dtype, int mode, bool worker_drift, int grid,
                        cudaStream_t s) {
    const FoldFn fn = dtype == kDtBF16 ? pick_fold<uint16_t>(mode, worker_drift)
                                       : pick_fold<float>(mode, worker_drift);
    void* args[] = {const_cast<FoldArgs*>(&a)};
    return cudaLaunchKernel(reinterpret_cast<const void*>(fn), dim3(grid), dim3(kThreads), args, 0, s);
}

cudaError_t launch_final(const FinalArgs& a, int dtype, int mode, bool ema, bool norm, bool pub,
                         bool swa, bool worker_drift, int grid, cudaStream_t s) {
    // without workers to fold here the dtype plays no part: one instance;
    // the workers' drift is computed here only for the workers folded here
    const int nl = !norm ? 0 : (worker_drift && a.P > 0) ? 2 : 1;
    const FinalFn fn = a.P == 0 ? pick_final_xt<float, false>(mode, ema, nl, pub, swa)
                     : dtype == kDtBF16 ? pick_final_xt<uint16_t, true>(mode, ema, nl, pub, swa)
                                        : pick_final_xt<float, true>(mode, ema, nl, pub, swa);
    void* args[] = {const_cast<FinalArgs*>(&a)};
    return cudaLaunchKernel(reinterpret_cast<const void*>(fn), dim3(grid), dim3(kThreads), args, 0, s);
}

}  // namespace cam
