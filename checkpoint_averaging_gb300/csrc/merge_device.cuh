// merge_device.cuh -- per-element arithmetic and memory access of the fused
// merge pass, shared by the kernels of libcam.
//
// The arithmetic is the fixed sequence of binary32 operations the C ABI
// documents (include/cam.h): plain mean in arrival order or token-weighted
// delta mean, plain replacement or outer Nesterov, EMA of the globals, squared
// drift. Explicit round-to-nearest intrinsics keep every multiply and add
// separately rounded. The argument block type A provides K, Kf, w[], W, lr,
// mu, beta and div (the division's DivPlan: by Kf or by W).
#pragma once

#include <cuda_runtime.h>

#include "cam_internal.h"

namespace cam {
namespace dev {

constexpr int kMean = CAM_MODE_MEAN_REPLACE;
constexpr int kDelta = CAM_MODE_DELTA_NESTEROV;

// ---- device-side chunk checks ------------------------------------------------

// The host builds every chunk table and checks it once (each tensor's chunks
// inside it, in order, without gaps); the passes check each chunk again as
// they take it, at the cost of a compare per chunk, so that a corrupted table
// is reported (kStatusBadChunk) and the chunk skipped instead of read or
// written through. A pass loads the chunk's slot once, from the launch's
// first tensor when the chunk names another, before checking it.

// Chunk ch's tensor is one of the launch's, [local0, local0 + n_local): only
// then may its slot be read.
__device__ __forceinline__ bool chunk_in_launch(const ChunkDesc& ch, int32_t local0,
                                                int32_t n_local) {
    return static_cast<uint32_t>(ch.local - local0) < static_cast<uint32_t>(n_local);
}

// At least one element, all of them inside the tensor of slot ts.
__device__ __forceinline__ bool chunk_in_tensor(const ChunkDesc& ch, const TensorSlot& ts) {
    return ch.start >= 0 && ch.len > 0 && ch.start <= ts.numel - ch.len;
}

// ---- memory access -----------------------------------------------------------

// Worker data: read once, never written by this pass. XVec<T> holds one
// thread's 8 consecutive elements of one worker as loaded (fp32 values, or
// bf16 pairs packed in 32-bit words) and widens on access; bf16 is the high
// half of a binary32, so widening is exact.
template <typename XT>
struct XVec;

template <>
struct XVec<float> {
    float v[8];
    __device__ __forceinline__ void load(const float* p) {
        asm volatile(
            "ld.global.nc.L1::no_allocate.L2::evict_first.v8.f32 "
            "{%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
            : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]),
              "=f"(v[6]), "=f"(v[7])
            : "l"(p));
    }
    __device__ __forceinline__ float get(int j) const { return v[j]; }
};

template <>
struct XVec<uint16_t> {
    uint32_t u[4];
    __device__ __forceinline__ void load(const uint16_t* p) {
        asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3])
                     : "l"(p));
    }
    __device__ __forceinline__ float get(int j) const {
        const uint32_t w = u[j >> 1];
        return __uint_as_float((j & 1) ? (w & 0xFFFF0000u) : (w << 16));
    }
};

__device__ __forceinline__ float load_x1(const float* p) {
    float v;
    asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float load_x1(const uint16_t* p) {
    unsigned short b;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(b) : "l"(p));
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// State (theta, m, e): read once and written back by the same thread.
__device__ __forceinline__ void load_s8(const float* p, float (&v)[8]) {
    asm volatile(
        "ld.global.L1::no_allocate.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]), "=f"(v[4]), "=f"(v[5]),
          "=f"(v[6]), "=f"(v[7])
        : "l"(p));
}

// N = 2 or 4 consecutive floats: state (read once, written back by the same
// thread) and fp32 worker elements, for the narrow steps below.
template <int N>
__device__ __forceinline__ void load_sn(const float* p, float (&v)[N]) {
    if constexpr (N == 4)
        asm volatile("ld.global.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                     : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3])
                     : "l"(p));
    else
        asm volatile("ld.global.L1::no_allocate.v2.f32 {%0,%1}, [%2];"
                     : "=f"(v[0]), "=f"(v[1])
                     : "l"(p));
}

template <int N>
__device__ __forceinline__ void store_sn(float* p, const float (&v)[N]) {
    if constexpr (N == 4)
        asm volatile("st.global.L1::no_allocate.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(v[0]),
                     "f"(v[1]), "f"(v[2]), "f"(v[3])
                     : "memory");
    else
        asm volatile("st.global.L1::no_allocate.v2.f32 [%0], {%1,%2};" ::"l"(p), "f"(v[0]),
                     "f"(v[1])
                     : "memory");
}

template <int N>
__device__ __forceinline__ void load_xn(const float* p, float (&v)[N]) {
    if constexpr (N == 4)
        asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                     : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3])
                     : "l"(p));
    else
        asm volatile("ld.global.nc.L1::no_allocate.v2.f32 {%0,%1}, [%2];"
                     : "=f"(v[0]), "=f"(v[1])
                     : "l"(p));
}

__device__ __forceinline__ void store_s8(float* p, const float (&v)[8]) {
    asm volatile(
        "st.global.L1::no_allocate.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p),
        "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]),
        "f"(v[7])
        : "memory");
}

// ---- division --------------------------------------------------------------

// s / d correctly rounded -- the bits __fdiv_rn(s, d) gives -- for the round's
// divisor d = p.d, from its reciprocal held as two binary32 terms, y = p.y =
// RN(1/d) and y_lo = p.y_lo = RN(1/d - y), and one of Markstein's
// corrections (P. Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Develop. 34(1), 1990; also Muller
// et al., "Handbook of Floating-Point Arithmetic", division with a fused
// multiply-add):
//   q0 = RN(s*y + RN(s*y_lo))   within one unit in the last place of s/d:
//                               the two terms carry 1/d to about 2^-47 of
//                               itself, so the sum is s/d to within
//                               |s/d| * 2^-46 before its one rounding
//   r  = s - d*q0               exact, q0 being faithful (one fused multiply-add)
//   q  = RN(q0 + r*y)           = RN(s/d) by Markstein's theorem (y within
//                               half a unit of 1/d, q0 faithful, r exact)
// All of it holds while nothing leaves the normal range. div_plan admits
// d in [2^(e-1), 2^e) inside [2^-100, 2^100] and |s| in
// [2^max(-100, e-124), 2^min(126, e+124)): then |s/d| lies in
// [2^-124, 2^125), so q0 and q are normal and d*q0 finite, s*y_lo loses at
// most 2^-150 to underflow (far below a unit of q0), and r is an integer
// multiple of ulp(d)*ulp(q0) >= 2^-148, fewer than 2^24 of them, so
// representable. A zero dividend gives itself (+-0 / d is +-0 for the plan's
// positive d). Every other s outside the range (smaller, larger, infinite,
// NaN), and every s of a divisor out of range (p.active 0), takes __fdiv_rn,
// out of line.

// |s| inside the plan's range (zeros are not).
__device__ __forceinline__ bool div_in_range(float s, const DivPlan& p) {
    return (__float_as_uint(s) & 0x7FFFFFFFu) - p.lo < p.span;
}

__device__ __forceinline__ float div_fast(float s, const DivPlan& p) {
    const float q0 = __fmaf_rn(s, p.y, __fmul_rn(s, p.y_lo));
    return __fmaf_rn(__fmaf_rn(-p.d, q0, s), p.y, q0);
}

static __device__ __noinline__ float div_rn_slow(float s, float d) { return __fdiv_rn(s, d); }

// A dividend outside the range.
__device__ __forceinline__ float div_outside(float s, const DivPlan& p) {
    return (s == 0.0f && p.active) ? s : div_rn_slow(s, p.d);
}

// One quotient (the passes' scalar tails).
__device__ __forceinline__ float div_rn(float s, const DivPlan& p) {
    return div_in_range(s, p) ? div_fast(s, p) : div_outside(s, p);
}

// N quotients: the reciprocal form for all of them, then one test of the N
// dividends against the range: t = 2|s| - 2^(lo_e + 1) as bit patterns
// (the sign shifted out) lies below 2*span for every |s| in range and at or
// above it for every other s (a zero wraps around to a large t), so the
// largest t decides for all N, at a shift-add and a maximum per element.
// Only when that test fails -- a zero, a dividend out of range, a divisor
// out of range -- are the N checked one by one and those outside the range
// taken again by div_outside. The merge loops so take one branch per N
// elements, and the N elements' arithmetic stays one straight run of code.
template <int N>
__device__ __forceinline__ void div_rn_n(const float (&s)[N], float (&q)[N], const DivPlan& p) {
    uint32_t tmax = 0u;
#pragma unroll
    for (int j = 0; j < N; ++j) {
        q[j] = div_fast(s[j], p);
        tmax = max(tmax, (__float_as_uint(s[j]) << 1) - (p.lo << 1));
    }
    if (tmax >= (p.span << 1)) {
#pragma unroll
        for (int j = 0; j < N; ++j)
            if (!div_in_range(s[j], p)) q[j] = div_outside(s[j], p);
    }
}

// ---- per-element arithmetic ----------------------------------------------------

// What follows the fold and the division for one element: q is the quotient
// (the mean s / K, or the token-weighted delta mean s / W); outer step and
// EMA update th, m, e in place, and acc collects the squared drift. Shared by
// every pass, so all produce the same bits.
template <int MODE, bool EMA, bool NORM, class A>
__device__ __forceinline__ void merge_update(const A& a, float q, float& th, float& m, float& e,
                                             float& acc) {
    if (MODE == kMean) {
        if (NORM) {
            const float d = __fsub_rn(q, th);
            acc = __fmaf_rn(d, d, acc);
        }
        th = q;  // plain replacement
    } else {
        const float delta = q;
        if (NORM) acc = __fmaf_rn(delta, delta, acc);
        const float g = -delta;  // pseudo-gradient theta - (theta + delta)
        const float m_new = __fadd_rn(__fmul_rn(a.mu, m), g);
        const float step = __fadd_rn(g, __fmul_rn(a.mu, m_new));
        th = __fsub_rn(th, __fmul_rn(a.lr, step));
        m = m_new;
    }
    if (EMA) {
        const float omb = __fsub_rn(1.0f, a.beta);
        e = __fadd_rn(__fmul_rn(a.beta, e), __fmul_rn(omb, th));
    }
}

// The division and merge_update for one element: s is the arrival-order sum
// (the plain sum of the workers, or the token-weighted sum of their deltas).
template <int MODE, bool EMA, bool NORM, class A>
__device__ __forceinline__ void merge_finish(const A& a, float s, float& th, float& m, float& e,
                                             float& acc) {
    merge_update<MODE, EMA, NORM>(a, div_rn(s, a.div), th, m, e, acc);
}

// One worker's term of the arrival-order fold: s + x (plain mean) or
// s + w * (x - theta) (token-weighted delta mean), one rounding per operation.
template <int MODE>
__device__ __forceinline__ float fold_term(float s, float x, float w, float th) {
    return MODE == kMean ? __fadd_rn(s, x) : __fadd_rn(s, __fmul_rn(w, __fsub_rn(x, th)));
}

// The arrival-order sum of one element: xk[k] (k < K) are the workers'
// values in arrival order.
template <int MODE, class A>
__device__ __forceinline__ float merge_fold(const A& a, const float (&xk)[CAM_KMAX], float th) {
    float s = 0.0f;
#pragma unroll
    for (int k = 0; k < CAM_KMAX; ++k)
        if (k < a.K) s = fold_term<MODE>(s, xk[k], MODE == kMean ? 1.0f : a.w[k], th);
    return s;
}

// One element of one round: th, m, e are updated in place; acc collects the
// squared drift.
template <int MODE, bool EMA, bool NORM, class A>
__device__ __forceinline__ void merge_elem(const A& a, const float (&xk)[CAM_KMAX],
                                           float& th, float& m, float& e, float& acc) {
    merge_finish<MODE, EMA, NORM>(a, merge_fold<MODE>(a, xk, th), th, m, e, acc);
}

// Folds the new global into the uniform running average: mu + (theta' - mu)/n,
// n = the number of globals in the average after this one.
template <class A>
__device__ __forceinline__ float swa_fold(const A& a, float mu, float th) {
    return __fadd_rn(mu, div_rn(__fsub_rn(th, mu), a.swa_div));
}

// Per-worker drift: accw[k] += (x_k - theta_old)^2 for k < K, before the
// outer step changes theta.
template <class A>
__device__ __forceinline__ void worker_drift(const A& a, const float (&xk)[CAM_KMAX], float th,
                                             float* accw) {
#pragma unroll
    for (int k = 0; k < CAM_KMAX; ++k)
        if (k < a.K) {
            const float d = __fsub_rn(xk[k], th);
            accw[k] = __fmaf_rn(d, d, accw[k]);
        }
}

// N elements whose sums s[] are formed: their quotients (div_rn_n), then
// merge_update element by element and, with SWA, the running average.
template <int N, int MODE, bool EMA, bool NORM, bool SWA, class A>
__device__ __forceinline__ void merge_finish_n(const A& a, const float (&s)[N], float (&th)[N],
                                               float (&m)[N], float (&e)[N], float (&sw)[N],
                                               float& acc) {
    float q[N];
    div_rn_n<N>(s, q, a.div);
#pragma unroll
    for (int j = 0; j < N; ++j) merge_update<MODE, EMA, NORM>(a, q[j], th[j], m[j], e[j], acc);
    if constexpr (SWA) {  // swa_fold's operations, the N divisions together
        float dv[N], qv[N];
#pragma unroll
        for (int j = 0; j < N; ++j) dv[j] = __fsub_rn(th[j], sw[j]);
        div_rn_n<N>(dv, qv, a.swa_div);
#pragma unroll
        for (int j = 0; j < N; ++j) sw[j] = __fadd_rn(sw[j], qv[j]);
    }
}

// N elements of one step, worker k's value of element j given by xv(k, j):
// in element order each worker's squared drift (WD) and the fold, then
// merge_finish_n. Per element the operations and their order are
// merge_elem's, and acc and accw collect in element order.
template <int N, int MODE, bool EMA, bool NORM, bool SWA, bool WD, class A, class XV>
__device__ __forceinline__ void merge_group(const A& a, const XV& xv, float (&th)[N],
                                            float (&m)[N], float (&e)[N], float (&sw)[N],
                                            float& acc, float* accw) {
    float s[N];
#pragma unroll
    for (int j = 0; j < N; ++j) {
        float xk[CAM_KMAX];
#pragma unroll
        for (int k = 0; k < CAM_KMAX; ++k) xk[k] = xv(k, j);
        if constexpr (WD) worker_drift(a, xk, th[j], accw);
        s[j] = merge_fold<MODE>(a, xk, th[j]);
    }
    merge_finish_n<N, MODE, EMA, NORM, SWA>(a, s, th, m, e, sw, acc);
}

// xs[0..K) are the workers' copies of the tensor; with PUB, xs[K] receives a
// copy of the new theta and xs[K+1] (when not null) a copy of the new EMA.
// With SWA the uniform running average ts.swa is updated from the new theta.
// With WD, accw[0..K) collect each worker's squared drift.
// N (2 or 4) consecutive elements from fp32 workers with narrower accesses:
// the register-heavy variants (a running average with norms, per-worker
// drift or published copies) take an 8-element step as 8 / N of these, which
// keeps them from spilling. Same operations in the same order per element
// as merge_vec8.
template <int N, int MODE, bool EMA, bool NORM, bool PUB, bool SWA, bool WD, class A>
__device__ __forceinline__ void merge_vecn_f32(const A& a, const void* const* xs,
                                               const TensorSlot& ts, int64_t i, float& acc,
                                               float* accw) {
    float x[CAM_KMAX][N];
#pragma unroll
    for (int k = 0; k < CAM_KMAX; ++k)
        if (k < a.K) load_xn<N>(static_cast<const float*>(xs[k]) + i, x[k]);
    float th[N], m[N], e[N], sw[N];
    if (MODE == kDelta || NORM || WD) load_sn<N>(ts.theta + i, th);
    if (MODE == kDelta) load_sn<N>(ts.m + i, m);
    if (EMA) load_sn<N>(ts.e + i, e);
    if constexpr (SWA) load_sn<N>(ts.swa + i, sw);
    merge_group<N, MODE, EMA, NORM, SWA, WD>(a, [&](int k, int j) { return x[k][j]; }, th, m, e, sw,
                                             acc, accw);
    store_sn<N>(ts.theta + i, th);
    if constexpr (SWA) store_sn<N>(ts.swa + i, sw);
    if (MODE == kDelta) store_sn<N>(ts.m + i, m);
    if (EMA) store_sn<N>(ts.e + i, e);
    if (PUB) {
        store_sn<N>(static_cast<float*>(const_cast<void*>(xs[a.K])) + i, th);
        if (EMA && xs[a.K + 1]) store_sn<N>(static_cast<float*>(const_cast<void*>(xs[a.K + 1])) + i, e);
    }
}

template <typename XT, int MODE, bool EMA, bool NORM, bool PUB = false, bool SWA = false,
          bool WD = false, class A>
__device__ __forceinline__ void merge_vec8(const A& a, const void* const* xs,
                                           const TensorSlot& ts, int64_t i, float& acc,
                                           float* accw = nullptr) {
    if constexpr (sizeof(XT) == 4 && SWA && (NORM || WD)) {
        // published copies or per-worker drift on top: 2 elements a step
        constexpr int N = (PUB || (WD && MODE == kMean && !EMA)) ? 2 : 4;
#pragma unroll
        for (int h = 0; h < 8; h += N)
            merge_vecn_f32<N, MODE, EMA, NORM, PUB, SWA, WD>(a, xs, ts, i + h, acc, accw);
        return;
    }
    XVec<XT> x[CAM_KMAX];
#pragma unroll
    for (int k = 0; k < CAM_KMAX; ++k)
        if (k < a.K) x[k].load(static_cast<const XT*>(xs[k]) + i);
    float th[8], m[8], e[8];
    if (MODE == kDelta || NORM || WD) load_s8(ts.theta + i, th);
    if (MODE == kDelta) load_s8(ts.m + i, m);
    if (EMA) load_s8(ts.e + i, e);
    float sw[8];
    if constexpr (SWA) load_s8(ts.swa + i, sw);
    if constexpr (EMA && !SWA) {
        // an EMA without a running average: element by element, each division
        // with its own range test (measured on GB300: the bf16 Nesterov + EMA
        // sweeps 1.5-2 % faster than with the eight divisions grouped; the
        // other variants as fast or faster grouped)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            float xk[CAM_KMAX];
#pragma unroll
            for (int k = 0; k < CAM_KMAX; ++k) xk[k] = x[k].get(j);
            if constexpr (WD) worker_drift(a, xk, th[j], accw);
            merge_elem<MODE, EMA, NORM>(a, xk, th[j], m[j], e[j], acc);
        }
    } else {
        merge_group<8, MODE, EMA, NORM, SWA, WD>(a, [&](int k, int j) { return x[k].get(j); }, th,
                                                 m, e, sw, acc, accw);
    }
    store_s8(ts.theta + i, th);
    if constexpr (SWA) store_s8(ts.swa + i, sw);
    if (MODE == kDelta) store_s8(ts.m + i, m);
    if (EMA) store_s8(ts.e + i, e);
    if (PUB) {
        store_s8(static_cast<float*>(const_cast<void*>(xs[a.K])) + i, th);
        if (EMA && xs[a.K + 1]) store_s8(static_cast<float*>(const_cast<void*>(xs[a.K + 1])) + i, e);
    }
}

template <typename XT, int MODE, bool EMA, bool NORM, bool PUB = false, bool SWA = false,
          bool WD = false, class A>
__device__ __forceinline__ void merge_one(const A& a, const void* const* xs,
                                          const TensorSlot& ts, int64_t i, float& acc,
                                          float* accw = nullptr) {
    float xk[CAM_KMAX];
#pragma unroll
    for (int k = 0; k < CAM_KMAX; ++k)
        xk[k] = (k < a.K) ? load_x1(static_cast<const XT*>(xs[k]) + i) : 0.0f;
    float th = ts.theta[i];
    float m = (MODE == kDelta) ? ts.m[i] : 0.0f;
    float e = EMA ? ts.e[i] : 0.0f;
    if constexpr (WD) worker_drift(a, xk, th, accw);
    merge_elem<MODE, EMA, NORM>(a, xk, th, m, e, acc);
    ts.theta[i] = th;
    if (MODE == kDelta) ts.m[i] = m;
    if (EMA) ts.e[i] = e;
    if constexpr (SWA) ts.swa[i] = swa_fold(a, ts.swa[i], th);
    if (PUB) {
        static_cast<float*>(const_cast<void*>(xs[a.K]))[i] = th;
        if (EMA && xs[a.K + 1]) static_cast<float*>(const_cast<void*>(xs[a.K + 1]))[i] = e;
    }
}

__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

}  // namespace dev
}  // namespace cam
