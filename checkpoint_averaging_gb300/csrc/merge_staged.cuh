// merge_staged.cuh -- the staged form of the fused merge pass, as a template,
// and its variant dispatch. Each worker dtype instantiates it in its own
// translation unit (merge_staged_f32.cu, merge_staged_bf16.cu).
//
// Same arithmetic, element by element, as merge_fused.cuh (merge_device.cuh's
// merge_elem), so theta, m, e and the running average come out bit for bit
// the same; only the way the bytes reach the SM differs. The fused pass is
// HBM-bound and its register-landed loads keep too few bytes in flight when a
// round reads few bytes per element (bf16 workers, no EMA). Here the loads
// land in shared memory instead:
//
//   * one block per SM: kStConsumerWarps consumer warps, one producer warp and
//     one reducer warp;
//   * the block walks its chunks (a persistent grid stride) in tiles of
//     kStTile elements; for every tile the producer's lane 0 issues one bulk
//     copy (cp.async.bulk, the TMA engine's 1-D form) per input array -- each
//     worker, and theta / m / e / swa where the variant reads them -- into one
//     stage of a ring of st_stages stages, and counts the bytes on that
//     stage's "full" mbarrier;
//   * with each tile the producer leaves a small descriptor in shared memory
//     (tensor, first element, length, last tile of its chunk), fetching the
//     next chunk's descriptor one chunk ahead; the consumers read no chunk
//     table (except with per-worker drift, where they walk the block's chunks
//     themselves, which measured faster there), and a stage of length 0 tells
//     them the work is done;
//   * consumers wait on "full", compute four elements each from shared
//     memory, store the results straight to global memory, and release the
//     stage on its "empty" mbarrier (one arrival per warp);
//   * the producer reuses a stage once all consumer warps released it.
//
// Up to st_stages - 1 tiles are in flight per SM while one is consumed, about
// 150 KB on the common variants against some 60 KB for the register path.
//
// A tile's ragged end (fewer than 8 elements, only at the end of a tensor) is
// not copied; the consumers read it from global memory directly.
//
// Drift partials per chunk: at the end of a chunk every consumer thread stores
// its fp32 sum(s) into one of kStRedSlots hand-over slots after the ring and
// its warp arrives on the slot's "red_full" mbarrier; a third warp, the
// reducer, adds the slot in a fixed order (lane-strided fp32, then an fp64
// xor butterfly), writes the partials and frees the slot on "red_empty". The
// consumers thus do no shuffles, atomics or fp64 arithmetic (scarce on this
// GPU), and the partials do not depend on timing.
//
// There is no block-wide barrier after the set-up, and every wait on an
// mbarrier gives up after kWaitLimitNs: it then sets kStatusWaitTimeout in the
// status word, and the producer waits (again with a limit) for the copies it
// has issued before the block exits.
//
// Checks of the protocol itself: the producer checks each chunk against the
// launch's tensors and a chunk that fails takes one empty stage marked as the
// last of its chunk instead of its tiles (kStatusBadChunk); the end marker
// carries the number of stages filled before it, which the consumers compare
// with their own count of stages taken; every drift hand-over carries the
// count of chunks handed over, which the reducer compares with its own. A
// mismatch sets kStatusProtocol and stops the block as a timeout does. (The
// consumers check the end marker only: they are issue-bound on some variants,
// where a compare per tile measured 1 %.)
#pragma once

#include <cuda_runtime.h>

#include "cam_internal.h"
#include "merge_device.cuh"

namespace cam {
namespace dev {

constexpr unsigned long long kWaitLimitNs = 4000000000ull;  // 4 s
constexpr unsigned long long kTestWaitLimitNs = 1000000ull;  // 1 ms (CAM_TEST_STALL_STAGED)

// ---- PTX: shared-memory addresses, mbarriers, bulk copies ---------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes the initialised barriers visible to the bulk-copy (async) proxy.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
        : "memory");
}

// Arrives and adds `bytes` to the transaction count of the current phase.
__device__ __forceinline__ void mbar_arrive_expect(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits until the phase with the given parity has completed; false when
// `limit` nanoseconds pass first.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          unsigned long long limit) {
    if (mbar_test(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_test(bar, parity))
        if (global_ns() - t0 > limit) return false;
    return true;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Global -> shared bulk copy of `bytes` (a multiple of 16; both addresses
// 16-byte aligned), completing on mbarrier `bar`. The hinted form marks the
// lines evict-first in L2 (worker data is read once).
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void bulk_load_once(uint32_t dst, const void* src, uint32_t bytes,
                                               uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// ---- shared-memory operands ---------------------------------------------------

// Four consecutive worker elements from a stage, widened to fp32 on access.
template <typename XT>
struct SVec4;

template <>
struct SVec4<float> {
    float v[4];
    __device__ __forceinline__ void load(uint32_t addr) {
        asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                     : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3])
                     : "r"(addr)
                     : "memory");
    }
    __device__ __forceinline__ float get(int j) const { return v[j]; }
};

template <>
struct SVec4<uint16_t> {
    uint32_t u[2];
    __device__ __forceinline__ void load(uint32_t addr) {
        asm volatile("ld.shared.v2.b32 {%0,%1}, [%2];"
                     : "=r"(u[0]), "=r"(u[1])
                     : "r"(addr)
                     : "memory");
    }
    __device__ __forceinline__ float get(int j) const {
        const uint32_t w = u[j >> 1];
        return __uint_as_float((j & 1) ? (w & 0xFFFF0000u) : (w << 16));
    }
};

__device__ __forceinline__ void lds4(uint32_t addr, float (&v)[4]) {
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3])
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void stg4(float* p, const float (&v)[4]) {
    asm volatile("st.global.L1::no_allocate.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(p), "f"(v[0]),
                 "f"(v[1]), "f"(v[2]), "f"(v[3])
                 : "memory");
}

// Where one stage keeps each array: K worker slabs of kStTile elements, then
// the state slabs the variant reads (theta, m, e, swa, in that order).
struct StageLayout {
    uint32_t x_slab;  // bytes per worker slab
    uint32_t th, m, e, sw;
};

// Four consecutive elements q..q+3 of the tile starting at global index i0.
template <typename XT, int MODE, bool EMA, bool NORM, bool PUB, bool SWA, bool WD>
__device__ __forceinline__ void staged_vec4(const MergeArgs& a, const void* const* xs,
                                            const TensorSlot& ts, uint32_t stage,
                                            const StageLayout& L, int64_t i, int q,
                                            float& acc, float* accw) {
    SVec4<XT> x[CAM_KMAX];
#pragma unroll
    for (int k = 0; k < CAM_KMAX; ++k)
        if (k < a.K) x[k].load(stage + k * L.x_slab + q * static_cast<int>(sizeof(XT)));
    float th[4], m[4], e[4], sw[4];
    if (MODE == kDelta || NORM || WD) lds4(stage + L.th + 4 * q, th);
    if (MODE == kDelta) lds4(stage + L.m + 4 * q, m);
    if (EMA) lds4(stage + L.e + 4 * q, e);
    if constexpr (SWA) lds4(stage + L.sw + 4 * q, sw);
    if constexpr (MODE == kMean) {
        // plain mean: element by element, each division with its own range
        // test (measured on GB300: the fp32 mean + EMA round 0.8 % faster
        // than with the four divisions grouped, while the bf16 Nesterov
        // rounds ran 8-9 % slower element by element)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            float xk[CAM_KMAX];
#pragma unroll
            for (int k = 0; k < CAM_KMAX; ++k) xk[k] = x[k].get(j);
            if constexpr (WD) worker_drift(a, xk, th[j], accw);
            merge_elem<MODE, EMA, NORM>(a, xk, th[j], m[j], e[j], acc);
            if constexpr (SWA) sw[j] = swa_fold(a, sw[j], th[j]);
        }
    } else {
        merge_group<4, MODE, EMA, NORM, SWA, WD>(a, [&](int k, int j) { return x[k].get(j); }, th,
                                                 m, e, sw, acc, accw);
    }
    stg4(ts.theta + i, th);
    if constexpr (SWA) stg4(ts.swa + i, sw);
    if (MODE == kDelta) stg4(ts.m + i, m);
    if (EMA) stg4(ts.e + i, e);
    if (PUB) {
        stg4(static_cast<float*>(const_cast<void*>(xs[a.K])) + i, th);
        if (EMA && xs[a.K + 1]) stg4(static_cast<float*>(const_cast<void*>(xs[a.K + 1])) + i, e);
    }
}

// Where fill number it lands in the ring of P stages: stage s = it mod P, in
// its use n = it / P (the mbarriers' phase parity is n & 1), advanced one
// fill at a time instead of dividing by the run-time P at every tile.
struct RingPos {
    int s = 0, n = 0;
    __device__ __forceinline__ void next(int P) {
        if (++s == P) {
            s = 0;
            ++n;
        }
    }
};

// What the producer tells the consumers about the tile in a stage (written
// before the stage's "full" arrival, read after the consumers' wait).
struct TileMeta {
    TensorSlot ts;
    int64_t i0;    // first element of the tile, within its tensor
    int32_t len;   // elements in the tile; 0 with last = 0 marks the end of the
                   // block's work, 0 with last = 1 a chunk that failed the
                   // device-side checks (nothing to compute, a zero partial)
    int32_t l;     // launch-local tensor index
    int32_t last;  // 1 on the last tile of a chunk
    int32_t seq;   // end marker only: the stages filled before it
};

template <typename XT, int MODE, bool EMA, int NL, bool PUB, bool SWA>
__global__ void __launch_bounds__(kStThreads, 1)
    merge_staged(const __grid_constant__ MergeArgs a) {
    constexpr bool NORM = NL >= 1;
    constexpr bool WD = NL >= 2;
    constexpr bool READ_TH = MODE == kDelta || NORM || WD;
    constexpr int kStateArrays = int(READ_TH) + int(MODE == kDelta) + int(EMA) + int(SWA);
    constexpr int kProducerWarp = kStConsumerWarps, kReducerWarp = kStConsumerWarps + 1;
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full[kStMaxStages];
    __shared__ __align__(8) uint64_t empty[kStMaxStages];
    __shared__ __align__(8) uint64_t red_full[kStRedSlots];
    __shared__ __align__(8) uint64_t red_empty[kStRedSlots];
    __shared__ TileMeta meta[kStMaxStages];
    __shared__ int red_tag[kStRedSlots];  // the hand-over's chunk count, checked by the reducer
    __shared__ int abort_flag;

    const int P = a.st_stages;
    const uint32_t stage_bytes = static_cast<uint32_t>(a.st_stage_bytes);
    StageLayout L;
    L.x_slab = kStTile * static_cast<uint32_t>(sizeof(XT));
    uint32_t off = a.K * L.x_slab;
    L.th = off;
    if (READ_TH) off += kStTile * 4;
    L.m = off;
    if (MODE == kDelta) off += kStTile * 4;
    L.e = off;
    if (EMA) off += kStTile * 4;
    L.sw = off;
    // drift hand-over: kStRedSlots slots of nq x kStConsumers floats after the ring
    const int nq = 1 + (WD ? a.K : 0);
    float* const red = reinterpret_cast<float*>(ring + static_cast<size_t>(P) * stage_bytes);

    if (threadIdx.x == 0) {
        for (int s = 0; s < P; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), kStConsumerWarps);
        }
        for (int s = 0; s < kStRedSlots; ++s) {
            mbar_init(smem_u32(&red_full[s]), kStConsumerWarps);
            mbar_init(smem_u32(&red_empty[s]), 1);
        }
        abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();  // the only block-wide barrier

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t ring0 = smem_u32(ring);
    volatile int* abort_v = &abort_flag;
    const unsigned long long lim = (a.test_stall || a.test_tag) ? kTestWaitLimitNs : kWaitLimitNs;

    if (warp == kProducerWarp) {
        // ---- producer: lane 0 walks the block's chunks and issues every
        // tile's copies; the next chunk's descriptor is fetched one chunk
        // ahead so that its latency hides behind the current chunk's tiles.
        if (lane != 0) return;
        const uint64_t once = policy_evict_first();
        int it = 0;  // stages filled so far (tiles, skips and the end marker)
        // Where fill number it lands. Measured on GB300 (alternating builds):
        // advancing it incrementally made the per-worker-drift rounds 6.5 %
        // faster and the bf16 rounds with the round's norms 6 % slower than
        // dividing by P at every tile, the others unchanged; so only the
        // former advance it.
        RingPos pp;
        auto at = [&]() -> RingPos {
            if constexpr (WD) return pp;
            else return RingPos{it % P, it / P};
        };
        bool ok = true;
        int c = blockIdx.x;
        ChunkDesc ch{}, chn{};
        TensorSlot ts{}, tsn{};
        if (c < a.n_chunks) {
            ch = a.chunks[c];
            if (chunk_in_launch(ch, a.local0, a.n_local)) ts = a.slots[ch.local];
        }
        for (; ok && c < a.n_chunks; c += gridDim.x) {
            const bool has_next = c + static_cast<int>(gridDim.x) < a.n_chunks;
            if (has_next) chn = a.chunks[c + gridDim.x];
            if (!chunk_in_launch(ch, a.local0, a.n_local) || !chunk_in_tensor(ch, ts)) {
                // a chunk that fails the checks: one empty stage, marked as
                // the last of its chunk, in place of its tiles
                atomicOr(a.status, kStatusBadChunk);
                const RingPos q = at();
                const int s = q.s, n = q.n;
                if ((n > 0 && !mbar_wait(smem_u32(&empty[s]), (n - 1) & 1, lim)) || *abort_v) {
                    ok = false;
                    break;
                }
                meta[s].len = 0;
                meta[s].last = 1;
                mbar_arrive(smem_u32(&full[s]));
                ++it;
                pp.next(P);
                if (has_next)
                    tsn = chunk_in_launch(chn, a.local0, a.n_local) ? a.slots[chn.local] : TensorSlot{};
                ch = chn;
                ts = tsn;
                continue;
            }
            const int l = ch.local - a.local0;
            const void* const* xs = a.x + static_cast<int64_t>(l) * a.stride;
            for (int t0 = 0; t0 < ch.len; t0 += kStTile, ++it, pp.next(P)) {
                const RingPos q = at();
                const int s = q.s, n = q.n;
                // the stage's previous tile must be released by every consumer warp
                if (n > 0 && !mbar_wait(smem_u32(&empty[s]), (n - 1) & 1, lim)) {
                    ok = false;
                    break;
                }
                if (*abort_v) {
                    ok = false;
                    break;
                }
                const int len = min(kStTile, ch.len - t0);
                const int len8 = len & ~7;
                const int64_t i0 = ch.start + t0;
                TileMeta& mt = meta[s];
                mt.ts = ts;
                mt.i0 = i0;
                mt.len = len;
                mt.l = l;
                mt.last = t0 + kStTile >= ch.len;
                const uint32_t bar = smem_u32(&full[s]);
                if (a.test_stall && it == 0) {
                    // test hook: the first tile is never issued, so its
                    // consumers' waits run out
                } else if (len8 == 0) {  // a tensor of fewer than 8 elements: nothing to copy
                    mbar_arrive(bar);
                } else {
                    const uint32_t st = ring0 + s * stage_bytes;
                    const uint32_t xb = len8 * static_cast<uint32_t>(sizeof(XT)), sb = len8 * 4u;
                    mbar_arrive_expect(bar, a.K * xb + kStateArrays * sb);
                    for (int k = 0; k < a.K; ++k)
                        bulk_load_once(st + k * L.x_slab, static_cast<const XT*>(xs[k]) + i0, xb,
                                       bar, once);
                    if (READ_TH) bulk_load(st + L.th, ts.theta + i0, sb, bar);
                    if (MODE == kDelta) bulk_load(st + L.m, ts.m + i0, sb, bar);
                    if (EMA) bulk_load(st + L.e, ts.e + i0, sb, bar);
                    if constexpr (SWA) bulk_load(st + L.sw, ts.swa + i0, sb, bar);
                }
                if (t0 == 0 && has_next)
                    tsn = chunk_in_launch(chn, a.local0, a.n_local) ? a.slots[chn.local] : TensorSlot{};
            }
            ch = chn;
            ts = tsn;
        }
        if (ok) {  // the end marker: a stage with len 0
            const RingPos q = at();
            const int s = q.s, n = q.n;
            if (n > 0 && !mbar_wait(smem_u32(&empty[s]), (n - 1) & 1, lim)) ok = false;
            if (ok) {
                meta[s].len = 0;
                meta[s].last = 0;
                meta[s].seq = a.test_tag ? -1 : it;  // (test hook: a wrong fill number)
                mbar_arrive(smem_u32(&full[s]));
                ++it;
            }
        }
        // Stay until the consumers have released every stage filled last, so
        // that no copy is in flight when the block exits.
        const int j0 = it > P ? it - P : 0;
        for (int j = j0; ok && j < it; ++j)
            if (!mbar_wait(smem_u32(&empty[j % P]), (j / P) & 1, lim)) ok = false;
        if (!ok) {
            *abort_v = 1;
            atomicOr(a.status, kStatusWaitTimeout);
            for (int j = j0; j < it; ++j) mbar_wait(smem_u32(&full[j % P]), (j / P) & 1, lim);
        }
        return;
    }

    if (warp == kReducerWarp) {
        // ---- reducer: one drift partial per chunk and quantity, in a fixed
        // order: lane l adds entries l, l + 32, ... (16 per-thread sums) in
        // fp32, then the warp adds the 32 lane sums in fp64 (xor butterfly,
        // lane 0's result). Quantity 0 is the round's drift, 1 + k worker k's.
        if constexpr (NORM) {
            int ci = 0;
            for (int c = blockIdx.x; c < a.n_chunks; c += gridDim.x, ++ci) {
                const int slot = ci % kStRedSlots, use = ci / kStRedSlots;
                if (*abort_v) return;
                if (!mbar_wait(smem_u32(&red_full[slot]), use & 1, lim)) {
                    *abort_v = 1;
                    atomicOr(a.status, kStatusWaitTimeout);
                    return;
                }
                if (red_tag[slot] != ci) {  // the consumers handed over another chunk
                    *abort_v = 1;
                    if (lane == 0) atomicOr(a.status, kStatusProtocol);
                    return;
                }
                const float* rb = red + slot * nq * kStConsumers;
                for (int q = 0; q < nq; ++q) {
                    float s = 0.0f;
#pragma unroll
                    for (int i = 0; i < kStConsumers / 32; ++i)
                        s = __fadd_rn(s, rb[q * kStConsumers + i * 32 + lane]);
                    const double d = warp_sum(static_cast<double>(s));
                    if (lane == 0) {
                        if (q == 0) a.partials[c] = d;
                        else a.worker_partials[static_cast<int64_t>(c) * CAM_KMAX + q - 1] = d;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&red_empty[slot]));
            }
        }
        return;
    }

    // ---- consumers: four elements per thread per tile ----
    const int g = threadIdx.x;
    float acc = 0.0f;
    float accw[CAM_KMAX];
#pragma unroll
    for (int k = 0; k < CAM_KMAX; ++k) accw[k] = 0.0f;
    // Hands chunk number ci's per-thread sums to the reducer warp; false when
    // the wait for a free slot gave up.
    auto hand_over = [&](int ci) -> bool {
        const int slot = ci % kStRedSlots, use = ci / kStRedSlots;
        if (use > 0 && !mbar_wait(smem_u32(&red_empty[slot]), (use - 1) & 1, lim)) {
            *abort_v = 1;
            atomicOr(a.status, kStatusWaitTimeout);
            return false;
        }
        float* rb = red + slot * nq * kStConsumers;
        rb[g] = acc;
        acc = 0.0f;
#pragma unroll
        for (int k = 0; k < CAM_KMAX; ++k) {
            if (WD && k < a.K) rb[(1 + k) * kStConsumers + g] = accw[k];
            accw[k] = 0.0f;
        }
        if (g == 0) red_tag[slot] = ci;  // before warp 0's arrival
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&red_full[slot]));
        return true;
    };
    // Waits for stage s's use n; false (with the abort flag set) on a timeout.
    auto wait_full = [&](int s, int n) -> bool {
        if (*abort_v) return false;
        if (!mbar_wait(smem_u32(&full[s]), n & 1, lim)) {
            *abort_v = 1;
            atomicOr(a.status, kStatusWaitTimeout);
            return false;
        }
        return true;
    };
    // The end marker must carry the consumers' own count of stages taken
    // (it = n P + s): otherwise they took a stage too many or too few, which
    // sets kStatusProtocol and stops the block like a timeout.
    auto end_in_sequence = [&](int s, int it) -> bool {
        if (meta[s].seq == it) return true;
        *abort_v = 1;
        if (lane == 0) atomicOr(a.status, kStatusProtocol);
        return false;
    };

    if constexpr (WD) {
        // With per-worker drift the arithmetic per element is heavy enough for
        // the pass to be issue-bound. Here the consumers walk the block's
        // chunks themselves and keep each chunk's pointers in registers, which
        // measured faster than reading the per-tile descriptor; they only
        // release the producer's end marker at the end.
        // They check each chunk as the producer does: one stage, nothing
        // computed, for a chunk that fails.
        int it = 0, ci = 0;
        RingPos cp;  // where stage number it lands
        for (int c = blockIdx.x; c < a.n_chunks; c += gridDim.x, ++ci) {
            const ChunkDesc ch = a.chunks[c];
            const bool in_launch = chunk_in_launch(ch, a.local0, a.n_local);
            const TensorSlot ts = a.slots[in_launch ? ch.local : a.local0];
            if (!in_launch || !chunk_in_tensor(ch, ts)) {  // the producer's one empty stage
                const int s = cp.s;
                if (!wait_full(s, cp.n)) return;
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
                ++it;
                cp.next(P);
                if (!hand_over(ci)) return;
                continue;
            }
            const void* const* xs = a.x + static_cast<int64_t>(ch.local - a.local0) * a.stride;
            for (int t0 = 0; t0 < ch.len; t0 += kStTile, ++it, cp.next(P)) {
                const int s = cp.s;
                if (!wait_full(s, cp.n)) return;
                const int len = min(kStTile, ch.len - t0);
                const int len8 = len & ~7;
                const int64_t i0 = ch.start + t0;
                if (4 * g < len8)
                    staged_vec4<XT, MODE, EMA, NORM, PUB, SWA, WD>(
                        a, xs, ts, ring0 + s * stage_bytes, L, i0 + 4 * g, 4 * g, acc, accw);
                if (g < len - len8)  // the ragged end, straight from global memory
                    merge_one<XT, MODE, EMA, NORM, PUB, SWA, WD>(a, xs, ts, i0 + len8 + g, acc, accw);
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
            }
            if (!hand_over(ci)) return;
        }
        const int s = cp.s;  // the end marker
        if (!wait_full(s, cp.n) || !end_in_sequence(s, it)) return;
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
    } else {
        // Otherwise they take the tiles in the order the producer filled the
        // stages, reading each tile's descriptor, until the end marker.
        RingPos cp;  // where stage number it lands
        for (int it = 0, ci = 0;; ++it, cp.next(P)) {
            const int s = cp.s;
            if (!wait_full(s, cp.n)) return;
            const int len = meta[s].len;
            if (len == 0 && !meta[s].last) {  // end marker: release it and stop
                if (!end_in_sequence(s, it)) return;
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
                return;
            }
            // (len 0 with last set: a chunk that failed the checks; nothing
            // below computes, and its partial is handed over as 0)
            const TensorSlot ts = meta[s].ts;
            const int64_t i0 = meta[s].i0;
            const int last = meta[s].last;
            const void* const* xs = a.x + static_cast<int64_t>(meta[s].l) * a.stride;
            const int len8 = len & ~7;
            if (4 * g < len8)
                staged_vec4<XT, MODE, EMA, NORM, PUB, SWA, WD>(a, xs, ts, ring0 + s * stage_bytes, L,
                                                               i0 + 4 * g, 4 * g, acc, accw);
            if (g < len - len8)  // the ragged end, straight from global memory
                merge_one<XT, MODE, EMA, NORM, PUB, SWA, WD>(a, xs, ts, i0 + len8 + g, acc, accw);
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
            if (NORM && last && !hand_over(ci++)) return;
        }
    }
}

template <typename XT, int MODE, bool PUB, bool SWA>
MergeFn staged_level(bool ema, int nl) {
    if (ema) {
        if (nl == 0) return merge_staged<XT, MODE, true, 0, PUB, SWA>;
        if (nl == 1) return merge_staged<XT, MODE, true, 1, PUB, SWA>;
        return merge_staged<XT, MODE, true, 2, PUB, SWA>;
    }
    if (nl == 0) return merge_staged<XT, MODE, false, 0, PUB, SWA>;
    if (nl == 1) return merge_staged<XT, MODE, false, 1, PUB, SWA>;
    return merge_staged<XT, MODE, false, 2, PUB, SWA>;
}

template <typename XT, bool PUB, bool SWA>
MergeFn staged_mode(const MergeVariant& v) {
    return v.mode == kDelta ? staged_level<XT, kDelta, PUB, SWA>(v.ema, v.norm_level)
                            : staged_level<XT, kMean, PUB, SWA>(v.ema, v.norm_level);
}

template <typename XT>
MergeFn staged_for_dtype(const MergeVariant& v) {
    if (v.pub) return v.swa ? staged_mode<XT, true, true>(v) : staged_mode<XT, true, false>(v);
    return v.swa ? staged_mode<XT, false, true>(v) : staged_mode<XT, false, false>(v);
}

}  // namespace dev
}  // namespace cam
