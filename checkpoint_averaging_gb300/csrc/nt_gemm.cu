// nt_gemm.cu -- batched NT GEMMs of the Newton-Schulz iteration (outer
// orthogonalisation, "DiffuRefill-1B" technical report, section 5.3) on the
// fifth-generation tensor cores of sm_103a, plus a CUDA-core fp32 form.
//
// Tensor-core kernel nt_gemm_tc<BF16, BN, EPI>: a persistent grid of one
// block per SM; block b takes the output tiles b, b + grid, ... Each block is
// six warps with fixed roles:
//
//   warp 0 (lane 0)  TMA producer: per K step, one 128-row box of A and BN/128
//                    boxes of B (128-byte rows, 128-byte swizzle) into a ring
//                    of shared-memory stages, counted on the stage's "full"
//                    mbarrier;
//   warp 1 (lane 0)  MMA issuer: four tcgen05.mma (M = 128, N = BN, K = 32
//                    bytes each) per stage into one of two TMEM accumulators
//                    (2 x BN fp32 columns), tcgen05.commit releasing the
//                    stage and, after a tile's last stage, the accumulator;
//                    warp 1 also allocates and frees the TMEM;
//   warps 2..5       epilogue: each owns 32 TMEM lanes (rows of the tile) and
//                    works in 32 x 32 boxes: tcgen05.ld of 32 columns, the
//                    scaling, the box (and, where asked, its transpose)
//                    written to a per-warp shared-memory staging buffer, and
//                    a TMA tensor store of each from lane 0. Two staging
//                    buffers per warp let one box's store overlap the next
//                    box's work; the accumulator is handed back as soon as
//                    its last columns are in registers.
//
// Two accumulators let the epilogue of one tile overlap the MMAs of the next.
// Shared-memory operands use the canonical K-major 128-byte-swizzled layout
// that TMA writes: 8-row groups of 1,024 bytes, so the matrix descriptors
// carry a stride of 1,024 bytes, and the four MMAs of a stage start 32 bytes
// apart inside each swizzled row.
//
// Every mbarrier wait is bounded (kTcWaitLimitNs of %globaltimer). A wait that
// runs out sets CAM_STATUS_GEMM_TIMEOUT in the status word and a block-wide
// abort flag; every role then leaves its loop, the producer waits (bounded)
// for the copies it issued, the MMA issuer for its MMAs, the epilogue for its
// stores, and warp 1 frees the TMEM before the block exits.
//
// CUDA-core kernel nt_gemm_simt: 128 x 128 tiles, 8 x 8 outputs per thread,
// fp32 fused multiply-adds; used for CAM_ORTHO_FP32.
#include "nt_gemm.h"

#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "cam_internal.h"

namespace cam {
namespace tc {

constexpr int kBM = 128;                 // tile rows (TMEM lanes)
constexpr int kTcThreads = 192;          // six warps
constexpr int kRowBytes = 128;           // one swizzled row of a stage: the K step
constexpr int kBoxBytes = kBM * kRowBytes;  // one 128-row TMA box: 16 KB
constexpr int kSmemBudget = 224 * 1024;  // the stage ring and the epilogue staging
constexpr unsigned long long kTcWaitLimitNs = 4000000000ull;
constexpr int kEpiAxpbyC = 2;            // kNtAxpby reading C (prefetched by TMA)
constexpr int kMaxProblems = 8;          // problems per launch
constexpr int kQueue = 4;                // unit queue of a Gram launch (slots)
constexpr int kOutBox = 32;              // epilogue boxes: 32 x 32 elements
constexpr int kEpiWarps = 4;

// ---- PTX wrappers ---------------------------------------------------------------

__device__ __forceinline__ uint32_t su32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void bar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void bar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void bar_expect(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
            bar),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool bar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long now_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase of the given parity; false if the block is aborting or
// the wait ran out (which starts the abort).
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         int32_t* status) {
    if (bar_test(bar, parity)) return true;
    const unsigned long long t0 = now_ns();
    while (!bar_test(bar, parity)) {
        if (*abort_flag) return false;
        if (now_ns() - t0 > kTcWaitLimitNs) {
            *abort_flag = 1;
            atomicOr(status, CAM_STATUS_GEMM_TIMEOUT);
            return false;
        }
    }
    return true;
}

// Three-dimensional tiled TMA load {x = K element, y = row, z = matrix}.
__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1,024 bytes apart (stride byte offset), leading byte offset unused (1),
// descriptor version 1 (bits 46-48), swizzle mode 2 = 128 B (bits 61-63).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
    return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (uint64_t(1) << 16) |
           (uint64_t(1024 >> 4) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// MN-major operand (M or N contiguous in memory, as TMA writes boxes of 128
// bytes of M (or N) by K rows under the 128-byte swizzle): 8-row groups along
// K 1,024 bytes apart (stride byte offset), and the next 128 bytes of M (or
// N) `lbo` bytes further (leading byte offset: one TMA box).
__device__ __forceinline__ uint64_t smem_desc_mn(uint32_t addr, uint32_t lbo) {
    return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (uint64_t(lbo >> 4) << 16) |
           (uint64_t(1024 >> 4) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// Instruction descriptor of kind::f16 (bf16 A and B) or kind::tf32: fp32
// accumulator (bits 4-5 = 1), A/B formats (bits 7-9, 10-12: bf16 = 1,
// tf32 = 2), K-major (bits 15, 16 = 0) or MN-major (1) operands, N >> 3
// (bits 17-22), M >> 4 (bits 24-28).
template <bool BF16, int BN, bool MNM>
__device__ __forceinline__ constexpr uint32_t instr_desc() {
    return (1u << 4) | ((BF16 ? 1u : 2u) << 7) | ((BF16 ? 1u : 2u) << 10) |
           (uint32_t(MNM ? 1 : 0) << 15) | (uint32_t(MNM ? 1 : 0) << 16) |
           (uint32_t(BN >> 3) << 17) | (uint32_t(kBM >> 4) << 24);
}

template <bool BF16>
__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                    uint32_t accumulate) {
    if constexpr (BF16)
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
            : "memory");
}

// Arrives on `bar` once every MMA this thread issued before has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Three-dimensional tiled TMA store of a shared-memory box, in this thread's
// bulk async-group.
__device__ __forceinline__ void tma_store(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(src), "r"(x), "r"(y), "r"(z)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Until at most one of this thread's groups still reads shared memory.
__device__ __forceinline__ void bulk_wait_read1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// Until every group of this thread has finished reading its source.
__device__ __forceinline__ void bulk_wait_read0() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Until every group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// Makes this thread's shared-memory writes visible to the TMA (async proxy).
__device__ __forceinline__ void fence_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- kernel arguments -------------------------------------------------------------

// One problem of a launch: a batch of equal-shape products with its own
// tensor maps. A launch runs up to kMaxProblems problems of one precision, one
// tile width and one epilogue kind, their units numbered one after another.
struct alignas(128) TcProblem {
    CUtensorMap ta;          // A: dims {K, M, batch}, box {K step, 128, 1}
    CUtensorMap tb;          // B: dims {K, N, batch}, box {K step, 128, 1}
    CUtensorMap ty;          // Y (or the Gram split partials): boxes of 32 x 32
    CUtensorMap tyt;         // Yt, or Y read transposed (Gram mirror): boxes of 32 x 32
    CUtensorMap tcm;         // C (kEpiAxpbyC): boxes of 32 x 32, swizzled as box_row
    const float* c;          // C (kEpiAxpbyC read directly, fp32): row stride ldc, matrix stride sc
    int64_t ldc, sc;
    int32_t batch;
    int32_t m_blocks;        // M / 128
    int32_t n_blocks;        // N / BN
    int32_t k_blocks;        // K / K step
    int32_t splits;          // Gram: K ranges per tile (> 1: fp32 partials)
    int32_t k_per_split;     // Gram: K steps per range
    int32_t n_tri;           // Gram: tiles per matrix reaching the upper triangle
    int32_t unit0;           // first unit of this problem in the launch
    int32_t has_y, has_yt;
};

struct alignas(128) TcArgs {
    TcProblem prob[kMaxProblems];
    int32_t n_problems;
    int32_t n_units;         // units of every problem
    float alpha, beta, diag;
    int32_t* status;
    // Gram launches: [0] the next unit to hand out, [1] blocks finished; both
    // 0 between launches (the last block to finish resets them)
    int32_t* sched;
};

// One unit of work: its problem, the tile's first rows in A and B, its
// matrix, its K steps and (Gram split) its range.
struct Unit {
    int p, b, rb, cb, split, k0, k1;
};

template <int BN, int EPI>
__device__ __forceinline__ Unit decode(const TcArgs& a, int u) {
    Unit t;
    int p = a.n_problems - 1;
    while (p > 0 && u < a.prob[p].unit0) --p;
    const TcProblem& P = a.prob[p];
    u -= P.unit0;
    t.p = p;
    if constexpr (EPI == kNtAxpby || EPI == kEpiAxpbyC) {
        const int per = P.m_blocks * P.n_blocks;
        t.b = u / per;
        const int rem = u - t.b * per;
        t.rb = rem / P.n_blocks;
        t.cb = rem - t.rb * P.n_blocks;
        t.split = 0;
        t.k0 = 0;
        t.k1 = P.k_blocks;
    } else {
        // ranges outermost: the units running at once share their K range
        const int per_split = P.n_tri * P.batch;
        t.split = u / per_split;
        int rem = u - t.split * per_split;
        t.b = rem / P.n_tri;
        int q = rem - t.b * P.n_tri;
        // column block cb holds row blocks 0 .. (BN cb + BN - 1) / 128
        int cb = 0;
        for (; cb < P.n_blocks - 1; ++cb) {
            const int cnt = min(P.m_blocks, (BN * cb + BN - 1) / kBM + 1);
            if (q < cnt) break;
            q -= cnt;
        }
        t.rb = q;
        t.cb = cb;
        t.k0 = t.split * P.k_per_split;
        t.k1 = min(P.k_blocks, t.k0 + P.k_per_split);
    }
    return t;
}

// ---- epilogue boxes ----------------------------------------------------------------

// One 32 x 32 box of results in shared memory, as the TMA store reads it.
// Row-major boxes (lane r writes its 32 values as row r): bf16 rows are 64
// bytes under the 64-byte swizzle (16-byte chunk q of row r at chunk
// q ^ ((r >> 1) & 3)), fp32 rows 128 bytes under the 128-byte swizzle (chunk
// q ^ (r & 7)), so a warp's 16-byte writes spread over all banks.
// Transposed boxes (value (r, c) at element c * 32 + r) are unswizzled: lane
// r's writes for one c are consecutive across the warp.
template <bool BF16OUT>
__device__ __forceinline__ void box_row(uint32_t buf, int r, const float* v) {
    if constexpr (BF16OUT) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(v[8 * q + 2 * e], v[8 * q + 2 * e + 1]);
                w[e] = *reinterpret_cast<const uint32_t*>(&h);
            }
            const uint32_t addr = buf + r * 64 + 16 * (q ^ ((r >> 1) & 3));
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]),
                         "r"(w[2]), "r"(w[3])
                         : "memory");
        }
    } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const uint32_t addr = buf + r * 128 + 16 * (q ^ (r & 7));
            asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v[4 * q]),
                         "f"(v[4 * q + 1]), "f"(v[4 * q + 2]), "f"(v[4 * q + 3])
                         : "memory");
        }
    }
}

// Row r of a row-major box as box_row lays it out (and TMA loads it).
template <bool BF16IN>
__device__ __forceinline__ void box_row_read(uint32_t buf, int r, float* v) {
    if constexpr (BF16IN) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t w[4];
            const uint32_t addr = buf + r * 64 + 16 * (q ^ ((r >> 1) & 3));
            asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                         : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                         : "r"(addr)
                         : "memory");
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                v[8 * q + 2 * e] = __uint_as_float(w[e] << 16);
                v[8 * q + 2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
            }
        }
    } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const uint32_t addr = buf + r * 128 + 16 * (q ^ (r & 7));
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(v[4 * q]), "=f"(v[4 * q + 1]), "=f"(v[4 * q + 2]), "=f"(v[4 * q + 3])
                         : "r"(addr)
                         : "memory");
        }
    }
}

template <bool BF16OUT>
__device__ __forceinline__ void box_col(uint32_t buf, int r, const float* v) {
#pragma unroll
    for (int c = 0; c < 32; ++c) {
        if constexpr (BF16OUT) {
            const __nv_bfloat16 h = __float2bfloat16_rn(v[c]);
            asm volatile("st.shared.b16 [%0], %1;" ::"r"(buf + (c * 32 + r) * 2),
                         "h"(*reinterpret_cast<const unsigned short*>(&h))
                         : "memory");
        } else {
            asm volatile("st.shared.f32 [%0], %1;" ::"r"(buf + (c * 32 + r) * 4), "f"(v[c]) : "memory");
        }
    }
}

// ---- the tensor-core kernel --------------------------------------------------------

template <bool BF16, int BN, int EPI, bool DC = false>
struct Geo {
    static constexpr int kBBytes = BN * kRowBytes;
    static constexpr int kStage = kBoxBytes + kBBytes;
    // epilogue staging: per warp kStgBufs buffers, each one box and its
    // transpose (a Gram split's fp32 partial box fits one buffer). bf16 boxes
    // are double-buffered; fp32 boxes, twice the bytes, single-buffered, which
    // leaves the TF32 ring four stages instead of three -- except for the
    // kEpiAxpbyC form that reads C through TMA (!DC, short K), which keeps
    // double buffers and one box of C per warp, prefetched a box ahead.
    static constexpr bool kTmaC = EPI == kEpiAxpbyC && !DC;
    static constexpr int kOutBytes = BF16 ? 2 : 4;
    static constexpr int kBox = kOutBox * kOutBox * kOutBytes;
    static constexpr int kStgBuf = 2 * kBox;
    static constexpr int kStgBufs = (BF16 || kTmaC) ? 2 : 1;
    static_assert(kStgBuf >= kOutBox * kOutBox * 4, "a partial box must fit a buffer");
    static constexpr int kCBox = kOutBox * kOutBox * (BF16 ? 2 : 4);
    static constexpr int kCRegion = kTmaC ? kEpiWarps * kCBox : 0;
    static constexpr int kStaging = kEpiWarps * kStgBufs * kStgBuf + kCRegion;
    static constexpr int kStagesFit = (kSmemBudget - kStaging) / kStage;
    static constexpr int kStages = kStagesFit < 8 ? kStagesFit : 8;
    static constexpr int kStgOffset = kStages * kStage;
    static constexpr int kBarOffset = kStgOffset + kStaging;
    // ring + staging + barriers (full, empty, tmem full, tmem empty, drain,
    // one "C full" per epilogue warp) + TMEM address + abort flag, plus 1 KB
    // to align the ring to 1,024 bytes
    static constexpr int kBars = 2 * kStages + 5 + kEpiWarps + 2 * kQueue;
    static constexpr int kSmem = kBarOffset + 8 * kBars + 16 + 4 * kQueue + 1024;
    static constexpr int kKStep = kRowBytes / (BF16 ? 2 : 4);  // elements per K step
    static_assert(kStages >= 2, "shared memory too small for the ring");
    static_assert(kSmem <= 232448, "over the per-block shared memory limit");
};

template <bool BF16, int BN, int EPI, bool MNM, bool DC = false>
__global__ void __launch_bounds__(kTcThreads, 1) nt_gemm_tc(const __grid_constant__ TcArgs a) {
    using G = Geo<BF16, BN, EPI, DC>;
    // MN-major operands: TMA boxes of 128 bytes of M (or N) by one K step of
    // rows; kMnBox bytes each, kMnCols elements of M (or N)
    constexpr int kMnCols = kRowBytes / (BF16 ? 2 : 4);
    constexpr int kMnBox = G::kKStep * kRowBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + G::kBarOffset);
    const uint32_t full0 = su32(bars);
    const uint32_t empty0 = full0 + 8 * G::kStages;
    const uint32_t tfull0 = empty0 + 8 * G::kStages;
    const uint32_t tempty0 = tfull0 + 16;
    const uint32_t drain = tempty0 + 16;
    const uint32_t cfull0 = drain + 8;
    const uint32_t qfull0 = cfull0 + 8 * kEpiWarps;  // unit queue (Gram launches)
    const uint32_t qempty0 = qfull0 + 8 * kQueue;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + G::kBars);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* qval = reinterpret_cast<volatile int*>(tmem_slot + 4);
    // Gram launches hand units out dynamically (their tiles' K ranges differ
    // from problem to problem); the others take u = block, block + grid, ...
    constexpr bool kDyn = EPI == kNtGram;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr uint32_t kCols = 2 * BN;  // two accumulators

    if (threadIdx.x == 0) {
        for (int s = 0; s < G::kStages; ++s) {
            bar_init(full0 + 8 * s, 1);
            bar_init(empty0 + 8 * s, 1);
        }
        for (int i = 0; i < 2; ++i) {
            bar_init(tfull0 + 8 * i, 1);
            bar_init(tempty0 + 8 * i, kEpiWarps);  // one arrival per epilogue warp
        }
        bar_init(drain, 1);
        for (int w = 0; w < kEpiWarps; ++w) bar_init(cfull0 + 8 * w, 1);
        for (int q = 0; q < kQueue; ++q) {
            bar_init(qfull0 + 8 * q, 1);
            bar_init(qempty0 + 8 * q, 1 + kEpiWarps);  // the MMA issuer and each epilogue warp
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         su32(tmem_slot)),
                     "r"(kCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // Launched as a programmatic dependent of the previous kernel on the
    // stream: everything above overlapped its tail; no global memory is
    // touched before it has completed. The next kernel may then start its
    // own set-up as soon as SMs free up.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0 && lane == 0) {
        // ---- producer ----
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued = 0;  // bit s: stage s has a fill whose phase is (filled_parity >> s) & 1
        uint32_t filled_parity = 0;
        int qslot = 0, iter = 0;
        uint32_t qphase = 0;
        for (;;) {
            int u;
            if constexpr (kDyn) {  // the next unit, published to the other roles
                if (*abort_flag) break;
                u = atomicAdd(a.sched, 1);
                if (u >= a.n_units) u = -1;
                if (!bar_wait(qempty0 + 8 * qslot, qphase ^ 1, abort_flag, a.status)) break;
                qval[qslot] = u;
                bar_arrive(qfull0 + 8 * qslot);
                if (++qslot == kQueue) {
                    qslot = 0;
                    qphase ^= 1;
                }
                if (u < 0) break;
            } else {
                u = blockIdx.x + iter++ * gridDim.x;
                if (u >= a.n_units || *abort_flag) break;
            }
            const Unit t = decode<BN, EPI>(a, u);
            const TcProblem& P = a.prob[t.p];
            const int arow = t.rb * kBM, brow = t.cb * BN;
            for (int kb = t.k0; kb < t.k1; ++kb) {
                if (!bar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, a.status)) break;
                const uint32_t sa = su32(smem + stage * G::kStage);
                const uint32_t fb = full0 + 8 * stage;
                bar_expect(fb, G::kStage);
                const int x = kb * G::kKStep;
                if constexpr (MNM) {  // boxes of kMnCols M (N) by one K step
#pragma unroll
                    for (int h = 0; h < kBM / kMnCols; ++h)
                        tma_load(sa + h * kMnBox, &P.ta, arow + h * kMnCols, x, t.b, fb);
#pragma unroll
                    for (int h = 0; h < BN / kMnCols; ++h)
                        tma_load(sa + kBoxBytes + h * kMnBox, &P.tb, brow + h * kMnCols, x, t.b, fb);
                } else {
                    tma_load(sa, &P.ta, x, arow, t.b, fb);
#pragma unroll
                    for (int h = 0; h < BN / kBM; ++h)
                        tma_load(sa + kBoxBytes + h * kBoxBytes, &P.tb, x, brow + h * kBM, t.b, fb);
                }
                issued |= 1u << stage;
                filled_parity = (filled_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == G::kStages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
        if constexpr (kDyn) {  // the last block out leaves the counters at 0
            if (!*abort_flag) {
                __threadfence();
                if (atomicAdd(a.sched + 1, 1) == int(gridDim.x) - 1) {
                    a.sched[0] = 0;
                    a.sched[1] = 0;
                    __threadfence();
                }
            }
        }
        if (*abort_flag) {  // let the copies in flight land before the block exits
            for (int s = 0; s < G::kStages; ++s)
                if ((issued >> s) & 1) {
                    const unsigned long long t0 = now_ns();
                    while (!bar_test(full0 + 8 * s, (filled_parity >> s) & 1))
                        if (now_ns() - t0 > kTcWaitLimitNs) break;
                }
        }
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer ----
        constexpr uint32_t idesc = instr_desc<BF16, BN, MNM>();
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        int qslot = 0, iter = 0;
        uint32_t qphase = 0;
        for (;;) {
            int u;
            if constexpr (kDyn) {
                if (!bar_wait(qfull0 + 8 * qslot, qphase, abort_flag, a.status)) break;
                u = qval[qslot];
                bar_arrive(qempty0 + 8 * qslot);
                if (++qslot == kQueue) {
                    qslot = 0;
                    qphase ^= 1;
                }
                if (u < 0) break;
            } else {
                u = blockIdx.x + iter++ * gridDim.x;
                if (u >= a.n_units) break;
            }
            const Unit t = decode<BN, EPI>(a, u);
            if (!bar_wait(tempty0 + 8 * acc, acc_phase ^ 1, abort_flag, a.status)) break;
            tc_fence_after();
            const uint32_t d = tmem + uint32_t(acc * BN);
            bool ok = true;
            for (int kb = t.k0; kb < t.k1; ++kb) {
                if (!bar_wait(full0 + 8 * stage, phase, abort_flag, a.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t sa = su32(smem + stage * G::kStage);
                // four MMAs of 32 bytes of K each: 32 bytes further along a
                // K-major row, or 32 bytes / element rows further down an
                // MN-major box
                constexpr uint32_t kAdv = MNM ? (32 / (BF16 ? 2 : 4)) * kRowBytes / 16 : 2;
                const uint64_t da = MNM ? smem_desc_mn(sa, kMnBox) : smem_desc(sa);
                const uint64_t db = MNM ? smem_desc_mn(sa + kBoxBytes, kMnBox) : smem_desc(sa + kBoxBytes);
#pragma unroll
                for (int k = 0; k < kRowBytes / 32; ++k)
                    mma<BF16>(d, da + uint64_t(kAdv * k), db + uint64_t(kAdv * k), idesc,
                              (kb > t.k0 || k > 0) ? 1u : 0u);
                mma_commit(empty0 + 8 * stage);
                if (++stage == G::kStages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok) break;
            mma_commit(tfull0 + 8 * acc);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
        if (*abort_flag) {  // every MMA issued so far completes before TMEM is freed
            mma_commit(drain);
            const unsigned long long t0 = now_ns();
            while (!bar_test(drain, 0))
                if (now_ns() - t0 > kTcWaitLimitNs) break;
        }
    } else if (warp >= 2) {
        // ---- epilogue ----
        const int quarter = warp & 3;  // TMEM lanes 32 quarter .. + 31: rows of the tile
        const uint32_t stg = su32(smem + G::kStgOffset + (warp - 2) * G::kStgBufs * G::kStgBuf);
        // kEpiAxpbyC through TMA (!DC): this warp's box of C, loaded one box ahead
        const uint32_t cbuf = su32(smem + G::kStgOffset + kEpiWarps * G::kStgBufs * G::kStgBuf +
                                   (warp - 2) * G::kCBox);
        const uint32_t cbar = cfull0 + 8 * (warp - 2);
        uint32_t c_phase = 0;
        bool c_pending = false;
        auto tma_c = [&](int u, int cc) {  // lane 0: the C box of unit u, column box cc
            const Unit n = decode<BN, EPI>(a, u);
            bar_expect(cbar, G::kCBox);
            tma_load(cbuf, &a.prob[n.p].tcm, n.cb * BN + cc * 32, n.rb * kBM + quarter * 32, n.b,
                     cbar);
        };
        if (G::kTmaC && lane == 0 && int(blockIdx.x) < a.n_units) {
            tma_c(blockIdx.x, 0);
            c_pending = true;
        }
        // kEpiAxpbyC read directly (DC, fp32 C, long K): this lane's row of the
        // next C box, 32 floats (one 128-byte line) from global memory a box
        // ahead, which frees the C boxes' shared memory for a fourth stage
        float cn[EPI == kEpiAxpbyC && DC ? 32 : 1];
        auto load_c = [&](int u, int cc) {
            if constexpr (EPI == kEpiAxpbyC && DC) {
                const Unit n = decode<BN, EPI>(a, u);
                const TcProblem& Q = a.prob[n.p];
                const float4* src = reinterpret_cast<const float4*>(
                    Q.c + n.b * Q.sc + int64_t(n.rb * kBM + quarter * 32 + lane) * Q.ldc +
                    n.cb * BN + cc * 32);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float4 x = __ldg(src + j);
                    cn[4 * j] = x.x;
                    cn[4 * j + 1] = x.y;
                    cn[4 * j + 2] = x.z;
                    cn[4 * j + 3] = x.w;
                }
            }
        };
        if (EPI == kEpiAxpbyC && DC && int(blockIdx.x) < a.n_units) load_c(blockIdx.x, 0);
        int acc = 0, buf = 0;
        uint32_t acc_phase = 0;
        int qslot = 0, iter = 0;
        uint32_t qphase = 0;
        for (;;) {
            int u;
            if constexpr (kDyn) {
                const bool okq = bar_wait(qfull0 + 8 * qslot, qphase, abort_flag, a.status);
                if (!__all_sync(0xffffffffu, okq)) break;
                u = qval[qslot];
                __syncwarp();
                if (lane == 0) bar_arrive(qempty0 + 8 * qslot);
                if (++qslot == kQueue) {
                    qslot = 0;
                    qphase ^= 1;
                }
                if (u < 0) break;
            } else {
                u = blockIdx.x + iter++ * gridDim.x;
                if (u >= a.n_units) break;
            }
            const Unit t = decode<BN, EPI>(a, u);
            const TcProblem& P = a.prob[t.p];
            // the whole warp leaves together: tcgen05.ld is warp-collective
            const bool ok = bar_wait(tfull0 + 8 * acc, acc_phase, abort_flag, a.status);
            if (!__all_sync(0xffffffffu, ok)) break;
            tc_fence_after();
            const int row0 = t.rb * kBM + quarter * 32;  // first row of this warp's boxes
            const uint32_t tbase = tmem + (uint32_t(quarter * 32) << 16) + uint32_t(acc * BN);
            // a Gram product split over K ranges writes fp32 partial boxes
            const bool part = EPI == kNtGram && P.splits > 1;
            const int z = part ? t.split * P.batch + t.b : t.b;
            bool aborted = false;
#pragma unroll 1
            for (int cc = 0; cc < BN / 32; ++cc) {
                float v[32];
                tmem_ld32(tbase + uint32_t(cc * 32), v);
                if (cc == BN / 32 - 1) {  // the accumulator is free for the next tile
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) bar_arrive(tempty0 + 8 * acc);
                }
                const int col0 = t.cb * BN + cc * 32;
                bool direct, mirror;
                if constexpr (EPI == kNtGram) {  // 32 x 32 boxes on / above the diagonal
                    direct = part || col0 >= row0;
                    mirror = !part && col0 > row0;
                } else {
                    direct = P.has_y != 0;
                    mirror = P.has_yt != 0;
                }
                if constexpr (EPI == kEpiAxpbyC) {
                    float c[32];
                    // the next box's C: this unit's next column box, or the
                    // first of the next unit this block takes (a static stride)
                    const int nu = cc + 1 < BN / 32 ? u : u + int(gridDim.x);
                    if constexpr (DC) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) c[i] = cn[i];
                        if (nu < a.n_units) load_c(nu, cc + 1 < BN / 32 ? cc + 1 : 0);
                    } else {
                        const bool cok = bar_wait(cbar, c_phase, abort_flag, a.status);
                        if (!__all_sync(0xffffffffu, cok)) {
                            aborted = true;
                            break;
                        }
                        c_phase ^= 1;
                        box_row_read<BF16>(cbuf, lane, c);
                        __syncwarp();  // every lane has read the box before it is refilled
                        c_pending = false;
                        if (lane == 0 && nu < a.n_units) {
                            tma_c(nu, cc + 1 < BN / 32 ? cc + 1 : 0);
                            c_pending = true;
                        }
                    }
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = fmaf(a.alpha, v[i], a.beta * c[i]);
                } else {
                    if (!part) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[i] *= a.alpha;
                    }
                }
                if (!direct && !mirror) continue;
                if (!part && col0 == row0) {  // this lane's diagonal element is column `lane`
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (i == lane) v[i] += a.diag;
                }
                // the buffer's store from kStgBufs boxes ago has finished reading it
                if (lane == 0) {
                    if constexpr (G::kStgBufs == 2) bulk_wait_read1();
                    else bulk_wait_read0();
                }
                __syncwarp();
                const uint32_t yb = stg + buf * G::kStgBuf;
                const uint32_t ytb = yb + G::kBox;
                if (part) {
                    box_row<false>(yb, lane, v);
                } else {
                    if (direct) box_row<BF16>(yb, lane, v);
                    if (mirror) box_col<BF16>(ytb, lane, v);
                }
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if (direct) tma_store(&P.ty, yb, col0, row0, z);
                    if (mirror) tma_store(&P.tyt, ytb, row0, col0, t.b);
                    bulk_commit();
                }
                if constexpr (G::kStgBufs == 2) buf ^= 1;
            }
            if (aborted) break;
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
        if (lane == 0) {
            if (c_pending) {  // a C box still in flight lands before the block exits
                const unsigned long long t0 = now_ns();
                while (!bar_test(cbar, c_phase))
                    if (now_ns() - t0 > kTcWaitLimitNs) break;
            }
            bulk_wait_all();  // stores done before the block (and its smem) goes
        }
        __syncwarp();
    }
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols)
                     : "memory");
    }
}

// Sums the split partials of Gram products in range order and writes
// Y = alpha sum + diag I, the whole symmetric matrix: element (i, j) takes the
// partials of (min, max), so both triangles carry the same bits. One block of
// 32 x 8 threads per 8-row quarter of a 32 x 32 tile on or above the diagonal
// (blockIdx.x: the tile, row by row, times four), one element per thread with
// its loads for several ranges in flight; the quarter is written, and
// mirrored, through shared memory.
template <typename T>
__global__ void __launch_bounds__(256) gram_reduce(const float* P, int splits, int batch,
                                                   int64_t M, float alpha, float diag, T* Y,
                                                   int64_t ldy, int64_t sY) {
    __shared__ float tile[8][33];
    const int b = blockIdx.y;
    // (tile, quarter) -> (ti, tj, rows 8 quarter .. + 7), tj >= ti
    const int64_t nt = M / 32;
    const int quarter = blockIdx.x & 3;
    int64_t q = blockIdx.x >> 2, ti = 0;
    while (q >= nt - ti) {
        q -= nt - ti;
        ++ti;
    }
    const int64_t tj = ti + q;
    const int tx = threadIdx.x, ty = threadIdx.y;  // 32 x 8
    const int64_t i = ti * 32 + quarter * 8 + ty, j = tj * 32 + tx;
    const int64_t split_stride = int64_t(batch) * M * M;
    // diagonal tile: the upper element of the pair
    const float* p = P + int64_t(b) * M * M + (j >= i ? i * M + j : j * M + i);
    float acc = 0.0f;
#pragma unroll 8
    for (int r = 0; r < splits; ++r) acc += p[r * split_stride];  // range order
    tile[ty][tx] = alpha * acc + (i == j ? diag : 0.0f);
    __syncthreads();
    T* y = Y + b * sY;
    y[i * ldy + j] = T(tile[ty][tx]);
    if (tj > ti) {  // the mirror: rows tj*32 + c, columns ti*32 + 8 quarter + r
        const int lin = ty * 32 + tx, c = lin >> 3, r = lin & 7;
        y[(tj * 32 + c) * ldy + ti * 32 + quarter * 8 + r] = T(tile[r][c]);
    }
}

// ---- the CUDA-core fp32 kernel -------------------------------------------------------

constexpr int kSimtThreads = 256;
constexpr int kSimtBK = 8;

struct SimtArgs {
    const float* A; int64_t lda, sA;
    const float* B; int64_t ldb, sB;
    int64_t K;
    int64_t k_len;      // K elements per range (blockIdx.z), a multiple of 8
    int32_t n_blocks;   // N / 128
    float alpha, beta, diag;
    const float* C; int64_t ldc, sC;
    float* Y; int64_t ldy, sY;
    float* Yt; int64_t ldyt, sYt;
    // split K: each range's raw sums, [range][matrix][M][N]; null: no split
    float* part; int64_t M, N;
};

// One 128 x 128 tile per block (blockIdx.x: tile, blockIdx.y: matrix,
// blockIdx.z: K range); thread (tx, ty) of a 16 x 16 grid owns rows
// ty*8 .. +7 and columns tx*4 .. +3 and 64 + tx*4 .. +3. K steps of 8, staged
// in shared memory with K outermost.
__global__ void __launch_bounds__(kSimtThreads) nt_gemm_simt(const __grid_constant__ SimtArgs a) {
    __shared__ __align__(16) float As[kSimtBK][128];
    __shared__ __align__(16) float Bs[kSimtBK][128];
    const int b = blockIdx.y;
    const int mb = blockIdx.x / a.n_blocks, nb = blockIdx.x % a.n_blocks;
    const float* A = a.A + b * a.sA + int64_t(mb) * 128 * a.lda;
    const float* B = a.B + b * a.sB + int64_t(nb) * 128 * a.ldb;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    // loads: thread t reads row t/2, K elements 4 (t%2) .. +3 of A and of B
    const int lr = tid >> 1, lk = (tid & 1) * 4;
    float acc[8][8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[i][j] = 0.0f;
    const int64_t k_begin = int64_t(blockIdx.z) * a.k_len;
    const int64_t k_end = k_begin + a.k_len < a.K ? k_begin + a.k_len : a.K;
    for (int64_t k0 = k_begin; k0 < k_end; k0 += kSimtBK) {
        const float4 av = *reinterpret_cast<const float4*>(A + lr * a.lda + k0 + lk);
        const float4 bv = *reinterpret_cast<const float4*>(B + lr * a.ldb + k0 + lk);
        __syncthreads();
        As[lk][lr] = av.x;
        As[lk + 1][lr] = av.y;
        As[lk + 2][lr] = av.z;
        As[lk + 3][lr] = av.w;
        Bs[lk][lr] = bv.x;
        Bs[lk + 1][lr] = bv.y;
        Bs[lk + 2][lr] = bv.z;
        Bs[lk + 3][lr] = bv.w;
        __syncthreads();
#pragma unroll
        for (int k = 0; k < kSimtBK; ++k) {
            const float4 a0 = *reinterpret_cast<const float4*>(&As[k][ty * 8]);
            const float4 a1 = *reinterpret_cast<const float4*>(&As[k][ty * 8 + 4]);
            const float4 b0 = *reinterpret_cast<const float4*>(&Bs[k][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4*>(&Bs[k][64 + tx * 4]);
            const float ar[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float br[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(ar[i], br[j], acc[i][j]);
        }
    }
    if (a.part) {  // a range's raw sums
        float* part = a.part + (int64_t(blockIdx.z) * gridDim.y + b) * a.M * a.N;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t row = int64_t(mb) * 128 + ty * 8 + i;
#pragma unroll
            for (int h = 0; h < 2; ++h)
                *reinterpret_cast<float4*>(part + row * a.N + int64_t(nb) * 128 + h * 64 + tx * 4) =
                    make_float4(acc[i][4 * h], acc[i][4 * h + 1], acc[i][4 * h + 2], acc[i][4 * h + 3]);
        }
        return;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int64_t row = int64_t(mb) * 128 + ty * 8 + i;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int64_t col = int64_t(nb) * 128 + h * 64 + tx * 4;
            float v[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = acc[i][4 * h + j];
            if (a.beta != 0.0f) {
                const float4 c = *reinterpret_cast<const float4*>(a.C + b * a.sC + row * a.ldc + col);
                const float cv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] = fmaf(a.alpha, v[j], a.beta * cv[j]);
            } else if (a.alpha != 1.0f) {
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] *= a.alpha;
            }
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (row == col + j) v[j] += a.diag;
            if (a.Y)
                *reinterpret_cast<float4*>(a.Y + b * a.sY + row * a.ldy + col) =
                    make_float4(v[0], v[1], v[2], v[3]);
            if (a.Yt)
#pragma unroll
                for (int j = 0; j < 4; ++j) a.Yt[b * a.sYt + (col + j) * a.ldyt + row] = v[j];
        }
    }
}

// The split CUDA-core product's epilogue: Y = alpha (sum of the ranges, in
// range order) + beta C + diag I, four elements per thread.
__global__ void simt_reduce(const __grid_constant__ SimtArgs a, int splits) {
    const int64_t quads = a.M * a.N / 4, per = int64_t(gridDim.y) * a.M * a.N;
    const int b = blockIdx.y;
    for (int64_t q = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; q < quads;
         q += int64_t(gridDim.x) * blockDim.x) {
        const int64_t row = 4 * q / a.N, col = 4 * q % a.N;
        const float* p = a.part + int64_t(b) * a.M * a.N + 4 * q;
        float4 t = *reinterpret_cast<const float4*>(p);
        for (int r = 1; r < splits; ++r) {
            const float4 u = *reinterpret_cast<const float4*>(p + r * per);
            t.x += u.x;
            t.y += u.y;
            t.z += u.z;
            t.w += u.w;
        }
        float v[4] = {t.x, t.y, t.z, t.w};
        if (a.beta != 0.0f) {
            const float4 c = *reinterpret_cast<const float4*>(a.C + b * a.sC + row * a.ldc + col);
            const float cv[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] = fmaf(a.alpha, v[j], a.beta * cv[j]);
        } else if (a.alpha != 1.0f) {
#pragma unroll
            for (int j = 0; j < 4; ++j) v[j] *= a.alpha;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (row == col + j) v[j] += a.diag;
        *reinterpret_cast<float4*>(a.Y + b * a.sY + row * a.ldy + col) =
            make_float4(v[0], v[1], v[2], v[3]);
    }
}

// ---- host side ---------------------------------------------------------------------

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        else
            cudaGetLastError();
    });
    return g_encode;
}

// Tensor map over `batch` row-major matrices of `rows` x `cols` elements
// (row stride ld, matrix stride sm, in elements), with boxes of
// box_cols x box_rows elements; zero fill outside.
int make_map(CUtensorMap* map, int64_t eb, const void* base, int64_t cols, int64_t rows,
             int64_t batch, int64_t ld, int64_t sm, int box_cols, int box_rows,
             CUtensorMapSwizzle swz) {
    const auto enc = encoder();
    if (!enc) return record_error(CAM_E_CUDA, "orthogonalisation: cuTensorMapEncodeTiled unavailable");
    const cuuint64_t dims[3] = {cuuint64_t(cols), cuuint64_t(rows), cuuint64_t(batch)};
    const cuuint64_t strides[2] = {cuuint64_t(ld * eb), cuuint64_t(sm * eb)};
    const cuuint32_t box[3] = {cuuint32_t(box_cols), cuuint32_t(box_rows), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r =
        enc(map, eb == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return record_error(CAM_E_CUDA, "orthogonalisation: cuTensorMapEncodeTiled failed (%d)",
                            static_cast<int>(r));
    return CAM_OK;
}

// Operand map: boxes of one K step (128 bytes) x 128 rows, 128-byte swizzle.
int operand_map(CUtensorMap* map, int64_t eb, const void* base, int64_t k, int64_t rows,
                int64_t batch, int64_t ld, int64_t sm) {
    return make_map(map, eb, base, k, rows, batch, ld, sm, static_cast<int>(kRowBytes / eb), kBM,
                    CU_TENSOR_MAP_SWIZZLE_128B);
}

// Output maps: 32 x 32 boxes; row-major boxes swizzled as box_row writes
// them, transposed boxes plain.
int out_map(CUtensorMap* map, int64_t eb, const void* base, int64_t cols, int64_t rows,
            int64_t batch, int64_t ld, int64_t sm, bool row_box) {
    const CUtensorMapSwizzle swz = !row_box ? CU_TENSOR_MAP_SWIZZLE_NONE
                                   : eb == 2 ? CU_TENSOR_MAP_SWIZZLE_64B
                                             : CU_TENSOR_MAP_SWIZZLE_128B;
    return make_map(map, eb, base, cols, rows, batch, ld, sm, kOutBox, kOutBox, swz);
}

// Launched as a programmatic dependent of the previous kernel on the stream
// (the kernel waits in griddepcontrol.wait before touching global memory).
template <bool BF16, int BN, int EPI, bool MNM = false, bool DC = false>
cudaError_t launch_tc(const TcArgs& a, int grid, cudaStream_t s) {
    using G = Geo<BF16, BN, EPI, DC>;
    static cudaError_t attr = cudaFuncSetAttribute(
        nt_gemm_tc<BF16, BN, EPI, MNM, DC>, cudaFuncAttributeMaxDynamicSharedMemorySize, G::kSmem);
    if (attr != cudaSuccess) return attr;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = G::kSmem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, nt_gemm_tc<BF16, BN, EPI, MNM, DC>, a);
}

template <bool BF16, int BN>
cudaError_t launch_tc_epi(const TcArgs& a, int epi, bool mn, bool dc, int grid, cudaStream_t s) {
    switch (epi) {
        case kNtAxpby: return launch_tc<BF16, BN, kNtAxpby>(a, grid, s);
        case kNtGram:
            return mn ? launch_tc<BF16, BN, kNtGram, true>(a, grid, s)
                      : launch_tc<BF16, BN, kNtGram>(a, grid, s);
        default:  // (C is fp32: TF32 products only, checked on the host)
            if constexpr (BF16) return cudaErrorInvalidValue;
            else return dc ? launch_tc<BF16, BN, kEpiAxpbyC, false, true>(a, grid, s)
                           : launch_tc<BF16, BN, kEpiAxpbyC>(a, grid, s);
    }
}

template <bool BF16>
cudaError_t launch_tc_any(const TcArgs& a, int bn, int epi, bool mn, bool dc, int grid,
                          cudaStream_t s) {
    return bn == 256 ? launch_tc_epi<BF16, 256>(a, epi, mn, dc, grid, s)
                     : launch_tc_epi<BF16, 128>(a, epi, mn, dc, grid, s);
}

int launch_fail(cudaError_t e) {
    return record_error(CAM_E_CUDA, "orthogonalisation: GEMM launch: %s", cudaGetErrorString(e));
}

// CUDA-core product; K split into ranges (summed by simt_reduce) when the
// tiles alone would leave most SMs idle, each range at least 128 long, within
// the partial buffer, and only for a row-major result.
int run_simt(const NtGemm& g, int sm_count, cudaStream_t s, int64_t* launches) {
    SimtArgs a;
    a.A = static_cast<const float*>(g.A);
    a.lda = g.lda;
    a.sA = g.sA;
    a.B = static_cast<const float*>(g.B);
    a.ldb = g.ldb;
    a.sB = g.sB;
    a.K = g.K;
    a.n_blocks = static_cast<int32_t>(g.N / 128);
    const bool gram = g.epilogue == kNtGram;
    a.alpha = g.alpha;
    a.beta = gram ? 0.0f : g.beta;
    a.diag = g.diag;
    a.C = static_cast<const float*>(g.C);
    a.ldc = g.ldc;
    a.sC = g.sC;
    a.Y = static_cast<float*>(g.Y);
    a.ldy = g.ldy;
    a.sY = g.sY;
    a.Yt = gram ? nullptr : static_cast<float*>(g.Yt);
    a.ldyt = g.ldyt;
    a.sYt = g.sYt;
    a.M = g.M;
    a.N = g.N;
    a.part = nullptr;
    const int64_t tiles = (g.M / 128) * (g.N / 128) * g.batch;
    int64_t splits = 1;
    if (g.partials && g.Y && !a.Yt) {
        const int64_t want = (2 * int64_t(sm_count) + tiles - 1) / tiles;
        const int64_t by_k = g.K / 128;
        const int64_t by_mem = g.partial_floats / (int64_t(g.batch) * g.M * g.N);
        splits = std::max<int64_t>(1, std::min(std::min(want, by_k), std::min<int64_t>(by_mem, 65535)));
    }
    // ranges of whole 128-element steps; no empty range
    a.k_len = ((g.K / 128 + splits - 1) / splits) * 128;
    splits = (g.K + a.k_len - 1) / a.k_len;
    if (splits > 1) a.part = g.partials;
    const dim3 grid(static_cast<unsigned>((g.M / 128) * (g.N / 128)), static_cast<unsigned>(g.batch),
                    static_cast<unsigned>(splits));
    nt_gemm_simt<<<grid, kSimtThreads, 0, s>>>(a);
    ++*launches;
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess && splits > 1) {
        const int64_t quads = g.M * g.N / 4;
        const unsigned rb = static_cast<unsigned>(std::min<int64_t>((quads + 255) / 256, 1024));
        simt_reduce<<<dim3(rb, static_cast<unsigned>(g.batch)), 256, 0, s>>>(a, static_cast<int>(splits));
        ++*launches;
        e = cudaGetLastError();
    }
    return e == cudaSuccess ? CAM_OK : launch_fail(e);
}

}  // namespace tc

int nt_gemm(const NtGemm* gs, int n, int sm_count, int32_t* status, cudaStream_t s,
            int64_t* launches) {
    using namespace tc;
    if (n < 1 || n > kMaxProblems)
        return record_error(CAM_E_ARG, "orthogonalisation: 1 to %d problems per GEMM launch",
                            kMaxProblems);
    const NtGemm& g0 = gs[0];
    bool all256 = true;
    for (int i = 0; i < n; ++i) {
        const NtGemm& g = gs[i];
        if (g.M % 128 || g.N % 128 || g.K % 128 || g.batch < 1)
            return record_error(CAM_E_ARG, "orthogonalisation: GEMM extents must be multiples of 128");
        if (g.precision != g0.precision || g.epilogue != g0.epilogue || g.alpha != g0.alpha ||
            g.beta != g0.beta || g.diag != g0.diag || (g.beta != 0.0f && !g.C))
            return record_error(CAM_E_ARG, "orthogonalisation: problems of one launch must agree");
        if (g.epilogue == kNtGram && (g.M != g.N || g.A != g.B))
            return record_error(CAM_E_ARG, "orthogonalisation: a Gram product takes one operand");
        if (g.mn_major != g0.mn_major ||
            (g.mn_major && (g.epilogue != kNtGram || g.precision != CAM_ORTHO_BF16)))
            return record_error(CAM_E_ARG,
                                "orthogonalisation: MN-major operands serve bf16 Gram products");
        all256 = all256 && g.N % 256 == 0;
    }
    if (g0.precision == CAM_ORTHO_BF16 && g0.beta != 0.0f)
        return record_error(CAM_E_ARG, "orthogonalisation: a bf16 product takes no C term");
    if (g0.precision == CAM_ORTHO_FP32) {
        for (int i = 0; i < n; ++i) {
            const int rc = run_simt(gs[i], sm_count, s, launches);
            if (rc != CAM_OK) return rc;
        }
        return CAM_OK;
    }
    const bool bf16 = g0.precision == CAM_ORTHO_BF16;
    const int64_t eb = bf16 ? 2 : 4;
    const int bn = all256 ? 256 : 128;
    const int64_t kstep = kRowBytes / eb;
    const bool gram = g0.epilogue == kNtGram;
    const bool mn = g0.mn_major;
    const int epi = gram ? kNtGram : (g0.beta != 0.0f ? kEpiAxpbyC : kNtAxpby);
    TcArgs a;
    std::memset(&a, 0, sizeof a);
    a.n_problems = n;
    a.alpha = g0.alpha;
    a.beta = g0.beta;
    a.diag = g0.diag;
    a.status = status;
    // Per problem (caller's order): tile counts and K steps; for Gram
    // products the tiles reaching the upper triangle and a K split for long
    // tiles, so that no unit is longer than one block's share of the launch
    // (ranges of at least 16 K steps, within the partial buffer; each range
    // costs a pass over the matrix in partials).
    int64_t work = 0;
    int n_blk[kMaxProblems], m_blk[kMaxProblems], k_blk[kMaxProblems], tri[kMaxProblems];
    for (int i = 0; i < n; ++i) {
        const NtGemm& g = gs[i];
        m_blk[i] = static_cast<int>(g.M / kBM);
        n_blk[i] = static_cast<int>(g.N / bn);
        k_blk[i] = static_cast<int>(g.K / kstep);
        tri[i] = 0;
        if (gram) {
            for (int cb = 0; cb < n_blk[i]; ++cb) tri[i] += std::min(m_blk[i], (bn * cb + bn - 1) / kBM + 1);
            work += int64_t(tri[i]) * g.batch * k_blk[i];
        } else {
            work += int64_t(m_blk[i]) * n_blk[i] * g.batch * k_blk[i];
        }
    }
    const int64_t longest = std::max<int64_t>(16, work / int64_t(sm_count));
    int splits[kMaxProblems], kps[kMaxProblems], ord[kMaxProblems];
    int64_t part_need = 0;
    for (int i = 0; i < n; ++i) {
        const NtGemm& g = gs[i];
        int sp = 1;
        if (gram && k_blk[i] > longest && g.partials) {
            const int64_t want = (k_blk[i] + longest - 1) / longest;
            const int64_t by_mem = (g.partial_floats - part_need) / (int64_t(g.batch) * g.M * g.M);
            sp = static_cast<int>(std::max<int64_t>(1, std::min(want, by_mem)));
        }
        kps[i] = (k_blk[i] + sp - 1) / sp;
        splits[i] = (k_blk[i] + kps[i] - 1) / kps[i];  // no empty range
        if (splits[i] > 1) part_need += int64_t(splits[i]) * g.batch * g.M * g.M;
        ord[i] = i;
    }
    // Gram launches hand their units out longest first: problems ordered by
    // the K steps of one unit
    if (gram)
        std::stable_sort(ord, ord + n, [&](int x, int y) { return kps[x] > kps[y]; });
    if (gram && !g0.sched)
        return record_error(CAM_E_ARG, "orthogonalisation: a Gram launch needs its unit counter");
    a.sched = g0.sched;
    int64_t part_used = 0;
    int32_t units = 0;
    for (int j = 0; j < n; ++j) {
        const int i = ord[j];
        TcProblem& P = a.prob[j];
        const NtGemm& g = gs[i];
        P.batch = g.batch;
        P.m_blocks = m_blk[i];
        P.n_blocks = n_blk[i];
        P.k_blocks = k_blk[i];
        P.n_tri = tri[i];
        P.splits = splits[i];
        P.k_per_split = kps[i];
        int rc;
        if (mn) {  // A stored K x M, B stored K x N: boxes of 128 bytes of M (N) by one K step
            rc = make_map(&P.ta, eb, g.A, g.M, g.K, g.batch, g.lda, g.sA,
                          static_cast<int>(kRowBytes / eb), static_cast<int>(kstep),
                          CU_TENSOR_MAP_SWIZZLE_128B);
            if (rc == CAM_OK)
                rc = make_map(&P.tb, eb, g.B, g.N, g.K, g.batch, g.ldb, g.sB,
                              static_cast<int>(kRowBytes / eb), static_cast<int>(kstep),
                              CU_TENSOR_MAP_SWIZZLE_128B);
        } else {
            rc = operand_map(&P.ta, eb, g.A, g.K, g.M, g.batch, g.lda, g.sA);
            if (rc == CAM_OK) rc = operand_map(&P.tb, eb, g.B, g.K, g.N, g.batch, g.ldb, g.sB);
        }
        if (rc != CAM_OK) return rc;
        P.unit0 = units;
        if (gram) {
            if (P.splits > 1) {
                float* part = g.partials + part_used;
                part_used += int64_t(P.splits) * g.batch * g.M * g.M;
                rc = out_map(&P.ty, 4, part, g.M, g.M, int64_t(P.splits) * g.batch, g.M, g.M * g.M,
                             true);
            } else {
                rc = out_map(&P.ty, eb, g.Y, g.N, g.M, g.batch, g.ldy, g.sY, true);
                if (rc == CAM_OK)  // the mirror: the same matrix, boxes written transposed
                    rc = out_map(&P.tyt, eb, g.Y, g.M, g.N, g.batch, g.ldy, g.sY, false);
            }
            units += P.n_tri * g.batch * P.splits;
        } else {
            P.has_y = g.Y != nullptr;
            P.has_yt = g.Yt != nullptr;
            if (P.has_y) rc = out_map(&P.ty, eb, g.Y, g.N, g.M, g.batch, g.ldy, g.sY, true);
            if (rc == CAM_OK && P.has_yt)
                rc = out_map(&P.tyt, eb, g.Yt, g.M, g.N, g.batch, g.ldyt, g.sYt, false);
            if (rc == CAM_OK && epi == kEpiAxpbyC) {  // C: in boxes like the row-major output, or directly
                rc = out_map(&P.tcm, eb, g.C, g.N, g.M, g.batch, g.ldc, g.sC, true);
                P.c = static_cast<const float*>(g.C);
                P.ldc = g.ldc;
                P.sc = g.sC;
            }
            units += P.m_blocks * P.n_blocks * g.batch;
        }
        if (rc != CAM_OK) return rc;
    }
    a.n_units = units;
    const int grid = std::min(units, sm_count);
    // the C term read directly, with a fourth ring stage, when every
    // product's K loop is long enough (1,024 or more) to hide the epilogue's
    // slower C reads; TMA boxes of C otherwise (measured: the 2,048-wide list
    // 6 % faster direct, the 512-wide stand 8 % slower)
    bool dc = true;
    for (int i = 0; i < n; ++i) dc = dc && gs[i].K >= 1024;
    const cudaError_t e = bf16 ? launch_tc_any<true>(a, bn, epi, mn, dc, grid, s)
                               : launch_tc_any<false>(a, bn, epi, mn, dc, grid, s);
    ++*launches;
    if (e != cudaSuccess) return launch_fail(e);
    // the split Gram products' partials, summed in range order
    int64_t part_off = 0;
    for (int j = 0; gram && j < n; ++j) {
        const TcProblem& P = a.prob[j];
        const NtGemm& g = gs[ord[j]];
        if (P.splits <= 1) continue;
        const float* part = g.partials + part_off;
        part_off += int64_t(P.splits) * g.batch * g.M * g.M;
        const int64_t nt = g.M / 32;  // tiles on or above the diagonal, per matrix
        const dim3 rgrid(static_cast<unsigned>(4 * nt * (nt + 1) / 2), static_cast<unsigned>(g.batch));
        if (bf16)
            gram_reduce<__nv_bfloat16><<<rgrid, dim3(32, 8), 0, s>>>(
                part, P.splits, g.batch, g.M, g.alpha, g.diag, static_cast<__nv_bfloat16*>(g.Y),
                g.ldy, g.sY);
        else
            gram_reduce<float><<<rgrid, dim3(32, 8), 0, s>>>(part, P.splits, g.batch, g.M, g.alpha,
                                                             g.diag, static_cast<float*>(g.Y), g.ldy,
                                                             g.sY);
        ++*launches;
        const cudaError_t r = cudaGetLastError();
        if (r != cudaSuccess) return launch_fail(r);
    }
    return CAM_OK;
}

}  // namespace cam
