// runtime.cu -- host side of libcam: contexts, fragment plans, the round state
// machine, argument validation and kernel launches (C ABI in include/cam.h).
//
// A context owns, per fragment (and once for "all tensors"), a plan: the
// fragment's tensors in order, its element space cut into chunks that never
// straddle a tensor, and small device tables (chunk list, state pointers,
// per-chunk drift partials). Chunk sizes are chosen per fragment from the
// device's SM count so that even a small fragment spreads over every SM.
//
// Rounds follow the merger described on the pages: a round collects the
// round's checkpoints as they arrive, closes once a quorum has arrived
// ("Pythia-14M on four rented GPUs and a bucket", "Getting updates through the
// bucket": quorum_size=3; "DiffuRefill-1B" technical report, section 3,
// Table 2, "Merger": wait for N fresh checkpoints of the current round tag),
// and round numbers only grow (same report, section 3, "Failure handling"
// (iii): a rollback is republished under a new round number). Accumulate only
// records the borrowed pointers; the commit runs the whole round as one fused
// pass, which visits every element's workers in the same arrival order as an
// eager fold would, so the result is the same bits.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <memory>
#include <new>
#include <string>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "cam_internal.h"
#include "side_internal.h"

#define CAM_API extern "C" __attribute__((visibility("default")))

using cam::ChunkDesc;
using cam::MergeArgs;
using cam::NormArgs;
using cam::TensorSlot;

namespace {

thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(CAM_E_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

// Makes `dev` current for the scope of one call and restores the caller's.
struct DeviceScope {
    int prev = -1;
    cudaError_t err = cudaSuccess;
    explicit DeviceScope(int dev) {
        err = cudaGetDevice(&prev);
        if (err == cudaSuccess && prev != dev) err = cudaSetDevice(dev);
    }
    ~DeviceScope() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// An NVTX range for profilers (a no-op unless a tool is attached).
struct NvtxRange {
    explicit NvtxRange(const char* label) { nvtxRangePushA(label); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace

int cam::record_error(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

struct Plan {
    std::vector<int32_t> tensors;      // global tensor ids, fragment order
    std::vector<int32_t> first_chunk;  // [T_f + 1]
    std::vector<ChunkDesc> chunks;     // host copy of the chunk list
    int64_t n_elems = 0;
    int32_t chunk_elems = 0;
    ChunkDesc* d_chunks = nullptr;
    TensorSlot* d_slots = nullptr;
    int32_t* d_first = nullptr;
    double* d_partials = nullptr;
    double* d_tsq = nullptr;
    double* d_worker_partials = nullptr;  // [n_chunks * CAM_KMAX]
    double* d_worker_tsq = nullptr;       // [n_tensors * CAM_KMAX]
    unsigned int* d_fin_counter = nullptr;  // blocks done, for a pass that finishes its norms
    int32_t n_chunks() const { return static_cast<int32_t>(chunks.size()); }
    int32_t n_tensors() const { return static_cast<int32_t>(tensors.size()); }
};

struct cam_round;

struct cam_ctx {
    int device = 0;
    int sm_count = 0;
    int32_t n_tensors = 0;
    int32_t n_fragments = 1;
    int32_t quorum = 1;
    std::vector<int64_t> numel;
    std::vector<int32_t> fragment_of;
    std::vector<float*> theta, m, e, swa;
    bool has_m = false, has_e = false, has_swa = false;
    std::vector<int64_t> swa_count;  // globals folded into each tensor's running average
    std::vector<int64_t> rows;       // matrix rows of each tensor (0: not a matrix)
    cam::OrthoWork* ortho = nullptr; // made at the first orthogonalised commit
    int64_t ortho_cap_elems = 0, ortho_cap_gram = 0;  // workspace sizing (padded elements)
    int64_t ortho_big_gram = 0;
    bool is_matrix(int32_t g) const {
        return rows[g] >= 2 && numel[g] % rows[g] == 0 && numel[g] / rows[g] >= 2;
    }
    bool pageable_access = false;  // the GPU reads pageable host memory directly
    bool staged = true;            // the staged form of the merge pass may be used
    bool test_stall = false;       // CAM_TEST_STALL_STAGED
    bool test_tag = false;         // CAM_TEST_BAD_TAG
    bool share_sms = false;        // CAM_SHARE_SMS: register form, at most 3/4 of its block slots
    bool time_commits = false;     // CAM_TIME_COMMITS: events around each commit
    cudaEvent_t commit_ev[2] = {nullptr, nullptr};
    cam_commit_record last_commit{};
    bool has_last_commit = false;
    bool last_commit_timed = false;  // its events were recorded (not inside a graph capture)
    // Running sums of eagerly folded rounds (cam_merge_fold): one fp32 buffer
    // over every tensor, made at the first fold. Open rounds cover disjoint
    // tensors, so they share it.
    float* d_sum = nullptr;
    std::vector<int64_t> sum_off;     // each tensor's offset in d_sum (8-element aligned)
    // Per plan: the last device work (fold, commit, reset) on its tensors.
    // Work on a plan waits for the events of every plan that shares tensors
    // with it, so rounds on overlapping tensors run in call order whatever
    // streams they are given, while rounds on disjoint fragments overlap.
    std::vector<cudaEvent_t> plan_ev;
    cudaEvent_t ortho_ev = nullptr;  // the last use of the orthogonalisation workspace
    int32_t* d_status = nullptr;   // device status word (CAM_STATUS_* bits), in dev_block
    std::vector<Plan> plans;  // [n_fragments] then "all"
    void* dev_block = nullptr;
    int64_t last_round = -1;
    int64_t launches = 0;
    int64_t staged_launches = 0;  // merge passes in the staged form
    std::vector<cam_round*> open;
    // resident blocks per SM: [dtype][mode][ema][norm level][publish][swa]
    int bps[2][2][2][3][2][2] = {};
    int bps_fin[2][2][2][2][2] = {};  // the same for norm level 1 with the finish fused
    bool fuse_finish = true;           // small rounds with norms finish them in the merge pass
    std::unique_ptr<MergeArgs> args;  // parameter block staging (copied at launch)
    std::unique_ptr<cam::MultiArgs> multi_args;  // the same for cam_merge_commit_many
    int bps_multi[2][2][2][2][2] = {};  // multi-round pass: [dtype][mode][ema][norms][publish]

    Plan& plan_of(int32_t fragment) { return plans[fragment < 0 ? n_fragments : fragment]; }
    const Plan& plan_of(int32_t fragment) const {
        return plans[fragment < 0 ? n_fragments : fragment];
    }
};

struct cam_round {
    cam_ctx* ctx = nullptr;
    int64_t round = 0;
    int32_t fragment = -1;
    int K = 0;
    int dtype = -1;
    std::vector<const void*> x;  // x[k * T_f + l]
    bool host_workers = false;   // some worker came through cam_merge_accumulate_host
    bool eager = false;          // workers are folded as they arrive (cam_merge_fold)
    int eager_mode = 0;          // the mode those folds used
    int n_folded = 0;            // workers folded so far; later ones are accumulated and
                                 // folded by the commit's final pass (x[(k - n_folded) * T_f + l])
    int64_t tokens[CAM_KMAX] = {};
    bool finalized = false;
    int mode = CAM_MODE_MEAN_REPLACE;
    float lr = 1.0f, mu = 0.0f;
    bool ema = false;
    float beta = 0.0f;
    bool norms = false;
    double* out_tensor = nullptr;
    double* out_fragment = nullptr;
    bool worker_norms = false;
    double* out_worker_tensor = nullptr;
    double* out_worker = nullptr;
    bool swa = false;
    bool publish = false;
    bool publish_ema = false;
    bool ortho = false;
    float ortho_lr = 0.0f;
    int ortho_scale = 0, ortho_precision = 0, ortho_iterations = 0;
    std::vector<void*> pub_theta, pub_ema;  // [T_f] device-visible addresses
};

namespace {

// Elements per chunk for a fragment of n elements: aim at >= 8 chunks per SM,
// within [one block-step, kMaxChunkElems], always a whole number of block-steps.
int32_t choose_chunk(int64_t n, int sm_count) {
    const int64_t q = cam::kChunkQuantum;
    const int64_t target = std::max<int64_t>(1, int64_t(sm_count) * 8);
    int64_t c = (n + target - 1) / target;
    c = ((c + q - 1) / q) * q;
    return static_cast<int32_t>(std::min<int64_t>(std::max<int64_t>(c, q), cam::kMaxChunkElems));
}

// Per-chunk cost of a register-form pass in element-equivalents (the chunk's
// table reads, its block barrier and drift-partial sum), for chunk_for_blocks.
constexpr int64_t kChunkCostElems = 1024;

// A fragment below kMaxChunkElems-sized chunks is spread over few waves of
// the register form's blocks, where the last wave's fill decides the time:
// among the whole numbers of block-steps, the chunk size with the smallest
// (waves x (chunk + kChunkCostElems)) for G blocks, tensors chunked one by
// one. Measured on the Pythia-14M step (6.4M-element fragment, G = 228):
// 14,336-element chunks (two per block) instead of 6,144 (four or five)
// took the graphed step from 0.0472 to 0.0448 ms.
int32_t chunk_for_blocks(const cam_ctx& c, const std::vector<int32_t>& tensors, int32_t chunk) {
    if (chunk >= cam::kMaxChunkElems) return chunk;
    const int64_t G = c.share_sms ? (2 * int64_t(c.sm_count) * 3) / 4 : 2 * int64_t(c.sm_count);
    auto cost = [&](int64_t ch) {
        int64_t n = 0;
        for (int32_t g : tensors) n += (c.numel[g] + ch - 1) / ch;
        return ((n + G - 1) / G) * (ch + kChunkCostElems);
    };
    int64_t best = chunk, best_cost = cost(chunk);
    for (int64_t ch = cam::kChunkQuantum; ch <= cam::kMaxChunkElems; ch += cam::kChunkQuantum)
        if (const int64_t k = cost(ch); k < best_cost) {
            best = ch;
            best_cost = k;
        }
    return static_cast<int32_t>(best);
}

void build_plan(Plan& p, const cam_ctx& c, int32_t fragment) {
    p.tensors.clear();
    for (int32_t t = 0; t < c.n_tensors; ++t)
        if (fragment < 0 || c.fragment_of[t] == fragment) p.tensors.push_back(t);
    p.n_elems = 0;
    for (int32_t g : p.tensors) p.n_elems += c.numel[g];
    p.chunk_elems = chunk_for_blocks(c, p.tensors, choose_chunk(p.n_elems, c.sm_count));
    p.chunks.clear();
    p.first_chunk.assign(1, 0);
    for (int32_t l = 0; l < p.n_tensors(); ++l) {
        const int64_t n = c.numel[p.tensors[l]];
        for (int64_t s = 0; s < n; s += p.chunk_elems)
            p.chunks.push_back(ChunkDesc{s, l, static_cast<int32_t>(std::min<int64_t>(p.chunk_elems, n - s))});
        p.first_chunk.push_back(static_cast<int32_t>(p.chunks.size()));
    }
}

// The invariants every kernel's indexing rests on, checked once on the host
// where the tables are made: each tensor's chunks lie inside it, in order,
// without gaps or overlap; chunk starts are multiples of the chunk quantum
// (so vectors stay aligned); first_chunk indexes them.
bool check_plan(const Plan& p, const cam_ctx& c) {
    if (p.first_chunk.size() != p.tensors.size() + 1 || p.first_chunk[0] != 0) return false;
    if (p.chunk_elems <= 0 || p.chunk_elems % cam::kChunkQuantum != 0) return false;
    for (int32_t l = 0; l < p.n_tensors(); ++l) {
        const int64_t n = c.numel[p.tensors[l]];
        int64_t next = 0;
        for (int32_t q = p.first_chunk[l]; q < p.first_chunk[l + 1]; ++q) {
            const ChunkDesc& ch = p.chunks[q];
            if (ch.local != l || ch.start != next || ch.len <= 0 || ch.len > p.chunk_elems ||
                ch.start % cam::kChunkQuantum != 0)
                return false;
            next = ch.start + ch.len;
        }
        if (next != n) return false;
    }
    return p.first_chunk.back() == p.n_chunks();
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Elements of the running-sum buffer (tensors in order, each rounded up to 8
// elements) after the end of tensor g's own.
int64_t sum_room_after(const cam_ctx& c, int32_t g) {
    int64_t room = (c.numel[g] + 7) / 8 * 8 - c.numel[g];
    for (int32_t t = g + 1; t < c.n_tensors; ++t) room += (c.numel[t] + 7) / 8 * 8;
    return room;
}

int validate_desc(const cam_ctx_desc* d) {
    if (!d) return fail(CAM_E_ARG, "cam_ctx_create: desc is NULL");
    if (d->n_tensors < 1) return fail(CAM_E_ARG, "cam_ctx_create: n_tensors must be >= 1");
    if (!d->numel || !d->master) return fail(CAM_E_ARG, "cam_ctx_create: numel and master are required");
    if (d->n_fragments < 1) return fail(CAM_E_ARG, "cam_ctx_create: n_fragments must be >= 1");
    if (d->quorum < 1 || d->quorum > CAM_KMAX)
        return fail(CAM_E_ARG, "cam_ctx_create: quorum must be in [1, %d]", CAM_KMAX);
    if (d->device < 0) return fail(CAM_E_ARG, "cam_ctx_create: device must be >= 0");
    if (d->flags & ~(CAM_INIT_EMA_FROM_MASTER | CAM_INIT_ZERO_MOMENTUM | CAM_INIT_ZERO_SWA |
                     CAM_NO_STAGING | CAM_TIME_COMMITS | CAM_NO_FUSED_FINISH |
                     CAM_TEST_STALL_STAGED | CAM_SHARE_SMS | CAM_TEST_BAD_CHUNK |
                     CAM_TEST_BAD_TAG))
        return fail(CAM_E_ARG, "cam_ctx_create: unknown flags 0x%x", d->flags);
    if ((d->flags & CAM_INIT_EMA_FROM_MASTER) && !d->ema)
        return fail(CAM_E_ARG, "cam_ctx_create: CAM_INIT_EMA_FROM_MASTER without EMA buffers");
    if ((d->flags & CAM_INIT_ZERO_MOMENTUM) && !d->momentum)
        return fail(CAM_E_ARG, "cam_ctx_create: CAM_INIT_ZERO_MOMENTUM without momentum buffers");
    if ((d->flags & CAM_INIT_ZERO_SWA) && !d->swa)
        return fail(CAM_E_ARG, "cam_ctx_create: CAM_INIT_ZERO_SWA without average buffers");
    for (int32_t t = 0; t < d->n_tensors; ++t) {
        const int64_t n = d->numel[t];
        if (n < 0) return fail(CAM_E_ARG, "cam_ctx_create: numel[%d] < 0", t);
        if (n > (int64_t(1) << 40)) return fail(CAM_E_ARG, "cam_ctx_create: numel[%d] too large", t);
        if (d->fragment_of && (d->fragment_of[t] < 0 || d->fragment_of[t] >= d->n_fragments))
            return fail(CAM_E_ARG, "cam_ctx_create: fragment_of[%d]=%d out of [0, %d)", t,
                        d->fragment_of[t], d->n_fragments);
        if (n > 0 && !d->master[t]) return fail(CAM_E_ARG, "cam_ctx_create: master[%d] is NULL", t);
        if (n > 0 && d->momentum && !d->momentum[t])
            return fail(CAM_E_ARG, "cam_ctx_create: momentum[%d] is NULL", t);
        if (n > 0 && d->ema && !d->ema[t])
            return fail(CAM_E_ARG, "cam_ctx_create: ema[%d] is NULL", t);
        if (n > 0 && d->swa && !d->swa[t])
            return fail(CAM_E_ARG, "cam_ctx_create: swa[%d] is NULL", t);
        if (d->rows && d->rows[t] < 0) return fail(CAM_E_ARG, "cam_ctx_create: rows[%d] < 0", t);
    }
    return CAM_OK;
}

}  // namespace

CAM_API const char* cam_last_error(void) { return g_err.c_str(); }

CAM_API const char* cam_version(void) { return "0.1.0"; }

CAM_API int cam_ctx_create(const cam_ctx_desc* d, cam_ctx** out) {
    if (!out) return fail(CAM_E_ARG, "cam_ctx_create: out is NULL");
    *out = nullptr;
    int rc = validate_desc(d);
    if (rc != CAM_OK) return rc;

    int n_dev = 0;
    cudaError_t ce = cudaGetDeviceCount(&n_dev);
    if (ce != cudaSuccess) return cuda_fail(ce, "cam_ctx_create: no usable CUDA device");
    if (d->device >= n_dev)
        return fail(CAM_E_CUDA, "cam_ctx_create: device %d not present (%d devices)", d->device, n_dev);
    DeviceScope scope(d->device);
    if (scope.err != cudaSuccess) return cuda_fail(scope.err, "cam_ctx_create: cudaSetDevice");

    std::unique_ptr<cam_ctx> c(new (std::nothrow) cam_ctx);
    if (!c) return fail(CAM_E_NOMEM, "cam_ctx_create: out of host memory");
    c->args.reset(new (std::nothrow) MergeArgs);
    c->multi_args.reset(new (std::nothrow) cam::MultiArgs);
    if (!c->args || !c->multi_args) return fail(CAM_E_NOMEM, "cam_ctx_create: out of host memory");
    c->device = d->device;
    ce = cudaDeviceGetAttribute(&c->sm_count, cudaDevAttrMultiProcessorCount, d->device);
    if (ce != cudaSuccess) return cuda_fail(ce, "cam_ctx_create: SM count");
    int pageable = 0;
    ce = cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, d->device);
    if (ce != cudaSuccess) return cuda_fail(ce, "cam_ctx_create: pageable memory access");
    c->pageable_access = pageable != 0;
    c->n_tensors = d->n_tensors;
    c->n_fragments = d->n_fragments;
    c->quorum = d->quorum;
    c->numel.assign(d->numel, d->numel + d->n_tensors);
    c->fragment_of.assign(d->n_tensors, 0);
    if (d->fragment_of) c->fragment_of.assign(d->fragment_of, d->fragment_of + d->n_tensors);
    c->theta.assign(d->master, d->master + d->n_tensors);
    c->has_m = d->momentum != nullptr;
    c->has_e = d->ema != nullptr;
    c->has_swa = d->swa != nullptr;
    c->m.assign(d->n_tensors, nullptr);
    c->e.assign(d->n_tensors, nullptr);
    c->swa.assign(d->n_tensors, nullptr);
    if (c->has_m) c->m.assign(d->momentum, d->momentum + d->n_tensors);
    if (c->has_e) c->e.assign(d->ema, d->ema + d->n_tensors);
    if (c->has_swa) c->swa.assign(d->swa, d->swa + d->n_tensors);
    c->swa_count.assign(d->n_tensors, 0);
    c->rows.assign(d->n_tensors, 0);
    if (d->rows) c->rows.assign(d->rows, d->rows + d->n_tensors);
    {   // iterate buffers hold a batch of equal-shape matrices in the GEMMs'
        // padded layout: at least the largest one, at most all of them,
        // capped at 2^29 elements (2^28 for Gram)
        int64_t big = 0, big_gram = 0, all = 0, all_gram = 0;
        auto pad = [](int64_t v) { return (v + 127) / 128 * 128; };
        for (int32_t t = 0; t < c->n_tensors; ++t)
            if (c->is_matrix(t)) {
                const int64_t rows = c->rows[t], cols = c->numel[t] / c->rows[t];
                const int64_t rp = pad(std::min(rows, cols)), lp = pad(std::max(rows, cols));
                big = std::max(big, rp * lp);
                big_gram = std::max(big_gram, rp * rp);
                all += rp * lp;
                all_gram += rp * rp;
            }
        c->ortho_cap_elems = std::max(big, std::min(all, int64_t(1) << 29));
        c->ortho_cap_gram = std::max(big_gram, std::min(all_gram, int64_t(1) << 28));
        c->ortho_big_gram = big_gram;
    }

    // Plans and one device block holding every plan's tables, after the
    // status word.
    c->share_sms = (d->flags & CAM_SHARE_SMS) != 0;  // (the plans' chunk sizes depend on it)
    c->plans.resize(c->n_fragments + 1);
    size_t bytes = 256;
    for (int32_t f = 0; f <= c->n_fragments; ++f) {
        Plan& p = c->plans[f];
        build_plan(p, *c, f < c->n_fragments ? f : -1);
        if (!check_plan(p, *c))
            return fail(CAM_E_ARG, "cam_ctx_create: internal error: inconsistent chunk plan");
        bytes += round_up(sizeof(ChunkDesc) * p.chunks.size(), 256);
        bytes += round_up(sizeof(TensorSlot) * p.tensors.size(), 256);
        bytes += round_up(sizeof(int32_t) * p.first_chunk.size(), 256);
        bytes += round_up(sizeof(double) * p.chunks.size(), 256);
        bytes += round_up(sizeof(double) * p.tensors.size(), 256);
        bytes += round_up(sizeof(double) * CAM_KMAX * p.chunks.size(), 256);
        bytes += round_up(sizeof(double) * CAM_KMAX * p.tensors.size(), 256);
        bytes += 256;  // the fused finish's block counter
    }
    ce = cudaMalloc(&c->dev_block, std::max<size_t>(bytes, 256));
    if (ce != cudaSuccess) {
        c->dev_block = nullptr;
        return fail(CAM_E_NOMEM, "cam_ctx_create: cudaMalloc(%zu): %s", bytes, cudaGetErrorString(ce));
    }
    std::vector<unsigned char> host(std::max<size_t>(bytes, 256), 0);
    c->d_status = static_cast<int32_t*>(c->dev_block);
    size_t off = 256;
    auto carve = [&](size_t n) {
        const size_t o = off;
        off += round_up(n, 256);
        return o;
    };
    for (Plan& p : c->plans) {
        std::vector<TensorSlot> slots;
        for (int32_t g : p.tensors)
            slots.push_back(TensorSlot{c->theta[g], c->m[g], c->e[g], c->swa[g], c->numel[g]});
        size_t o;
        o = carve(sizeof(ChunkDesc) * p.chunks.size());
        if (!p.chunks.empty()) std::memcpy(&host[o], p.chunks.data(), sizeof(ChunkDesc) * p.chunks.size());
        if ((d->flags & CAM_TEST_BAD_CHUNK) && p.tensors.size() >= 2 && p.first_chunk[1] > 0 &&
            sum_room_after(*c, p.tensors[0]) >= cam::kChunkQuantum) {
            // test hook: the device copy of the first tensor's last chunk runs
            // one chunk quantum past the tensor's end (inside the running-sum
            // buffer too, which holds the tensors in order)
            ChunkDesc bad = p.chunks[p.first_chunk[1] - 1];
            bad.len += cam::kChunkQuantum;
            std::memcpy(&host[o + sizeof(ChunkDesc) * (p.first_chunk[1] - 1)], &bad, sizeof bad);
        }
        p.d_chunks = reinterpret_cast<ChunkDesc*>(static_cast<unsigned char*>(c->dev_block) + o);
        o = carve(sizeof(TensorSlot) * slots.size());
        if (!slots.empty()) std::memcpy(&host[o], slots.data(), sizeof(TensorSlot) * slots.size());
        p.d_slots = reinterpret_cast<TensorSlot*>(static_cast<unsigned char*>(c->dev_block) + o);
        o = carve(sizeof(int32_t) * p.first_chunk.size());
        std::memcpy(&host[o], p.first_chunk.data(), sizeof(int32_t) * p.first_chunk.size());
        p.d_first = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(c->dev_block) + o);
        o = carve(sizeof(double) * p.chunks.size());
        p.d_partials = reinterpret_cast<double*>(static_cast<unsigned char*>(c->dev_block) + o);
        o = carve(sizeof(double) * p.tensors.size());
        p.d_tsq = reinterpret_cast<double*>(static_cast<unsigned char*>(c->dev_block) + o);
        o = carve(sizeof(double) * CAM_KMAX * p.chunks.size());
        p.d_worker_partials = reinterpret_cast<double*>(static_cast<unsigned char*>(c->dev_block) + o);
        o = carve(sizeof(double) * CAM_KMAX * p.tensors.size());
        p.d_worker_tsq = reinterpret_cast<double*>(static_cast<unsigned char*>(c->dev_block) + o);
        o = carve(sizeof(unsigned int));  // zero from the upload below
        p.d_fin_counter = reinterpret_cast<unsigned int*>(static_cast<unsigned char*>(c->dev_block) + o);
    }
    ce = cudaMemcpy(c->dev_block, host.data(), bytes, cudaMemcpyHostToDevice);
    if (ce != cudaSuccess) {
        cudaFree(c->dev_block);
        return cuda_fail(ce, "cam_ctx_create: table upload");
    }
    for (int dt = 0; dt < 2; ++dt)
        for (int md = 0; md < 2; ++md)
            for (int em = 0; em < 2; ++em)
                for (int nl = 0; nl < 3; ++nl)
                    for (int pb = 0; pb < 2; ++pb)
                        for (int sw = 0; sw < 2; ++sw)
                            c->bps[dt][md][em][nl][pb][sw] = std::max(
                                1, cam::merge_blocks_per_sm(cam::MergeVariant{
                                       dt, md, em != 0, nl, pb != 0, sw != 0}));

    for (int dt = 0; dt < 2; ++dt)
        for (int md = 0; md < 2; ++md)
            for (int em = 0; em < 2; ++em)
                for (int pb = 0; pb < 2; ++pb)
                    for (int sw = 0; sw < 2; ++sw) {
                        cam::MergeVariant v{dt, md, em != 0, 1, pb != 0, sw != 0};
                        v.fin = true;
                        c->bps_fin[dt][md][em][pb][sw] = std::max(1, cam::merge_blocks_per_sm(v));
                    }
    for (int dt = 0; dt < 2; ++dt)
        for (int md = 0; md < 2; ++md)
            for (int em = 0; em < 2; ++em)
                for (int nl = 0; nl < 2; ++nl)
                    for (int pb = 0; pb < 2; ++pb)
                        c->bps_multi[dt][md][em][nl][pb] = std::max(
                            1, cam::multi_blocks_per_sm(cam::MergeVariant{
                                   dt, md, em != 0, nl, pb != 0, false}));
    c->fuse_finish = !(d->flags & CAM_NO_FUSED_FINISH);
    c->staged = !(d->flags & CAM_NO_STAGING);
    c->test_stall = (d->flags & CAM_TEST_STALL_STAGED) != 0;
    c->test_tag = (d->flags & CAM_TEST_BAD_TAG) != 0;
    c->share_sms = (d->flags & CAM_SHARE_SMS) != 0;
    c->time_commits = (d->flags & CAM_TIME_COMMITS) != 0;
    for (int i = 0; c->time_commits && i < 2 && ce == cudaSuccess; ++i)
        ce = cudaEventCreate(&c->commit_ev[i]);
    c->plan_ev.assign(c->n_fragments + 1, nullptr);
    for (size_t i = 0; i < c->plan_ev.size() && ce == cudaSuccess; ++i)
        ce = cudaEventCreateWithFlags(&c->plan_ev[i], cudaEventDisableTiming);
    if (ce == cudaSuccess) ce = cudaEventCreateWithFlags(&c->ortho_ev, cudaEventDisableTiming);
    if (ce != cudaSuccess) {
        cam_ctx_destroy(c.release());
        return cuda_fail(ce, "cam_ctx_create: events");
    }
    if (c->staged) {
        ce = cam::staged_prepare();
        if (ce != cudaSuccess) {
            cam_ctx_destroy(c.release());
            return cuda_fail(ce, "cam_ctx_create: staged pass set-up");
        }
    }

    cudaStream_t s = static_cast<cudaStream_t>(d->stream);
    for (int32_t t = 0; t < c->n_tensors && ce == cudaSuccess; ++t) {
        if (c->numel[t] == 0) continue;
        if (d->flags & CAM_INIT_ZERO_MOMENTUM) {
            ce = cam::launch_fill(c->m[t], c->numel[t], 0.0f, s);
            ++c->launches;
        }
        if (ce == cudaSuccess && (d->flags & CAM_INIT_EMA_FROM_MASTER)) {
            ce = cam::launch_copy(c->e[t], c->theta[t], c->numel[t], s);
            ++c->launches;
        }
        if (ce == cudaSuccess && (d->flags & CAM_INIT_ZERO_SWA)) {
            ce = cam::launch_fill(c->swa[t], c->numel[t], 0.0f, s);
            ++c->launches;
        }
    }
    if (ce != cudaSuccess) {
        cam_ctx_destroy(c.release());
        return cuda_fail(ce, "cam_ctx_create: init kernels");
    }
    *out = c.release();
    return CAM_OK;
}

CAM_API void cam_ctx_destroy(cam_ctx* c) {
    if (!c) return;
    for (cam_round* r : c->open) delete r;
    c->open.clear();
    {
        DeviceScope scope(c->device);
        if (c->dev_block) cudaFree(c->dev_block);
        cam::ortho_destroy(c->ortho);
        if (c->d_sum) cudaFree(c->d_sum);
        for (cudaEvent_t ev : c->plan_ev)
            if (ev) cudaEventDestroy(ev);
        if (c->ortho_ev) cudaEventDestroy(c->ortho_ev);
        for (cudaEvent_t ev : c->commit_ev)
            if (ev) cudaEventDestroy(ev);
    }
    delete c;
}

CAM_API int cam_merge_begin(cam_ctx* c, int64_t round, int32_t fragment, cam_round** out) {
    if (!c || !out) return fail(CAM_E_ARG, "cam_merge_begin: NULL argument");
    *out = nullptr;
    if (fragment < -1 || fragment >= c->n_fragments)
        return fail(CAM_E_ARG, "cam_merge_begin: fragment %d out of [-1, %d)", fragment, c->n_fragments);
    if (round <= c->last_round)
        return fail(CAM_E_STALE, "cam_merge_begin: round %lld is not newer than %lld",
                    static_cast<long long>(round), static_cast<long long>(c->last_round));
    for (const cam_round* r : c->open)
        if (r->fragment == -1 || fragment == -1 || r->fragment == fragment)
            return fail(CAM_E_BUSY, "cam_merge_begin: fragment %d overlaps open round %lld (fragment %d)",
                        fragment, static_cast<long long>(r->round), r->fragment);
    if (static_cast<int>(c->open.size()) >= CAM_MAX_OPEN_ROUNDS)
        return fail(CAM_E_BUSY, "cam_merge_begin: %d rounds already open", CAM_MAX_OPEN_ROUNDS);
    cam_round* r = new (std::nothrow) cam_round;
    if (!r) return fail(CAM_E_NOMEM, "cam_merge_begin: out of host memory");
    r->ctx = c;
    r->round = round;
    r->fragment = fragment;
    try {
        r->x.reserve(size_t(CAM_KMAX) * c->plan_of(fragment).tensors.size());
        c->open.push_back(r);
    } catch (...) {
        delete r;
        return fail(CAM_E_NOMEM, "cam_merge_begin: out of host memory");
    }
    c->last_round = round;
    *out = r;
    return CAM_OK;
}

namespace {

// Device address under which the GPU reaches host buffer p, or nullptr when
// it cannot: page-locked memory mapped for the device (cudaHostAlloc,
// cudaHostRegister, pinned torch tensors), managed memory, or ordinary pageable
// memory on systems whose GPU reads host page tables (Grace: NVLink-C2C with
// address translation). Device memory of the context's device is accepted too.
const void* device_view_of_host(const cam_ctx* c, const void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();  // the failed query must not linger as the last error
        return nullptr;
    }
    switch (at.type) {
        case cudaMemoryTypeHost:
            return at.devicePointer;
        case cudaMemoryTypeManaged:
            return p;
        case cudaMemoryTypeDevice:
            return at.device == c->device ? p : nullptr;
        default:  // unregistered pageable memory
            return c->pageable_access ? p : nullptr;
    }
}

int accumulate(cam_round* r, const void* const* ckpt, cam_dtype dtype, int64_t tokens,
               bool host, const char* fn) {
    if (!r) return fail(CAM_E_ARG, "%s: round is NULL", fn);
    if (r->finalized) return fail(CAM_E_STATE, "%s: round already finalized", fn);
    if (r->K >= CAM_KMAX) return fail(CAM_E_KMAX, "%s: more than %d workers", fn, CAM_KMAX);
    if (dtype != CAM_F32 && dtype != CAM_BF16)
        return fail(CAM_E_ARG, "%s: unknown dtype %d", fn, static_cast<int>(dtype));
    if (r->K > 0 && dtype != r->dtype)
        return fail(CAM_E_ARG, "%s: dtype %d differs from the round's %d", fn,
                    static_cast<int>(dtype), r->dtype);
    if (tokens < 0 || tokens > (int64_t(1) << 56))
        return fail(CAM_E_ARG, "%s: tokens %lld out of range", fn, static_cast<long long>(tokens));
    const cam_ctx* c = r->ctx;
    const Plan& p = c->plan_of(r->fragment);
    if (!ckpt && p.n_tensors() > 0) return fail(CAM_E_ARG, "%s: ckpt is NULL", fn);
    for (int32_t l = 0; l < p.n_tensors(); ++l)
        if (!ckpt[l] && c->numel[p.tensors[l]] > 0)
            return fail(CAM_E_ARG, "%s: ckpt[%d] is NULL", fn, l);
    const size_t base = r->x.size();
    for (int32_t l = 0; l < p.n_tensors(); ++l) {
        const void* q = ckpt[l];
        if (host && c->numel[p.tensors[l]] > 0) {
            q = device_view_of_host(c, ckpt[l]);
            if (!q) {
                r->x.resize(base);
                return fail(CAM_E_ARG,
                            "%s: ckpt[%d] is host memory the GPU cannot read (pin it or "
                            "register it with the CUDA driver)", fn, l);
            }
        }
        r->x.push_back(q);
    }
    r->tokens[r->K] = tokens;
    r->dtype = dtype;
    r->host_workers = r->host_workers || host;
    ++r->K;
    return CAM_OK;
}

}  // namespace

CAM_API int cam_merge_accumulate(cam_round* r, const void* const* ckpt, cam_dtype dtype,
                                 int64_t tokens) {
    return accumulate(r, ckpt, dtype, tokens, false, "cam_merge_accumulate");
}

CAM_API int cam_merge_accumulate_host(cam_round* r, const void* const* ckpt, cam_dtype dtype,
                                      int64_t tokens) {
    return accumulate(r, ckpt, dtype, tokens, true, "cam_merge_accumulate_host");
}

namespace {

// Makes the context's running-sum buffer and its per-plan events.
int ensure_sum(cam_ctx* c, const char* fn) {
    if (c->d_sum) return CAM_OK;
    std::vector<int64_t> off(c->n_tensors);
    int64_t total = 0;
    for (int32_t t = 0; t < c->n_tensors; ++t) {
        off[t] = total;
        total += (c->numel[t] + 7) / 8 * 8;
    }
    float* buf = nullptr;
    cudaError_t ce = cudaMalloc(&buf, sizeof(float) * size_t(std::max<int64_t>(total, 8)));
    if (ce != cudaSuccess) {
        cudaGetLastError();
        return fail(CAM_E_NOMEM, "%s: cudaMalloc of the running sums (%lld floats): %s", fn,
                    static_cast<long long>(total), cudaGetErrorString(ce));
    }
    c->d_sum = buf;
    c->sum_off.swap(off);
    return CAM_OK;
}

// True while `s` is being captured into a CUDA graph. Captured work is
// ordered by the capture alone: the per-plan events, recorded by work outside
// any graph, are neither waited on nor recorded inside one.
bool capturing(cudaStream_t s) {
    cudaStreamCaptureStatus st = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &st) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return st != cudaStreamCaptureStatusNone;
}

// Orders stream s after the last device work that touched any of a
// fragment's tensors: its own plan and the whole-list plan, or every plan
// for a whole-list round. An event not yet recorded is no wait.
cudaError_t plan_order(cam_ctx* c, int32_t fragment, cudaStream_t s, bool cap) {
    cudaError_t ce = cudaSuccess;
    for (int32_t f = 0; !cap && f <= c->n_fragments && ce == cudaSuccess; ++f)
        if (fragment < 0 || f == fragment || f == c->n_fragments)
            ce = cudaStreamWaitEvent(s, c->plan_ev[f], 0);
    return ce;
}

cudaError_t plan_mark(cam_ctx* c, int32_t fragment, cudaStream_t s, bool cap) {
    if (cap) return cudaSuccess;
    return cudaEventRecord(c->plan_ev[fragment < 0 ? c->n_fragments : fragment], s);
}

// Bit l of vec[]: tensor l0 + l of the plan takes the vector path in a
// launch covering [l0, l0 + n), given its pointers' alignment.
template <class F>
void set_vec(uint32_t* vec, int n, F&& ok) {
    std::fill(vec, vec + cam::kEagerTensors / 32, 0u);
    for (int l = 0; l < n; ++l)
        if (ok(l)) vec[l >> 5] |= 1u << (l & 31);
}

}  // namespace

CAM_API int cam_merge_fold(cam_round* r, const void* const* ckpt, cam_dtype dtype, int64_t tokens,
                           cam_mode mode, void* stream) {
    const char* fn = "cam_merge_fold";
    if (!r) return fail(CAM_E_ARG, "%s: round is NULL", fn);
    if (r->finalized) return fail(CAM_E_STATE, "%s: round already finalized", fn);
    if (r->K > r->n_folded)
        return fail(CAM_E_STATE, "%s: the round already holds accumulated workers (folds come first)", fn);
    if (r->ortho) return fail(CAM_E_STATE, "%s: an orthogonalised round needs its workers at commit", fn);
    if (r->K >= CAM_KMAX) return fail(CAM_E_KMAX, "%s: more than %d workers", fn, CAM_KMAX);
    if (dtype != CAM_F32 && dtype != CAM_BF16)
        return fail(CAM_E_ARG, "%s: unknown dtype %d", fn, static_cast<int>(dtype));
    if (r->K > 0 && dtype != r->dtype)
        return fail(CAM_E_ARG, "%s: dtype %d differs from the round's %d", fn,
                    static_cast<int>(dtype), r->dtype);
    if (mode != CAM_MODE_MEAN_REPLACE && mode != CAM_MODE_DELTA_NESTEROV)
        return fail(CAM_E_ARG, "%s: unknown mode %d", fn, static_cast<int>(mode));
    if (r->eager && mode != r->eager_mode)
        return fail(CAM_E_ARG, "%s: mode %d differs from the earlier folds' %d", fn,
                    static_cast<int>(mode), r->eager_mode);
    if (tokens < 0 || tokens > (int64_t(1) << 56))
        return fail(CAM_E_ARG, "%s: tokens %lld out of range", fn, static_cast<long long>(tokens));
    cam_ctx* c = r->ctx;
    const Plan& p = c->plan_of(r->fragment);
    const int T = p.n_tensors();
    if (!ckpt && T > 0) return fail(CAM_E_ARG, "%s: ckpt is NULL", fn);
    std::vector<const void*> xs(T, nullptr);
    for (int32_t l = 0; l < T; ++l) {
        if (c->numel[p.tensors[l]] == 0) continue;
        if (!ckpt[l]) return fail(CAM_E_ARG, "%s: ckpt[%d] is NULL", fn, l);
        xs[l] = device_view_of_host(c, ckpt[l]);
        if (!xs[l])
            return fail(CAM_E_ARG, "%s: ckpt[%d] is memory the GPU cannot read", fn, l);
    }
    DeviceScope scope(c->device);
    if (scope.err != cudaSuccess) return cuda_fail(scope.err, "cam_merge_fold: cudaSetDevice");
    char label[80];
    std::snprintf(label, sizeof label, "cam_merge_fold round %lld worker %d",
                  static_cast<long long>(r->round), r->K);
    NvtxRange nvtx(label);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool cap = capturing(s);
    if (cap && !c->d_sum)
        return fail(CAM_E_STATE, "%s: the context's first fold allocates; make it outside a graph capture", fn);
    int rc = ensure_sum(c, fn);
    if (rc != CAM_OK) return rc;
    cudaError_t ce = plan_order(c, r->fragment, s, cap);
    const int k = r->K;
    const uintptr_t xa = dtype == CAM_F32 ? 32 : 16;
    const bool wd = r->worker_norms;
    cam::FoldArgs a;
    a.slots = p.d_slots;
    a.status = c->d_status;
    a.k = k;
    a.first = k == 0;
    a.w = static_cast<float>(tokens);
    int64_t launched = 0;
    for (int l0 = 0; l0 < T && ce == cudaSuccess; l0 += cam::kEagerTensors) {
        const int n = std::min(cam::kEagerTensors, T - l0);
        const int32_t c0 = p.first_chunk[l0], c1 = p.first_chunk[l0 + n];
        if (c1 == c0) continue;
        for (int l = 0; l < n; ++l) {
            const int32_t g = p.tensors[l0 + l];
            a.x[l] = xs[l0 + l];
            a.sum[l] = c->d_sum + c->sum_off[g];
        }
        set_vec(a.vec, n, [&](int l) {
            const int32_t g = p.tensors[l0 + l];
            return aligned(a.x[l], xa) && aligned(c->theta[g], 32);
        });
        a.chunks = p.d_chunks + c0;
        a.worker_partials = wd ? p.d_worker_partials + static_cast<int64_t>(c0) * CAM_KMAX : nullptr;
        a.n_chunks = c1 - c0;
        a.local0 = l0;
        a.n_local = n;
        const int grid = static_cast<int>(std::min<int64_t>(a.n_chunks, int64_t(c->sm_count) * 2));
        ce = cam::launch_fold(a, dtype, mode, wd, grid, s);
        ++launched;
    }
    if (ce == cudaSuccess) ce = plan_mark(c, r->fragment, s, cap);
    if (ce != cudaSuccess) return cuda_fail(ce, "cam_merge_fold: launch");
    c->launches += launched;
    r->eager = true;
    r->eager_mode = mode;
    r->tokens[k] = tokens;
    r->dtype = dtype;
    ++r->K;
    ++r->n_folded;
    return CAM_OK;
}

CAM_API int cam_merge_finalize(cam_round* r, cam_mode mode, float lr, float mu) {
    if (!r) return fail(CAM_E_ARG, "cam_merge_finalize: round is NULL");
    if (r->finalized) return fail(CAM_E_STATE, "cam_merge_finalize: finalized twice");
    if (mode != CAM_MODE_MEAN_REPLACE && mode != CAM_MODE_DELTA_NESTEROV)
        return fail(CAM_E_ARG, "cam_merge_finalize: unknown mode %d", static_cast<int>(mode));
    if (!std::isfinite(lr) || !std::isfinite(mu))
        return fail(CAM_E_ARG, "cam_merge_finalize: lr and mu must be finite");
    if (mode == CAM_MODE_DELTA_NESTEROV && !r->ctx->has_m)
        return fail(CAM_E_ARG, "cam_merge_finalize: Nesterov needs momentum buffers");
    if (r->eager && mode != r->eager_mode)
        return fail(CAM_E_STATE, "cam_merge_finalize: mode %d differs from the folds' mode %d",
                    static_cast<int>(mode), r->eager_mode);
    r->finalized = true;
    r->mode = mode;
    r->lr = lr;
    r->mu = mu;
    return CAM_OK;
}

CAM_API int cam_ema_update(cam_round* r, float beta) {
    if (!r) return fail(CAM_E_ARG, "cam_ema_update: round is NULL");
    if (r->ema) return fail(CAM_E_STATE, "cam_ema_update: asked twice");
    if (!std::isfinite(beta)) return fail(CAM_E_ARG, "cam_ema_update: beta must be finite");
    if (!r->ctx->has_e) return fail(CAM_E_ARG, "cam_ema_update: context has no EMA buffers");
    r->ema = true;
    r->beta = beta;
    return CAM_OK;
}

CAM_API int cam_worker_drift_norm(cam_round* r, double* per_worker_tensor, double* per_worker) {
    if (!r) return fail(CAM_E_ARG, "cam_worker_drift_norm: round is NULL");
    if (r->worker_norms) return fail(CAM_E_STATE, "cam_worker_drift_norm: asked twice");
    if (r->eager)
        return fail(CAM_E_STATE,
                    "cam_worker_drift_norm: ask before the first fold (each fold computes its own)");
    if (!per_worker_tensor && !per_worker)
        return fail(CAM_E_ARG, "cam_worker_drift_norm: both outputs NULL");
    r->worker_norms = true;
    r->out_worker_tensor = per_worker_tensor;
    r->out_worker = per_worker;
    return CAM_OK;
}

CAM_API int cam_merge_orthogonalize(cam_round* r, float lr, int32_t scale_mode, int32_t precision,
                                    int32_t iterations) {
    const char* fn = "cam_merge_orthogonalize";
    if (!r) return fail(CAM_E_ARG, "%s: round is NULL", fn);
    if (r->ortho) return fail(CAM_E_STATE, "%s: asked twice", fn);
    if (r->eager) return fail(CAM_E_STATE, "%s: needs the workers at commit, not folded", fn);
    if (!std::isfinite(lr)) return fail(CAM_E_ARG, "%s: lr must be finite", fn);
    if (scale_mode != CAM_ORTHO_SCALE_FIXED && scale_mode != CAM_ORTHO_SCALE_MATCH_NORM)
        return fail(CAM_E_ARG, "%s: unknown scale mode %d", fn, scale_mode);
    const int32_t base = precision & ~int32_t(CAM_ORTHO_SHORT_SIDE);
    const bool short_side = (precision & CAM_ORTHO_SHORT_SIDE) != 0;
    if (base != CAM_ORTHO_TF32 && base != CAM_ORTHO_FP32 && !(base == CAM_ORTHO_BF16 && !short_side))
        return fail(CAM_E_ARG, "%s: unknown precision %d", fn, precision);
    if (iterations < 1 || iterations > 1000)
        return fail(CAM_E_ARG, "%s: iterations %d outside [1, 1000]", fn, iterations);
    r->ortho = true;
    r->ortho_lr = lr;
    r->ortho_scale = scale_mode;
    r->ortho_precision = precision;
    r->ortho_iterations = iterations;
    return CAM_OK;
}

CAM_API int cam_swa_update(cam_round* r) {
    if (!r) return fail(CAM_E_ARG, "cam_swa_update: round is NULL");
    if (r->swa) return fail(CAM_E_STATE, "cam_swa_update: asked twice");
    if (!r->ctx->has_swa) return fail(CAM_E_ARG, "cam_swa_update: context has no average buffers");
    r->swa = true;
    return CAM_OK;
}

CAM_API int cam_drift_norm(cam_round* r, double* per_tensor, double* per_fragment) {
    if (!r) return fail(CAM_E_ARG, "cam_drift_norm: round is NULL");
    if (r->norms) return fail(CAM_E_STATE, "cam_drift_norm: asked twice");
    if (!per_tensor && !per_fragment) return fail(CAM_E_ARG, "cam_drift_norm: both outputs NULL");
    r->norms = true;
    r->out_tensor = per_tensor;
    r->out_fragment = per_fragment;
    return CAM_OK;
}

CAM_API int cam_merge_publish(cam_round* r, float* const* theta_out, float* const* ema_out) {
    const char* fn = "cam_merge_publish";
    if (!r) return fail(CAM_E_ARG, "%s: round is NULL", fn);
    if (r->publish) return fail(CAM_E_STATE, "%s: asked twice", fn);
    const cam_ctx* c = r->ctx;
    const Plan& p = c->plan_of(r->fragment);
    if (!theta_out && p.n_tensors() > 0) return fail(CAM_E_ARG, "%s: theta_out is NULL", fn);
    std::vector<void*> th(p.n_tensors(), nullptr), em;
    if (ema_out) em.assign(p.n_tensors(), nullptr);
    for (int32_t l = 0; l < p.n_tensors(); ++l) {
        if (c->numel[p.tensors[l]] == 0) continue;
        for (int which = 0; which < (ema_out ? 2 : 1); ++which) {
            float* q = which == 0 ? theta_out[l] : ema_out[l];
            if (!q) return fail(CAM_E_ARG, "%s: %s[%d] is NULL", fn, which ? "ema_out" : "theta_out", l);
            const void* d = device_view_of_host(c, q);
            if (!d)
                return fail(CAM_E_ARG, "%s: %s[%d] is memory the GPU cannot write", fn,
                            which ? "ema_out" : "theta_out", l);
            (which == 0 ? th : em)[l] = const_cast<void*>(d);
        }
    }
    r->publish = true;
    r->publish_ema = ema_out != nullptr;
    r->pub_theta.swap(th);
    r->pub_ema.swap(em);
    return CAM_OK;
}

namespace {

void close_round(cam_round* r) {
    auto& open = r->ctx->open;
    open.erase(std::remove(open.begin(), open.end(), r), open.end());
    delete r;
}

}  // namespace

CAM_API int cam_merge_abort(cam_round* r) {
    if (!r) return fail(CAM_E_ARG, "cam_merge_abort: round is NULL");
    close_round(r);
    return CAM_OK;
}

namespace {

// Whether round r can be committed (on a stream that is or is not being
// captured): the checks cam_merge_commit makes before anything runs.
// Records the message for `fn` and returns the error, else CAM_OK.
int commit_checks(const cam_round* r, bool cap, const char* fn) {
    const cam_ctx* c = r->ctx;
    if (!r->finalized) return fail(CAM_E_STATE, "%s: round not finalized", fn);
    if (r->K < c->quorum)
        return fail(CAM_E_QUORUM, "%s: %d participants < quorum %d", fn, r->K, c->quorum);
    if (r->K < 1) return fail(CAM_E_QUORUM, "%s: no participants", fn);
    if (r->publish_ema && !r->ema)
        return fail(CAM_E_STATE, "%s: an EMA copy was asked for without an EMA update", fn);
    int64_t W = 0;
    for (int k = 0; k < r->K; ++k) W += r->tokens[k];
    if (r->mode == CAM_MODE_DELTA_NESTEROV && W <= 0)
        return fail(CAM_E_ARG, "%s: total token count must be > 0", fn);
    if (r->ortho) {
        if (r->mode != CAM_MODE_MEAN_REPLACE)
            return fail(CAM_E_STATE, "%s: orthogonalisation applies to plain-mean rounds", fn);
        if (r->norms || r->worker_norms || r->publish || r->swa)
            return fail(CAM_E_STATE, "%s: an orthogonalised round takes only an EMA update", fn);
    }
    if (cap && r->swa)
        return fail(CAM_E_STATE,
                    "%s: a running-average update cannot be captured (its count would not "
                    "advance on replay)", fn);
    if (cap && r->ortho && !c->ortho)
        return fail(CAM_E_STATE,
                    "%s: the first orthogonalised commit allocates; make it outside a graph capture",
                    fn);
    if (r->swa) {
        int64_t prev = -1;
        for (int32_t g : c->plan_of(r->fragment).tensors) {
            if (c->numel[g] == 0) continue;
            if (prev >= 0 && c->swa_count[g] != prev)
                return fail(CAM_E_STATE,
                            "%s: the fragment's running averages hold different numbers of "
                            "globals (reset them together)", fn);
            prev = c->swa_count[g];
        }
    }
    return CAM_OK;
}

}  // namespace

CAM_API int cam_merge_commit(cam_round* r, void* stream) {
    if (!r) return fail(CAM_E_ARG, "cam_merge_commit: round is NULL");
    cam_ctx* c = r->ctx;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool cap = capturing(s);
    if (const int rc = commit_checks(r, cap, "cam_merge_commit"); rc != CAM_OK) return rc;
    int64_t W = 0;
    for (int k = 0; k < r->K; ++k) W += r->tokens[k];

    const Plan& p = c->plan_of(r->fragment);
    const int K = r->K;
    const int T = p.n_tensors();
    int64_t swa_prev = -1;
    if (r->swa) {
        for (int32_t g : p.tensors) {
            if (c->numel[g] == 0) continue;
            if (swa_prev >= 0 && c->swa_count[g] != swa_prev)
                return fail(CAM_E_STATE,
                            "cam_merge_commit: the fragment's running averages hold different "
                            "numbers of globals (reset them together)");
            swa_prev = c->swa_count[g];
        }
        if (swa_prev < 0) swa_prev = 0;
    }
    const bool delta = r->mode == CAM_MODE_DELTA_NESTEROV;
    const uintptr_t xa = r->dtype == CAM_F32 ? 32 : 16;
    MergeArgs& a = *c->args;
    a.slots = p.d_slots;
    a.K = K;
    a.Kf = static_cast<float>(K);
    for (int k = 0; k < CAM_KMAX; ++k) a.w[k] = k < K ? static_cast<float>(r->tokens[k]) : 0.0f;
    a.W = static_cast<float>(W);
    a.div = cam::div_plan(delta ? a.W : a.Kf);
    a.lr = r->lr;
    a.mu = r->mu;
    a.beta = r->beta;
    a.swa_n = static_cast<float>(swa_prev + 1);
    a.swa_div = cam::div_plan(a.swa_n);
    const int norm_level = r->worker_norms ? 2 : (r->norms ? 1 : 0);
    const int bps = c->bps[r->dtype][r->mode][r->ema][norm_level][r->publish][r->swa];
    // CAM_SHARE_SMS: a pass takes at most three quarters of the register
    // form's block slots, so that a round in flight on another stream starts
    // beside it. (Measured on the Pythia-14M step, two streams: 55 us against
    // 65 us with one block per SM; 7/8, 5/8 and 1/2 of the slots were slower.)
    auto grid_for = [&](int64_t n_chunks, int per_sm) -> int {
        int64_t slots = int64_t(c->sm_count) * per_sm;
        if (c->share_sms) slots -= slots / 4;
        return static_cast<int>(std::min<int64_t>(n_chunks, std::max<int64_t>(1, slots)));
    };
    const cam::MergeVariant variant{r->dtype, r->mode, r->ema, norm_level, r->publish, r->swa};
    const int stride = K + (r->publish ? 2 : 0);
    a.stride = stride;

    DeviceScope scope(c->device);
    if (scope.err != cudaSuccess) {
        close_round(r);
        return cuda_fail(scope.err, "cam_merge_commit: cudaSetDevice");
    }
    if (r->ortho && !c->ortho) {  // workspace of the orthogonalisation, made once per context
        const int rc = cam::ortho_create(&c->ortho, c->ortho_cap_elems, c->ortho_cap_gram,
                                         c->ortho_big_gram);
        if (rc == CAM_E_CUDA) close_round(r);  // a CUDA failure frees the round, as below
        if (rc != CAM_OK) return rc;            // CAM_E_NOMEM: nothing ran, the round stays open
    }
    cudaError_t ce = cudaSuccess;
    char label[96];
    std::snprintf(label, sizeof label, "cam_merge_commit round %lld fragment %d K %d",
                  static_cast<long long>(r->round), r->fragment, K);
    NvtxRange nvtx(label);
    const int64_t launches0 = c->launches, staged0 = c->staged_launches;
    ce = plan_order(c, r->fragment, s, cap);  // after earlier work on these tensors
    const bool timed = c->time_commits && !cap;
    if (ce == cudaSuccess && timed) ce = cudaEventRecord(c->commit_ev[0], s);
    const int per_launch = cam::kXCap / stride;
    // The staged form: a ring of as many stages as fit (at least 2, at most
    // kStMaxStages), for launches whose workers are device memory.
    const int64_t st_bytes = cam::staged_stage_bytes(variant, K);
    const int st_stages = static_cast<int>(std::min<int64_t>(
        cam::kStMaxStages, (cam::kStSmemBytes - cam::staged_red_bytes(variant, K)) / st_bytes));
    // Measured on GB300 (1.08B lists, 4B sweep): the staged form is ahead
    // when a round writes at most two state arrays (theta plus m or e) and
    // behind when it writes three (theta, m, e or theta, e, swa), where the
    // register form is kept.
    const int state_writes = 1 + int(delta) + int(r->ema) + int(r->swa);
    // (a staged block takes its SM's shared memory: with CAM_SHARE_SMS the
    // register form leaves room for another round's blocks)
    const bool staged_ok = c->staged && !c->share_sms && !r->host_workers && st_stages >= 2 &&
                           state_writes <= 2;
    // Small rounds with the round's drift norms finish them in the merge pass
    // itself (register form, last block): one launch fewer, the same sums.
    const int32_t fin_shared =
        cam::finish_smem_bytes(T, p.n_chunks()) <= cam::kFinishSmemMax ? 1 : 0;
    const NormArgs na{p.d_partials, p.d_first, T, p.d_tsq, r->out_tensor, r->out_fragment,
                      norm_level >= 2 ? K : 0, p.d_worker_partials, p.d_worker_tsq,
                      r->out_worker_tensor, r->out_worker, p.n_chunks(), fin_shared};
    const bool fuse = c->fuse_finish && norm_level == 1 && !r->eager && !r->ortho &&
                      p.n_chunks() > 0 && p.n_chunks() <= cam::kFuseMaxChunks && T <= per_launch;
    cam::MergeVariant variant_fin = variant;
    variant_fin.fin = true;
    a.fin = na;
    a.fin_counter = p.d_fin_counter;
    a.status = c->d_status;
    a.st_stages = st_stages;
    a.st_stage_bytes = static_cast<int32_t>(st_bytes);
    a.test_stall = c->test_stall ? 1 : 0;
    a.test_tag = c->test_tag ? 1 : 0;
    // Fused pass over the fragment's local tensors [lb, le).
    auto launch_range = [&](int lb, int le) {
        for (int l0 = lb; l0 < le && ce == cudaSuccess; l0 += per_launch) {
            const int n = std::min(per_launch, le - l0);
            const int32_t c0 = p.first_chunk[l0], c1 = p.first_chunk[l0 + n];
            if (c1 == c0) continue;
            bool all_vec = true;
            std::memset(a.vec, 0, sizeof a.vec);
            for (int l = 0; l < n; ++l) {
                const int32_t g = p.tensors[l0 + l];
                bool v = aligned(c->theta[g], 32) && (!delta || aligned(c->m[g], 32)) &&
                         (!r->ema || aligned(c->e[g], 32)) && (!r->swa || aligned(c->swa[g], 32));
                for (int k = 0; k < K; ++k) {
                    const void* xp = r->x[size_t(k) * T + l0 + l];
                    a.x[size_t(l) * stride + k] = xp;
                    v = v && aligned(xp, xa);
                }
                if (r->publish) {
                    void* pt = r->pub_theta[l0 + l];
                    void* pe = r->publish_ema ? r->pub_ema[l0 + l] : nullptr;
                    a.x[size_t(l) * stride + K] = pt;
                    a.x[size_t(l) * stride + K + 1] = pe;
                    v = v && aligned(pt, 32) && aligned(pe, 32);
                }
                if (v) a.vec[l >> 5] |= 1u << (l & 31);
                all_vec = all_vec && v;
            }
            a.chunks = p.d_chunks + c0;
            a.partials = norm_level >= 1 ? p.d_partials + c0 : nullptr;
            a.worker_partials =
                norm_level >= 2 ? p.d_worker_partials + static_cast<int64_t>(c0) * CAM_KMAX : nullptr;
            a.n_chunks = c1 - c0;
            a.local0 = l0;
            a.n_local = n;
            if (fuse) {  // a single launch covering the whole fragment
                const int grid =
                    grid_for(a.n_chunks, c->bps_fin[r->dtype][r->mode][r->ema][r->publish][r->swa]);
                ce = cam::launch_merge(a, variant_fin, grid, s);
            } else if (staged_ok && all_vec) {  // one block per SM
                const int grid = static_cast<int>(std::min<int64_t>(a.n_chunks, c->sm_count));
                ce = cam::launch_merge_staged(a, variant, grid, s);
                ++c->staged_launches;
            } else {
                ce = cam::launch_merge(a, variant, grid_for(a.n_chunks, bps), s);
            }
            ++c->launches;
        }
    };
    // Final pass of an eagerly folded round: from the running sums.
    auto launch_final = [&]() {
        cam::FinalArgs fa;
        fa.slots = p.d_slots;
        fa.status = c->d_status;
        fa.K = K;
        fa.Kf = a.Kf;
        fa.W = a.W;
        fa.div = a.div;
        fa.lr = a.lr;
        fa.mu = a.mu;
        fa.beta = a.beta;
        fa.swa_n = a.swa_n;
        fa.swa_div = a.swa_div;
        const int P = K - r->n_folded;  // accumulated after the folds: folded here
        fa.P = P;
        fa.first_k = r->n_folded;
        fa.stride = 3 + P;
        for (int q = 0; q < CAM_KMAX; ++q)
            fa.wp[q] = q < P ? static_cast<float>(r->tokens[r->n_folded + q]) : 0.0f;
        const int per = std::min(cam::kEagerTensors, cam::kFinalPtrs / fa.stride);
        for (int l0 = 0; l0 < T && ce == cudaSuccess; l0 += per) {
            const int n = std::min(per, T - l0);
            const int32_t c0 = p.first_chunk[l0], c1 = p.first_chunk[l0 + n];
            if (c1 == c0) continue;
            for (int l = 0; l < n; ++l) {
                const int32_t g = p.tensors[l0 + l];
                const void** tp = fa.ptr + static_cast<size_t>(l) * fa.stride;
                tp[0] = c->d_sum + c->sum_off[g];
                tp[1] = r->publish ? r->pub_theta[l0 + l] : nullptr;
                tp[2] = r->publish_ema ? r->pub_ema[l0 + l] : nullptr;
                for (int q = 0; q < P; ++q) tp[3 + q] = r->x[size_t(q) * T + l0 + l];
            }
            set_vec(fa.vec, n, [&](int l) {
                const int32_t g = p.tensors[l0 + l];
                const void* const* tp = fa.ptr + static_cast<size_t>(l) * fa.stride;
                bool v = aligned(c->theta[g], 32) && (!delta || aligned(c->m[g], 32)) &&
                         (!r->ema || aligned(c->e[g], 32)) && (!r->swa || aligned(c->swa[g], 32)) &&
                         aligned(tp[1], 32) && aligned(tp[2], 32);
                for (int q = 0; q < P; ++q) v = v && aligned(tp[3 + q], xa);
                return v;
            });
            fa.chunks = p.d_chunks + c0;
            fa.partials = norm_level >= 1 ? p.d_partials + c0 : nullptr;
            fa.worker_partials =
                norm_level >= 2 ? p.d_worker_partials + static_cast<int64_t>(c0) * CAM_KMAX : nullptr;
            fa.n_chunks = c1 - c0;
            fa.local0 = l0;
            fa.n_local = n;
            const int grid = static_cast<int>(std::min<int64_t>(fa.n_chunks, int64_t(c->sm_count) * 2));
            ce = cam::launch_final(fa, r->dtype, r->mode, r->ema, norm_level >= 1, r->publish, r->swa,
                                   norm_level >= 2, grid, s);
            ++c->launches;
        }
    };
    if (r->eager) {
        launch_final();
    } else if (!r->ortho) {
        launch_range(0, T);
    } else {
        // the vectors and other non-matrix tensors take the fused pass ...
        int run = -1;
        for (int l = 0; l <= T; ++l) {
            const bool mat = l < T && c->is_matrix(p.tensors[l]);
            if (l < T && !mat) {
                if (run < 0) run = l;
            } else if (run >= 0) {
                launch_range(run, l);
                run = -1;
            }
        }
        // ... and each matrix has its averaged update replaced by its polar
        // factor, equal shapes batched together (first-appearance order)
        const cam::OrthoParams op{K,
                                  r->dtype,
                                  r->ortho_lr,
                                  r->ortho_scale,
                                  r->ortho_precision & ~int32_t(CAM_ORTHO_SHORT_SIDE),
                                  r->ortho_iterations,
                                  r->ema,
                                  r->beta,
                                  (r->ortho_precision & CAM_ORTHO_SHORT_SIDE) != 0,
                                  c->d_status};
        // the workspace is the context's: after its last use on any stream
        if (ce == cudaSuccess && !cap) ce = cudaStreamWaitEvent(s, c->ortho_ev, 0);
        std::vector<char> done(T, 0);
        std::vector<std::vector<cam::OrthoMatrix>> groups;
        for (int l = 0; l < T && ce == cudaSuccess; ++l) {
            const int32_t g0 = p.tensors[l];
            if (done[l] || !c->is_matrix(g0)) continue;
            groups.emplace_back();
            for (int q = l; q < T; ++q) {
                const int32_t g = p.tensors[q];
                if (done[q] || !c->is_matrix(g) || c->rows[g] != c->rows[g0] ||
                    c->numel[g] != c->numel[g0])
                    continue;
                done[q] = 1;
                cam::OrthoMatrix om;
                om.theta = c->theta[g];
                om.e = c->e[g];
                om.rows = c->rows[g];
                om.cols = c->numel[g] / c->rows[g];
                for (int k = 0; k < CAM_KMAX; ++k) om.x[k] = k < K ? r->x[size_t(k) * T + q] : nullptr;
                groups.back().push_back(om);
            }
        }
        if (ce == cudaSuccess) {
            const int rc = cam::ortho_round(c->ortho, groups, op, s, c->sm_count, &c->launches);
            if (rc != CAM_OK) {
                close_round(r);
                return rc;
            }
        }
        if (ce == cudaSuccess && !cap) ce = cudaEventRecord(c->ortho_ev, s);
    }
    if (ce == cudaSuccess && norm_level >= 1 && !fuse) {
        ce = cam::launch_norm_finish(na, s);
        ++c->launches;
    }
    if (ce == cudaSuccess) ce = plan_mark(c, r->fragment, s, cap);
    if (ce == cudaSuccess && timed) ce = cudaEventRecord(c->commit_ev[1], s);
    if (ce == cudaSuccess) {
        cam_commit_record& rec = c->last_commit;
        rec.round = r->round;
        rec.fragment = r->fragment;
        rec.K = K;
        rec.mode = r->mode;
        rec.form = r->eager ? CAM_FORM_FOLDED
                 : r->ortho ? CAM_FORM_ORTHO
                            : (c->staged_launches > staged0 ? CAM_FORM_STAGED : CAM_FORM_REGISTER);
        rec.elements = p.n_elems;
        const int64_t xb = r->dtype == CAM_BF16 ? 2 : 4;
        const int64_t per = (r->eager ? 4 + (K - r->n_folded) * xb : K * xb) + 4 +
                            ((delta || norm_level >= 1) ? 4 : 0) +
                            (delta ? 8 : 0) + (r->ema ? 8 : 0) + (r->swa ? 8 : 0) +
                            (r->publish ? 4 : 0) + (r->publish_ema ? 4 : 0);
        rec.bytes = r->ortho ? 0 : per * p.n_elems;
        rec.launches = c->launches - launches0;
        rec.ms = -1.0f;
        c->has_last_commit = true;
        c->last_commit_timed = timed;
    }
    if (ce == cudaSuccess && r->swa)
        for (int32_t g : p.tensors) c->swa_count[g] = swa_prev + 1;
    close_round(r);
    if (ce != cudaSuccess) return cuda_fail(ce, "cam_merge_commit: launch");
    return CAM_OK;
}

CAM_API int cam_merge_commit_many(cam_round* const* rounds, int32_t n, void* stream) {
    const char* fn = "cam_merge_commit_many";
    if (!rounds || n < 1) return fail(CAM_E_ARG, "%s: no rounds", fn);
    if (n > cam::kMultiMax) return fail(CAM_E_ARG, "%s: at most %d rounds", fn, cam::kMultiMax);
    for (int i = 0; i < n; ++i) {
        if (!rounds[i]) return fail(CAM_E_ARG, "%s: round %d is NULL", fn, i);
        if (rounds[i]->ctx != rounds[0]->ctx)
            return fail(CAM_E_ARG, "%s: the rounds belong to different contexts", fn);
        for (int j = 0; j < i; ++j)
            if (rounds[j] == rounds[i]) return fail(CAM_E_ARG, "%s: round %d given twice", fn, i);
    }
    cam_ctx* c = rounds[0]->ctx;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool cap = capturing(s);
    // every round's checks before anything runs (open rounds never overlap:
    // cam_merge_begin refuses a fragment that shares tensors with one)
    for (int i = 0; i < n; ++i)
        if (const int rc = commit_checks(rounds[i], cap, fn); rc != CAM_OK) return rc;

    // One register-form pass for all of them when they are the same variant,
    // their norms (if any) finished in the pass, and their pointers fit;
    // otherwise one commit after another, in the given order.
    const cam_round* r0 = rounds[0];
    bool one_pass = n > 1 && c->fuse_finish;
    int64_t ptrs = 0;
    for (int i = 0; i < n && one_pass; ++i) {
        const cam_round* r = rounds[i];
        const Plan& p = c->plan_of(r->fragment);
        one_pass = !r->eager && !r->ortho && !r->swa && !r->worker_norms && r->dtype == r0->dtype &&
                   r->mode == r0->mode && r->ema == r0->ema && r->norms == r0->norms &&
                   r->publish == r0->publish &&
                   (!r->norms || (p.n_chunks() > 0 && p.n_chunks() <= cam::kFuseMaxChunks));
        ptrs += int64_t(p.n_tensors()) * (r->K + (r->publish ? 2 : 0));
    }
    if (!one_pass || ptrs > cam::kMultiXCap) {
        for (int i = 0; i < n; ++i)
            if (const int rc = cam_merge_commit(rounds[i], stream); rc != CAM_OK) return rc;
        return CAM_OK;
    }

    DeviceScope scope(c->device);
    if (scope.err != cudaSuccess) {
        for (int i = 0; i < n; ++i) close_round(rounds[i]);
        return cuda_fail(scope.err, "cam_merge_commit_many: cudaSetDevice");
    }
    const bool delta = r0->mode == CAM_MODE_DELTA_NESTEROV;
    const int norm_level = r0->norms ? 1 : 0;
    const uintptr_t xa = r0->dtype == CAM_F32 ? 32 : 16;
    cam::MultiArgs& a = *c->multi_args;
    a.n_rounds = n;
    a.status = c->d_status;
    std::memset(a.vec, 0, sizeof a.vec);
    // the rounds with fewest chunks first: their finishes then run while the
    // blocks still stream the longer rounds
    std::vector<int> ord(n);
    for (int i = 0; i < n; ++i) ord[i] = i;
    std::stable_sort(ord.begin(), ord.end(), [&](int x, int y) {
        return c->plan_of(rounds[x]->fragment).n_chunks() < c->plan_of(rounds[y]->fragment).n_chunks();
    });
    int32_t chunks = 0, xp = 0;
    size_t smem = 0;
    int64_t elems = 0, bytes = 0;
    for (int j = 0; j < n; ++j) {
        const cam_round* r = rounds[ord[j]];
        const Plan& p = c->plan_of(r->fragment);
        const int K = r->K, T = p.n_tensors(), stride = K + (r->publish ? 2 : 0);
        int64_t W = 0;
        for (int k = 0; k < K; ++k) W += r->tokens[k];
        cam::MultiRound& R = a.r[j];
        R.chunks = p.d_chunks;
        R.slots = p.d_slots;
        R.partials = norm_level ? p.d_partials : nullptr;
        R.fin_counter = p.d_fin_counter;
        const int32_t shared = cam::finish_smem_bytes(T, p.n_chunks()) <= cam::kFinishSmemMax ? 1 : 0;
        R.fin = NormArgs{p.d_partials, p.d_first, T, p.d_tsq, r->out_tensor, r->out_fragment,
                         0, nullptr, nullptr, nullptr, nullptr, p.n_chunks(), shared};
        if (norm_level && shared) smem = std::max(smem, cam::finish_smem_bytes(T, p.n_chunks()));
        R.c_begin = chunks;
        R.n_chunks = p.n_chunks();
        R.x0 = xp;
        R.vec0 = 0;  // (set below: one bit per tensor)
        R.n_local = T;
        R.stride = stride;
        R.K = K;
        R.Kf = static_cast<float>(K);
        for (int k = 0; k < CAM_KMAX; ++k) R.w[k] = k < K ? static_cast<float>(r->tokens[k]) : 0.0f;
        R.W = static_cast<float>(W);
        R.div = cam::div_plan(r->mode == CAM_MODE_DELTA_NESTEROV ? R.W : R.Kf);
        R.lr = r->lr;
        R.mu = r->mu;
        R.beta = r->beta;
        chunks += p.n_chunks();
        xp += T * stride;
        elems += p.n_elems;
        const int64_t xb = r->dtype == CAM_BF16 ? 2 : 4;
        bytes += (K * xb + 4 + ((delta || norm_level >= 1) ? 4 : 0) + (delta ? 8 : 0) +
                  (r->ema ? 8 : 0) + (r->publish ? 4 : 0) + (r->publish_ema ? 4 : 0)) *
                 p.n_elems;
    }
    // pointers and the vector-path bits, one bit per tensor over the rounds
    int32_t vb = 0;
    for (int j = 0; j < n; ++j) {
        const cam_round* r = rounds[ord[j]];
        const Plan& p = c->plan_of(r->fragment);
        cam::MultiRound& R = a.r[j];
        const int K = r->K, T = p.n_tensors();
        R.vec0 = vb;
        for (int l = 0; l < T; ++l) {
            const int32_t g = p.tensors[l];
            const void** xs = a.x + R.x0 + static_cast<size_t>(l) * R.stride;
            bool v = aligned(c->theta[g], 32) && (!delta || aligned(c->m[g], 32)) &&
                     (!r->ema || aligned(c->e[g], 32));
            for (int k = 0; k < K; ++k) {
                xs[k] = r->x[size_t(k) * T + l];
                v = v && aligned(xs[k], xa);
            }
            if (r->publish) {
                xs[K] = r->pub_theta[l];
                xs[K + 1] = r->publish_ema ? r->pub_ema[l] : nullptr;
                v = v && aligned(xs[K], 32) && aligned(xs[K + 1], 32);
            }
            if (v) a.vec[(vb + l) >> 5] |= 1u << ((vb + l) & 31);
        }
        vb += T;
    }
    a.n_chunks = chunks;  // (vb <= ptrs <= kMultiXCap: every tensor has a pointer)

    char label[96];
    std::snprintf(label, sizeof label, "cam_merge_commit_many %d rounds", n);
    NvtxRange nvtx(label);
    const int64_t launches0 = c->launches;
    cudaError_t ce = cudaSuccess;
    for (int i = 0; i < n && ce == cudaSuccess; ++i)
        ce = plan_order(c, rounds[i]->fragment, s, cap);  // after earlier work on these tensors
    const bool timed = c->time_commits && !cap;
    if (ce == cudaSuccess && timed) ce = cudaEventRecord(c->commit_ev[0], s);
    if (ce == cudaSuccess && chunks > 0) {
        const cam::MergeVariant v{r0->dtype, r0->mode, r0->ema, norm_level, r0->publish, false};
        // (all the rounds are in this launch: CAM_SHARE_SMS has nothing to leave room for)
        const int b = c->bps_multi[r0->dtype][r0->mode][r0->ema][norm_level][r0->publish];
        const int grid = static_cast<int>(std::min<int64_t>(chunks, int64_t(c->sm_count) * b));
        ce = cam::launch_merge_multi(a, v, grid, smem, s);
        ++c->launches;
    }
    for (int i = 0; i < n && ce == cudaSuccess; ++i) ce = plan_mark(c, rounds[i]->fragment, s, cap);
    if (ce == cudaSuccess && timed) ce = cudaEventRecord(c->commit_ev[1], s);
    if (ce == cudaSuccess) {
        const cam_round* rl = rounds[n - 1];
        cam_commit_record& rec = c->last_commit;
        rec.round = rl->round;
        rec.fragment = rl->fragment;
        rec.K = rl->K;
        rec.mode = rl->mode;
        rec.form = CAM_FORM_REGISTER;
        rec.elements = elems;
        rec.bytes = bytes;
        rec.launches = c->launches - launches0;
        rec.ms = -1.0f;
        c->has_last_commit = true;
        c->last_commit_timed = timed;
    }
    for (int i = 0; i < n; ++i) close_round(rounds[i]);
    if (ce != cudaSuccess) return cuda_fail(ce, "cam_merge_commit_many: launch");
    return CAM_OK;
}

CAM_API int cam_swa_reset(cam_ctx* c, int32_t fragment, void* stream) {
    if (!c) return fail(CAM_E_ARG, "cam_swa_reset: ctx is NULL");
    if (!c->has_swa) return fail(CAM_E_ARG, "cam_swa_reset: context has no average buffers");
    if (fragment < -1 || fragment >= c->n_fragments)
        return fail(CAM_E_ARG, "cam_swa_reset: fragment %d out of [-1, %d)", fragment, c->n_fragments);
    for (const cam_round* r : c->open)
        if (r->fragment == -1 || fragment == -1 || r->fragment == fragment)
            return fail(CAM_E_BUSY, "cam_swa_reset: fragment %d overlaps open round %lld", fragment,
                        static_cast<long long>(r->round));
    DeviceScope scope(c->device);
    if (scope.err != cudaSuccess) return cuda_fail(scope.err, "cam_swa_reset: cudaSetDevice");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (capturing(s))
        return fail(CAM_E_STATE, "cam_swa_reset: the counts it resets live on the host; not in a "
                                 "graph capture");
    const Plan& p = c->plan_of(fragment);
    cudaError_t ce = plan_order(c, fragment, s, false);
    for (int32_t g : p.tensors) {
        if (ce != cudaSuccess) break;
        if (c->numel[g] == 0) continue;
        ce = cam::launch_fill(c->swa[g], c->numel[g], 0.0f, s);
        ++c->launches;
    }
    if (ce == cudaSuccess) ce = plan_mark(c, fragment, s, false);
    if (ce != cudaSuccess) return cuda_fail(ce, "cam_swa_reset: launch");
    for (int32_t g : p.tensors) c->swa_count[g] = 0;
    return CAM_OK;
}

CAM_API int cam_swa_counts(const cam_ctx* c, int64_t* counts) {
    if (!c || !counts) return fail(CAM_E_ARG, "cam_swa_counts: NULL argument");
    std::memcpy(counts, c->swa_count.data(), sizeof(int64_t) * c->swa_count.size());
    return CAM_OK;
}

CAM_API int cam_swa_set_counts(cam_ctx* c, const int64_t* counts) {
    if (!c || !counts) return fail(CAM_E_ARG, "cam_swa_set_counts: NULL argument");
    if (!c->open.empty()) return fail(CAM_E_STATE, "cam_swa_set_counts: a round is open");
    for (int32_t t = 0; t < c->n_tensors; ++t)
        if (counts[t] < 0) return fail(CAM_E_ARG, "cam_swa_set_counts: counts[%d] < 0", t);
    c->swa_count.assign(counts, counts + c->n_tensors);
    return CAM_OK;
}

CAM_API int cam_fragment_info(const cam_ctx* c, int32_t fragment, int32_t* n_tensors,
                              int64_t* n_elems, int32_t* tensor_ids) {
    if (!c) return fail(CAM_E_ARG, "cam_fragment_info: ctx is NULL");
    if (fragment < -1 || fragment >= c->n_fragments)
        return fail(CAM_E_ARG, "cam_fragment_info: fragment %d out of [-1, %d)", fragment, c->n_fragments);
    const Plan& p = c->plan_of(fragment);
    if (n_tensors) *n_tensors = p.n_tensors();
    if (n_elems) *n_elems = p.n_elems;
    if (tensor_ids && !p.tensors.empty())
        std::memcpy(tensor_ids, p.tensors.data(), sizeof(int32_t) * p.tensors.size());
    return CAM_OK;
}

CAM_API int cam_ctx_launch_count(const cam_ctx* c, int64_t* out) {
    if (!c || !out) return fail(CAM_E_ARG, "cam_ctx_launch_count: NULL argument");
    *out = c->launches;
    return CAM_OK;
}

CAM_API int cam_ctx_status(cam_ctx* c, int32_t* out) {
    if (!c || !out) return fail(CAM_E_ARG, "cam_ctx_status: NULL argument");
    DeviceScope scope(c->device);
    if (scope.err != cudaSuccess) return cuda_fail(scope.err, "cam_ctx_status: cudaSetDevice");
    cudaError_t ce = cudaDeviceSynchronize();
    int32_t v = 0;
    if (ce == cudaSuccess) ce = cudaMemcpy(&v, c->d_status, sizeof v, cudaMemcpyDeviceToHost);
    if (ce != cudaSuccess) return cuda_fail(ce, "cam_ctx_status");
    *out = v;
    return CAM_OK;
}

CAM_API int cam_ctx_last_commit(cam_ctx* c, cam_commit_record* out) {
    if (!c || !out) return fail(CAM_E_ARG, "cam_ctx_last_commit: NULL argument");
    if (!c->has_last_commit) return fail(CAM_E_ARG, "cam_ctx_last_commit: no commit yet");
    *out = c->last_commit;
    if (c->last_commit_timed) {
        DeviceScope scope(c->device);
        float ms = 0.0f;
        cudaError_t ce = scope.err;
        if (ce == cudaSuccess) ce = cudaEventSynchronize(c->commit_ev[1]);
        if (ce == cudaSuccess) ce = cudaEventElapsedTime(&ms, c->commit_ev[0], c->commit_ev[1]);
        if (ce != cudaSuccess) return cuda_fail(ce, "cam_ctx_last_commit");
        out->ms = ms;
    }
    return CAM_OK;
}

CAM_API int cam_stream_capturing(void* stream, int32_t* out) {
    if (!out) return fail(CAM_E_ARG, "cam_stream_capturing: out is NULL");
    *out = capturing(static_cast<cudaStream_t>(stream)) ? 1 : 0;
    return CAM_OK;
}

CAM_API int cam_ctx_staged_count(const cam_ctx* c, int64_t* out) {
    if (!c || !out) return fail(CAM_E_ARG, "cam_ctx_staged_count: NULL argument");
    *out = c->staged_launches;
    return CAM_OK;
}

CAM_API int cam_ctx_get_last_round(const cam_ctx* c, int64_t* out) {
    if (!c || !out) return fail(CAM_E_ARG, "cam_ctx_get_last_round: NULL argument");
    *out = c->last_round;
    return CAM_OK;
}

CAM_API int cam_ctx_get_quorum(const cam_ctx* c, int32_t* out) {
    if (!c || !out) return fail(CAM_E_ARG, "cam_ctx_get_quorum: NULL argument");
    *out = c->quorum;
    return CAM_OK;
}

CAM_API int cam_ctx_set_quorum(cam_ctx* c, int32_t quorum) {
    if (!c) return fail(CAM_E_ARG, "cam_ctx_set_quorum: ctx is NULL");
    if (quorum < 1 || quorum > CAM_KMAX)
        return fail(CAM_E_ARG, "cam_ctx_set_quorum: quorum %d outside [1, %d]", quorum, CAM_KMAX);
    c->quorum = quorum;
    return CAM_OK;
}

CAM_API int cam_ctx_set_last_round(cam_ctx* c, int64_t round) {
    if (!c) return fail(CAM_E_ARG, "cam_ctx_set_last_round: ctx is NULL");
    if (!c->open.empty()) return fail(CAM_E_STATE, "cam_ctx_set_last_round: a round is open");
    if (round < c->last_round)
        return fail(CAM_E_STALE, "cam_ctx_set_last_round: %lld would lower %lld",
                    static_cast<long long>(round), static_cast<long long>(c->last_round));
    c->last_round = round;
    return CAM_OK;
}

CAM_API int cam_merge_round(cam_ctx* c, int64_t round, int32_t fragment, int32_t n_workers,
                            const void* const* const* ckpt, cam_dtype dtype,
                            const int64_t* tokens, cam_mode mode, float lr, float mu,
                            int32_t do_ema, float beta, double* per_tensor, double* per_fragment,
                            void* stream) {
    const char* fn = "cam_merge_round";
    if (!c) return fail(CAM_E_ARG, "%s: ctx is NULL", fn);
    if (!ckpt || n_workers < 1 || n_workers > CAM_KMAX)
        return fail(CAM_E_ARG, "%s: %d workers (1 to %d, with their pointer arrays)", fn,
                    static_cast<int>(n_workers), CAM_KMAX);
    cam_round* r = nullptr;
    if (const int rc = cam_merge_begin(c, round, fragment, &r); rc != CAM_OK) return rc;
    int rc = CAM_OK;
    for (int32_t k = 0; rc == CAM_OK && k < n_workers; ++k)
        rc = cam_merge_accumulate(r, ckpt[k], dtype, tokens ? tokens[k] : 0);
    if (rc == CAM_OK) rc = cam_merge_finalize(r, mode, lr, mu);
    if (rc == CAM_OK && do_ema) rc = cam_ema_update(r, beta);
    if (rc == CAM_OK && (per_tensor || per_fragment))
        rc = cam_drift_norm(r, per_tensor, per_fragment);
    // the commit's own checks first, so that a round that fails them is dropped
    // here (cam_merge_commit leaves such a round open for its caller)
    if (rc == CAM_OK) rc = commit_checks(r, capturing(static_cast<cudaStream_t>(stream)), fn);
    if (rc != CAM_OK) {
        close_round(r);  // nothing launched; the failing step's message stays
        return rc;
    }
    return cam_merge_commit(r, stream);  // closes the round, launched or not
}
