/*
 * cam.h -- C ABI of libcam, the GB300 DiLoCo outer-merge library.
 *
 * One merge round takes the round's worker checkpoints and moves the global
 * model (fp32 master weights theta) one outer step:
 *
 *   - plain replacement: theta' = mean of the workers, folded into a running
 *     fp32 sum in arrival order ("DiffuRefill-1B" model card, "How it is
 *     trained", Merging; "DiffuRefill-1B: Pretraining a Masked Diffusion
 *     Language Model on Free, Preemptible Notebook GPUs", section 3, Table 2,
 *     "Outer step": outer learning rate 1, no momentum);
 *   - outer Nesterov on the token-weighted mean of the deltas
 *     ("Pythia-14M on four rented GPUs and a bucket", "Getting updates through
 *     the bucket": learning rate 0.7, momentum 0.9);
 *
 * then optionally updates the EMA of the globals (same report, Table 2, "Side
 * averages", beta 0.9) and reports L2 drift norms. A round may be restricted to
 * one of F parameter fragments and closes only with a quorum of participants
 * (Pythia page, same section: fragments=4, quorum_size=3; two rounds may be in
 * flight at once).
 *
 * Element arithmetic (fixed, so results are reproducible bit for bit): every
 * operation is one IEEE binary32 operation rounded to nearest-even, no fused
 * multiply-add, correctly rounded division. With x_k the k-th worker's value
 * widened to fp32 (bf16 widening is exact), in accumulate- or fold-call order
 * k = 1..K:
 *   MEAN_REPLACE:    s = sum_k x_k;  theta' = s / K
 *   DELTA_NESTEROV:  s = sum_k w_k * (x_k - theta);  Delta = s / W,
 *                    w_k = (float)tokens_k, W = (float)(sum_k tokens_k);
 *                    g = -Delta;  m' = mu*m + g;  theta' = theta - lr*(g + mu*m')
 *   EMA:             e' = beta*e + (1 - beta)*theta'
 *   drift norm:      per tensor sqrt(sum_i delta_i^2), delta = Delta (DELTA mode)
 *                    or theta' - theta (MEAN mode), squares summed in a fixed
 *                    order (fp32 over runs of at most a few dozen squares,
 *                    then fp64), so they are reproducible bit for bit; per
 *                    fragment sqrt(sum over its tensors).
 *
 * Conventions:
 *   - Every call returns CAM_OK (0) or a negative cam_status. On any error the
 *     library state is unchanged unless the call's comment says otherwise, and
 *     cam_last_error() returns a message for the calling thread.
 *   - "device pointer" means memory on the context's CUDA device; "host
 *     pointer" means ordinary CPU memory read during the call only.
 *   - Device work is stream-ordered: a round's work on the stream passed to
 *     cam_merge_commit, a fold's on the stream passed to cam_merge_fold.
 *     Across streams the library orders, by CUDA events, work that shares
 *     tensors (commits, folds and cam_swa_reset of overlapping fragments run
 *     in call order) and orthogonalised commits (which share one workspace);
 *     rounds on disjoint fragments may overlap. Work the caller issues on
 *     the same buffers (reading theta, refilling a worker) is the caller's to
 *     order against the stream it passed.
 *     Only cam_ctx_create, cam_ctx_status and a timed cam_ctx_last_commit
 *     wait for the device, and the context's first fold or first
 *     orthogonalised commit, which allocate (cudaMalloc).
 *   - CUDA graphs: commits and folds issued on a stream that is being
 *     captured are recorded into the graph (kernel launches only, no event
 *     of the library), and every replay repeats them with the arguments of
 *     the capture, reading and writing the same buffers again. This removes
 *     the host cost of small rounds issued in a loop. Refused inside a
 *     capture (CAM_E_STATE), because a replay could not repeat them
 *     faithfully or they allocate: a running-average update or reset (its
 *     count lives on the host), a context's first fold and first
 *     orthogonalised commit. A timed context does not time captured commits.
 *   - Not thread-safe per context: calls on one context must not overlap.
 */
#ifndef CAM_H
#define CAM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define CAM_KMAX 8            /* most workers one round may accumulate */
#define CAM_MAX_OPEN_ROUNDS 8 /* rounds begun and not yet committed, per context */

typedef enum {
    CAM_OK = 0,
    CAM_E_ARG = -1,    /* null/invalid argument, size or dtype mismatch, non-finite scalar */
    CAM_E_STATE = -2,  /* call out of order (e.g. commit before finalize) */
    CAM_E_STALE = -3,  /* round number not newer than every round already begun */
    CAM_E_BUSY = -4,   /* the fragment overlaps a round that is open */
    CAM_E_QUORUM = -5, /* fewer accumulated workers than the quorum */
    CAM_E_KMAX = -6,   /* more than CAM_KMAX accumulate calls */
    CAM_E_CUDA = -7,   /* a CUDA call failed (no device, launch error, ...) */
    CAM_E_NOMEM = -8   /* host or device allocation failed */
} cam_status;

typedef enum { CAM_F32 = 0, CAM_BF16 = 1 } cam_dtype;

typedef enum {
    CAM_MODE_MEAN_REPLACE = 0,   /* plain mean, plain replacement */
    CAM_MODE_DELTA_NESTEROV = 1  /* token-weighted delta mean, outer Nesterov */
} cam_mode;

/* cam_ctx_desc.flags */
#define CAM_INIT_EMA_FROM_MASTER 1u /* at create: e <- theta (EMA starts at the first global) */
#define CAM_INIT_ZERO_MOMENTUM 2u   /* at create: m <- 0 */
#define CAM_INIT_ZERO_SWA 4u        /* at create: running averages <- 0, no globals folded */
#define CAM_NO_STAGING 8u           /* never use the staged (bulk-copy) form of the merge pass */
#define CAM_TIME_COMMITS 16u        /* time each commit's device work (cam_ctx_last_commit) */
#define CAM_NO_FUSED_FINISH 32u     /* always finish drift norms in a separate norm pass */
#define CAM_TEST_STALL_STAGED 64u   /* test hook, never for real rounds: every staged merge pass
                                       withholds its first tile and gives up waiting after
                                       about 1 ms (see cam_ctx_status) */
#define CAM_SHARE_SMS 128u          /* merge passes take at most three quarters of the register
                                       form's block slots, so rounds in flight on other streams
                                       start alongside */
#define CAM_TEST_BAD_CHUNK 256u     /* test hook, never for real rounds: the device copy of the
                                       chunk table runs the first tensor's last chunk 2,048
                                       elements past that tensor's end (see cam_ctx_status) */
#define CAM_TEST_BAD_TAG 512u       /* test hook, never for real rounds: every staged merge pass
                                       gives its end marker a wrong fill number and gives up
                                       waiting after about 1 ms (see cam_ctx_status) */

/* Bits of the device status word (cam_ctx_status) */
#define CAM_STATUS_WAIT_TIMEOUT 1 /* a staged merge pass gave up waiting for its copies */
#define CAM_STATUS_GEMM_TIMEOUT 2 /* a tensor-core GEMM of the orthogonalisation gave up waiting */
#define CAM_STATUS_BAD_CHUNK 4    /* a merge or fold pass met a chunk outside its tensor and
                                     skipped it */
#define CAM_STATUS_PROTOCOL 8     /* a staged merge pass found a stage or a drift hand-over out
                                     of sequence and stopped */

/* cam_merge_orthogonalize */
#define CAM_ORTHO_SCALE_FIXED 0      /* theta' = theta + lr * polar(Delta) */
#define CAM_ORTHO_SCALE_MATCH_NORM 1 /* ... + lr * |Delta|_F / sqrt(min(m, n)) * polar(Delta) */
#define CAM_ORTHO_TF32 0             /* GEMMs on the tensor cores, TF32 inputs, fp32 accumulation */
#define CAM_ORTHO_FP32 1             /* GEMMs in full fp32 on the CUDA cores */
#define CAM_ORTHO_BF16 2             /* iterate and GEMM inputs in bf16, fp32 accumulation */
#define CAM_ORTHO_SHORT_SIDE 4       /* OR into precision: iterate in the short side's space */

typedef struct cam_ctx cam_ctx;     /* opaque */
typedef struct cam_round cam_round; /* opaque */

/*
 * The merger's parameter list. Tensor t has numel[t] fp32 elements at
 * master[t] (theta), momentum[t] (m) and ema[t] (e); each is a contiguous
 * device buffer owned by the caller for the life of the context. momentum may
 * be NULL (Nesterov rounds are then rejected) and so may ema (ema_update is
 * then rejected). fragment_of[t] in [0, n_fragments) assigns tensors to
 * fragments (NULL: every tensor in fragment 0). A fragment's tensors are
 * always taken in increasing t: that is the "fragment order" of every
 * per-tensor array below. numel[t] may be 0. Buffers need no particular
 * alignment; 32-byte aligned buffers take the vectorised path.
 */
typedef struct {
    int32_t n_tensors;
    const int64_t* numel;       /* host, [n_tensors] */
    const int32_t* fragment_of; /* host, [n_tensors] or NULL */
    int32_t n_fragments;        /* >= 1 */
    int32_t quorum;             /* >= 1: accumulate calls needed to commit */
    float* const* master;       /* host array of n_tensors device pointers */
    float* const* momentum;     /* host array of n_tensors device pointers, or NULL */
    float* const* ema;          /* host array of n_tensors device pointers, or NULL */
    int32_t device;             /* CUDA device ordinal holding the buffers */
    uint32_t flags;             /* CAM_INIT_* */
    void* stream;               /* cudaStream_t for the CAM_INIT_* work; NULL = default */
    float* const* swa;          /* host array of n_tensors device pointers, or NULL:
                                   uniform running averages of the globals */
    const int64_t* rows;        /* host, [n_tensors] or NULL: tensor t is a row-major
                                   rows[t] x (numel[t] / rows[t]) matrix when both are >= 2
                                   and divide evenly; it matters only to orthogonalised
                                   rounds (cam_merge_orthogonalize) */
} cam_ctx_desc;

/*
 * Creates a context: validates the description, plans the chunking of every
 * fragment for the device, allocates the library's small device tables and
 * runs the CAM_INIT_* work on desc->stream. Copies every host array it reads.
 * Errors: CAM_E_ARG (invalid description, checked before any CUDA call),
 * CAM_E_CUDA (no usable device), CAM_E_NOMEM.
 */
int cam_ctx_create(const cam_ctx_desc* desc, cam_ctx** out);

/* Frees the context and every round still open on it. The caller makes sure
 * no committed work of the context is still running on the device. NULL is a
 * no-op. */
void cam_ctx_destroy(cam_ctx* ctx);

/*
 * Opens round `round` on `fragment` (or -1: every tensor). Round numbers must
 * strictly increase over the context's life, so a republished global always
 * carries a new number ("DiffuRefill-1B" technical report, section 3,
 * "Failure handling" (iii)). Errors: CAM_E_ARG (fragment out of range),
 * CAM_E_STALE (round not above every round begun so far), CAM_E_BUSY (an open
 * round covers an overlapping fragment), CAM_E_NOMEM.
 */
int cam_merge_begin(cam_ctx* ctx, int64_t round, int32_t fragment, cam_round** out);

/*
 * Adds one worker to the round, in arrival order: the merger sums the
 * downloaded checkpoints in the order they come in ("DiffuRefill-1B" model
 * card, "How it is trained", Merging), and in the token-weighted form each
 * worker's delta counts by the tokens it trained on ("Pythia-14M on four
 * rented GPUs and a bucket", "Getting updates through the bucket"). Nothing
 * is read here; the commit's pass reads every worker once. ckpt is a host array of
 * T_f device pointers, the worker's copy of each tensor of the fragment in
 * fragment order (each numel[t] contiguous elements of `dtype`). tokens is
 * the worker's token count (>= 0; used as its weight in DELTA_NESTEROV mode,
 * ignored in MEAN_REPLACE). The buffers are BORROWED: they must stay valid
 * and unmodified until the committed work has run on the commit stream.
 * Every accumulate of one round must use the same dtype. On a round that
 * has folded workers (cam_merge_fold), accumulated workers come after the
 * folds and are folded, in their order, by the commit's final pass.
 * Errors: CAM_E_ARG, CAM_E_STATE (already finalized), CAM_E_KMAX.
 */
int cam_merge_accumulate(cam_round* rd, const void* const* ckpt, cam_dtype dtype,
                         int64_t tokens);

/*
 * Like cam_merge_accumulate, but ckpt holds HOST pointers: the worker's
 * tensors stay in CPU memory and the fused pass streams them to the GPU itself
 * (over NVLink-C2C on Grace systems), so no staging copy or device buffer is
 * needed. This is the merger of the DiffuRefill-1B pages folding each
 * downloaded checkpoint as it arrives ("DiffuRefill-1B" model card, "How it
 * is trained", Merging), with the checkpoint in host RAM. Each buffer must be
 * readable by the device: page-locked memory mapped for it (cudaHostAlloc,
 * cudaHostRegister, pinned torch tensors), managed memory, or pageable memory
 * on systems where cudaDevAttrPageableMemoryAccess is 1. Anything else is
 * rejected with CAM_E_ARG before any work and the round is unchanged. Host
 * and device checkpoints may be mixed within a round. Borrowed like device
 * checkpoints. Errors: as cam_merge_accumulate.
 */
int cam_merge_accumulate_host(cam_round* rd, const void* const* ckpt, cam_dtype dtype,
                              int64_t tokens);

/*
 * Folds one arriving worker into the round at once ("DiffuRefill-1B" model
 * card, "How it is trained", Merging: each checkpoint is added to the running
 * fp32 sum as it comes in). ckpt holds the worker's T_f tensors in fragment
 * order, in device memory or in host memory the device can read (as for
 * cam_merge_accumulate_host). The fold runs on `stream` (a cudaStream_t, NULL
 * for the default stream):
 *
 * - MEAN_REPLACE: s <- s + x_k;
 * - DELTA_NESTEROV: s <- s + w_k * (x_k - theta);
 *
 * with s an fp32 running sum that starts at +0 with the first fold. The
 * buffers are borrowed only until this fold has run on `stream`, not until
 * commit.
 *
 * Rules of a folded round:
 *
 * - every fold of a round uses the same mode and dtype;
 * - cam_merge_finalize must later name that mode;
 * - folds come first: once a worker has been accumulated, no more folds;
 * - per-worker drift (cam_worker_drift_norm) must be asked for before the
 *   first fold;
 * - orthogonalisation is not available.
 *
 * Successive folds of a round may use different streams; the library orders
 * them, and the commit, after one another. cam_merge_commit then runs one
 * pass over the sums instead of over the workers, folding first any workers
 * accumulated after the folds. Per element, every operation and its order
 * are those of an accumulated round, so the results are the same bits.
 *
 * Folding all but the last arrival and accumulating the last one gives the
 * shortest time from the last arrival to the new global: its fold, the
 * finish and the published copies (cam_merge_publish) are one pass, whose
 * host-to-device reads and device-to-host writes share the link at once.
 *
 * The first fold of a context allocates one fp32 buffer as large as the
 * whole tensor list (CAM_E_NOMEM if it cannot).
 *
 * Errors: CAM_E_ARG, CAM_E_STATE (finalized, accumulated, or orthogonalised
 * round), CAM_E_KMAX, CAM_E_NOMEM, CAM_E_CUDA.
 */
int cam_merge_fold(cam_round* rd, const void* const* ckpt, cam_dtype dtype, int64_t tokens,
                   cam_mode mode, void* stream);

/*
 * Chooses the outer step. MEAN_REPLACE is plain replacement by the mean
 * ("DiffuRefill-1B" technical report, section 3, Table 2, "Outer step": outer
 * learning rate 1, no momentum) and ignores lr, mu and the token counts.
 * DELTA_NESTEROV is outer Nesterov on the token-weighted mean of the deltas
 * ("Pythia-14M on four rented GPUs and a bucket", "Getting updates through
 * the bucket": lr 0.7, momentum 0.9) and needs momentum buffers. lr and mu
 * must be finite.
 * Errors: CAM_E_ARG, CAM_E_STATE (finalized twice).
 */
int cam_merge_finalize(cam_round* rd, cam_mode mode, float lr, float mu);

/*
 * Asks for the EMA update e' = beta*e + (1-beta)*theta' on the round's
 * tensors, fused into the same pass: the EMA of the globals the merger keeps
 * beside them ("DiffuRefill-1B" technical report, section 3, Table 2, "Side
 * averages", beta 0.9; model card, "How it is trained", EMA). beta must be
 * finite. Needs EMA buffers.
 * Errors: CAM_E_ARG, CAM_E_STATE (asked twice).
 */
int cam_ema_update(cam_round* rd, float beta);

/*
 * Outer orthogonalisation ("DiffuRefill-1B" technical report, section 5.3,
 * where swapping the averaged update for its polar factor improved a
 * four-worker stand run). For every matrix-shaped tensor of the round (cam_ctx_desc.rows), the
 * plain-mean update Delta = mean_k(x_k) - theta (the same fp32 arithmetic as
 * a plain-mean round) is replaced by its polar factor U V^T, and
 * theta' = theta + s * U V^T with s = lr (CAM_ORTHO_SCALE_FIXED) or
 * s = lr * |Delta|_F / sqrt(min(m, n)) (CAM_ORTHO_SCALE_MATCH_NORM: the
 * update keeps Delta's Frobenius norm). Other tensors are merged by plain
 * replacement. The polar factor is reached by `iterations` Newton-Schulz
 * steps from Delta / |Delta|_F (X <- 1.5 X - 0.5 X X^T X in `precision`,
 * this library's own GEMM kernels: the tensor cores for CAM_ORTHO_TF32 and
 * CAM_ORTHO_BF16, the CUDA cores for CAM_ORTHO_FP32); singular values of
 * Delta below about 1.5^-(iterations - 8) of the largest have not converged
 * by then. Only plain-mean rounds, and only with an EMA update (no drift
 * norms, publish or running average: CAM_E_STATE at commit). The first
 * orthogonalised commit of a context allocates its workspace (Delta, two
 * iterates and their transposes with each side padded to a multiple of 128,
 * the Gram matrices, and 128 MiB of split partials; all equal-shape
 * matrices of the round at once, up to 2^29 elements per buffer).
 * Errors: CAM_E_ARG, CAM_E_STATE (asked twice).
 *
 * CAM_ORTHO_BF16 keeps the iterate and the Gram matrix in bf16 between
 * steps (fp32 accumulation inside each GEMM, tensor cores at bf16 rate).
 * Delta, its norm and the final step stay fp32. The polar factor carries
 * bf16 rounding, a few units of 2^-8 relative.
 *
 * CAM_ORTHO_SHORT_SIDE, OR-ed into precision, changes where the iteration
 * runs for matrices whose long side is at least 4 times the short side r.
 * Writing the iterate as X_k = X_0 P_k (tall) or P_k X_0 (wide), each step
 * becomes P <- 1.5 P - 0.5 P (P^T G P) on r x r matrices, with
 * G = X_0^T X_0 (tall) or X_0 X_0^T (wide). The iterates are the same in
 * exact arithmetic; the polar factor is then one product with X_0. Per
 * step that costs 6 r^3 flops instead of 4 m n r. G and the r x r steps run
 * in full fp32 whatever the precision; the final product uses `precision`.
 * G squares Delta's condition number, so rounding grows like
 * u * cond(Delta)^2: the option suits well-conditioned tall updates (token
 * embeddings), not ill-conditioned ones. Other shapes take the plain
 * iteration. It combines with CAM_ORTHO_TF32 or CAM_ORTHO_FP32 only.
 */
int cam_merge_orthogonalize(cam_round* rd, float lr, int32_t scale_mode, int32_t precision,
                            int32_t iterations);

/*
 * Asks for each worker's own drift, written on the commit stream: worker k
 * (arrival order) moved sqrt(sum_i (x_k - theta)^2) away from the global it
 * started from, theta being the global before this round. per_worker_tensor
 * (device, [K * T_f], worker-major: [k * T_f + t]) holds it per tensor and
 * per_worker (device, [K]) over the fragment; either may be NULL but not
 * both. K is the number of workers accumulated when the round commits.
 * This is the per-worker form of the local drift the DiffuRefill-1B report
 * tracks ("DiffuRefill-1B" technical report, section 5.1); a worker far from
 * the others shows up here. Computed in the same pass, squares summed in fp32
 * within a thread and fp64 above, in a fixed order. Errors: CAM_E_ARG,
 * CAM_E_STATE (asked twice).
 */
int cam_worker_drift_norm(cam_round* rd, double* per_worker_tensor, double* per_worker);

/*
 * Asks the same pass to fold the new global into each tensor's uniform
 * running average: swa' = swa + (theta' - swa) / n, n = the globals in the
 * average after this round (the first fold after a reset copies theta'
 * exactly). The DiffuRefill-1B run released the uniform average of the 130
 * globals of its final stretch ("DiffuRefill-1B" technical report, section 4
 * and Table 5). Needs average buffers; all tensors of the round's fragment
 * must hold the same number of globals (CAM_E_STATE at commit otherwise).
 * Errors: CAM_E_ARG, CAM_E_STATE (asked twice).
 */
int cam_swa_update(cam_round* rd);

/*
 * Asks for drift norms, written on the commit stream: per_tensor[T_f] (device
 * pointer, fragment order) and per_fragment[1] (device pointer); either may be
 * NULL but not both. Local drift is the workers' movement away from the last
 * global ("DiffuRefill-1B" technical report, section 5.1). Errors: CAM_E_ARG,
 * CAM_E_STATE (asked twice).
 */
int cam_drift_norm(cam_round* rd, double* per_tensor, double* per_fragment);

/*
 * Asks the fused pass to also write the new global theta' (and, when ema_out
 * is not NULL, the new EMA e') into theta_out[T_f] / ema_out[T_f], fragment
 * order, in the same pass that computes them. These are typically pinned host
 * buffers from which the merger publishes the new global and its EMA
 * ("DiffuRefill-1B" technical report, section 3, Table 2, "Merger" and "Side
 * averages"; the model card's Files: global_b.pt, global_ema.pt), so no
 * separate device-to-host copy follows the round. Each buffer holds numel[t]
 * floats and must be writable by the GPU (device memory of the context's
 * device, or host memory as for cam_merge_accumulate_host). ema_out needs an
 * EMA update in the same round (checked at commit, CAM_E_STATE). Errors:
 * CAM_E_ARG, CAM_E_STATE (asked twice).
 */
int cam_merge_publish(cam_round* rd, float* const* theta_out, float* const* ema_out);

/*
 * Closes the round: the merger publishes only once enough fresh checkpoints
 * are in ("DiffuRefill-1B" technical report, section 3, Table 2, "Merger";
 * "Pythia-14M on four rented GPUs and a bucket", "Getting updates through the
 * bucket": quorum_size). It checks the round (finalized, quorum met, weights valid), then
 * launches the fused merge pass (and the norm pass if asked, unless the round
 * is small enough for the merge pass to finish the norms itself) on `stream`
 * (a cudaStream_t; NULL = legacy default stream) and frees the round handle.
 * Returns before the device work finishes. On CAM_E_STATE / CAM_E_QUORUM /
 * CAM_E_ARG, and CAM_E_NOMEM (the workspace of a context's first
 * orthogonalised round), nothing is launched and the round stays open. On
 * CAM_E_CUDA the round is freed and the fragment's buffers are undefined.
 * So the handle is gone exactly when the call returns CAM_OK or CAM_E_CUDA.
 */
int cam_merge_commit(cam_round* rd, void* stream);

/*
 * Commits n open rounds of one context (n <= CAM_MAX_OPEN_ROUNDS; open rounds
 * never share tensors) as if cam_merge_commit were called for each in array
 * order on `stream`, with the same results bit for bit. "Pythia-14M on four
 * rented GPUs and a bucket", "Getting updates through the bucket": fragments
 * have rounds of their own and two may be in flight at once, so rounds can
 * close together; their merges then share one pass. When the rounds are the
 * same variant of the register form -- the same worker dtype, mode, EMA
 * update, drift norms or none (no per-worker drift), published copies or
 * none, no running-average update, eager folds or orthogonalisation, norms
 * finished in the pass (at most 4,096 chunks per fragment, the context not
 * created with CAM_NO_FUSED_FINISH) -- and their worker and copy pointers
 * number at most 3,584 together, one launch merges all of them: its blocks
 * take every round's chunks, a round's norms are finished by the block that
 * completes its last chunk, and short rounds end while long ones still
 * stream. Otherwise the rounds are committed one after another.
 *
 * Every round is checked as cam_merge_commit checks it before anything runs:
 * on CAM_E_ARG (NULL or repeated handles, rounds of different contexts, more
 * than CAM_MAX_OPEN_ROUNDS), CAM_E_STATE or CAM_E_QUORUM nothing is launched
 * and every round stays open. On CAM_E_CUDA the rounds of a shared pass are
 * freed and their buffers undefined; rounds committed one after another
 * behave as cam_merge_commit, in order, and a failure leaves the later ones
 * open. cam_ctx_last_commit then describes the last round of the array, with
 * the elements, bytes, launches and time of the whole call.
 */
int cam_merge_commit_many(cam_round* const* rounds, int32_t n, void* stream);

/* Drops an open round without touching any buffer. The round number stays
 * used. */
int cam_merge_abort(cam_round* rd);

/*
 * One whole round in one call, for callers whose host time per round counts
 * (small fragment rounds committed back to back, as in the Pythia-14M run:
 * "Pythia-14M on four rented GPUs and a bucket", "Getting updates through
 * the bucket"). It is cam_merge_begin(round, fragment); cam_merge_accumulate
 * of workers 0 .. n_workers-1, in that (arrival) order; cam_merge_finalize
 * (mode, lr, mu); cam_ema_update(beta) when do_ema is nonzero;
 * cam_drift_norm(per_tensor, per_fragment) when either is non-NULL; and
 * cam_merge_commit(stream): the same checks, launches and results, in one
 * host call.
 *
 * ckpt is a host array of n_workers (1 .. CAM_KMAX) pointers, ckpt[k] worker
 * k's host array of T_f device pointers in fragment order (as for
 * cam_merge_accumulate), every worker of `dtype`. tokens is a host array of
 * n_workers token counts, or NULL for none (then only MEAN_REPLACE can
 * commit). per_tensor and per_fragment are device arrays as for
 * cam_drift_norm, or NULL. The workers' buffers and the norm outputs are
 * borrowed as for those calls, until the work has run on `stream`.
 *
 * On an error before the commit's launches nothing is launched, the round
 * is dropped as by cam_merge_abort (its number counts as used) and the
 * failing step's error is returned; an error in the launches is returned as
 * cam_merge_commit returns it. Errors: those of the calls above.
 */
int cam_merge_round(cam_ctx* ctx, int64_t round, int32_t fragment, int32_t n_workers,
                    const void* const* const* ckpt, cam_dtype dtype, const int64_t* tokens,
                    cam_mode mode, float lr, float mu, int32_t do_ema, float beta,
                    double* per_tensor, double* per_fragment, void* stream);

/* Number of tensors and elements of `fragment` (-1: all), and its tensor
 * indices in fragment order when `tensor_ids` (host, [T_f]) is not NULL. */
int cam_fragment_info(const cam_ctx* ctx, int32_t fragment, int32_t* n_tensors,
                      int64_t* n_elems, int32_t* tensor_ids);

/* Highest round number begun so far (-1 before the first), and restoring it
 * when a merger restarts from saved state. set fails with CAM_E_STATE while a
 * round is open and with CAM_E_STALE when it would lower the number. */
int cam_ctx_get_last_round(const cam_ctx* ctx, int64_t* out);
int cam_ctx_set_last_round(cam_ctx* ctx, int64_t round);

/* The quorum later commits require, changed without rebuilding the context:
 * a merger left with fewer live workers merges the leftovers with a lower
 * quorum, down to a single participant ("Pythia-14M on four rented GPUs and a
 * bucket", the run's last round had one participant; "DiffuRefill-1B"
 * technical report, section 3, "Failure handling": the merger can go on with
 * N = 1). Applies to rounds committed afterwards, open ones included.
 * Errors: CAM_E_ARG (NULL, or quorum outside [1, CAM_KMAX]). */
int cam_ctx_get_quorum(const cam_ctx* ctx, int32_t* out);
int cam_ctx_set_quorum(cam_ctx* ctx, int32_t quorum);

/* Kernels this context has launched so far (merge passes, norm passes and
 * the CAM_INIT_* work), for accounting what a timed region ran. */
int cam_ctx_launch_count(const cam_ctx* ctx, int64_t* out);

/*
 * The merge pass has two forms with the same results, element for element.
 *
 * - The register form loads each thread's elements into registers.
 * - The staged form streams tiles of every input array into a ring of
 *   shared-memory stages with the TMA engine's bulk copies. It keeps more
 *   bytes in flight per SM.
 *
 * A commit uses the staged form for every launch that meets all of these:
 *
 * - its workers came through cam_merge_accumulate;
 * - its buffers are all vector-aligned;
 * - the round writes at most two state arrays: theta plus m or e.
 *
 * Rounds that write three state arrays (Nesterov with an EMA update, or an
 * EMA update with a running-average update) measure faster in the register
 * form, so they keep it. Rounds with workers from cam_merge_accumulate_host
 * always use the register form, and so does a context created with
 * CAM_NO_STAGING.
 *
 * Small rounds that ask for the round's drift norms (not per-worker drift),
 * whose fragment has at most 4,096 chunks (about 64M elements) and fits one
 * launch, take the register form and finish the norms in that same pass: the
 * pass's last block to finish sums the per-chunk partials exactly as the norm
 * pass would, so the results are the same bits, one launch fewer. A context
 * created with CAM_NO_FUSED_FINISH always launches the separate norm pass.
 *
 * A context created with CAM_SHARE_SMS keeps every merge pass in the
 * register form with at most three quarters of the form's block slots (the
 * blocks the device holds at once). The pass of a round in flight on another
 * stream then starts beside it instead of after it: a long round and short
 * rounds of other fragments overlap. The results are the same bits.
 *
 * Every wait of the staged form on one of its barriers gives up after a few
 * seconds. It then sets CAM_STATUS_WAIT_TIMEOUT in the context's device status
 * word, and the results of that commit are undefined. A context created with
 * CAM_TEST_STALL_STAGED exercises that path on purpose: its staged passes
 * never issue their first tile's copies, their waits give up after about
 * 1 ms instead, every copy they did issue lands before the pass returns, and
 * the status word reports the timeout. It exists to test this failure path
 * without hanging or faulting the GPU; the buffers of such a round are
 * left partly written.
 *
 * The merge and fold passes also check every chunk of the context's tables
 * as they take it: its tensor among the launch's, at least one element, all
 * of them inside the tensor. The tables are built and checked on the host at
 * cam_ctx_create, so a chunk fails only if its table was corrupted in device
 * memory; the pass then reads and writes nothing for that chunk, counts its
 * drift as 0, and sets CAM_STATUS_BAD_CHUNK. A context created with
 * CAM_TEST_BAD_CHUNK plants such a chunk (in every table of two or more
 * tensors, the first tensor's last chunk reaches 2,048 elements past its
 * end) to test this; the caller gives that tensor's buffers (state, workers
 * and published copies) 2,048 spare elements past its end, so that even an
 * unchecked pass would stay inside them. The staged form further checks its
 * own protocol: the marker that ends a block's stages carries the number of
 * stages filled, which its consumers compare with the number they took, and
 * each drift hand-over carries its chunk count, which the reducer compares
 * with its own; a mismatch sets CAM_STATUS_PROTOCOL and stops the pass as a
 * timeout does. A context created with CAM_TEST_BAD_TAG has every staged pass
 * mislabel its end marker to test this (its waits give up after about 1 ms,
 * as with CAM_TEST_STALL_STAGED).
 *
 * cam_ctx_status waits for all work on the context's device, then writes the
 * word (0: nothing went wrong) to *out. The word stays set once set.
 * Errors: CAM_E_ARG, CAM_E_CUDA.
 */
int cam_ctx_status(cam_ctx* ctx, int32_t* out);

/* What the last successful cam_merge_commit of a context did. */
typedef struct {
    int64_t round;
    int32_t fragment;   /* -1: every tensor */
    int32_t K;          /* workers merged */
    int32_t mode;       /* cam_mode */
    int32_t form;       /* CAM_FORM_* of the merge pass */
    int64_t elements;   /* elements of the round's tensors */
    int64_t bytes;      /* algorithmic bytes of the merge pass (0 for orthogonalised rounds) */
    int64_t launches;   /* kernels the commit launched */
    float ms;           /* device time of the commit's work, or -1 without CAM_TIME_COMMITS */
} cam_commit_record;

#define CAM_FORM_REGISTER 0 /* the register form of the merge pass */
#define CAM_FORM_STAGED 1   /* the staged (bulk-copy) form */
#define CAM_FORM_FOLDED 2   /* the final pass of an eagerly folded round */
#define CAM_FORM_ORTHO 3    /* an orthogonalised round */

/*
 * Copies the record of the context's last successful commit to *out. The
 * algorithmic bytes count every byte the pass must move once:
 *
 * - per element, K worker elements (4 B fp32, 2 B bf16), or the 4-byte
 *   running sum of a folded round;
 * - theta written (4 B), and read (4 B) in delta mode or with drift norms;
 * - m read and written (8 B) in delta mode;
 * - e read and written (8 B) with an EMA update;
 * - the running average read and written (8 B);
 * - 4 B for each published copy.
 *
 * With CAM_TIME_COMMITS, ms is the device time between events recorded
 * before the commit's first launch and after its last; the call then waits
 * for that commit to finish. Errors: CAM_E_ARG (NULL, or no commit yet),
 * CAM_E_CUDA.
 */
int cam_ctx_last_commit(cam_ctx* ctx, cam_commit_record* out);

/* Merge passes this context has launched in the staged form (a subset of
 * cam_ctx_launch_count), so a caller can tell which form a round took. */
int cam_ctx_staged_count(const cam_ctx* ctx, int64_t* out);

/* *out = 1 while `stream` (a cudaStream_t, NULL = legacy default stream) is
 * being captured into a CUDA graph, else 0: what a binding needs to know to
 * skip its own per-stream bookkeeping for captured work. Errors: CAM_E_ARG
 * (out NULL). */
int cam_stream_capturing(void* stream, int32_t* out);

/*
 * cam_merge_round_noalloc -- a whole round (accumulate, finalize, optional
 * EMA update and drift norms, commit) in one call that allocates no memory.
 * The pages have no counterpart to this call: it exists for callers that may
 * not allocate device memory. One example is code embedded in a host
 * framework whose memory pool has reserved the device's memory up front, so a
 * cudaMalloc outside it fails or fragments the pool. Another is a merge issued
 * on a path where cudaMalloc/cudaFree would synchronise the device and stall
 * other streams. cam_ctx_create allocates its tables; this call needs no
 * context.
 *
 * Arguments, all plain pointers: n_tensors in [0, CAM_NOALLOC_MAX_TENSORS];
 * numel (host, [n_tensors]); master / momentum / ema (host arrays of device
 * pointers to fp32 buffers, as in cam_ctx_desc; momentum is needed for
 * DELTA_NESTEROV, ema when ema_update != 0); n_workers in [1, CAM_KMAX];
 * ckpt (host, [n_workers * n_tensors] device pointers, worker-major in arrival
 * order: ckpt[k * n_tensors + t]); dtype of every checkpoint; tokens (host,
 * [n_workers], read in DELTA_NESTEROV mode only); mode, lr, mu, beta as for
 * the context calls; per_tensor ([n_tensors]) and per_round ([1]) are device
 * pointers for the drift norms, either or both NULL. The element arithmetic
 * is the one documented at the top of this header, so the results equal those
 * of a context round on the same inputs. Buffers must live on the current
 * CUDA device; the work is queued on `stream` and the call returns before it
 * runs.
 *
 * Memory: the drift partials live in one fixed array in the library's device
 * memory: (CAM_NOALLOC_MAX_CHUNKS + CAM_NOALLOC_MAX_TENSORS) doubles, about
 * 1.1 MB, held on every GPU that loads the library until the process exits.
 * A round is cut into chunks of at most 16,384 elements, so one call covers
 * at most CAM_NOALLOC_MAX_CHUNKS chunks (about 2.1e9 elements). Larger rounds,
 * and more than CAM_NOALLOC_MAX_TENSORS tensors, are rejected with CAM_E_ARG
 * before any CUDA call. (Rounds under about 2e7 elements use shorter chunks,
 * chosen from the device's SM count; their exact chunk count is checked after
 * the device lookup, still before any launch, and stays far below the limit.)
 * The array keeps the previous call's contents; every
 * entry a call reads is written by that call first, so nothing needs
 * clearing. All calls share the one array: calls whose device work overlaps
 * (different streams without ordering, or several host threads) race on it
 * whenever one of them asks for norms. Calls on one stream are ordered and safe.
 *
 * The first call on each device looks up the array's device address and the
 * device's properties, with that device current; make that first call before
 * any stream capture. The address is kept for the life of the process: after
 * cudaDeviceReset on a device (a new context, where the array may sit
 * elsewhere) the process must not call this entry point on that device again.
 * Errors: CAM_E_ARG (argument and size checks, before any CUDA call),
 * CAM_E_CUDA.
 */
#define CAM_NOALLOC_MAX_TENSORS 4096
#define CAM_NOALLOC_MAX_CHUNKS 131072
int cam_merge_round_noalloc(int32_t n_tensors, const int64_t* numel, float* const* master,
                            float* const* momentum, float* const* ema, int32_t n_workers,
                            const void* const* ckpt, cam_dtype dtype, const int64_t* tokens,
                            cam_mode mode, float lr, float mu, int32_t ema_update, float beta,
                            double* per_tensor, double* per_round, void* stream);

/*
 * A worker adopting the new global while keeping the progress it made since
 * its last push: theta_w <- theta_w + (g - theta_pushed), per element a
 * binary32 subtraction then addition. The DiffuRefill-1B run tried this and
 * found it worse than plain replacement in 60 of 63 probes ("DiffuRefill-1B"
 * technical report, section 5.1), so plain replacement (copying g) remains
 * the default; this call exists to run and measure the alternative.
 * theta_w[t] (fp32, updated in place), global[t] (fp32) and pushed[t] (the
 * checkpoint as pushed, fp32 or bf16) are device pointers to numel[t]
 * elements, all arrays host arrays of n_tensors entries. No context and no
 * allocation; queued on `stream`. Errors: CAM_E_ARG (checked before any CUDA
 * call), CAM_E_CUDA.
 */
int cam_adopt_keep_drift(int32_t n_tensors, const int64_t* numel, float* const* theta_w,
                         const float* const* global, const void* const* pushed,
                         cam_dtype pushed_dtype, void* stream);

/* Message describing the calling thread's last error ("" if none). */
const char* cam_last_error(void);

/* Starts the running averages of `fragment` (-1: all) afresh: zeroes them on
 * `stream` and sets their counts to 0. Errors: CAM_E_ARG, CAM_E_BUSY (an open
 * round overlaps the fragment), CAM_E_CUDA. */
int cam_swa_reset(cam_ctx* ctx, int32_t fragment, void* stream);

/* The number of globals in each tensor's running average (counts, host,
 * [n_tensors]), and restoring it when a merger restarts from saved state
 * (CAM_E_STATE while a round is open). */
int cam_swa_counts(const cam_ctx* ctx, int64_t* counts);
int cam_swa_set_counts(cam_ctx* ctx, const int64_t* counts);

/* Library version, e.g. "0.1.0". */
const char* cam_version(void);

#ifdef __cplusplus
}
#endif

#endif /* CAM_H */
