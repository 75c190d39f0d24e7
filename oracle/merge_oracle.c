/*
 * merge_oracle.c -- the DiLoCo outer merge, restated as plain, slow CPU loops.
 *
 * TEST INFRASTRUCTURE. This file is the oracle that the CUDA path is checked
 * against; it is not part of the product. Only the test suite, the package's
 * smoke check and the benchmark's CPU-baseline and reference arms may load or
 * call it. It shares no code, header, table or helper with the CUDA library.
 *
 * What it follows (sources are the pages' titles and sections):
 *   [MC]  "DiffuRefill-1B" model card, "How it is trained", Merging bullet:
 *         the round's checkpoints are averaged as a plain mean, folded into a
 *         running fp32 sum as they arrive.  EMA bullet: an exponential average
 *         of the globals with beta 0.9.
 *   [TR]  "DiffuRefill-1B: Pretraining a Masked Diffusion Language Model on
 *         Free, Preemptible Notebook GPUs", section 3 (Training system),
 *         Table 2: "Outer step" row -- plain replacement, the new global is the
 *         mean of the workers (outer learning rate 1, no momentum);
 *         "Side averages" row -- EMA of the globals, beta 0.9.
 *   [GM]  "Pythia-14M on four rented GPUs and a bucket", section "Getting
 *         updates through the bucket": the merge takes a token-weighted mean
 *         of the deltas and applies an outer Nesterov optimizer (learning rate
 *         0.7, momentum 0.9).
 *   [TR 4] same report, section 4 (Data and schedule): the released weights
 *         are the uniform average of the 130 merged globals of the final
 *         stretch; section 5.4 / Table 5: uniform average and averages of
 *         the last 3 and 5 snapshots.
 *   [TR 5.1] same report, section 5.1 (Distributed optimisation): local
 *         drift, the movement of the workers away from the last global, and
 *         the rejected alternative to plain replacement, adopting the global
 *         as theta <- theta + (g - theta_pushed), which keeps each worker's
 *         progress since its last push.
 *
 * Readings where the pages leave a step open (each is listed with its reason
 * in the design notes of the repository):
 *   - delta sign: a worker's delta is x_k - theta; the outer pseudo-gradient is
 *     g = theta - (theta + Delta) = -Delta, so lr 1 / momentum 0 lands exactly
 *     on the token-weighted mean of the workers;
 *   - Nesterov form: momentum buffer m' = mu*m + g, step g + mu*m',
 *     theta' = theta - lr*step, m starting at zero (dampening 0);
 *   - weighted mean: weights are the token counts w_k, summed first
 *     (s = sum_k w_k*(x_k - theta), arrival order), then divided by W = sum w_k;
 *   - plain mean ignores token counts;
 *   - EMA input is the new global theta' (after the outer step), no bias
 *     correction;
 *   - uniform average of the globals (SWA): kept as a running mean,
 *     mu_n = mu_{n-1} + (theta_n - mu_{n-1}) / n, n counting the globals
 *     folded since the average was last reset (mu_1 = theta_1 exactly);
 *   - drift: per tensor the L2 norm of the mean worker displacement
 *     (Delta in the token-weighted mode, mean - theta_old in the plain mode),
 *     squares summed in fp64 in index order; per worker, the L2 norm of that
 *     worker's displacement x_k - theta_old;
 *   - keeping local drift on adoption: theta_w + (g - theta_pushed), the
 *     difference taken first, as the report writes it.
 *
 * Arithmetic: every operation below is one IEEE binary32 operation rounded to
 * nearest-even (the build passes -ffp-contract=off so no multiply-add is
 * fused). bf16 storage is widened by placing its 16 bits above 16 zero bits.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORA_F32 0
#define ORA_BF16 1

#define ORA_MEAN_REPLACE 0
#define ORA_DELTA_NESTEROV 1

#define ORA_OK 0
#define ORA_EARG (-1)

#define ORA_KMAX 64

/* ---- step: widen one stored value to fp32 ------------------------------- */

/* A bf16 value is the high half of a binary32, so widening is exact. */
static float widen_bf16(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

static float load_elem(const void* base, int dtype, int64_t i) {
    if (dtype == ORA_BF16) return widen_bf16(((const uint16_t*)base)[i]);
    return ((const float*)base)[i];
}

/* ---- step: plain mean, folded into a running fp32 sum [MC], [TR Tab.2] --- */

static float plain_mean(int K, const float* xs) {
    float s = 0.0f;
    for (int k = 0; k < K; ++k) s = s + xs[k]; /* arrival order */
    return s / (float)K;
}

/* ---- step: token-weighted mean of the deltas [GM] ------------------------ */

static float weighted_delta(int K, const float* xs, const float* w, float W,
                            float theta) {
    float s = 0.0f;
    for (int k = 0; k < K; ++k) {
        float d = xs[k] - theta;  /* worker k's delta against the global */
        float wd = w[k] * d;
        s = s + wd;               /* arrival order */
    }
    return s / W;
}

/* ---- step: outer Nesterov on the pseudo-gradient g = -Delta [GM] --------- */

static void outer_nesterov(float delta, float lr, float mu, float* theta,
                           float* m) {
    float g = -delta;
    float m_new = mu * (*m) + g;
    float step = g + mu * m_new;
    *theta = *theta - lr * step;
    *m = m_new;
}

/* ---- step: EMA of the globals [MC], [TR Tab.2] --------------------------- */

static float ema_step(float e, float theta_new, float beta) {
    float one_minus_beta = 1.0f - beta;
    return beta * e + one_minus_beta * theta_new;
}

/* ---- step: uniform running average of the globals [TR 4], [TR Tab.5] ---- */

static float swa_step(float mu, float theta_new, float n) {
    float d = theta_new - mu;
    return mu + d / n;
}

/* ---- exported single-step entry points (used to pin each step) ----------- */

int ora_widen_bf16(int64_t n, const uint16_t* in, float* out) {
    if (n < 0 || (n > 0 && (!in || !out))) return ORA_EARG;
    for (int64_t i = 0; i < n; ++i) out[i] = widen_bf16(in[i]);
    return ORA_OK;
}

int ora_plain_mean(int64_t n, int K, const void* const* x, int dtype,
                   float* out) {
    if (n < 0 || K < 1 || K > ORA_KMAX || !x || !out) return ORA_EARG;
    float xs[ORA_KMAX];
    for (int64_t i = 0; i < n; ++i) {
        for (int k = 0; k < K; ++k) xs[k] = load_elem(x[k], dtype, i);
        out[i] = plain_mean(K, xs);
    }
    return ORA_OK;
}

static int weights_of(int K, const int64_t* tokens, float* w, float* W) {
    int64_t total = 0;
    for (int k = 0; k < K; ++k) {
        if (tokens[k] < 0) return ORA_EARG;
        total += tokens[k];
        w[k] = (float)tokens[k];
    }
    if (total <= 0) return ORA_EARG;
    *W = (float)total;
    return ORA_OK;
}

int ora_weighted_delta(int64_t n, int K, const void* const* x, int dtype,
                       const int64_t* tokens, const float* theta, float* out) {
    if (n < 0 || K < 1 || K > ORA_KMAX || !x || !tokens || !theta || !out)
        return ORA_EARG;
    float w[ORA_KMAX], W;
    if (weights_of(K, tokens, w, &W) != ORA_OK) return ORA_EARG;
    float xs[ORA_KMAX];
    for (int64_t i = 0; i < n; ++i) {
        for (int k = 0; k < K; ++k) xs[k] = load_elem(x[k], dtype, i);
        out[i] = weighted_delta(K, xs, w, W, theta[i]);
    }
    return ORA_OK;
}

int ora_outer_nesterov(int64_t n, const float* delta, float lr, float mu,
                       float* theta, float* m) {
    if (n < 0 || !delta || !theta || !m) return ORA_EARG;
    for (int64_t i = 0; i < n; ++i) outer_nesterov(delta[i], lr, mu, &theta[i], &m[i]);
    return ORA_OK;
}

int ora_ema(int64_t n, const float* theta_new, float beta, float* e) {
    if (n < 0 || !theta_new || !e) return ORA_EARG;
    for (int64_t i = 0; i < n; ++i) e[i] = ema_step(e[i], theta_new[i], beta);
    return ORA_OK;
}

/* Folds one more global into the running average: swa <- swa + (theta_new -
 * swa) / count, where count >= 1 is the number of globals in the average
 * after this one. */
int ora_swa(int64_t n, const float* theta_new, int64_t count, float* swa) {
    if (n < 0 || count < 1 || !theta_new || !swa) return ORA_EARG;
    float nf = (float)count;
    for (int64_t i = 0; i < n; ++i) swa[i] = swa_step(swa[i], theta_new[i], nf);
    return ORA_OK;
}

/* Sum over elements of (x_k - theta)^2 for every worker k, each difference one
 * fp32 subtraction, the squares summed in fp64 in index order [TR 5.1]. */
int ora_worker_drift(int64_t n, int K, const void* const* x, int dtype,
                     const float* theta, double* sumsq) {
    if (n < 0 || K < 1 || K > ORA_KMAX || !x || !theta || !sumsq) return ORA_EARG;
    for (int k = 0; k < K; ++k) {
        double acc = 0.0;
        for (int64_t i = 0; i < n; ++i) {
            float d = load_elem(x[k], dtype, i) - theta[i];
            acc += (double)d * (double)d;
        }
        sumsq[k] = acc;
    }
    return ORA_OK;
}

/* Adopting the new global g while keeping the progress made since the push:
 * theta_w <- theta_w + (g - theta_pushed) [TR 5.1]. theta_pushed has dtype
 * `dtype` (the checkpoint as pushed); theta_w and g are fp32. */
int ora_adopt_keep_drift(int64_t n, float* theta_w, const float* g, const void* pushed,
                         int dtype) {
    if (n < 0 || !theta_w || !g || !pushed) return ORA_EARG;
    for (int64_t i = 0; i < n; ++i) {
        float d = g[i] - load_elem(pushed, dtype, i);
        theta_w[i] = theta_w[i] + d;
    }
    return ORA_OK;
}

/* ---- one tensor of one merge round -------------------------------------- */

/*
 * Applies one round to one tensor of numel elements, in place on theta (and
 * m, e when used).  x[0..K-1] are the included workers' copies of the tensor
 * in arrival order, all of dtype `dtype`.  tokens[k] is worker k's token count
 * (read only in the token-weighted mode).  When do_ema is non-zero the EMA is
 * updated from the new theta.  When sumsq is not NULL it receives the sum over
 * elements of the squared drift, accumulated in fp64 in index order.
 */
int ora_merge_tensor(int64_t numel, int K, const void* const* x, int dtype,
                     const int64_t* tokens, int mode, float lr, float mu,
                     int do_ema, float beta, float* theta, float* m, float* e,
                     double* sumsq) {
    if (numel < 0 || K < 1 || K > ORA_KMAX || !x || !theta) return ORA_EARG;
    if (dtype != ORA_F32 && dtype != ORA_BF16) return ORA_EARG;
    if (mode != ORA_MEAN_REPLACE && mode != ORA_DELTA_NESTEROV) return ORA_EARG;
    if (do_ema && !e) return ORA_EARG;
    float w[ORA_KMAX], W = 0.0f;
    if (mode == ORA_DELTA_NESTEROV) {
        if (!m || !tokens) return ORA_EARG;
        if (weights_of(K, tokens, w, &W) != ORA_OK) return ORA_EARG;
    }
    double acc = 0.0;
    float xs[ORA_KMAX];
    for (int64_t i = 0; i < numel; ++i) {
        for (int k = 0; k < K; ++k) xs[k] = load_elem(x[k], dtype, i);
        float theta_old = theta[i];
        float drift;
        if (mode == ORA_MEAN_REPLACE) {
            float mean = plain_mean(K, xs);
            drift = mean - theta_old;
            theta[i] = mean;               /* plain replacement */
        } else {
            float delta = weighted_delta(K, xs, w, W, theta_old);
            drift = delta;
            outer_nesterov(delta, lr, mu, &theta[i], &m[i]);
        }
        if (do_ema) e[i] = ema_step(e[i], theta[i], beta);
        acc += (double)drift * (double)drift;
    }
    if (sumsq) *sumsq = acc;
    return ORA_OK;
}
