/*
 * CPU oracle for the ZeRO / FSDP sharded mixed-precision step over a
 * FlatParameter.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline and reference legs may load this library.  The
 * product path never calls it, and it shares no code, header or constant with
 * the CUDA library.
 *
 * Everything here is a plain scalar loop in the order the method is stated:
 * flatten/pad/shard, reduce-scatter by averaging, AdamW on each rank's shard
 * with fp32 state, round to bf16, all-gather.  Arithmetic is done in double;
 * every stored value (gradient mean, master, m, v) is rounded to fp32 with
 * round-to-nearest-even, and parameters are rounded to bf16 with the bit
 * method below.  Build with -ffp-contract=off so that no multiply-add is fused
 * behind the reader's back (the arithmetic is exactly what is written).
 *
 * Sources (page title, section):
 *   [L5]  "Lesson 5: ZeRO and FSDP (including the FSDP2 architecture)",
 *         hpc.payai.win -- section 2 (stage memory), section 3 (communication
 *         ledger: reduce-scatter, local update + cast to BF16, all-gather),
 *         section 7.1 (FlatParameter flatten + tail padding).
 *   [DZ]  "Data parallelism and ZeRO memory sharding", jefxiong.cn --
 *         section 3.1 (mean of per-rank means), section 4.2 and the appendix
 *         update simulator (Adam with bias correction on each rank's slice,
 *         then concatenation of the updated slices).
 *   [LA]  "FSDP", Latent Atlas (process-cxr.github.io) -- section 5.1
 *         (each unit's parameters flattened and split evenly over the ranks),
 *         section 8.2 (bf16 gradients handed to an fp32 master update),
 *         section 9.5 (FSDP2 splits every parameter on its own).
 *   [A03] "03 · FSDP (ZeRO-3): per-layer all-gather and reshard"
 *         (llm-infra-atlas) -- section 4 (FSDP2: each parameter marked as
 *         split along dim 0 over the data-parallel mesh).
 *   Further sections used by single functions below: [L5] section 7.2
 *   (per-parameter Shard(0)), [L5] section 3 on gradient accumulation
 *   (ZeRO-1 accumulates locally and reduce-scatters once), [DZ] section 6
 *   (a global gradient norm needs a reduction across shards).
 *
 * Readings where the pages leave a step open (each is also listed with the
 * design notes): decoupled weight decay theta*(1 - lr*wd) applied to the old
 * weights (AdamW); eps added after the square root of the bias-corrected v;
 * the reduction is a mean (sum / N_d) over ranks; micro-step accumulation
 * averages the K micro-batch means (acc / K).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- bf16 ---- */

/* Widen a bf16 bit pattern to fp32: bf16 is the top half of an fp32 word. */
float oracle_bf16_to_f32(uint16_t h)
{
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/*
 * Round fp32 to bf16, round-to-nearest, ties to even, by the bit method:
 * add 0x7FFF plus the lowest kept bit, then drop the low 16 bits.  A carry
 * out of the mantissa correctly bumps the exponent (and overflows to inf).
 * NaN is kept a quiet NaN.
 */
uint16_t oracle_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7FFFFFFFu) > 0x7F800000u) {
        return (uint16_t)((u >> 16) | 0x0040u);
    }
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

void oracle_round_to_bf16(const float* x, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) {
        out[i] = oracle_f32_to_bf16(x[i]);
    }
}

/* -------------------------------------------------------------- layout ---- */

/*
 * FlatParameter layout ([L5] section 7.1, [LA] section 5.1): tensors are
 * concatenated in registration order with no gaps, so tensor i starts at the
 * sum of the sizes before it.  The flat buffer is padded at the tail only, up
 * to the next multiple of the rank count, and split into n_ranks equal
 * contiguous shards; rank r owns [r*S, (r+1)*S).
 *
 * Returns 0, or -1 when a size is negative, the total is zero or n_ranks < 1
 * (the pages reject non-positive sizes with an error).
 * out3 receives {P, P_pad, S}.
 */
int oracle_flat_layout(const int64_t* numels, int64_t n_tensors, int32_t n_ranks,
                       int64_t* offsets, int64_t* out3)
{
    if (n_tensors < 1 || n_ranks < 1) {
        return -1;
    }
    int64_t running = 0;
    for (int64_t i = 0; i < n_tensors; ++i) {
        if (numels[i] < 0) {
            return -1;
        }
        offsets[i] = running;
        running = running + numels[i];
    }
    if (running <= 0) {
        return -1;
    }
    int64_t P = running;
    int64_t pad = 0;
    while ((P + pad) % n_ranks != 0) {
        pad = pad + 1;
    }
    int64_t P_pad = P + pad;
    out3[0] = P;
    out3[1] = P_pad;
    out3[2] = P_pad / n_ranks;
    return 0;
}

/* ------------------------------------------------------ reduce-scatter ---- */

/*
 * Mean over ranks of one element ([DZ] section 3.1: g = (1/N) sum_r g_r).
 * The sum of bf16 values is formed in double, then divided by N and rounded
 * once to fp32.
 */
static float mean_over_ranks(const uint16_t* grads, int32_t n_ranks, int64_t rank_stride,
                             int64_t index)
{
    double sum = 0.0;
    for (int32_t k = 0; k < n_ranks; ++k) {
        sum = sum + (double)oracle_bf16_to_f32(grads[(int64_t)k * rank_stride + index]);
    }
    return (float)(sum / (double)n_ranks);
}

/*
 * Element-wise mean over ranks of n elements.  grads holds n_ranks rows,
 * row k starting at grads + k*rank_stride.  Used both for whole buffers and for
 * sampled elements gathered from large runs.
 */
void oracle_rank_mean(const uint16_t* grads, int32_t n_ranks, int64_t rank_stride, int64_t n,
                      float* out)
{
    for (int64_t i = 0; i < n; ++i) {
        out[i] = mean_over_ranks(grads, n_ranks, rank_stride, i);
    }
}

/*
 * Reduce-scatter by averaging ([L5] section 3, step 1): rank r receives only its
 * slice [r*S, (r+1)*S) of the mean of the n_ranks full gradient buffers.
 * grads: n_ranks rows of P_pad = n_ranks*S bf16 values.
 * shards_out: n_ranks rows of S fp32 values.
 */
void oracle_reduce_scatter(const uint16_t* grads, int32_t n_ranks, int64_t S, float* shards_out)
{
    int64_t P_pad = (int64_t)n_ranks * S;
    for (int32_t r = 0; r < n_ranks; ++r) {
        for (int64_t i = 0; i < S; ++i) {
            int64_t e = (int64_t)r * S + i;
            shards_out[(int64_t)r * S + i] = mean_over_ranks(grads, n_ranks, P_pad, e);
        }
    }
}

/*
 * All-reduce by averaging: every rank receives the whole mean vector.
 * This is the data-parallel baseline the sharded path must reproduce.
 */
void oracle_all_reduce(const uint16_t* grads, int32_t n_ranks, int64_t P_pad, float* full_out)
{
    for (int64_t e = 0; e < P_pad; ++e) {
        full_out[e] = mean_over_ranks(grads, n_ranks, P_pad, e);
    }
}

/* ------------------------------------------------------- accumulation ----- */

/*
 * fp32 gradient accumulation over micro-steps ([L5] section 2 note and
 * section 3: a sharded fp32 accumulator of 4*Psi/N_d bytes; the gradient shard is
 * reduce-scattered at every micro-batch).  first != 0 starts from zero.
 */
void oracle_accumulate(float* acc, const float* g, int64_t n, int32_t first)
{
    for (int64_t i = 0; i < n; ++i) {
        if (first) {
            acc[i] = (float)(0.0 + (double)g[i]);
        } else {
            acc[i] = (float)((double)acc[i] + (double)g[i]);
        }
    }
}

/* Average of K micro-batch means: g = acc / K, rounded once to fp32. */
void oracle_average_micro(const float* acc, int64_t n, int32_t n_micro, float* g_out)
{
    for (int64_t i = 0; i < n; ++i) {
        g_out[i] = (float)((double)acc[i] / (double)n_micro);
    }
}

/* -------------------------------------------------------------- AdamW ----- */

/*
 * One AdamW step on n fp32 elements, in place ([DZ] section 4.2 and the
 * appendix simulator: m = b1*m + (1-b1)*g, v = b2*v + (1-b2)*g^2,
 * m_hat = m/(1-b1^t), v_hat = v/(1-b2^t), w -= lr*m_hat/(sqrt(v_hat)+eps);
 * [LA] section 8.2: the fp32 master weights are what Adam updates).
 * Weight decay is the decoupled AdamW form applied to the old weights.
 * All arithmetic is double; m, v and theta are each rounded once to fp32 when
 * stored, and the update of theta uses the stored (fp32) m and v.
 */
void oracle_adamw(float* theta, float* m, float* v, const float* g, int64_t n, double lr,
                  double beta1, double beta2, double eps, double weight_decay, int64_t step)
{
    double bc1 = 1.0 - pow(beta1, (double)step);
    double bc2 = 1.0 - pow(beta2, (double)step);
    for (int64_t i = 0; i < n; ++i) {
        double gi = (double)g[i];
        float m_new = (float)(beta1 * (double)m[i] + (1.0 - beta1) * gi);
        float v_new = (float)(beta2 * (double)v[i] + (1.0 - beta2) * gi * gi);
        double m_hat = (double)m_new / bc1;
        double v_hat = (double)v_new / bc2;
        double decayed = (double)theta[i] * (1.0 - lr * weight_decay);
        double updated = decayed - lr * m_hat / (sqrt(v_hat) + eps);
        m[i] = m_new;
        v[i] = v_new;
        theta[i] = (float)updated;
    }
}

/* ------------------------------------ FSDP2 per-parameter Shard(0) ------- */

/*
 * FSDP2 per-parameter sharding ([L5] section 7.2: every parameter keeps its
 * own shape and is split along dim 0 over the data-parallel ranks, with no
 * FlatParameter and no padding; [A03] section 4; [LA] section 9.5).  Reading:
 * the rows are split the way a tensor is cut into n_ranks chunks -- chunk =
 * ceil(dim0 / n_ranks) rows, rank r owns rows [r*chunk, min((r+1)*chunk, dim0))
 * (possibly none).  Returns the element range [*begin, *end) of rank r.
 */
void oracle_param_shard_bounds(int64_t dim0, int64_t row_numel, int32_t n_ranks, int32_t rank,
                               int64_t* begin, int64_t* end)
{
    int64_t chunk = (dim0 + n_ranks - 1) / n_ranks;
    int64_t first_row = (int64_t)rank * chunk;
    int64_t last_row = first_row + chunk;
    if (first_row > dim0) {
        first_row = dim0;
    }
    if (last_row > dim0) {
        last_row = dim0;
    }
    *begin = first_row * row_numel;
    *end = last_row * row_numel;
}

/* ------------------------------------- ZeRO-1 local accumulation --------- */

/*
 * ZeRO-1 gradient accumulation ([L5] section 3, on gradient accumulation:
 * with ZeRO-1 each rank still holds the full gradient, so it can accumulate
 * the micro-batches locally and reduce-scatter only once, at the last one;
 * section 2 note: the fp32 accumulator then costs the full +4 Psi per rank).
 * acc_full: n_ranks rows of P_pad fp32 (each rank's own full accumulator);
 * acc = (first ? 0 : acc) + widen(grad), rounded once to fp32.
 */
void oracle_zero1_accumulate(const uint16_t* grads, float* acc_full, int32_t n_ranks, int64_t P_pad,
                             int32_t first)
{
    for (int32_t k = 0; k < n_ranks; ++k) {
        for (int64_t e = 0; e < P_pad; ++e) {
            int64_t idx = (int64_t)k * P_pad + e;
            double g = (double)oracle_bf16_to_f32(grads[idx]);
            double prev = first ? 0.0 : (double)acc_full[idx];
            acc_full[idx] = (float)(prev + g);
        }
    }
}

/*
 * ZeRO-1 optimizer step after n_micro accumulated micro-batches: the one
 * reduce-scatter averages the ranks' fp32 accumulators (sum in double, one
 * rounding), the result is divided by n_micro (one rounding), then every rank
 * runs AdamW on its shard, rounds to bf16, and the shards are all-gathered.
 */
int oracle_zero1_step(const float* acc_full, int32_t n_ranks, int64_t S, int32_t n_micro,
                      float* master, float* m, float* v, uint16_t* full_out, double lr,
                      double beta1, double beta2, double eps, double weight_decay, int64_t step)
{
    if (n_ranks < 1 || S < 1 || n_micro < 1 || step < 1) {
        return -1;
    }
    int64_t P_pad = (int64_t)n_ranks * S;
    float* g = (float*)malloc((size_t)P_pad * sizeof(float));
    uint16_t* p_shards = (uint16_t*)malloc((size_t)P_pad * sizeof(uint16_t));
    if (g == NULL || p_shards == NULL) {
        free(g);
        free(p_shards);
        return -1;
    }
    for (int32_t r = 0; r < n_ranks; ++r) {
        for (int64_t i = 0; i < S; ++i) {
            int64_t e = (int64_t)r * S + i;
            double sum = 0.0;
            for (int32_t k = 0; k < n_ranks; ++k) {
                sum = sum + (double)acc_full[(int64_t)k * P_pad + e];
            }
            float mean = (float)(sum / (double)n_ranks);
            g[e] = (float)((double)mean / (double)n_micro);
        }
    }
    for (int32_t r = 0; r < n_ranks; ++r) {
        int64_t off = (int64_t)r * S;
        oracle_adamw(master + off, m + off, v + off, g + off, S, lr, beta1, beta2, eps,
                     weight_decay, step);
        oracle_round_to_bf16(master + off, S, p_shards + off);
    }
    oracle_all_gather(p_shards, n_ranks, S, full_out);
    free(g);
    free(p_shards);
    return 0;
}

/* ------------------------------------------------ gradient clipping ------- */

/*
 * Global gradient-norm clipping ([DZ] section 6: a global norm needs a
 * reduction across every shard).  Reading: the clip-by-total-L2-norm rule of
 * data-parallel training -- the norm is taken over the averaged gradient of
 * every element of every unit, coef = max_norm / (norm + 1e-6), and the
 * gradient is multiplied by coef only when coef < 1.
 */

/* Sum of squares of n fp32 values, in double. */
double oracle_sum_squares(const float* g, int64_t n)
{
    double acc = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        acc = acc + (double)g[i] * (double)g[i];
    }
    return acc;
}

/* The clip coefficient from the total sum of squares, rounded once to fp32
 * (the gradient it multiplies is fp32); 1 when no clipping is needed. */
float oracle_clip_coefficient(double total_sum_squares, double max_norm)
{
    double norm = sqrt(total_sum_squares);
    double coef = max_norm / (norm + 1e-6);
    if (coef >= 1.0) {
        return 1.0f;
    }
    return (float)coef;
}

/* g = fp32(g * coef), in place (left unchanged when coef == 1). */
void oracle_scale(float* g, int64_t n, float coef)
{
    if (coef == 1.0f) {
        return;
    }
    for (int64_t i = 0; i < n; ++i) {
        g[i] = (float)((double)g[i] * (double)coef);
    }
}

/* --------------------------------------------------------- all-gather ----- */

/*
 * All-gather ([L5] section 3, step 3; [DZ] appendix simulator: the updated
 * slices are concatenated once): full[r*S + i] = shard_r[i].
 */
void oracle_all_gather(const uint16_t* shards, int32_t n_ranks, int64_t S, uint16_t* full)
{
    for (int32_t r = 0; r < n_ranks; ++r) {
        for (int64_t i = 0; i < S; ++i) {
            full[(int64_t)r * S + i] = shards[(int64_t)r * S + i];
        }
    }
}

/* ------------------------------------------------------ composed step ----- */

/*
 * One sharded step over all logical ranks, composed from the pieces above in
 * the order [L5] section 3 gives for ZeRO-1/2:
 *   1. reduce-scatter the n_ranks bf16 gradient buffers by averaging;
 *   2. (micro-stepping only) fold the mean into the rank's fp32 accumulator;
 *      at the last micro-step the gradient is acc / n_micro;
 *   3. each rank runs AdamW on its fp32 master/m/v shard and rounds it to bf16;
 *   4. all-gather the bf16 shards into the full parameter buffer.
 *
 * grads:  n_ranks rows of P_pad bf16.
 * master, m, v: n_ranks rows of S fp32 (rank r's shard at r*S), updated in
 *               place when the optimizer runs.
 * accum:  NULL, or n_ranks rows of S fp32 (micro-step accumulator).
 * full_out: P_pad bf16, written when the optimizer runs.
 * Returns 1 if the optimizer ran, 0 if this was an accumulation-only micro-step,
 * -1 on bad arguments.
 */
int oracle_zero_step(const uint16_t* grads, float* master, float* m, float* v, float* accum,
                     int32_t micro_step, int32_t n_micro, uint16_t* full_out, int32_t n_ranks,
                     int64_t S, double lr, double beta1, double beta2, double eps,
                     double weight_decay, int64_t step)
{
    if (n_ranks < 1 || S < 1 || step < 1) {
        return -1;
    }
    if (accum == NULL && !(micro_step == 1 && n_micro == 1)) {
        return -1;
    }
    if (n_micro < 1 || micro_step < 1 || micro_step > n_micro) {
        return -1;
    }
    int64_t P_pad = (int64_t)n_ranks * S;
    float* g_shards = (float*)malloc((size_t)P_pad * sizeof(float));
    uint16_t* p_shards = (uint16_t*)malloc((size_t)P_pad * sizeof(uint16_t));
    if (g_shards == NULL || p_shards == NULL) {
        free(g_shards);
        free(p_shards);
        return -1;
    }

    oracle_reduce_scatter(grads, n_ranks, S, g_shards);

    if (accum != NULL && n_micro > 1) {
        oracle_accumulate(accum, g_shards, P_pad, micro_step == 1);
        if (micro_step < n_micro) {
            free(g_shards);
            free(p_shards);
            return 0;
        }
        oracle_average_micro(accum, P_pad, n_micro, g_shards);
    }

    for (int32_t r = 0; r < n_ranks; ++r) {
        int64_t off = (int64_t)r * S;
        oracle_adamw(master + off, m + off, v + off, g_shards + off, S, lr, beta1, beta2, eps,
                     weight_decay, step);
        oracle_round_to_bf16(master + off, S, p_shards + off);
    }

    oracle_all_gather(p_shards, n_ranks, S, full_out);
    free(g_shards);
    free(p_shards);
    return 1;
}

/*
 * The unsharded data-parallel step the sharded one must equal ([DZ] section
 * 4.2: all-reduce to the full mean gradient, then one Adam update of the whole
 * vector): theta, m, v are full P_pad vectors.
 */
int oracle_ddp_step(const uint16_t* grads, float* theta, float* m, float* v, uint16_t* full_out,
                    int32_t n_ranks, int64_t P_pad, double lr, double beta1, double beta2,
                    double eps, double weight_decay, int64_t step)
{
    if (n_ranks < 1 || P_pad < 1 || step < 1) {
        return -1;
    }
    float* g = (float*)malloc((size_t)P_pad * sizeof(float));
    if (g == NULL) {
        return -1;
    }
    oracle_all_reduce(grads, n_ranks, P_pad, g);
    oracle_adamw(theta, m, v, g, P_pad, lr, beta1, beta2, eps, weight_decay, step);
    oracle_round_to_bf16(theta, P_pad, full_out);
    free(g);
    return 0;
}
