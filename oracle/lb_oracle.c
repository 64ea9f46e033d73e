/*
 * Layer-boundary oracle: a plain, slow, single-threaded CPU statement of what the
 * boundary hot path computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may include, link or call
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code, header, table or constant with the CUDA library.
 *
 * Sources ("Layer boundaries", sglang developer guide):
 *   - section "Residual stream", state table: an Initial stream has no residual, so
 *     the consumer's enter initialises it; a Written stream is only read; a Pending
 *     stream completes owed work, applies the producer update, then reads.
 *   - section "Residual stream", helper table: complete_output finishes the owed sum
 *     and leaves the update pending; fold adds a completed plain contribution to the
 *     residual.
 *   - section "Token layouts and sums": the owed sum runs over a SumGroup (attention
 *     TP, full TP or the MoE output reduction); ATTN_DP rows are per-set with padding
 *     and counts taken from batch metadata.
 *   - section "Residual update and input read": the fused add+norm read keeps its
 *     FP32 accumulation and normalises that, not a separately rounded snapshot.
 *   - section "Auxiliary capture and extra contributions": a BF16 snapshot followed by
 *     a norm differs from the fused FP32 path, so the norm input here is the FP32 sum.
 *   - section "Execute a layer": prepare() returns the consumer's input format, which
 *     can be quantized (here per-token dynamic FP8 E4M3).
 *   - section "Producer contracts and output state" and "Enter and leave the layer
 *     stack": a HandoffOutput carries a deferred MoE finalize; the fused
 *     finalize(handoff, residual, gamma) does finalize + sum + residual add + norm.
 *   - section "Choose a reduction policy", value rs: fixed-size reduce-scatter, and
 *     "SGLang flashinfer_allreduce_fusion精读", section forward: with reduce-scatter
 *     each rank normalises only its own row slice.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   RMSNorm is y = o * (1 / sqrt(mean(o^2) + eps)) * gamma, eps inside the root,
 *   gamma a plain multiplier; partials are summed k ascending from +0.0f, then the
 *   residual is added; FP8 is OCP E4M3 ("fn": bias 7, max 448, no infinities) with
 *   round-to-nearest-even and saturation, scale = max|yf| / 448 over the FP32 yf;
 *   an all-zero row gets scale 0 and all codes 0x00.
 *
 * Arithmetic: IEEE binary32 for the owed sum, the residual fold and the normalised
 * output (the fused read keeps FP32 accumulation); the RMSNorm's sum of squares and
 * its scalar 1/sqrt are taken in binary64 and rounded once, since the pages leave
 * their precision open.  Every operation is written separately; build with
 * -ffp-contract=off -fno-fast-math so that no multiply-add is contracted.
 *
 * Parity status: every function below is pinned by the CPU tests (hand-computed
 * cases, closed forms, invariants, library cross-checks); none is unpinned.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------------ */
/* Number formats                                                                  */
/* ------------------------------------------------------------------------------ */

/* bfloat16 is the upper half of an IEEE binary32: widening is exact. */
float ora_bf16_to_f32(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary32 -> bfloat16, round to nearest, ties to even.  The kept half is the upper
 * 16 bits; the dropped half decides the rounding.  NaN stays NaN (quiet bit set). */
uint16_t ora_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint32_t upper = u >> 16;
    uint32_t dropped = u & 0xFFFFu;
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)(upper | 0x0040u);
    if (dropped > 0x8000u)
        upper += 1u;                       /* above the midpoint: round up */
    else if (dropped == 0x8000u && (upper & 1u))
        upper += 1u;                       /* exact tie: go to the even neighbour */
    return (uint16_t)upper;                /* a carry into the exponent is correct */
}

/* OCP 8-bit floating point, E4M3 ("fn" flavour): 1 sign, 4 exponent bits (bias 7),
 * 3 mantissa bits; exponent 0 is subnormal (m * 2^-9); S.1111.111 is NaN; there is
 * no infinity, so the largest finite magnitude is S.1111.110 = 1.75 * 2^8 = 448. */
float ora_e4m3_to_f32(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    float mag;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        mag = (float)m * ldexpf(1.0f, -9);
    else
        mag = (1.0f + (float)m / 8.0f) * ldexpf(1.0f, e - 7);
    return sign ? -mag : mag;
}

/* binary32 -> E4M3, round to nearest with ties to even, saturating to +-448
 * (infinities included); NaN -> 0x7F.  The non-negative finite codes 0x00..0x7E are
 * in increasing order of value, so the encoder finds the largest code whose value is
 * <= |x| by bisection and then rounds between it and the next code. */
uint8_t ora_f32_to_e4m3(float x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    int lo = 0, hi = 0x7E;                 /* invariant: value(lo) <= a < value(hi) */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if ((double)ora_e4m3_to_f32((uint8_t)mid) <= a)
            lo = mid;
        else
            hi = mid;
    }
    double vlo = (double)ora_e4m3_to_f32((uint8_t)lo);
    double vhi = (double)ora_e4m3_to_f32((uint8_t)hi);
    double below = a - vlo, above = vhi - a;    /* exact in binary64 */
    int code;
    if (below < above)
        code = lo;
    else if (above < below)
        code = hi;
    else
        code = (lo % 2 == 0) ? lo : hi;         /* tie: even mantissa (even code) */
    return (uint8_t)(sign | code);
}

/* ------------------------------------------------------------------------------ */
/* Per-row steps                                                                   */
/* ------------------------------------------------------------------------------ */

/* Consumer read: RMSNorm of the FP32 row o[0..H) with weight gamma.
 *   ms = (sum_h o[h]^2) / H            binary64 (exact squares, h order)
 *   r  = (float)(1 / sqrt(ms + eps))   binary64, rounded once to binary32
 *   yf[h] = (o[h] * r) * weight[h]     binary32
 * weight = gamma, or 1 + gamma (binary32) for the Gemma form of the norm that the
 * fused final-norm handoff expects ("Layer boundaries", section "Enter and leave the
 * layer stack": the fused path reads a GemmaRMSNorm's weight).
 * The pages fix FP32 for the accumulated residual o, which is what is normalised;
 * they say nothing about the precision of the norm's own sum of squares, so it is
 * taken in binary64: a sequential binary32 sum over a long row would carry an error
 * growing with H that belongs to no reading of the method. */
static void rmsnorm_row(const float *o, const float *gamma, int gemma, int64_t H,
                        float eps, float *yf)
{
    double ss = 0.0;
    for (int64_t h = 0; h < H; ++h) {
        double sq = (double)o[h] * (double)o[h];
        ss = ss + sq;
    }
    double ms = ss / (double)H;
    float r = (float)(1.0 / sqrt(ms + (double)eps));
    for (int64_t h = 0; h < H; ++h) {
        float weight = gemma ? 1.0f + gamma[h] : gamma[h];
        float t = o[h] * r;
        yf[h] = t * weight;
    }
}

/* Per-token dynamic FP8: amax over the FP32 yf (before any bf16 rounding),
 * scale = amax / 448, q = E4M3(yf / scale); an all-zero row has scale 0, codes 0. */
static void quantize_row(const float *yf, int64_t H, uint8_t *q, float *scale)
{
    float amax = 0.0f;
    for (int64_t h = 0; h < H; ++h) {
        float a = fabsf(yf[h]);
        if (a > amax)
            amax = a;
    }
    float s = amax / 448.0f;
    *scale = s;
    for (int64_t h = 0; h < H; ++h)
        q[h] = (amax == 0.0f) ? (uint8_t)0x00 : ora_f32_to_e4m3(yf[h] / s);
}

/* Writes every requested output of one row from its FP32 sum o.  NULL = not wanted. */
static void emit_row(const float *o, int64_t H, float eps, const float *gamma, int gemma,
                     uint16_t *res_out, uint16_t *y_out, uint8_t *q_out,
                     float *scale_out, float *yf_buf)
{
    if (res_out)
        for (int64_t h = 0; h < H; ++h)
            res_out[h] = ora_f32_to_bf16(o[h]);
    if (y_out || q_out) {
        rmsnorm_row(o, gamma, gemma, H, eps, yf_buf);
        if (y_out)
            for (int64_t h = 0; h < H; ++h)
                y_out[h] = ora_f32_to_bf16(yf_buf[h]);
        if (q_out)
            quantize_row(yf_buf, H, q_out, scale_out);
    }
}

/* Complete the owed sum of K partial rows and fold it into the residual row:
 *   o[h] = (((+0 + p_0[h]) + p_1[h]) + ... + p_{K-1}[h]) + res[h]
 * with the residual term absent in the Initial state (res == NULL). */
static void fold_row(const uint16_t *const *prow, int K, const uint16_t *res,
                     int64_t H, float *o)
{
    for (int64_t h = 0; h < H; ++h) {
        float acc = 0.0f;
        for (int k = 0; k < K; ++k)
            acc = acc + ora_bf16_to_f32(prow[k][h]);
        if (res)
            acc = acc + ora_bf16_to_f32(res[h]);
        o[h] = acc;
    }
}

/* ------------------------------------------------------------------------------ */
/* Whole-batch entry points (called through ctypes by the tests)                   */
/* ------------------------------------------------------------------------------ */

/* Dense boundary over T rows of width H.  partials: K row-major bf16 [T,H] arrays;
 * res_in: bf16 [T,H] or NULL (Initial); outputs bf16 [T,H] / u8 [T,H] / f32 [T], each
 * NULL when not wanted.  work: caller scratch of 2*H floats.  Returns 0. */
int ora_fold_norm(const uint16_t *const *partials, int K, const uint16_t *res_in,
                  const float *gamma, int gemma, int64_t T, int64_t H, float eps,
                  uint16_t *res_out, uint16_t *y_out, uint8_t *q_out,
                  float *scale_out, float *work)
{
    const uint16_t *prow[64];
    if (K < 0 || K > 64)
        return -1;
    float *o = work, *yf = work + H;
    for (int64_t t = 0; t < T; ++t) {
        for (int k = 0; k < K; ++k)
            prow[k] = partials[k] + t * H;
        fold_row(prow, K, res_in ? res_in + t * H : NULL, H, o);
        emit_row(o, H, eps, gamma, gemma,
                 res_out ? res_out + t * H : NULL,
                 y_out ? y_out + t * H : NULL,
                 q_out ? q_out + t * H : NULL,
                 scale_out ? scale_out + t : NULL, yf);
    }
    return 0;
}

/* Deferred MoE finalize folded into the residual, then read:
 *   o[t,h] = (sum_{j ascending} w[t,j] * E[idx[t,j], h]) + res[t,h]
 * each product rounded to FP32 before it is added (no multiply-add).  E is the
 * expert-sorted bf16 [n_rows, H] output; idx/w are [T, topk].  An index outside
 * [0, n_rows) contributes nothing and makes the return value 1. */
int ora_moe_finalize_fold_norm(const uint16_t *E, int64_t n_rows, const int32_t *idx,
                               const float *w, int topk, const uint16_t *res_in,
                               const float *gamma, int gemma, int64_t T, int64_t H,
                               float eps,
                               uint16_t *res_out, uint16_t *y_out, uint8_t *q_out,
                               float *scale_out, float *work)
{
    int bad = 0;
    float *o = work, *yf = work + H;
    for (int64_t t = 0; t < T; ++t) {
        for (int64_t h = 0; h < H; ++h) {
            float acc = 0.0f;
            for (int j = 0; j < topk; ++j) {
                int32_t p = idx[t * topk + j];
                if (p < 0 || (int64_t)p >= n_rows) {
                    bad = 1;
                    continue;
                }
                float term = w[t * topk + j] * ora_bf16_to_f32(E[(int64_t)p * H + h]);
                acc = acc + term;
            }
            if (res_in)
                acc = acc + ora_bf16_to_f32(res_in[t * H + h]);
            o[h] = acc;
        }
        emit_row(o, H, eps, gamma, gemma,
                 res_out ? res_out + t * H : NULL,
                 y_out ? y_out + t * H : NULL,
                 q_out ? q_out + t * H : NULL,
                 scale_out ? scale_out + t : NULL, yf);
    }
    return bad;
}

/* Row slice of a padded, ragged batch (fixed-size reduce-scatter).  The padded batch
 * has T_pad rows split into num_slices equal slices of S = T_pad / num_slices rows;
 * this computes slice `slice` only.  Token set i holds valid rows
 * [offsets[i], offsets[i] + counts[i]); every other row is padding.  Local row
 * i in [0,S) maps to global row g = slice*S + i of the partials; the residual input
 * and all outputs are compact [S, ...] arrays.  Padding rows are neither computed
 * nor written.  num_sets == 0 means that every row is valid.  Returns the number of
 * rows written, or -1 on bad metadata. */
int64_t ora_slice_fold_norm(const uint16_t *const *partials, int K, int64_t T_pad,
                            int num_slices, int slice, const int32_t *offsets,
                            const int32_t *counts, int num_sets,
                            const uint16_t *res_in, const float *gamma, int gemma,
                            int64_t H, float eps, uint16_t *res_out, uint16_t *y_out,
                            uint8_t *q_out, float *scale_out, float *work)
{
    const uint16_t *prow[64];
    if (K < 0 || K > 64 || num_slices <= 0 || T_pad % num_slices != 0 || slice < 0 ||
        slice >= num_slices)
        return -1;
    int64_t S = T_pad / num_slices;
    float *o = work, *yf = work + H;
    int64_t written = 0;
    for (int64_t i = 0; i < S; ++i) {
        int64_t g = (int64_t)slice * S + i;
        int valid = (num_sets == 0);
        for (int s = 0; s < num_sets; ++s)
            if (g >= offsets[s] && g < (int64_t)offsets[s] + counts[s])
                valid = 1;
        if (!valid)
            continue;
        for (int k = 0; k < K; ++k)
            prow[k] = partials[k] + g * H;
        fold_row(prow, K, res_in ? res_in + i * H : NULL, H, o);
        emit_row(o, H, eps, gamma, gemma,
                 res_out ? res_out + i * H : NULL,
                 y_out ? y_out + i * H : NULL,
                 q_out ? q_out + i * H : NULL,
                 scale_out ? scale_out + i : NULL, yf);
        ++written;
    }
    return written;
}

/* One rank's rows of a padded, ragged batch under a variable-size reduce-scatter
 * ("Layer boundaries", section "Choose a reduction policy", value rsv; section "Token
 * layouts and sums": ATTN_DP token sets).  Rank `set` receives exactly the valid rows
 * of its own token set, [offsets[set], offsets[set] + counts[set]), as compact
 * [counts[set], ...] arrays; local row i is global row offsets[set] + i.  Returns the
 * number of rows written, or -1 on bad metadata. */
int64_t ora_set_slice_fold_norm(const uint16_t *const *partials, int K, int64_t T_pad,
                                int set, const int32_t *offsets, const int32_t *counts,
                                int num_sets, const uint16_t *res_in, const float *gamma,
                                int gemma, int64_t H, float eps, uint16_t *res_out,
                                uint16_t *y_out, uint8_t *q_out, float *scale_out,
                                float *work)
{
    const uint16_t *prow[64];
    if (K < 0 || K > 64 || set < 0 || set >= num_sets || counts[set] < 0 ||
        (int64_t)offsets[set] + counts[set] > T_pad)
        return -1;
    float *o = work, *yf = work + H;
    for (int64_t i = 0; i < counts[set]; ++i) {
        int64_t g = (int64_t)offsets[set] + i;
        for (int k = 0; k < K; ++k)
            prow[k] = partials[k] + g * H;
        fold_row(prow, K, res_in ? res_in + i * H : NULL, H, o);
        emit_row(o, H, eps, gamma, gemma,
                 res_out ? res_out + i * H : NULL,
                 y_out ? y_out + i * H : NULL,
                 q_out ? q_out + i * H : NULL,
                 scale_out ? scale_out + i : NULL, yf);
    }
    return counts[set];
}

/* Elementwise format helpers over arrays, for the tests. */
void ora_bf16_to_f32_array(const uint16_t *in, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = ora_bf16_to_f32(in[i]);
}

void ora_f32_to_bf16_array(const float *in, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = ora_f32_to_bf16(in[i]);
}

void ora_f32_to_e4m3_array(const float *in, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = ora_f32_to_e4m3(in[i]);
}

void ora_e4m3_to_f32_array(const uint8_t *in, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = ora_e4m3_to_f32(in[i]);
}
