/*
 * oracle.c -- plain, slow, single-threaded CPU reference for the fused Q4_K
 * SwiGLU feed-forward block.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant with the CUDA
 * library.
 *
 * What it computes (sources):
 *   - The block:  y = W_down . (silu(W_gate . x) (*) (W_up . x)), hidden width H
 *     projected up twice to the intermediate width I, combined by SwiGLU and
 *     projected back down.  "Fused SwiGLU MLP: ZINC RDNA4 Down-Projection
 *     Bandwidth", section "The MLP is two trips up to a wider width".
 *   - Weights in Q4_K super-blocks ("Fused SwiGLU MLP...", FAQ "Why is fusing
 *     the SwiGLU intermediate harder..."; "VGPR pressure caps the fused RDNA4
 *     prefill GEMM at nine waves", section "What the fused GEMM actually spends
 *     registers on").  The pages name the format but do not lay out its bytes;
 *     the reading used here is the GGUF Q4_K arrangement:
 *       bytes 0..1   d     (IEEE binary16, little endian)
 *       bytes 2..3   dmin  (IEEE binary16)
 *       bytes 4..15  scales[12]: eight 6-bit (sc, m) pairs, one per sub-block
 *                    of 32 weights
 *       bytes 16..143 qs[128]: 4-bit quants; byte qs[32g+l] holds weight 64g+l
 *                    in its low nibble and weight 64g+32+l in its high nibble
 *       w = d*sc*q - dmin*m
 *   - Mixture of experts: y_t = sum_j w_{t,j} FFN_{e_{t,j}}(x_t), expert ids and
 *     weights given per token ("Four bottlenecks, one CUDA backend...",
 *     section "Bottleneck 2 -- MoE decode was paying for its routing twice").
 *   - The normalisation before the block and the residual connection around
 *     it: x = RMSNorm(h) * gamma feeds the block and h += block(x) ("Four
 *     bottlenecks, one CUDA backend...", section "Bottleneck 3 -- Gemma
 *     decode is launch-latency bound": rms_norm and the residual accumulate
 *     as one launch).  The pages do not write RMSNorm out; the reading is the
 *     usual x = h / sqrt(mean(h^2) + eps) * gamma, rounded once to bf16.
 *   - The router that chooses them: per token, the top_k experts by logit,
 *     then softmax weights over the chosen logits (same page and section:
 *     the layer computes router logits and picks the top-k experts; the
 *     softmax over the chosen k is the reading used throughout).
 *
 * Precision: Q4_K dequantisation is done in fp32 exactly as the format states
 * (both products are exact in fp32, so only the final subtraction rounds); the
 * matrix products, silu and the down projection are evaluated in fp64.  The
 * quantiser decides integer codes, so it works in fp32 step by step (see
 * oracle_q4k_quantize_row).
 *
 * Compile with -O2 -ffp-contract=off (no fast-math).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QK 256        /* weights per super-block            */
#define QK_BYTES 144  /* bytes per super-block              */

/* ---- scalar formats ---------------------------------------------------- */

/* IEEE binary16 -> float, written out from the format's definition:
 * sign, 5-bit biased exponent (bias 15), 10-bit fraction. */
float oracle_f16_to_f32(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);               /* subnormal: f * 2^-14 / 1024 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp(1024.0 + f, e - 25);           /* (1 + f/1024) * 2^(e-15) */
    return (float)(sign ? -v : v);
}

/* float -> IEEE binary16, round to nearest even (the C compiler's _Float16
 * conversion is correctly rounded). */
uint16_t oracle_f32_to_f16(float x)
{
    _Float16 v = (_Float16)x;
    uint16_t h;
    memcpy(&h, &v, 2);
    return h;
}

/* bfloat16 bits -> float: the upper half of an IEEE binary32. */
float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* ---- Q4_K block ------------------------------------------------------------ */

/* 6-bit scale and min of sub-block j (0..7) from the 12 packed bytes.
 * Sub-blocks 0..3 keep their 6 bits in the low bits of scales[j] (scale) and
 * scales[j+4] (min).  Sub-blocks 4..7 keep their low 4 bits in the nibbles of
 * scales[j+4] (scale: low nibble, min: high nibble) and their top 2 bits in
 * the two spare top bits of scales[j-4] (scale) and scales[j] (min). */
void oracle_q4k_scale_min(const uint8_t *scales, int j, int *sc, int *m)
{
    if (j < 4) {
        *sc = scales[j] & 63;
        *m = scales[j + 4] & 63;
    } else {
        *sc = (scales[j + 4] & 15) | ((scales[j - 4] >> 6) << 4);
        *m = (scales[j + 4] >> 4) | ((scales[j] >> 6) << 4);
    }
}

/* 4-bit code of weight k (0..255) of a block. */
static int q4k_code(const uint8_t *qs, int k)
{
    int g = k / 64, r = k % 64;
    uint8_t byte = qs[32 * g + (r % 32)];
    return r < 32 ? (byte & 15) : (byte >> 4);
}

/* Dequantise one row of ceil(cols/256) consecutive blocks into cols floats.
 * Weights at positions >= cols in the last block are not written. */
void oracle_q4k_dequant_row(const uint8_t *row, int64_t cols, float *out)
{
    int64_t nb = (cols + QK - 1) / QK;
    for (int64_t b = 0; b < nb; ++b) {
        const uint8_t *blk = row + b * QK_BYTES;
        float d = oracle_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
        float dmin = oracle_f16_to_f32((uint16_t)(blk[2] | (blk[3] << 8)));
        const uint8_t *scales = blk + 4;
        const uint8_t *qs = blk + 16;
        for (int k = 0; k < QK; ++k) {
            int64_t col = b * QK + k;
            if (col >= cols)
                break;
            int sc, m;
            oracle_q4k_scale_min(scales, k / 32, &sc, &m);
            float ds = d * (float)sc;      /* exact: 11 x 6 significant bits */
            float dm = dmin * (float)m;    /* exact                          */
            float wq = ds * (float)q4k_code(qs, k); /* exact: 17 x 4 bits    */
            out[col] = wq - dm;            /* the only rounding              */
        }
    }
}

void oracle_q4k_dequant(const uint8_t *blocks, float *out, int64_t rows, int64_t cols)
{
    int64_t rb = ((cols + QK - 1) / QK) * QK_BYTES;
    /* rows are independent: a build with OpenMP takes them in parallel */
    #pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        oracle_q4k_dequant_row(blocks + r * rb, cols, out + r * cols);
}

/* ---- other block formats (W_down of the routed and single-token paths) -----
 * The pages name Q5_K, Q6_K and Q5_1 expert matrices ("Four bottlenecks, one
 * CUDA backend...", section "Bottleneck 2": the down projection of the routed
 * layers runs in Q5_K or Q5_1; section "Bottleneck 4": Q5_K and Q6_K GEMMs)
 * without laying out their bytes.  Reading: the GGUF arrangements.
 *   Q5_K (176 bytes / 256 weights): d, dmin (fp16), 12 scale bytes as Q4_K,
 *     qh[32], qs[128].  Weight k: 4-bit code as Q4_K plus 16 * bit (k / 32)
 *     of qh[k % 32]; w = d*sc*q - dmin*m, sub-block k / 32.
 *   Q6_K (210 bytes / 256 weights): ql[128], qh[64], scales[16] (int8), d
 *     (fp16).  Weight k in half n = k / 128 (r = k % 128, i = r / 32,
 *     l = r % 32): low 4 bits from ql[64n + l + 32 (i & 1)] (low nibble for
 *     i < 2, high for i >= 2), high 2 bits = bits 2i, 2i+1 of qh[32n + l];
 *     w = d * scales[k / 16] * (q - 32).
 *   Q5_1 (24 bytes / 32 weights): d, m (fp16), qh (32 bits, little endian),
 *     qs[16].  Weight j < 16: low nibble of qs[j] plus 16 * bit j of qh;
 *     weight 16 + j: high nibble of qs[j] plus 16 * bit 16 + j; w = d*q + m.
 * In every format the products are exact in fp32 (Q5_K: 11 x 6 x 5 bits;
 * Q6_K: 11 bits x |sc * (q - 32)| <= 4096; Q5_1: 11 x 5 bits), so the value
 * is the exact product (Q6_K) or the exact product with one rounding of the
 * final addition (Q5_K, Q5_1): bit-exact whatever the evaluation order, as
 * long as the products are not rounded. */
enum { FMT_Q4_K = 0, FMT_Q5_K = 1, FMT_Q6_K = 2, FMT_Q5_1 = 3 };

int64_t oracle_fmt_block_weights(int fmt) { return fmt == FMT_Q5_1 ? 32 : 256; }

int64_t oracle_fmt_block_bytes(int fmt)
{
    switch (fmt) {
    case FMT_Q4_K: return 144;
    case FMT_Q5_K: return 176;
    case FMT_Q6_K: return 210;
    case FMT_Q5_1: return 24;
    default: return 0;
    }
}

int64_t oracle_fmt_row_bytes(int fmt, int64_t cols)
{
    int64_t bw = oracle_fmt_block_weights(fmt);
    return ((cols + bw - 1) / bw) * oracle_fmt_block_bytes(fmt);
}

static float fp16_at(const uint8_t *p) { return oracle_f16_to_f32((uint16_t)(p[0] | (p[1] << 8))); }

/* value of weight k of one block */
static float q5k_weight(const uint8_t *blk, int k)
{
    float d = fp16_at(blk), dmin = fp16_at(blk + 2);
    const uint8_t *scales = blk + 4, *qh = blk + 16, *qs = blk + 48;
    int sc, m;
    oracle_q4k_scale_min(scales, k / 32, &sc, &m);
    int q = q4k_code(qs, k) + 16 * ((qh[k % 32] >> (k / 32)) & 1);
    float wq = (d * (float)sc) * (float)q;   /* exact: 11 x 6 x 5 bits */
    return wq - dmin * (float)m;             /* one rounding           */
}

static float q6k_weight(const uint8_t *blk, int k)
{
    const uint8_t *ql = blk, *qh = blk + 128;
    const int8_t *scales = (const int8_t *)(blk + 192);
    float d = fp16_at(blk + 208);
    int n = k / 128, r = k % 128, i = r / 32, l = r % 32;
    uint8_t lb = ql[64 * n + l + 32 * (i & 1)];
    int lo = i < 2 ? (lb & 15) : (lb >> 4);
    int hi = (qh[32 * n + l] >> (2 * i)) & 3;
    int q = (lo | (hi << 4)) - 32;
    return (float)((double)d * (double)(scales[k / 16] * q));   /* exact */
}

static float q51_weight(const uint8_t *blk, int j)
{
    float d = fp16_at(blk), m = fp16_at(blk + 2);
    uint32_t qh = (uint32_t)blk[4] | ((uint32_t)blk[5] << 8) | ((uint32_t)blk[6] << 16) |
                  ((uint32_t)blk[7] << 24);
    const uint8_t *qs = blk + 8;
    int q = j < 16 ? ((qs[j] & 15) | (((qh >> j) & 1) << 4))
                   : ((qs[j - 16] >> 4) | (((qh >> j) & 1) << 4));
    return d * (float)q + m;                 /* d*q exact; one rounding */
}

void oracle_dequant_row_fmt(int fmt, const uint8_t *row, int64_t cols, float *out)
{
    if (fmt == FMT_Q4_K) {
        oracle_q4k_dequant_row(row, cols, out);
        return;
    }
    int64_t bw = oracle_fmt_block_weights(fmt), bb = oracle_fmt_block_bytes(fmt);
    for (int64_t col = 0; col < cols; ++col) {
        const uint8_t *blk = row + (col / bw) * bb;
        int k = (int)(col % bw);
        out[col] = fmt == FMT_Q5_K ? q5k_weight(blk, k)
                 : fmt == FMT_Q6_K ? q6k_weight(blk, k) : q51_weight(blk, k);
    }
}

void oracle_dequant_fmt(int fmt, const uint8_t *blocks, float *out, int64_t rows, int64_t cols)
{
    int64_t rb = oracle_fmt_row_bytes(fmt, cols);
    for (int64_t r = 0; r < rows; ++r)
        oracle_dequant_row_fmt(fmt, blocks + r * rb, cols, out + r * cols);
}

/* ---- min/max quantiser ------------------------------------------------------
 * The pages do not give a quantiser; this library's reading of a "min/max"
 * Q4_K quantiser, every step in fp32 round-to-nearest (no fused operations,
 * IEEE division), rint = round half to even:
 *   per sub-block j of 32 weights:  lo = min(0, min w), hi = max w,
 *                                   scale_j = (hi - lo) / 15, min_j = -lo
 *   per block:   d = f16(max_j scale_j / 63), dmin = f16(max_j min_j / 63)
 *                sc_j = clamp(rint(scale_j / d), 0, 63)   (0 when d == 0)
 *                m_j  = clamp(rint(min_j / dmin), 0, 63)  (0 when dmin == 0)
 *   per weight:  q = clamp(rint((w + dmin*m_j) / (d*sc_j)), 0, 15)
 *                                                       (0 when d*sc_j == 0)
 * Positions >= cols in the last block are quantised as zeros. */
static int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

static void q4k_pack_scales(uint8_t *scales, const int *sc, const int *m)
{
    memset(scales, 0, 12);
    for (int j = 0; j < 4; ++j) {
        scales[j] = (uint8_t)(sc[j] & 63);
        scales[j + 4] = (uint8_t)(m[j] & 63);
    }
    for (int j = 4; j < 8; ++j) {
        scales[j + 4] = (uint8_t)((sc[j] & 15) | ((m[j] & 15) << 4));
        scales[j - 4] |= (uint8_t)((sc[j] >> 4) << 6);
        scales[j] |= (uint8_t)((m[j] >> 4) << 6);
    }
}

void oracle_q4k_quantize_row(const float *w, int64_t cols, uint8_t *row)
{
    int64_t nb = (cols + QK - 1) / QK;
    for (int64_t b = 0; b < nb; ++b) {
        float x[QK];
        for (int k = 0; k < QK; ++k) {
            int64_t col = b * QK + k;
            x[k] = col < cols ? w[col] : 0.0f;
        }
        float scale[8], mn[8];
        float max_scale = 0.0f, max_min = 0.0f;
        for (int j = 0; j < 8; ++j) {
            float lo = 0.0f, hi = x[32 * j];
            for (int l = 0; l < 32; ++l) {
                float v = x[32 * j + l];
                if (v < lo) lo = v;
                if (v > hi) hi = v;
            }
            float diff = hi - lo;
            scale[j] = diff / 15.0f;
            mn[j] = -lo;
            if (scale[j] > max_scale) max_scale = scale[j];
            if (mn[j] > max_min) max_min = mn[j];
        }
        float dq = max_scale / 63.0f;
        float dmq = max_min / 63.0f;
        uint16_t d16 = oracle_f32_to_f16(dq);
        uint16_t dm16 = oracle_f32_to_f16(dmq);
        float d = oracle_f16_to_f32(d16);
        float dmin = oracle_f16_to_f32(dm16);
        int sc[8], m[8];
        for (int j = 0; j < 8; ++j) {
            float rs = d > 0.0f ? scale[j] / d : 0.0f;
            float rm = dmin > 0.0f ? mn[j] / dmin : 0.0f;
            sc[j] = clampi((int)rintf(rs), 0, 63);
            m[j] = clampi((int)rintf(rm), 0, 63);
        }
        uint8_t *blk = row + b * QK_BYTES;
        blk[0] = (uint8_t)(d16 & 255);
        blk[1] = (uint8_t)(d16 >> 8);
        blk[2] = (uint8_t)(dm16 & 255);
        blk[3] = (uint8_t)(dm16 >> 8);
        q4k_pack_scales(blk + 4, sc, m);
        uint8_t *qs = blk + 16;
        memset(qs, 0, 128);
        for (int k = 0; k < QK; ++k) {
            int j = k / 32;
            float ds = d * (float)sc[j];
            float dm = dmin * (float)m[j];
            int q = 0;
            if (ds > 0.0f) {
                float t = x[k] + dm;
                float r = t / ds;
                q = clampi((int)rintf(r), 0, 15);
            }
            int g = k / 64, r = k % 64;
            if (r < 32)
                qs[32 * g + r] |= (uint8_t)q;
            else
                qs[32 * g + (r - 32)] |= (uint8_t)(q << 4);
        }
    }
}

void oracle_q4k_quantize(const float *w, uint8_t *blocks, int64_t rows, int64_t cols)
{
    int64_t rb = ((cols + QK - 1) / QK) * QK_BYTES;
    for (int64_t r = 0; r < rows; ++r)
        oracle_q4k_quantize_row(w + r * cols, cols, blocks + r * rb);
}

/* ---- the feed-forward block ------------------------------------------------ */

double oracle_silu(double g) { return g / (1.0 + exp(-g)); }

/* y[T x H] (fp64) = W_down . (silu(W_gate . x) * (W_up . x)) for each token row
 * of x[T x H] (bf16 bits, row-major).
 *   Wg, Wu: I rows of H/256 blocks;  Wd: H rows of ceil(I/256) blocks.
 * Each weight row is dequantised once (fp32), the sums run in fp64 in
 * ascending index order. */
void oracle_swiglu_ffn_fmt(const uint16_t *x, const uint8_t *Wg, const uint8_t *Wu,
                           const uint8_t *Wd, int wd_fmt, int64_t T, int64_t H, int64_t I,
                           double *y)
{
    int64_t rb_in = ((H + QK - 1) / QK) * QK_BYTES;
    int64_t rb_dn = oracle_fmt_row_bytes(wd_fmt, I);
    double *xf = (double *)malloc(sizeof(double) * (size_t)(T * H));
    double *h = (double *)malloc(sizeof(double) * (size_t)(T * I));
    for (int64_t i = 0; i < T * H; ++i)
        xf[i] = (double)oracle_bf16_to_f32(x[i]);
    /* g = Wg x, u = Wu x, h = silu(g) * u.  Each row i has its own scratch,
     * so a build with OpenMP may take the rows in parallel; every sum keeps
     * its order, so the result is the same either way. */
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < I; ++i) {
        float *wg = (float *)malloc(sizeof(float) * (size_t)H);
        float *wu = (float *)malloc(sizeof(float) * (size_t)H);
        oracle_q4k_dequant_row(Wg + i * rb_in, H, wg);
        oracle_q4k_dequant_row(Wu + i * rb_in, H, wu);
        for (int64_t t = 0; t < T; ++t) {
            const double *xt = xf + t * H;
            double g = 0.0, u = 0.0;
            for (int64_t k = 0; k < H; ++k) {
                g += (double)wg[k] * xt[k];
                u += (double)wu[k] * xt[k];
            }
            h[t * I + i] = oracle_silu(g) * u;
        }
        free(wg); free(wu);
    }
    /* y = Wd h (rows n independent, as above) */
    #pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < H; ++n) {
        float *wd = (float *)malloc(sizeof(float) * (size_t)I);
        oracle_dequant_row_fmt(wd_fmt, Wd + n * rb_dn, I, wd);
        for (int64_t t = 0; t < T; ++t) {
            const double *ht = h + t * I;
            double acc = 0.0;
            for (int64_t i = 0; i < I; ++i)
                acc += (double)wd[i] * ht[i];
            y[t * H + n] = acc;
        }
        free(wd);
    }
    free(xf); free(h);
}

/* The block with all three matrices in Q4_K. */
void oracle_swiglu_ffn(const uint16_t *x, const uint8_t *Wg, const uint8_t *Wu,
                       const uint8_t *Wd, int64_t T, int64_t H, int64_t I, double *y)
{
    oracle_swiglu_ffn_fmt(x, Wg, Wu, Wd, FMT_Q4_K, T, H, I, y);
}

/* Mixture of experts: y_t = sum_{j < top_k} w[t][j] * FFN_{ids[t][j]}(x_t).
 * Experts are stacked: expert e's W_gate starts at Wg + e * I * rowbytes(H),
 * likewise W_up; its W_down at Wd + e * H * rowbytes(I).  An id outside
 * [0, E) contributes nothing. */
/* Routed block with a per-expert scale on the down projection ("Four
 * bottlenecks, one CUDA backend...", section "Bottleneck 2": a routed layer's
 * per-expert down projection carries a scale applied inside the batched path):
 *     y_t = sum_j w_tj * s_e * FFN_e(x_t),   e = ids[t][j],
 * s one fp32 value per expert (down_scale NULL: every s_e = 1).  The products
 * w_tj * s_e * FFN_e are formed in fp64. */
void oracle_moe_swiglu_ffn_scaled(const uint16_t *x, const int32_t *ids, const float *wts,
                                  const float *down_scale, const uint8_t *Wg, const uint8_t *Wu,
                                  const uint8_t *Wd, int wd_fmt, int64_t T, int64_t H, int64_t I,
                                  int64_t E, int64_t top_k, double *y)
{
    int64_t rb_in = ((H + QK - 1) / QK) * QK_BYTES;
    int64_t rb_dn = oracle_fmt_row_bytes(wd_fmt, I);
    double *yt = (double *)malloc(sizeof(double) * (size_t)H);
    for (int64_t t = 0; t < T; ++t) {
        double *out = y + t * H;
        for (int64_t n = 0; n < H; ++n)
            out[n] = 0.0;
        for (int64_t j = 0; j < top_k; ++j) {
            int64_t e = ids[t * top_k + j];
            if (e < 0 || e >= E)
                continue;
            oracle_swiglu_ffn_fmt(x + t * H, Wg + e * I * rb_in, Wu + e * I * rb_in,
                                  Wd + e * H * rb_dn, wd_fmt, 1, H, I, yt);
            double w = (double)wts[t * top_k + j];
            if (down_scale)
                w *= (double)down_scale[e];
            for (int64_t n = 0; n < H; ++n)
                out[n] += w * yt[n];
        }
    }
    free(yt);
}

void oracle_moe_swiglu_ffn_fmt(const uint16_t *x, const int32_t *ids, const float *wts,
                               const uint8_t *Wg, const uint8_t *Wu, const uint8_t *Wd,
                               int wd_fmt, int64_t T, int64_t H, int64_t I, int64_t E,
                               int64_t top_k, double *y)
{
    oracle_moe_swiglu_ffn_scaled(x, ids, wts, NULL, Wg, Wu, Wd, wd_fmt, T, H, I, E, top_k, y);
}

void oracle_moe_swiglu_ffn(const uint16_t *x, const int32_t *ids, const float *wts,
                           const uint8_t *Wg, const uint8_t *Wu, const uint8_t *Wd,
                           int64_t T, int64_t H, int64_t I, int64_t E, int64_t top_k,
                           double *y)
{
    oracle_moe_swiglu_ffn_fmt(x, ids, wts, Wg, Wu, Wd, FMT_Q4_K, T, H, I, E, top_k, y);
}

/* Router: for each token t, the top_k of its E logits and their softmax
 * weights.  Order: a ranks above b when a's logit is larger, or the logits
 * are equal and a's index is lower; a NaN logit ranks below every number
 * (-inf included) and NaNs among themselves by index; -0 equals +0.  ids[t]
 * lists the chosen experts from the highest rank down.  weights[t][j] =
 * exp(l_j - l_0) / sum_i exp(l_i - l_0) over the chosen logits (l_0 the
 * highest), evaluated in fp64 and rounded once to fp32.  Selection is plain:
 * top_k passes, each taking the best expert not taken yet. */
static int router_ranks_above(float a, int64_t ia, float b, int64_t ib)
{
    int na = isnan(a), nb = isnan(b);
    if (na || nb) {
        if (na && nb)
            return ia < ib;
        return nb; /* the number ranks above the NaN */
    }
    if (a != b)
        return a > b;
    return ia < ib;
}

void oracle_route_top_k(const float *logits, int64_t T, int64_t E, int64_t top_k,
                        int32_t *ids, float *weights)
{
    unsigned char *taken = (unsigned char *)malloc((size_t)(E > 0 ? E : 1));
    double *ex = (double *)malloc(sizeof(double) * (size_t)(top_k > 0 ? top_k : 1));
    for (int64_t t = 0; t < T; ++t) {
        const float *l = logits + t * E;
        for (int64_t e = 0; e < E; ++e)
            taken[e] = 0;
        for (int64_t j = 0; j < top_k; ++j) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e) {
                if (taken[e])
                    continue;
                if (best < 0 || router_ranks_above(l[e], e, l[best], best))
                    best = e;
            }
            taken[best] = 1;
            ids[t * top_k + j] = (int32_t)best;
        }
        double top = (double)l[ids[t * top_k]];
        double sum = 0.0;
        for (int64_t j = 0; j < top_k; ++j) {
            ex[j] = exp((double)l[ids[t * top_k + j]] - top);
            sum += ex[j];
        }
        for (int64_t j = 0; j < top_k; ++j)
            weights[t * top_k + j] = (float)(ex[j] / sum);
    }
    free(taken);
    free(ex);
}

/* double -> bfloat16 bits, rounded once to nearest even: the value is split
 * as m * 2^e with 0.5 <= |m| < 1, m is rounded to 8 significant bits and
 * scaled back.  Covers the normal range of bf16 (the only range the tests
 * use); zero keeps its sign. */
uint16_t oracle_bf16_from_f64(double v)
{
    if (v == 0.0 || isnan(v) || isinf(v)) {
        float f = (float)v;
        uint32_t u;
        memcpy(&u, &f, 4);
        return (uint16_t)(u >> 16 | (isnan(v) ? 0x40u : 0u));
    }
    int e;
    double m = frexp(v, &e);
    double q = nearbyint(ldexp(m, 8));       /* default rounding: nearest even */
    float f = (float)ldexp(q, e - 8);        /* exact: 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

/* RMSNorm of the rows of h [T][H] (fp32) into bf16 bits:
 *     x[t][c] = bf16( h[t][c] / sqrt(sum_c' h[t][c']^2 / H + eps) * gamma[c] )
 * with the sum, the root and the products in fp64 and one rounding. */
void oracle_rmsnorm_bf16(const float *h, const float *gamma, double eps, int64_t T, int64_t H,
                         uint16_t *x)
{
    for (int64_t t = 0; t < T; ++t) {
        const float *row = h + t * H;
        double ss = 0.0;
        for (int64_t c = 0; c < H; ++c)
            ss += (double)row[c] * (double)row[c];
        double r = 1.0 / sqrt(ss / (double)H + eps);
        for (int64_t c = 0; c < H; ++c)
            x[t * H + c] = oracle_bf16_from_f64((double)row[c] * r * (double)gamma[c]);
    }
}
