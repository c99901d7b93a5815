/*
 * q8_oracle.c -- plain, slow, obviously correct CPU oracle for the
 * Q8_0-weight x Q8_0-activation matrix multiply.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code with the CUDA library.
 *
 * What it follows (ds4 study guide pages):
 *   - "Q8_0 quantised matmul" (GPU code walkthrough, trace 3): the operation
 *     out = W x over Q8_0 weights and Q8_0 activations, with in_dim % 32 == 0
 *     (32-element blocks), W given as out_dim rows of in_dim weights.
 *   - "Q8_K quantisation (8-bit)" (model-architecture page, quantisation
 *     section 1): per block amax = max |x_i|, scale = amax / 127,
 *     q_i = (int8) roundf(x_i / scale).  The Q8_0 activation quantiser is this
 *     formula on 32-element blocks with the scale stored as IEEE binary16.
 *   - "fixed-point dot product" (same page, quantisation section 4): a block's
 *     contribution is the product of the two blocks' scales and the integer
 *     dot product of their quants, summed over blocks in fp32.
 *   - "routed MoE" (GPU code walkthrough, trace 5) and the expert pointer
 *     array (MoE C notes, section 1): each selected expert is a separate
 *     weight matrix; only the selected ones are read.
 *   - the expert FFN around it (the same trace's four steps: gate and up
 *     projections of the selected experts, SwiGLU, down projection, weighted
 *     sum; the MoE study page's "SwiGLU activation" section for
 *     mid = silu(gate) * up and the clamp of gate from above and of up to
 *     [-limit, limit]).
 *
 * Readings where the pages are silent (each one also listed in the design notes):
 *   - block layout: 34 bytes, fp16 d little-endian then int8 q[32] (GGUF Q8_0);
 *   - x / d is an IEEE fp32 division by the fp32 d (not the fp16-rounded one),
 *     rounding is roundf (half away from zero), d is stored rounded to binary16
 *     (to nearest, ties to even, subnormals kept) and the dot uses that stored d;
 *   - an all-zero block (or one whose fp32 d underflows to 0) stores d = +0 and
 *     q = 0;
 *   - accumulation is fp32 in block order b = 0..nb-1, each block adding
 *     (d_w * d_x) * (float) isum;
 *   - an expert id outside [0, n_expert) yields a zero output row and raises
 *     the error flag;
 *   - SwiGLU: silu(g) = g / (1 + e^-g) (the pages print silu's use, not its
 *     body), evaluated in double from the fp32 gate and up and rounded once
 *     to fp32; the clamp applies when limit > 0 (limit = 0: none);
 *   - the down projection's activations are the fp32 mid rows quantised with
 *     the activation quantiser above, one row per pair;
 *   - the weighted sum adds the k experts of a token in slot order, in double;
 *   - the second weight format (Q2_K and Q4_K super-blocks against Q8_K
 *     activations): see its own section at the end of this file;
 *   - RMSNorm (the model's attn_norm / ffn_norm scales, model-architecture page,
 *     weight table): y_i = x_i / sqrt(mean_j x_j^2 + eps) * gamma_i, the usual
 *     definition (the pages name the norm but print no formula), evaluated in
 *     double from the fp32 inputs and rounded once to fp32; eps > 0 is an argument.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math -shared -fPIC.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define QK 32
#define QBYTES 34

/* ---- IEEE-754 binary16 <-> binary32, from the format's definition ---------- */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Normal: (-1)^s * 2^(e-15) * (1 + f/1024); subnormal (e = 0): 2^-14 * f/1024. */
uint16_t q8o_f32_to_f16(float value) {
    uint32_t u;
    memcpy(&u, &value, 4);
    uint32_t sign = (u >> 16) & 0x8000u;
    uint32_t exp32 = (u >> 23) & 0xffu;
    uint32_t frac32 = u & 0x7fffffu;
    if (exp32 == 0xffu)                                 /* inf or NaN */
        return (uint16_t)(sign | 0x7c00u | (frac32 ? 0x200u : 0u));
    if (exp32 == 0u)                                     /* fp32 zero/subnormal: < 2^-126 -> 0 */
        return (uint16_t)sign;
    int e = (int)exp32 - 127;                            /* value = 1.frac * 2^e */
    if (e > 15)
        return (uint16_t)(sign | 0x7c00u);               /* overflow -> inf */
    uint32_t sig = frac32 | 0x800000u;                   /* 24-bit significand */
    if (e >= -14) {
        /* normal: keep 10 fraction bits, drop 13, round to nearest even */
        uint32_t keep = frac32 >> 13;
        uint32_t rest = frac32 & 0x1fffu;
        uint32_t h = ((uint32_t)(e + 15) << 10) | keep;
        if (rest > 0x1000u || (rest == 0x1000u && (keep & 1u)))
            h += 1u;                                     /* carry may reach inf: correct */
        return (uint16_t)(sign | h);
    }
    /* subnormal result: count in units of 2^-24; value / 2^-24 = sig * 2^(e+1) */
    int shift = -(e + 1);                                /* >= 14 here */
    if (shift > 31)
        return (uint16_t)sign;
    uint32_t keep = sig >> shift;
    uint32_t rest = sig & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rest > half || (rest == half && (keep & 1u)))
        keep += 1u;                                      /* 0x400 = smallest normal: correct */
    return (uint16_t)(sign | keep);
}

float q8o_f16_to_f32(uint16_t h) {
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    float v;
    if (e == 0)
        v = ldexpf((float)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexpf((float)(1024 + f), e - 25);
    return s ? -v : v;
}

/* ---- block access ------------------------------------------------------------ */

static float blk_d(const uint8_t *blk) {
    return q8o_f16_to_f32((uint16_t)(blk[0] | ((uint16_t)blk[1] << 8)));
}

static int8_t blk_q(const uint8_t *blk, int i) {
    return (int8_t)blk[2 + i];
}

/* ---- activation quantiser ----------------------------------------------------- */

/* One 32-element block of x -> one 34-byte block. */
void q8o_quantize_block(uint8_t *out, const float *x) {
    float amax = 0.0f;
    for (int i = 0; i < QK; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float d = amax / 127.0f;
    uint16_t dh = 0;
    if (d != 0.0f) {
        for (int i = 0; i < QK; ++i)
            out[2 + i] = (uint8_t)(int8_t)(int)roundf(x[i] / d);   /* through int: defined at +-128 */
        dh = q8o_f32_to_f16(d);
    } else {
        for (int i = 0; i < QK; ++i) out[2 + i] = 0;
    }
    out[0] = (uint8_t)(dh & 0xffu);
    out[1] = (uint8_t)(dh >> 8);
}

/* x [n_tok][in_dim] fp32 -> xq [n_tok][in_dim/32] blocks. */
int q8o_quantize(uint8_t *xq, const float *x, uint64_t in_dim, uint64_t n_tok) {
    if (in_dim == 0 || in_dim % QK) return -1;
    uint64_t nb = in_dim / QK;
    for (uint64_t t = 0; t < n_tok; ++t)
        for (uint64_t b = 0; b < nb; ++b)
            q8o_quantize_block(xq + (t * nb + b) * QBYTES, x + t * in_dim + b * QK);
    return 0;
}

/* ---- dot product -------------------------------------------------------------- */

/* One output: row w (nb blocks) against activation row a (nb blocks).
 * Returns the fp32 sum; *bound receives sum_b |d_w d_x isum_b| in double. */
float q8o_dot_row(const uint8_t *w, const uint8_t *a, uint64_t nb, double *bound) {
    float acc = 0.0f;
    double bsum = 0.0;
    for (uint64_t b = 0; b < nb; ++b) {
        const uint8_t *wb = w + b * QBYTES;
        const uint8_t *ab = a + b * QBYTES;
        int32_t isum = 0;
        for (int i = 0; i < QK; ++i)
            isum += (int32_t)blk_q(wb, i) * (int32_t)blk_q(ab, i);
        float dw = blk_d(wb), dx = blk_d(ab);
        acc += (dw * dx) * (float)isum;
        bsum += fabs((double)dw * (double)dx * (double)isum);
    }
    if (bound) *bound = bsum;
    return acc;
}

/* out[t][o] = sum_b d_w d_x sum_i q_w q_x, W [out_dim][nb] blocks,
 * xq [n_tok][nb] blocks.  bound (optional) gets the same shape as out. */
int q8o_matmul(float *out, double *bound, const uint8_t *W, uint64_t in_dim,
               uint64_t out_dim, const uint8_t *xq, uint64_t n_tok) {
    if (in_dim == 0 || in_dim % QK) return -1;
    uint64_t nb = in_dim / QK;
    for (uint64_t t = 0; t < n_tok; ++t)
        for (uint64_t o = 0; o < out_dim; ++o) {
            double bd = 0.0;
            out[t * out_dim + o] = q8o_dot_row(W + o * nb * QBYTES, xq + t * nb * QBYTES, nb, &bd);
            if (bound) bound[t * out_dim + o] = bd;
        }
    return 0;
}

/* Selected outputs only: out[s] = (tok[s], row[s]) of the full product. */
int q8o_matmul_sample(float *out, double *bound, const uint8_t *W, uint64_t in_dim,
                      uint64_t out_dim, const uint8_t *xq, uint64_t n_tok,
                      const int64_t *tok, const int64_t *row, uint64_t n_sample) {
    if (in_dim == 0 || in_dim % QK) return -1;
    uint64_t nb = in_dim / QK;
    for (uint64_t s = 0; s < n_sample; ++s) {
        if (tok[s] < 0 || (uint64_t)tok[s] >= n_tok || row[s] < 0 || (uint64_t)row[s] >= out_dim)
            return -1;
        double bd = 0.0;
        out[s] = q8o_dot_row(W + (uint64_t)row[s] * nb * QBYTES, xq + (uint64_t)tok[s] * nb * QBYTES, nb, &bd);
        if (bound) bound[s] = bd;
    }
    return 0;
}

/* ---- routed experts ------------------------------------------------------------ */

/* Pairs p = t*k + j select expert e = ids[p]; out[p][o] = W_e[o] . x_row, where
 * W_e = W_experts + e * expert_stride bytes, and x_row is activation row t
 * (x_per_pair == 0: xq has n_tok rows) or row p (x_per_pair != 0: n_tok*k rows).
 * Returns 0, or 1 when some id was out of range (its output row is zero). */
int q8o_moe(float *out, double *bound, const uint8_t *W_experts, uint32_t n_expert,
            uint64_t expert_stride, const int32_t *ids, uint32_t k, uint64_t in_dim,
            uint64_t out_dim, const uint8_t *xq, int x_per_pair, uint64_t n_tok) {
    if (in_dim == 0 || in_dim % QK || k == 0) return -1;
    uint64_t nb = in_dim / QK;
    int flag = 0;
    for (uint64_t t = 0; t < n_tok; ++t)
        for (uint32_t j = 0; j < k; ++j) {
            uint64_t p = t * k + j;
            int32_t e = ids[p];
            const uint8_t *xrow = xq + (x_per_pair ? p : t) * nb * QBYTES;
            for (uint64_t o = 0; o < out_dim; ++o) {
                double bd = 0.0;
                float v = 0.0f;
                if (e < 0 || (uint32_t)e >= n_expert) {
                    flag = 1;
                } else {
                    const uint8_t *w = W_experts + (uint64_t)e * expert_stride + o * nb * QBYTES;
                    v = q8o_dot_row(w, xrow, nb, &bd);
                }
                out[p * out_dim + o] = v;
                if (bound) bound[p * out_dim + o] = bd;
            }
        }
    return flag;
}

/* Selected outputs of the routed product: (pair[s], row[s]). */
int q8o_moe_sample(float *out, double *bound, const uint8_t *W_experts, uint32_t n_expert,
                   uint64_t expert_stride, const int32_t *ids, uint32_t k, uint64_t in_dim,
                   uint64_t out_dim, const uint8_t *xq, int x_per_pair, uint64_t n_tok,
                   const int64_t *pair, const int64_t *row, uint64_t n_sample) {
    if (in_dim == 0 || in_dim % QK || k == 0) return -1;
    uint64_t nb = in_dim / QK;
    int flag = 0;
    for (uint64_t s = 0; s < n_sample; ++s) {
        if (pair[s] < 0 || (uint64_t)pair[s] >= n_tok * k || row[s] < 0 || (uint64_t)row[s] >= out_dim)
            return -1;
        uint64_t p = (uint64_t)pair[s];
        int32_t e = ids[p];
        double bd = 0.0;
        float v = 0.0f;
        if (e < 0 || (uint32_t)e >= n_expert) {
            flag = 1;
        } else {
            const uint8_t *xrow = xq + (x_per_pair ? p : p / k) * nb * QBYTES;
            v = q8o_dot_row(W_experts + (uint64_t)e * expert_stride + (uint64_t)row[s] * nb * QBYTES,
                            xrow, nb, &bd);
        }
        out[s] = v;
        if (bound) bound[s] = bd;
    }
    return flag;
}

/* ---- the expert FFN around the routed product --------------------------------- */

/* SwiGLU with the optional clamp, element by element:
 *   limit > 0: gate = min(gate, limit), up = min(max(up, -limit), limit)
 *   mid = silu(gate) * up,  silu(g) = g / (1 + e^-g). */
void q8o_swiglu(float *mid, const float *gate, const float *up, uint64_t n, float limit) {
    for (uint64_t i = 0; i < n; ++i) {
        double g = gate[i], u = up[i];
        if (limit > 0.0f) {
            if (g > limit) g = limit;
            if (u > limit) u = limit;
            if (u < -limit) u = -limit;
        }
        mid[i] = (float)(g / (1.0 + exp(-g)) * u);
    }
}

/* Weighted sum of each token's k expert outputs: out[t][o] = sum_j w[t*k+j] *
 * y[t*k+j][o] (j = 0..k-1, in double); bound[t][o] = sum_j |w y|. */
void q8o_combine(double *out, double *bound, const float *y, const float *w, uint64_t n_tok, uint32_t k,
                 uint64_t dim) {
    for (uint64_t t = 0; t < n_tok; ++t)
        for (uint64_t o = 0; o < dim; ++o) {
            double s = 0.0, b = 0.0;
            for (uint32_t j = 0; j < k; ++j) {
                uint64_t p = t * k + j;
                double v = (double)w[p] * (double)y[p * dim + o];
                s += v;
                b += fabs(v);
            }
            out[t * dim + o] = s;
            if (bound) bound[t * dim + o] = b;
        }
}

/* The routed expert FFN of n_tok tokens, k experts each (pair p = t*k + j,
 * expert ids[p], weight w[p]):
 *   gate[p] = W_gate[e] . xq[t],  up[p] = W_up[e] . xq[t]      (in_dim -> mid_dim)
 *   mid[p]  = swiglu(gate[p], up[p])
 *   y[p]    = W_down[e] . quantise(mid[p])                     (mid_dim -> out_dim)
 *   out[t]  = sum_j w[t*k+j] y[t*k+j]
 * x is fp32 [n_tok][in_dim] and is quantised here.  Expert e's gate and up
 * matrices start at e * gate_up_stride bytes, its down matrix at e * down_stride.
 * Returned besides out (double [n_tok][out_dim]) and its bound: y and y_bound
 * ([n_pairs][out_dim]), mid ([n_pairs][mid_dim]) and its quantised blocks midq
 * ([n_pairs][mid_dim/32] blocks).  Returns 1 when an id was out of range (that
 * pair's gate, up, mid and y rows are zero), 0 otherwise, -1 on bad dimensions
 * or allocation failure. */
int q8o_moe_ffn(double *out, double *out_bound, float *y, double *y_bound, float *mid, uint8_t *midq,
                const uint8_t *W_gate, const uint8_t *W_up, const uint8_t *W_down, uint32_t n_expert,
                uint64_t gate_up_stride, uint64_t down_stride, const int32_t *ids, const float *w, uint32_t k,
                uint64_t in_dim, uint64_t mid_dim, uint64_t out_dim, float limit, const float *x,
                uint64_t n_tok) {
    if (in_dim == 0 || in_dim % QK || mid_dim == 0 || mid_dim % QK || k == 0) return -1;
    uint64_t n_pairs = n_tok * k;
    uint8_t *xq = malloc(n_tok * (in_dim / QK) * QBYTES + 1);
    float *gate = malloc(n_pairs * mid_dim * sizeof(float) + 1);
    float *up = malloc(n_pairs * mid_dim * sizeof(float) + 1);
    int rc = -1;
    if (xq && gate && up) {
        q8o_quantize(xq, x, in_dim, n_tok);
        int f1 = q8o_moe(gate, NULL, W_gate, n_expert, gate_up_stride, ids, k, in_dim, mid_dim, xq, 0, n_tok);
        int f2 = q8o_moe(up, NULL, W_up, n_expert, gate_up_stride, ids, k, in_dim, mid_dim, xq, 0, n_tok);
        q8o_swiglu(mid, gate, up, n_pairs * mid_dim, limit);
        q8o_quantize(midq, mid, mid_dim, n_pairs);
        int f3 = q8o_moe(y, y_bound, W_down, n_expert, down_stride, ids, k, mid_dim, out_dim, midq, 1, n_tok);
        q8o_combine(out, out_bound, y, w, n_tok, k, out_dim);
        rc = (f1 < 0 || f2 < 0 || f3 < 0) ? -1 : (f1 | f2 | f3);
    }
    free(xq);
    free(gate);
    free(up);
    return rc;
}

/* ---- RMSNorm feeding the quantiser ------------------------------------------- */

/* Per token row t: r = 1 / sqrt(mean_i x_i^2 + eps), y_i = x_i * r * gamma_i
 * (gamma == NULL: all ones), then xq = the activation quantiser of y.  y is
 * fp32 [n_tok][dim], xq [n_tok][dim/32] blocks.  Returns -1 on bad dimensions. */
int q8o_rmsnorm_quantize(uint8_t *xq, float *y, const float *x, const float *gamma, uint64_t dim,
                         uint64_t n_tok, double eps) {
    if (dim == 0 || dim % QK) return -1;
    for (uint64_t t = 0; t < n_tok; ++t) {
        const float *xr = x + t * dim;
        double s = 0.0;
        for (uint64_t i = 0; i < dim; ++i) s += (double)xr[i] * (double)xr[i];
        double r = 1.0 / sqrt(s / (double)dim + eps);
        for (uint64_t i = 0; i < dim; ++i)
            y[t * dim + i] = (float)((double)xr[i] * r * (gamma ? (double)gamma[i] : 1.0));
    }
    return q8o_quantize(xq, y, dim, n_tok);
}

/* ---- second weight format: K-quant super-blocks x Q8_K activations -----------
 *
 * Model-architecture page, quantisation section 3 ("Block layout"): 256 weights
 * per block; Q2_K is 84 bytes (scales[16], qs[64] of 2-bit values, d, dmin) and
 * Q4_K 144 bytes (d, dmin, scales[12] holding scales and mins, qs[128] of 4-bit
 * values).  Section 1 prints the 2-bit field order inside a byte (field k is
 * (byte >> 2k) & 3) and the Q8_K quantiser; section 4 the dot product of a
 * K-quant row with a Q8_K row, whose value is the sum of dequantised weight
 * times dequantised activation.  The routed experts of the code walkthrough
 * (trace 5) and the MoE page's Q4_K expert path use these blocks.
 *
 * Readings where the pages are silent (each one also listed in the design notes):
 *   - the pages name these blocks llama.cpp/GGML formats and print their field
 *     order and sizes, not the packing inside them; the packing is GGML's k-quant
 *     layout:
 *       Q2_K: d, dmin binary16 little-endian at bytes 80 and 82; 16 sub-blocks of
 *         16 weights; scales[i] holds sub-block i's scale (low nibble) and min
 *         (high nibble); weight 128h + 32j + 16s + l (h < 2, j < 4, s < 2, l < 16)
 *         is field j of byte qs[32h + 16s + l], in sub-block 8h + 2j + s.
 *       Q4_K: d, dmin at bytes 0 and 2, scales[12] at 4, qs at 16; 8 sub-blocks of
 *         32 weights with 6-bit scale sc and min m: for j < 4, sc = s[j] & 63 and
 *         m = s[j+4] & 63; for j >= 4, sc = (s[j+4] & 15) | ((s[j-4] >> 6) << 4) and
 *         m = (s[j+4] >> 4) | ((s[j] >> 6) << 4); weight 64c + l (c < 4, l < 32) is
 *         the low nibble of qs[32c + l] (sub-block 2c), weight 64c + 32 + l its high
 *         nibble (sub-block 2c + 1);
 *   - a weight's value is d * sc * q - dmin * m (the printed comment's
 *     "d * (scale * q + dmin * offset)" is garbled; a min offset is subtracted);
 *   - Q8_K: fp32 d = amax / 127 and q = (int8) roundf(x / d) per 256-value block as
 *     printed; an all-zero block stores d = 0 and q = 0;
 *   - the product is the plain definition: out = sum_i w_i * (d_x * q_x,i) over the
 *     dequantised values, evaluated in double and rounded once to fp32.
 */
#define QKK 256
#define KQ_Q2 2
#define KQ_Q4 4

uint64_t q8o_kq_block_bytes(int fmt) {
    return fmt == KQ_Q2 ? 84u : (fmt == KQ_Q4 ? 144u : 0u);
}

static uint16_t le16(const uint8_t *p) { return (uint16_t)(p[0] | ((uint16_t)p[1] << 8)); }

/* Scale, min and 2- or 4-bit value of weight i (0..255) of one block. */
static void kq_fields(const uint8_t *blk, int fmt, int i, int *sc, int *m, int *q, double *d, double *dmin) {
    if (fmt == KQ_Q2) {
        int h = i / 128, j = (i % 128) / 32, s = (i % 32) / 16, l = i % 16;
        int sb = 8 * h + 2 * j + s;
        *sc = blk[sb] & 15;
        *m = blk[sb] >> 4;
        *q = (blk[16 + 32 * h + 16 * s + l] >> (2 * j)) & 3;
        *d = q8o_f16_to_f32(le16(blk + 80));
        *dmin = q8o_f16_to_f32(le16(blk + 82));
    } else {
        const uint8_t *s = blk + 4;
        int c = i / 64, hi = (i % 64) / 32, l = i % 32;
        int j = 2 * c + hi;
        if (j < 4) {
            *sc = s[j] & 63;
            *m = s[j + 4] & 63;
        } else {
            *sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
            *m = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
        }
        uint8_t byte = blk[16 + 32 * c + l];
        *q = hi ? (byte >> 4) : (byte & 15);
        *d = q8o_f16_to_f32(le16(blk));
        *dmin = q8o_f16_to_f32(le16(blk + 2));
    }
}

/* The 256 weights of one block as doubles: d * sc * q - dmin * m. */
static void kq_dequant_block(double *w, const uint8_t *blk, int fmt) {
    for (int i = 0; i < QKK; ++i) {
        int sc, m, q;
        double d, dmin;
        kq_fields(blk, fmt, i, &sc, &m, &q, &d, &dmin);
        w[i] = d * (double)sc * (double)q - dmin * (double)m;
    }
}

/* W [rows][in_dim/256 blocks] -> out [rows][in_dim] doubles. */
int q8o_kq_dequant(double *out, const uint8_t *W, int fmt, uint64_t in_dim, uint64_t rows) {
    uint64_t bb = q8o_kq_block_bytes(fmt);
    if (!bb || in_dim == 0 || in_dim % QKK) return -1;
    uint64_t nsb = in_dim / QKK;
    for (uint64_t r = 0; r < rows; ++r)
        for (uint64_t b = 0; b < nsb; ++b)
            kq_dequant_block(out + r * in_dim + b * QKK, W + (r * nsb + b) * bb, fmt);
    return 0;
}

/* Q8_K: x [n_tok][in_dim] -> d [n_tok][in_dim/256] (fp32) and q [n_tok][in_dim]. */
int q8o_quantize_q8k(float *d, int8_t *q, const float *x, uint64_t in_dim, uint64_t n_tok) {
    if (in_dim == 0 || in_dim % QKK) return -1;
    uint64_t nsb = in_dim / QKK;
    for (uint64_t t = 0; t < n_tok; ++t)
        for (uint64_t b = 0; b < nsb; ++b) {
            const float *xb = x + t * in_dim + b * QKK;
            int8_t *qb = q + t * in_dim + b * QKK;
            float amax = 0.0f;
            for (int i = 0; i < QKK; ++i) {
                float a = fabsf(xb[i]);
                if (a > amax) amax = a;
            }
            float scale = amax / 127.0f;
            d[t * nsb + b] = scale;
            for (int i = 0; i < QKK; ++i)
                qb[i] = scale != 0.0f ? (int8_t)(int)roundf(xb[i] / scale) : 0;
        }
    return 0;
}

/* Sub-block of weight i: Q2_K 16 sub-blocks of 16, Q4_K 8 of 32 (layout above). */
static int kq_subblock(int fmt, int i) {
    if (fmt == KQ_Q2) return 8 * (i / 128) + 2 * ((i % 128) / 32) + (i % 32) / 16;
    return 2 * (i / 64) + (i % 64) / 32;
}

/* One output: K-quant row w (nsb blocks) against Q8_K row (dx [nsb], qx [nsb*256]).
 * Returns the fp32 rounding of the double sum; *bound gets
 * sum_b sum_j |d_x| (|d sc_j isum_j| + |dmin m_j xsum_j|) over the blocks' sub-blocks j
 * (isum_j = sum q_w q_x, xsum_j = sum q_x): the terms a fixed-point evaluation
 * adds in fp32, one per sub-block as the Q8_0 bound has one per 32-value block. */
float q8o_kq_dot_row(const uint8_t *w, int fmt, const float *dx, const int8_t *qx, uint64_t nsb, double *bound) {
    uint64_t bb = q8o_kq_block_bytes(fmt);
    double acc = 0.0, bsum = 0.0;
    double wv[QKK];
    for (uint64_t b = 0; b < nsb; ++b) {
        const uint8_t *blk = w + b * bb;
        kq_dequant_block(wv, blk, fmt);
        double xd = (double)dx[b];
        double dot = 0.0, d = 0.0, dmin = 0.0;
        double t_sc[16] = {0}, t_m[16] = {0};
        for (int i = 0; i < QKK; ++i) {
            int sc, m, q;
            kq_fields(blk, fmt, i, &sc, &m, &q, &d, &dmin);
            int qxi = qx[b * QKK + i];
            int j = kq_subblock(fmt, i);
            dot += wv[i] * (xd * (double)qxi);
            t_sc[j] += (double)sc * (double)q * (double)qxi;
            t_m[j] += (double)m * (double)qxi;
        }
        acc += dot;
        for (int j = 0; j < 16; ++j) bsum += fabs(xd) * (fabs(d * t_sc[j]) + fabs(dmin * t_m[j]));
    }
    if (bound) *bound = bsum;
    return (float)acc;
}

/* out[t][o] = row o of W against Q8_K row t. */
int q8o_kq_matmul_q(float *out, double *bound, const uint8_t *W, int fmt, uint64_t in_dim, uint64_t out_dim,
                    const float *dx, const int8_t *qx, uint64_t n_tok) {
    uint64_t bb = q8o_kq_block_bytes(fmt);
    if (!bb || in_dim == 0 || in_dim % QKK) return -1;
    uint64_t nsb = in_dim / QKK;
    for (uint64_t t = 0; t < n_tok; ++t)
        for (uint64_t o = 0; o < out_dim; ++o) {
            double bd = 0.0;
            out[t * out_dim + o] = q8o_kq_dot_row(W + o * nsb * bb, fmt, dx + t * nsb, qx + t * in_dim, nsb, &bd);
            if (bound) bound[t * out_dim + o] = bd;
        }
    return 0;
}

/* Routed K-quant experts: pair p = t*k + j multiplies expert ids[p]'s matrix
 * (at W_experts + ids[p] * expert_stride bytes) by Q8_K row p (x_per_pair) or t.
 * An id outside [0, n_expert) gives a zero row and return value 1. */
int q8o_kq_moe(float *out, double *bound, const uint8_t *W_experts, int fmt, uint32_t n_expert,
               uint64_t expert_stride, const int32_t *ids, uint32_t k, uint64_t in_dim, uint64_t out_dim,
               const float *dx, const int8_t *qx, int x_per_pair, uint64_t n_tok) {
    uint64_t bb = q8o_kq_block_bytes(fmt);
    if (!bb || in_dim == 0 || in_dim % QKK || k == 0) return -1;
    uint64_t nsb = in_dim / QKK;
    int flag = 0;
    for (uint64_t p = 0; p < n_tok * k; ++p) {
        int32_t e = ids[p];
        uint64_t xr = x_per_pair ? p : p / k;
        for (uint64_t o = 0; o < out_dim; ++o) {
            double bd = 0.0;
            float v = 0.0f;
            if (e < 0 || (uint32_t)e >= n_expert)
                flag = 1;
            else
                v = q8o_kq_dot_row(W_experts + (uint64_t)e * expert_stride + o * nsb * bb, fmt, dx + xr * nsb,
                                   qx + xr * in_dim, nsb, &bd);
            out[p * out_dim + o] = v;
            if (bound) bound[p * out_dim + o] = bd;
        }
    }
    return flag;
}
