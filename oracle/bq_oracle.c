/*
 * bq_oracle.c -- the oracle: plain, slow CPU statement of block-quantized
 * weight packing and the batch-1 dequant + matrix-vector product.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  The GPU library never
 * includes, links or calls it, and the two share no source.
 *
 * Everything here is single-threaded scalar C.  Packing follows fp32 IEEE-754
 * arithmetic exactly (build with -ffp-contract=off, no fast-math) because the
 * packed bytes are compared bit for bit.  Dequantization and the dot products
 * are done in fp64, summed in index order.
 *
 * Sources (the pages give the formats only by their byte cost and name):
 *  - RunIT README, "Quantization" table and "Key Technique" column: Q8_0 at
 *    1.06 B/elem, Q4_0 at 0.56 B/elem, dequantized on the fly inside the dot
 *    product.  1.0625 = 34/32 and 0.5625 = 18/32: one fp16 scale per 32
 *    weights plus 8 or 4 bits per weight, the GGUF block formats the README
 *    names under its GGUF Format link.
 *  - EdgeRunner blog post, "What worked" #2: the fused kernel reads the
 *    quantized weights directly; no fp32 weights are materialised.
 *  - Block layouts, scale rules and nibble order (the plainest reading of the
 *    GGUF-style formats):
 *      Q8_0 block, 34 B: fp16 d (little-endian) at bytes 0-1, then q[0..31]
 *           as int8.  d = fp16(max|w| / 127); q = round(w / d); w' = d * q.
 *      Q4_0 block, 18 B: fp16 d at bytes 0-1, then qs[0..15]; element j < 16
 *           is qs[j] & 0xF and element j+16 is qs[j] >> 4.
 *           d = fp16(max|w| / 8); n = clamp(round(w / d) + 8, 0, 15);
 *           w' = d * (n - 8).
 *    "round" is round-half-away-from-zero (C roundf); the divisions are fp32
 *    and correctly rounded; w / d divides by the STORED fp16 scale; d == 0
 *    gives q = 0 (Q8_0) or n = 8 (Q4_0).
 *  - Q4_K (RunIT README kernel table, gemv_q4k_f16 / "gemv_q4k.metal", and
 *    "Quantization" table, Q4_K_M; EdgeRunner forum summary, 核心特性, the
 *    K-quant formats).  The pages name the format but do not define it; the
 *    reading here is the public GGUF Q4_K super-block:
 *      256 weights in 144 bytes: fp16 d at bytes 0-1, fp16 dmin at bytes 2-3,
 *      12 bytes s[0..11] holding eight 6-bit sub-block scales sc[j] and mins
 *      m[j] (j < 4: sc = s[j] & 63, m = s[j+4] & 63; j >= 4: sc = (s[j+4] &
 *      15) | (s[j-4] >> 6) << 4, m = (s[j+4] >> 4) | (s[j] >> 6) << 4), then
 *      128 bytes qs: sub-blocks 2g and 2g+1 (32 weights each) share
 *      qs[32g .. 32g+31], element i of sub-block 2g the low nibble of
 *      qs[32g+i] and element i of sub-block 2g+1 its high nibble;
 *      w = d*sc[j]*q - dmin*m[j] for sub-block j.
 *    The quantizer is not on the pages either; the plainest reading that
 *    fills this layout, per sub-block j: lo = min(0, min w), hi = max w,
 *    scale_j = (hi - lo) / 15, min_j = -lo; per super-block d =
 *    fp16(max_j scale_j / 63), dmin = fp16(max_j min_j / 63); sc[j] =
 *    clamp(round(scale_j / d), 0, 63), m[j] = clamp(round(min_j / dmin), 0,
 *    63) (0 when the divisor is 0); q = clamp(round((w + dmin*m[j]) /
 *    (d*sc[j])), 0, 15) (0 when d*sc[j] is 0).  fp32 arithmetic, correctly
 *    rounded divisions, round half away from zero, as for Q8_0 / Q4_0.
 *  - RMSNorm and SiLU for the fused gate+up kernel (RunIT README kernel table
 *    rows rms_norm_f32_f32_f32g, silu_mul_f32 and fused_ffn_q4_0_f32 "gate+up+
 *    silu fused"; EdgeRunner "The progression", RMSNorm+GEMV fusion stage):
 *    xn = x * gamma / sqrt(mean(x^2) + eps); y = silu(Wg xn) * (Wu xn),
 *    silu(z) = z / (1 + exp(-z)).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define BQO_Q4_0 2
#define BQO_Q8_0 8
#define BQO_Q4_K 12

/* ------------------------------------------------------------------------ */
/* IEEE-754 binary16 conversion, written from the format definition.        */
/* ------------------------------------------------------------------------ */

static int floor_log2_u32(uint32_t v) { /* v > 0 */
    int e = -1;
    while (v) { v >>= 1; ++e; }
    return e;
}

/* fp32 -> fp16 bits, round to nearest, ties to even; overflow gives +-Inf;
 * binary16 subnormals are produced (gradual underflow); NaN stays NaN. */
uint16_t bqo_f32_to_f16_bits(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t sgn = (uint16_t)((u >> 16) & 0x8000u);
    uint32_t bexp = (u >> 23) & 0xFFu;
    uint32_t frac = u & 0x7FFFFFu;
    if (bexp == 0xFFu) /* Inf or NaN */
        return (uint16_t)(sgn | 0x7C00u | (frac ? (0x200u | (frac >> 13)) : 0u));
    if (bexp == 0 && frac == 0) return sgn; /* signed zero */
    /* |f| = sig * 2^ex with sig an integer */
    uint32_t sig = bexp ? (frac | 0x800000u) : frac;
    int ex = bexp ? (int)bexp - 150 : -149;
    int e = floor_log2_u32(sig) + ex; /* exponent of the leading bit */
    /* quantum of the binary16 result: 2^(e-10) for normal halves, and the
     * subnormal quantum 2^-24 below the normal range */
    int qe = (e < -14) ? -24 : e - 10;
    int shift = qe - ex; /* bits of sig below the quantum, always > 0 here */
    uint32_t m;
    if (shift >= 32) {
        m = 0; /* |f| < 2^-32 of a quantum: rounds to zero */
    } else {
        m = sig >> shift;
        uint32_t rem = sig & ((1u << shift) - 1u);
        uint32_t half = 1u << (shift - 1);
        if (rem > half || (rem == half && (m & 1u))) m += 1u;
    }
    if (m < 1024u) return (uint16_t)(sgn | m); /* subnormal (or zero) half */
    if (m == 2048u) { m = 1024u; qe += 1; }   /* rounding carried */
    int hexp = qe + 10 + 15;                  /* biased exponent */
    if (hexp >= 31) return (uint16_t)(sgn | 0x7C00u);
    return (uint16_t)(sgn | ((uint32_t)hexp << 10) | (m - 1024u));
}

/* fp16 bits -> fp64, exact. */
double bqo_f16_bits_to_f64(uint16_t h) {
    int s = (h >> 15) & 1;
    int be = (h >> 10) & 0x1F;
    int man = h & 0x3FF;
    double v;
    if (be == 0x1F) v = man ? NAN : INFINITY;
    else if (be == 0) v = ldexp((double)man, -24);
    else v = ldexp((double)(man + 1024), be - 25);
    return s ? -v : v;
}

void bqo_f32_to_f16_array(const float *in, uint16_t *out, int64_t n) {
    for (int64_t i = 0; i < n; ++i) out[i] = bqo_f32_to_f16_bits(in[i]);
}

/* ------------------------------------------------------------------------ */
/* Q4_K super-blocks (the reading in the header comment)                    */
/* ------------------------------------------------------------------------ */

static float q4k_stored(uint16_t h) { return (float)bqo_f16_bits_to_f64(h); }

static float q4k_round_clamp(float v, float hi) {
    float r = roundf(v);
    if (r > hi) r = hi;
    if (r < 0.0f) r = 0.0f;
    return r;
}

/* sub-block j's 6-bit scale and min from the 12 scale bytes */
static void q4k_scale_min(const uint8_t *s, int j, int *sc, int *mn) {
    if (j < 4) {
        *sc = s[j] & 63;
        *mn = s[j + 4] & 63;
    } else {
        *sc = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
        *mn = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
    }
}

/* One super-block of 256 fp32 weights into 144 bytes. */
static void pack_superblock_q4_k(const float *w, uint8_t *sb) {
    float scale[8], mins[8], smax = 0.0f, mmax = 0.0f;
    for (int j = 0; j < 8; ++j) {
        float lo = 0.0f, hi = w[32 * j];
        for (int i = 0; i < 32; ++i) {
            float v = w[32 * j + i];
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
        scale[j] = (hi - lo) / 15.0f;
        mins[j] = -lo;
        if (scale[j] > smax) smax = scale[j];
        if (mins[j] > mmax) mmax = mins[j];
    }
    uint16_t dh = bqo_f32_to_f16_bits(smax / 63.0f);
    uint16_t mh = bqo_f32_to_f16_bits(mmax / 63.0f);
    float d = q4k_stored(dh), dmin = q4k_stored(mh);
    int sc[8], mn[8];
    for (int j = 0; j < 8; ++j) {
        sc[j] = d != 0.0f ? (int)q4k_round_clamp(scale[j] / d, 63.0f) : 0;
        mn[j] = dmin != 0.0f ? (int)q4k_round_clamp(mins[j] / dmin, 63.0f) : 0;
    }
    sb[0] = (uint8_t)(dh & 0xFFu);
    sb[1] = (uint8_t)(dh >> 8);
    sb[2] = (uint8_t)(mh & 0xFFu);
    sb[3] = (uint8_t)(mh >> 8);
    uint8_t *s = sb + 4;
    for (int j = 0; j < 4; ++j) {
        s[j] = (uint8_t)(sc[j] | ((sc[j + 4] >> 4) << 6));
        s[j + 4] = (uint8_t)(mn[j] | ((mn[j + 4] >> 4) << 6));
        s[j + 8] = (uint8_t)((sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4));
    }
    uint8_t *qs = sb + 16;
    memset(qs, 0, 128);
    for (int j = 0; j < 8; ++j) {
        float D = d * (float)sc[j], Mf = dmin * (float)mn[j];
        for (int i = 0; i < 32; ++i) {
            int q = D != 0.0f ? (int)q4k_round_clamp((w[32 * j + i] + Mf) / D, 15.0f) : 0;
            qs[32 * (j / 2) + i] |= (uint8_t)((j & 1) ? q << 4 : q);
        }
    }
}

/* code q (0..15), D = d*sc and Mf = dmin*m (fp64, exact) of element e (0..255) */
static void q4k_elem(const uint8_t *sb, int e, int *q, double *D, double *Mf) {
    int j = e / 32, i = e % 32, sc, mn;
    q4k_scale_min(sb + 4, j, &sc, &mn);
    int byte = sb[16 + 32 * (j / 2) + i];
    *q = (j & 1) ? (byte >> 4) : (byte & 0xF);
    *D = bqo_f16_bits_to_f64((uint16_t)(sb[0] | (sb[1] << 8))) * (double)sc;
    *Mf = bqo_f16_bits_to_f64((uint16_t)(sb[2] | (sb[3] << 8))) * (double)mn;
}

static double q4k_weight(const uint8_t *row, int64_t k) {
    int q;
    double D, Mf;
    q4k_elem(row + (k / 256) * 144, (int)(k % 256), &q, &D, &Mf);
    return D * (double)q - Mf;
}

static int q4k_pack(const float *W, int64_t M, int64_t K, uint8_t *out) {
    if (M < 0 || K < 0 || K % 256) return -1;
    int64_t ns = K / 256;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t b = 0; b < ns; ++b) pack_superblock_q4_k(W + m * K + 256 * b, out + (m * ns + b) * 144);
    return 0;
}

static int q4k_dequant(const uint8_t *Wq, int64_t M, int64_t K, double *out) {
    if (M < 0 || K < 0 || K % 256) return -1;
    int64_t rb = K / 256 * 144;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k) out[m * K + k] = q4k_weight(Wq + m * rb, k);
    return 0;
}

static int q4k_gemv(const uint8_t *Wq, int64_t M, int64_t K, const double *x, double *y, double *S) {
    if (M < 0 || K < 0 || K % 256) return -1;
    int64_t rb = K / 256 * 144;
    for (int64_t m = 0; m < M; ++m) {
        double acc = 0.0, sacc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = q4k_weight(Wq + m * rb, k) * x[k];
            acc += p;
            sacc += fabs(p);
        }
        y[m] = acc;
        if (S) S[m] = sacc;
    }
    return 0;
}

/* The bound's scale for Q4_K rows: SK[m] = sum over sub-blocks j of
 * (d*sc_j * sum_i |q_i x_i| + dmin*m_j * sum_i |x_i|), the sums of the
 * magnitudes of the two terms w = d*sc*q - dmin*m splits each weight into
 * (SK >= sum_k |w x|). */
int bqo_q4_k_split_scale(const uint8_t *Wq, int64_t M, int64_t K, const double *x, double *SK) {
    if (M < 0 || K < 0 || K % 256) return -1;
    int64_t rb = K / 256 * 144;
    for (int64_t m = 0; m < M; ++m) {
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            int q;
            double D, Mf;
            q4k_elem(Wq + m * rb + (k / 256) * 144, (int)(k % 256), &q, &D, &Mf);
            acc += D * fabs((double)q * x[k]) + Mf * fabs(x[k]);
        }
        SK[m] = acc;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Block formats                                                            */
/* ------------------------------------------------------------------------ */

int64_t bqo_block_bytes(int qtype) {
    if (qtype == BQO_Q8_0) return 34;
    if (qtype == BQO_Q4_0) return 18;
    return -1;
}

int64_t bqo_packed_bytes(int qtype, int64_t M, int64_t K) {
    if (qtype == BQO_Q4_K) return (M < 0 || K < 0 || K % 256) ? -1 : M * (K / 256) * 144;
    int64_t bb = bqo_block_bytes(qtype);
    if (bb < 0 || M < 0 || K < 0 || K % 32) return -1;
    return M * (K / 32) * bb;
}

static float stored_scale(uint16_t dh) { return (float)bqo_f16_bits_to_f64(dh); }

/* One Q8_0 block from 32 fp32 weights. */
static void pack_block_q8_0(const float *w, uint8_t *blk) {
    float amax = 0.0f;
    for (int j = 0; j < 32; ++j) {
        float a = fabsf(w[j]);
        if (a > amax) amax = a;
    }
    float d32 = amax / 127.0f;
    uint16_t dh = bqo_f32_to_f16_bits(d32);
    float df = stored_scale(dh);
    blk[0] = (uint8_t)(dh & 0xFFu);
    blk[1] = (uint8_t)(dh >> 8);
    for (int j = 0; j < 32; ++j) {
        int q = 0;
        if (df != 0.0f) {
            float r = roundf(w[j] / df);
            if (r > 127.0f) r = 127.0f;
            if (r < -127.0f) r = -127.0f;
            q = (int)r;
        }
        blk[2 + j] = (uint8_t)(int8_t)q;
    }
}

/* One Q4_0 block from 32 fp32 weights. */
static void pack_block_q4_0(const float *w, uint8_t *blk) {
    float amax = 0.0f;
    for (int j = 0; j < 32; ++j) {
        float a = fabsf(w[j]);
        if (a > amax) amax = a;
    }
    float d32 = amax / 8.0f;
    uint16_t dh = bqo_f32_to_f16_bits(d32);
    float df = stored_scale(dh);
    int n[32];
    for (int j = 0; j < 32; ++j) {
        float r = 8.0f;
        if (df != 0.0f) r = roundf(w[j] / df) + 8.0f;
        if (r > 15.0f) r = 15.0f;
        if (r < 0.0f) r = 0.0f;
        n[j] = (int)r;
    }
    blk[0] = (uint8_t)(dh & 0xFFu);
    blk[1] = (uint8_t)(dh >> 8);
    for (int j = 0; j < 16; ++j) blk[2 + j] = (uint8_t)(n[j] | (n[j + 16] << 4));
}

/* W: fp32 [M, K] row-major; out: M rows of K/32 blocks.  Returns 0, or -1 on
 * a bad qtype or shape. */
int bqo_quantize_pack(int qtype, const float *W, int64_t M, int64_t K, uint8_t *out) {
    if (qtype == BQO_Q4_K) return q4k_pack(W, M, K, out);
    int64_t bb = bqo_block_bytes(qtype);
    if (bb < 0 || M < 0 || K < 0 || K % 32) return -1;
    int64_t nb = K / 32;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t b = 0; b < nb; ++b) {
            const float *w = W + m * K + 32 * b;
            uint8_t *blk = out + (m * nb + b) * bb;
            if (qtype == BQO_Q8_0) pack_block_q8_0(w, blk);
            else pack_block_q4_0(w, blk);
        }
    return 0;
}

/* Dequantized weight of element j (0..31) of one block, in fp64 (exact). */
static double dequant_elem(int qtype, const uint8_t *blk, int j) {
    uint16_t dh = (uint16_t)(blk[0] | (blk[1] << 8));
    double d = bqo_f16_bits_to_f64(dh);
    if (qtype == BQO_Q8_0) return d * (double)(int8_t)blk[2 + j];
    int byte = blk[2 + (j & 15)];
    int nib = (j < 16) ? (byte & 0xF) : (byte >> 4);
    return d * (double)(nib - 8);
}

/* Wq: M packed rows -> fp64 [M, K]. */
int bqo_dequant(int qtype, const uint8_t *Wq, int64_t M, int64_t K, double *out) {
    if (qtype == BQO_Q4_K) return q4k_dequant(Wq, M, K, out);
    int64_t bb = bqo_block_bytes(qtype);
    if (bb < 0 || M < 0 || K < 0 || K % 32) return -1;
    int64_t nb = K / 32;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t k = 0; k < K; ++k)
            out[m * K + k] = dequant_elem(qtype, Wq + (m * nb + k / 32) * bb, (int)(k % 32));
    return 0;
}

/* y[m] = sum_k w[m,k] * x[k]; S[m] = sum_k |w[m,k] * x[k]| (S may be NULL).
 * fp64, summed in index order.  x is fp64 so that fp32 inputs pass exactly
 * and an fp64 RMSNorm output can be fed in. */
int bqo_gemv(int qtype, const uint8_t *Wq, int64_t M, int64_t K, const double *x,
             double *y, double *S) {
    if (qtype == BQO_Q4_K) return q4k_gemv(Wq, M, K, x, y, S);
    int64_t bb = bqo_block_bytes(qtype);
    if (bb < 0 || M < 0 || K < 0 || K % 32) return -1;
    int64_t nb = K / 32;
    for (int64_t m = 0; m < M; ++m) {
        double acc = 0.0, sacc = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = dequant_elem(qtype, Wq + (m * nb + k / 32) * bb, (int)(k % 32)) * x[k];
            acc += p;
            sacc += fabs(p);
        }
        y[m] = acc;
        if (S) S[m] = sacc;
    }
    return 0;
}

/* The fused q|k|v + bias projection (RunIT README kernel table,
 * fused_qkv_bias_q8_0_f32, "Q+K+V+bias in ONE dispatch"), read as the plain
 * definition: y[m] = sum_k w[m,k] * x[k] + bias[m] over the q, k and v rows
 * concatenated, in fp64; S[m] = sum_k |w[m,k] * x[k]| + |bias[m]| (S may be
 * NULL; bias NULL means zeros). */
int bqo_gemv_bias(int qtype, const uint8_t *Wq, int64_t M, int64_t K, const double *x,
                  const double *bias, double *y, double *S) {
    if (bqo_gemv(qtype, Wq, M, K, x, y, S)) return -1;
    if (bias)
        for (int64_t m = 0; m < M; ++m) {
            y[m] += bias[m];
            if (S) S[m] += fabs(bias[m]);
        }
    return 0;
}

/* The unquantized fp16-weight GEMV ("We Wrote Our Own Inference Engine",
 * "What actually moved it" #4: a GEMV for the unquantized fp16 matrices;
 * RunIT README, kernel table, gemv_f16w_f32in_f32out: fp16 weights, fp32 in
 * and out), read as the plain definition: W is fp16 [M, K] row-major (bits),
 * y[m] = sum_k w[m,k] * x[k] in fp64, summed in index order; S[m] =
 * sum_k |w[m,k] * x[k]| (S may be NULL). */
int bqo_gemv_f16(const uint16_t *W, int64_t M, int64_t K, const double *x, double *y, double *S) {
    if (M < 0 || K < 0) return -1;
    for (int64_t m = 0; m < M; ++m) {
        double acc = 0.0, sacc = 0.0;
        for (int64_t k = 0; k < K; k++) {
            double p = bqo_f16_bits_to_f64(W[m * K + k]) * x[k];
            acc += p;
            sacc += fabs(p); /* sum of |w x| */
        }
        y[m] = acc;
        if (S) S[m] = sacc;
    }
    return 0;
}

/* xn[k] = x[k] * gamma[k] / sqrt(mean(x^2) + eps); gamma NULL means ones. */
int bqo_rmsnorm(const double *x, const double *gamma, int64_t K, double eps, double *xn) {
    if (K <= 0) return -1;
    double ss = 0.0;
    for (int64_t k = 0; k < K; ++k) ss += x[k] * x[k];
    double r = 1.0 / sqrt(ss / (double)K + eps);
    for (int64_t k = 0; k < K; ++k) xn[k] = x[k] * r * (gamma ? gamma[k] : 1.0);
    return 0;
}

double bqo_silu(double z) { return z / (1.0 + exp(-z)); }

/* g = Wg xn, u = Wu xn, y = silu(g) * u.  g, u, Sg, Su may be NULL. */
int bqo_gate_up_silu(int qtype, const uint8_t *Wg, const uint8_t *Wu, int64_t M, int64_t K,
                     const double *xn, double *y, double *g, double *u, double *Sg,
                     double *Su) {
    int64_t rb = bqo_packed_bytes(qtype, 1, K); /* bytes of one packed row */
    if (rb < 0 || M < 0) return -1;
    for (int64_t m = 0; m < M; ++m) {
        double gm, um, sg, su;
        bqo_gemv(qtype, Wg + m * rb, 1, K, xn, &gm, &sg);
        bqo_gemv(qtype, Wu + m * rb, 1, K, xn, &um, &su);
        y[m] = bqo_silu(gm) * um;
        if (g) g[m] = gm;
        if (u) u[m] = um;
        if (Sg) Sg[m] = sg;
        if (Su) Su[m] = su;
    }
    return 0;
}
