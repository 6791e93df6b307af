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
/* Block formats                                                            */
/* ------------------------------------------------------------------------ */

int64_t bqo_block_bytes(int qtype) {
    if (qtype == BQO_Q8_0) return 34;
    if (qtype == BQO_Q4_0) return 18;
    return -1;
}

int64_t bqo_packed_bytes(int qtype, int64_t M, int64_t K) {
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
    int64_t bb = bqo_block_bytes(qtype);
    if (bb < 0 || M < 0 || K < 0 || K % 32) return -1;
    int64_t rb = (K / 32) * bb;
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
