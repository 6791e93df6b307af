// bq_dot.cuh -- the fixed-order arithmetic of one row of a block-quantized
// GEMV: on-the-fly dequant of 8-block units and their dot products with x.
//
// Every GEMV kernel in this library (single-row, gate+up, multi-row verify,
// streaming or generic) reaches each output through these functions, so the
// rounding of a row depends only on (qtype, K).  That is what makes a verify
// row memcmp-equal to the single-row result ("We Wrote Our Own Inference
// Engine", "Correctness first": verify is checked against decode with memcmp,
// because kernels with different summation orders drift).
//
// The tree, for one row:
//   unit     = 8 consecutive blocks (256 weights; 272 B in Q8_0, 144 B in Q4_0)
//   block b  : a_i = sum over t = 0..7 of q[4t+i] * x[4t+i]  (fma chain, i = 0..3)
//              s_b = (a_0 + a_1) + (a_2 + a_3)
//   unit     : c = sum over b of d_b * s_b                    (fma chain, b = 0..7)
//   lane l   : p_l = c_l + c_{l+G} + c_{l+2G} + ...           (in order, G lanes)
//   row      : p folded pairwise by xor-butterfly over the G lanes
// All steps use explicit _rn intrinsics, so the compiler cannot contract or
// reassociate them differently in different kernels.  Every code is converted
// to fp32 exactly (q and n-8 are small integers), so dequantisation itself
// adds no rounding; the per-block scale multiplies the block's partial sum
// once, as w = d*q factors out of the block's dot product.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

namespace bq {

constexpr int QT_Q4_0 = 2;
constexpr int QT_Q8_0 = 8;
constexpr int QT_Q4_K = 12;

template <int QT> struct Fmt;
template <> struct Fmt<QT_Q8_0> {
    static constexpr int block_bytes = 34;
    static constexpr int unit_bytes = 272;  // 8 blocks = 17 x 16 B
    static constexpr int unit_words = 68;
};
template <> struct Fmt<QT_Q4_0> {
    static constexpr int block_bytes = 18;
    static constexpr int unit_bytes = 144;  // 8 blocks = 9 x 16 B
    static constexpr int unit_words = 36;
};
// Q4_K: the unit is one super-block of 256 weights (144 B = 9 x 16 B); its
// bytes per 32 weights (18) are given as block_bytes for size arithmetic only
template <> struct Fmt<QT_Q4_K> {
    static constexpr int block_bytes = 18;
    static constexpr int unit_bytes = 144;
    static constexpr int unit_words = 36;
};

// ---------------------------------------------------------------------------
// exact code -> fp32 conversion
// ---------------------------------------------------------------------------
// Q8_0: flip the sign bit of every byte (q + 128 as an unsigned byte) and
// place that byte in the low mantissa of 2^23: the float 2^23 + q + 128, from
// which subtracting 2^23 + 128 leaves q exactly.
constexpr float Q8_MAGIC = 8388736.0f;  // 2^23 + 128
__device__ __forceinline__ float q8_raw(uint32_t word, int pos) {
    const uint32_t flipped = word ^ 0x80808080u;
    return __uint_as_float(__byte_perm(flipped, 0x4B000000u, 0x7540u | (uint32_t)pos));
}
// Q4_0: the nibbles of a word are masked in place once (low nibbles, or high
// nibbles), and the byte at `pos` goes into the low mantissa byte of a magic
// float.  A low nibble n under 2^23 gives 2^23 + n; a high nibble stays in
// bits 4..7 (the byte holds 16n) under 2^19, whose mantissa step is 2^-4, so
// it gives 2^19 + 16n * 2^-4 = 2^19 + n without a shift.  Subtracting
// 2^23 + 8 or 2^19 + 8 leaves n - 8 exactly.
constexpr float Q4_MAGIC = 8388616.0f;     // 2^23 + 8
constexpr float Q4_MAGIC_HI = 524296.0f;   // 2^19 + 8
__device__ __forceinline__ float q4_raw(uint32_t word, bool high, int pos) {
    const uint32_t nib = word & (high ? 0xF0F0F0F0u : 0x0F0F0F0Fu);
    return __uint_as_float(
        __byte_perm(nib, high ? 0x49000000u : 0x4B000000u, 0x7540u | (uint32_t)pos));
}

__device__ __forceinline__ float scale_at(const uint32_t *w, int byte_off) {
    const uint32_t h = (w[byte_off >> 2] >> (8 * (byte_off & 3))) & 0xFFFFu;
    return __half2float(__ushort_as_half((unsigned short)h));
}

// ---------------------------------------------------------------------------
// x sources.  xs.at(e0) returns a view of the x elements from e0 on;
// view.get(r, B, t) is the float4 of elements e0 + 32B + 4t .. +3 of input
// row r.  Either e0 is a multiple of 256 (a unit), or only B = 0 is read.
// ---------------------------------------------------------------------------
// x staged in shared memory with its 16-byte chunks permuted within each
// 128-byte line: chunk c (elements 4c..4c+3) sits at chunk position
// (c & ~7) | ((c ^ c >> 3 ^ c >> 6) & 7).  With c = 64u + 8b + t (unit u,
// block b, step t) the bank group is t ^ b ^ u (mod 8), so eight lanes that
// read different units of one block position, or different blocks of one
// unit, all hit different banks.
__host__ __device__ constexpr int x_chunk_pos(int c) { return (c & ~7) | ((c ^ (c >> 3) ^ (c >> 6)) & 7); }
// float offset of element e (any e) in the permuted layout
__host__ __device__ constexpr int x_pos(int e) { return 4 * x_chunk_pos(e >> 2) + (e & 3); }
struct XSmem {
    const float *base;
    int rstride;  // floats between rows
    // Q4_K: the staged 32-element block sums of x (xblock_sum), block k of
    // row r at sums[r * sstride + k]; unused by the other formats
    const float *sums = nullptr;
    int sstride = 0;
    // Step t of block B of the view sits at p[t ^ B] + 32 B floats: with
    // c0 = e0 / 4 (a multiple of 8) the chunk of (B, t) is at position
    // c0 + 8B + (t ^ B ^ key), key = (c0 >> 3 ^ c0 >> 6) & 7, when e0 is a
    // multiple of 256 (then c0 >> 3 has zero low bits) or B = 0.  The eight
    // pointers are formed once per view, so each load is a register plus an
    // immediate offset.
    struct View {
        const float *p[8];
        int rstride;
        const float *s;
        int sstride;
        __device__ __forceinline__ float4 get(int r, int B, int t) const {
            return *reinterpret_cast<const float4 *>(p[(t ^ B) & 7] + r * rstride + 32 * B);
        }
        // the staged sum of block B of the view (Q4_K)
        __device__ __forceinline__ float bsum(int r, int B) const { return s[r * sstride + B]; }
    };
    __device__ __forceinline__ View at(int e0) const {
        const int c0 = e0 >> 2;
        const int k0 = 4 * (c0 ^ (((c0 >> 3) ^ (c0 >> 6)) & 7));
        View v;
#pragma unroll
        for (int j = 0; j < 8; ++j) v.p[j] = base + (k0 ^ (4 * j));
        v.rstride = rstride;
        v.s = sums + (e0 >> 5);
        v.sstride = sstride;
        return v;
    }
};
// floats of shared memory one staged x of K elements takes (K rounded up to 128 B)
__host__ __device__ constexpr int x_padded_floats(int K) { return (K + 31) / 32 * 32; }

// The sum of the 32 x elements of block B of a view, in a fixed order that
// every kernel shares: u_i = x[i] + x[4+i] + ... + x[28+i] in order (i = 0..3),
// then (u_0 + u_1) + (u_2 + u_3).  Q4_K subtracts dmin*m times this sum per
// sub-block; staged x computes it once per CTA, global x recomputes it inline,
// and both give the same bits.
template <class XV>
__device__ __forceinline__ float xblock_sum(const XV &xv, int r, int B) {
    float2 u01 = make_float2(-0.0f, -0.0f), u23 = make_float2(-0.0f, -0.0f);
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        const float4 v = xv.get(r, B, t);
        u01 = __fadd2_rn(u01, make_float2(v.x, v.y));
        u23 = __fadd2_rn(u23, make_float2(v.z, v.w));
    }
    return __fadd_rn(__fadd_rn(u01.x, u01.y), __fadd_rn(u23.x, u23.y));
}

// x read from global memory (through L1)
struct XGlobal {
    const float *x;
    int K;
    struct View {
        const float *p;
        int K;
        __device__ __forceinline__ float4 get(int r, int B, int t) const {
            return __ldg(reinterpret_cast<const float4 *>(p + (size_t)r * K + 32 * B + 4 * t));
        }
        __device__ __forceinline__ float bsum(int r, int B) const { return xblock_sum(*this, r, B); }
    };
    __device__ __forceinline__ View at(int e0) const { return View{x + e0, K}; }
};

// RMSNorm applied while reading: xn = (x * rs) * gamma, rs from rms_scale()
struct XGlobalNorm {
    const float *x;
    const float *gamma;
    float rs;
    struct View {
        const float *x, *gamma;
        float rs;
        __device__ __forceinline__ float4 get(int, int B, int t) const {
            const int e = 32 * B + 4 * t;
            const float4 v = __ldg(reinterpret_cast<const float4 *>(x + e));
            const float4 g = __ldg(reinterpret_cast<const float4 *>(gamma + e));
            return make_float4(__fmul_rn(__fmul_rn(v.x, rs), g.x), __fmul_rn(__fmul_rn(v.y, rs), g.y),
                               __fmul_rn(__fmul_rn(v.z, rs), g.z), __fmul_rn(__fmul_rn(v.w, rs), g.w));
        }
        __device__ __forceinline__ float bsum(int r, int B) const { return xblock_sum(*this, r, B); }
    };
    __device__ __forceinline__ View at(int e0) const { return View{x + e0, gamma + e0, rs}; }
};

__device__ __forceinline__ float f4(const float4 &v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// ---------------------------------------------------------------------------
// one block of NW weight sets against R input rows:
//   c[v][r] = fma(d_b(v), s_b(v, r), c[v][r])
// NW = 1 serves the single-row GEMV (R = 1) and verify (R > 1); NW = 2 serves
// gate+up (two matrices, one x).  Each (v, r) pair sees exactly the operation
// sequence of the NW = 1, R = 1 case, so results do not depend on NW or R.
// ---------------------------------------------------------------------------
// code j of the block whose first byte (its scale) is byte `base` of w
template <int QT>
__device__ __forceinline__ float raw_at_byte(const uint32_t *w, int base, int j) {
    if constexpr (QT == QT_Q8_0) {
        const int byte = base + 2 + j;
        return q8_raw(w[byte >> 2], byte & 3);
    } else {
        const int byte = base + 2 + (j & 15);
        return q4_raw(w[byte >> 2], j >= 16, byte & 3);
    }
}

// The block's scale d and code-x sums s[v][r] = (a_0 + a_1) + (a_2 + a_3),
// a_i the in-order FMA chain over t of q[4t+i] * x[4t+i].  With BQ_F32X2 the
// chains run in pairs (a_0, a_1) and (a_2, a_3) on packed fp32x2 FMAs: each
// half is an IEEE fp32 fma with round-to-nearest, so the bits are the same.
#ifndef BQ_F32X2
#define BQ_F32X2 1
#endif
template <int QT, int NW, int R, int B, int WB, class XV>
__device__ __forceinline__ void block_sum_at(const uint32_t *const (&w)[NW], const XV &xv_,
                                             float (&s)[NW][R], float (&d)[NW]) {
    constexpr float M = QT == QT_Q8_0 ? Q8_MAGIC : Q4_MAGIC;
#if BQ_F32X2
    // codes 4t..4t+3 are low nibbles for t < 4 and high nibbles for t >= 4
    // (Q4_0), so each pair takes one magic
    const float2 mneg = make_float2(-M, -M);
    const float2 mneg_hi = QT == QT_Q8_0 ? mneg : make_float2(-Q4_MAGIC_HI, -Q4_MAGIC_HI);
    float2 a[NW][R][2];
#pragma unroll
    for (int v = 0; v < NW; ++v)
#pragma unroll
        for (int r = 0; r < R; ++r) a[v][r][0] = a[v][r][1] = make_float2(-0.0f, -0.0f);
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        float4 xv[R];
#pragma unroll
        for (int r = 0; r < R; ++r) xv[r] = xv_.get(r, B, t);
#pragma unroll
        for (int v = 0; v < NW; ++v) {
            const float2 mt = t < 4 ? mneg : mneg_hi;
            const float2 q01 = __fadd2_rn(
                make_float2(raw_at_byte<QT>(w[v], WB, 4 * t), raw_at_byte<QT>(w[v], WB, 4 * t + 1)),
                mt);
            const float2 q23 = __fadd2_rn(
                make_float2(raw_at_byte<QT>(w[v], WB, 4 * t + 2), raw_at_byte<QT>(w[v], WB, 4 * t + 3)),
                mt);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                a[v][r][0] = __ffma2_rn(q01, make_float2(xv[r].x, xv[r].y), a[v][r][0]);
                a[v][r][1] = __ffma2_rn(q23, make_float2(xv[r].z, xv[r].w), a[v][r][1]);
            }
        }
    }
#pragma unroll
    for (int v = 0; v < NW; ++v) {
        d[v] = scale_at(w[v], WB);
#pragma unroll
        for (int r = 0; r < R; ++r)
            s[v][r] = __fadd_rn(__fadd_rn(a[v][r][0].x, a[v][r][0].y),
                                __fadd_rn(a[v][r][1].x, a[v][r][1].y));
    }
#else
    float a[NW][R][4];
#pragma unroll
    for (int v = 0; v < NW; ++v)
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int i = 0; i < 4; ++i) a[v][r][i] = -0.0f;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        float4 xv[R];
#pragma unroll
        for (int r = 0; r < R; ++r) xv[r] = xv_.get(r, B, t);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int v = 0; v < NW; ++v) {
                const float q = __fsub_rn(raw_at_byte<QT>(w[v], WB, 4 * t + i),
                                          QT == QT_Q4_0 && t >= 4 ? Q4_MAGIC_HI : M);
#pragma unroll
                for (int r = 0; r < R; ++r) a[v][r][i] = __fmaf_rn(q, f4(xv[r], i), a[v][r][i]);
            }
        }
    }
#pragma unroll
    for (int v = 0; v < NW; ++v) {
        d[v] = scale_at(w[v], WB);
#pragma unroll
        for (int r = 0; r < R; ++r)
            s[v][r] = __fadd_rn(__fadd_rn(a[v][r][0], a[v][r][1]), __fadd_rn(a[v][r][2], a[v][r][3]));
    }
#endif
}

// block B of a unit whose bytes w holds from the unit's start
template <int QT, int NW, int R, int B, class XV>
__device__ __forceinline__ void block_sum(const uint32_t *const (&w)[NW], const XV &xv,
                                          float (&s)[NW][R], float (&d)[NW]) {
    block_sum_at<QT, NW, R, B, Fmt<QT>::block_bytes * B>(w, xv, s, d);
}

template <int QT, int NW, int R, int B, class XV>
__device__ __forceinline__ void block_dot(const uint32_t *const (&w)[NW], const XV &xv,
                                          float (&c)[NW][R]) {
    float s[NW][R], d[NW];
    block_sum<QT, NW, R, B>(w, xv, s, d);
#pragma unroll
    for (int v = 0; v < NW; ++v)
#pragma unroll
        for (int r = 0; r < R; ++r) c[v][r] = __fmaf_rn(d[v], s[v][r], c[v][r]);
}

// ---------------------------------------------------------------------------
// Q4_K: the unit is one super-block (256 weights, 144 bytes): fp16 d, fp16
// dmin, 12 bytes of eight 6-bit sub-block scales sc_j and mins m_j, then 128
// bytes of nibbles, sub-blocks 2g (low nibbles) and 2g+1 (high nibbles)
// sharing bytes 32g..32g+31; w = d*sc_j*q - dmin*m_j (RunIT README kernel
// table, gemv_q4k_f16, read with the public GGUF Q4_K layout).  The tree of
// one unit, per weight set v and input row r:
//   sub-block j: s_j = (a_0 + a_1) + (a_2 + a_3), a_i the in-order FMA chain
//                over t = 0..7 of q[4t+i] * x[4t+i]   (q = 0..15, exact)
//   cq = in-order FMA chain over j of (d*sc_j) * s_j
//   cm = in-order FMA chain over j of (dmin*m_j) * xblock_sum_j
//   c  = cq - cm
// d*sc_j and dmin*m_j are exact in fp32 (an 11-bit by a 6-bit significand),
// so the dequantization itself adds no rounding; the x block sums are shared
// by every row.
// ---------------------------------------------------------------------------
constexpr float Q4K_MAGIC = 8388608.0f;  // 2^23: low nibble n -> 2^23 + n
constexpr float Q4K_MAGIC_HI = 524288.0f;  // 2^19: a high nibble 16n -> 2^19 + n

// sub-block scales d*sc_j and offsets dmin*m_j from a super-block's first 16 bytes
__device__ __forceinline__ void q4k_scales(uint4 h, float (&D)[8], float (&Mn)[8]) {
    const float d = __half2float(__ushort_as_half((unsigned short)(h.x & 0xFFFFu)));
    const float dm = __half2float(__ushort_as_half((unsigned short)(h.x >> 16)));
    const uint32_t sc_lo = h.y & 0x3F3F3F3Fu, mn_lo = h.z & 0x3F3F3F3Fu;
    const uint32_t sc_hi = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
    const uint32_t mn_hi = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        D[k] = __fmul_rn(d, __uint2float_rn((sc_lo >> (8 * k)) & 0xFFu));
        D[4 + k] = __fmul_rn(d, __uint2float_rn((sc_hi >> (8 * k)) & 0xFFu));
        Mn[k] = __fmul_rn(dm, __uint2float_rn((mn_lo >> (8 * k)) & 0xFFu));
        Mn[4 + k] = __fmul_rn(dm, __uint2float_rn((mn_hi >> (8 * k)) & 0xFFu));
    }
}

// the scale and offset of sub-block j alone (j may differ between lanes)
__device__ __forceinline__ void q4k_scale_of(uint4 h, int j, float &D, float &Mn) {
    const float d = __half2float(__ushort_as_half((unsigned short)(h.x & 0xFFFFu)));
    const float dm = __half2float(__ushort_as_half((unsigned short)(h.x >> 16)));
    const int k = 8 * (j & 3);
    const uint32_t y = h.y >> k, z = h.z >> k, w = h.w >> k;
    const uint32_t sc = j < 4 ? (y & 63u) : ((w & 15u) | (((y >> 6) & 3u) << 4));
    const uint32_t mn = j < 4 ? (z & 63u) : (((w >> 4) & 15u) | (((z >> 6) & 3u) << 4));
    D = __fmul_rn(d, __uint2float_rn(sc));
    Mn = __fmul_rn(dm, __uint2float_rn(mn));
}

// s[v][r] = sum over sub-block j's 32 elements of q * x, its codes in the
// nibbles (low: hi == 0, high: hi == 1) of the 8 words wq[v][0..7] of its
// byte pair group; x from block B of the view.  With the packed fp32x2 FMAs
// each half is an IEEE fp32 fma, so the bits equal the scalar chains'.
template <int NW, int R, class XV>
__device__ __forceinline__ void q4k_sub_sum(const uint32_t (&wq)[NW][8], int hi, const XV &xv, int B,
                                            float (&s)[NW][R]) {
    const uint32_t mask = hi ? 0xF0F0F0F0u : 0x0F0F0F0Fu;
    const uint32_t magic = hi ? 0x49000000u : 0x4B000000u;
    const float m = hi ? Q4K_MAGIC_HI : Q4K_MAGIC;
    const float2 mneg = make_float2(-m, -m);
    float2 a[NW][R][2];
#pragma unroll
    for (int v = 0; v < NW; ++v)
#pragma unroll
        for (int r = 0; r < R; ++r) a[v][r][0] = a[v][r][1] = make_float2(-0.0f, -0.0f);
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        float4 xv4[R];
#pragma unroll
        for (int r = 0; r < R; ++r) xv4[r] = xv.get(r, B, t);
#pragma unroll
        for (int v = 0; v < NW; ++v) {
            const uint32_t nib = wq[v][t] & mask;
            const float2 q01 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(nib, magic, 0x7540u)),
                                                      __uint_as_float(__byte_perm(nib, magic, 0x7541u))),
                                          mneg);
            const float2 q23 = __fadd2_rn(make_float2(__uint_as_float(__byte_perm(nib, magic, 0x7542u)),
                                                      __uint_as_float(__byte_perm(nib, magic, 0x7543u))),
                                          mneg);
#pragma unroll
            for (int r = 0; r < R; ++r) {
                a[v][r][0] = __ffma2_rn(q01, make_float2(xv4[r].x, xv4[r].y), a[v][r][0]);
                a[v][r][1] = __ffma2_rn(q23, make_float2(xv4[r].z, xv4[r].w), a[v][r][1]);
            }
        }
    }
#pragma unroll
    for (int v = 0; v < NW; ++v)
#pragma unroll
        for (int r = 0; r < R; ++r)
            s[v][r] = __fadd_rn(__fadd_rn(a[v][r][0].x, a[v][r][0].y),
                                __fadd_rn(a[v][r][1].x, a[v][r][1].y));
}

// One super-block of NW weight sets against R input rows of the view at e0:
// header(v) returns weight set v's first 16 bytes, pair(v, g, wq) fills the 8
// words of its byte pair group g.
template <int NW, int R, class XV, class Header, class Pair>
__device__ __forceinline__ void q4k_unit(const XV &xv, Header header, Pair pair, float (&c)[NW][R]) {
    float D[NW][8], Mn[NW][8], cq[NW][R], cm[NW][R];
#pragma unroll
    for (int v = 0; v < NW; ++v) {
        q4k_scales(header(v), D[v], Mn[v]);
#pragma unroll
        for (int r = 0; r < R; ++r) cq[v][r] = cm[v][r] = -0.0f;
    }
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        uint32_t wq[NW][8];
#pragma unroll
        for (int v = 0; v < NW; ++v) pair(v, g, wq[v]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float sj[NW][R];
            q4k_sub_sum<NW, R>(wq, h, xv, 2 * g + h, sj);
#pragma unroll
            for (int v = 0; v < NW; ++v)
#pragma unroll
                for (int r = 0; r < R; ++r) cq[v][r] = __fmaf_rn(D[v][2 * g + h], sj[v][r], cq[v][r]);
        }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float sx = xv.bsum(r, j);
#pragma unroll
            for (int v = 0; v < NW; ++v) cm[v][r] = __fmaf_rn(Mn[v][j], sx, cm[v][r]);
        }
#pragma unroll
    for (int v = 0; v < NW; ++v)
#pragma unroll
        for (int r = 0; r < R; ++r) c[v][r] = __fsub_rn(cq[v][r], cm[v][r]);
}

// the unit from words in registers (w[v][0..35], the unit's bytes little-endian)
template <int NW, int R, class XS>
__device__ __forceinline__ void q4k_unit_words(const uint32_t *const (&w)[NW], const XS &xs, int e0,
                                               float (&c)[NW][R]) {
    q4k_unit<NW, R>(
        xs.at(e0), [&](int v) { return make_uint4(w[v][0], w[v][1], w[v][2], w[v][3]); },
        [&](int v, int g, uint32_t (&wq)[8]) {
#pragma unroll
            for (int t = 0; t < 8; ++t) wq[t] = w[v][4 + 8 * g + t];
        },
        c);
}

// the unit from shared memory (up[v]: the unit's first byte, 16-byte aligned)
template <int NR, int R, class XS>
__device__ __forceinline__ void q4k_unit_rows(const uint8_t *const (&up)[NR], const XS &xs, int e0,
                                              float (&c)[NR][R]) {
    q4k_unit<NR, R>(
        xs.at(e0), [&](int v) { return *reinterpret_cast<const uint4 *>(up[v]); },
        [&](int v, int g, uint32_t (&wq)[8]) {
            const uint4 a = *reinterpret_cast<const uint4 *>(up[v] + 16 + 32 * g);
            const uint4 b = *reinterpret_cast<const uint4 *>(up[v] + 32 + 32 * g);
            wq[0] = a.x, wq[1] = a.y, wq[2] = a.z, wq[3] = a.w;
            wq[4] = b.x, wq[5] = b.y, wq[6] = b.z, wq[7] = b.w;
        },
        c);
}

// One unit (nbk <= 8 blocks; w[v] holds the unit's bytes little-endian from
// its start) against x elements from e0.  c[v][r] receives the unit partials.
template <int QT, int NW, int R, class XS>
__device__ __forceinline__ void unit_dot(const uint32_t *const (&w)[NW], int nbk, const XS &xs,
                                         int e0, float (&c)[NW][R]) {
    if constexpr (QT == QT_Q4_K) {
        q4k_unit_words<NW, R>(w, xs, e0, c);  // a super-block is always whole
        return;
    }
#pragma unroll
    for (int v = 0; v < NW; ++v)
#pragma unroll
        for (int r = 0; r < R; ++r) c[v][r] = -0.0f;
    const auto xv = xs.at(e0);
    block_dot<QT, NW, R, 0>(w, xv, c);
    if (nbk > 1) block_dot<QT, NW, R, 1>(w, xv, c);
    if (nbk > 2) block_dot<QT, NW, R, 2>(w, xv, c);
    if (nbk > 3) block_dot<QT, NW, R, 3>(w, xv, c);
    if (nbk > 4) block_dot<QT, NW, R, 4>(w, xv, c);
    if (nbk > 5) block_dot<QT, NW, R, 5>(w, xv, c);
    if (nbk > 6) block_dot<QT, NW, R, 6>(w, xv, c);
    if (nbk > 7) block_dot<QT, NW, R, 7>(w, xv, c);
}

// NR weight rows against R input rows of one x view, one full unit each:
// c[v][r] receives the unit partial of weight row v against input row r with
// exactly unit_dot's operation sequence, so the bits depend on neither NR nor
// R.  up[v] is the unit's first byte in shared memory (16-byte aligned).
// Weights are read block by block: the bytes of block b lie in the 16-byte
// chunks floor(34b/16) .. +2 for Q8_0 (always three chunks) and
// floor(18b/16) .. +1 for Q4_0 (always two), so a row holds one block's words
// in registers while every x value read from shared memory serves NR rows.
// (A chunk shared by two blocks is loaded once: the compiler reuses the load.)
template <int QT, int NR, int R, int B, class XV>
__device__ __forceinline__ void rows_block(const uint8_t *const (&up)[NR], const XV &xv,
                                           float (&c)[NR][R]) {
    constexpr int bb = Fmt<QT>::block_bytes;
    constexpr int off = bb * B;
    constexpr int c0 = off / 16;
    constexpr int nch = (off + bb - 1) / 16 - c0 + 1;
    uint32_t w[NR][4 * nch];
#pragma unroll
    for (int v = 0; v < NR; ++v)
#pragma unroll
        for (int k = 0; k < nch; ++k) {
            const uint4 q = *reinterpret_cast<const uint4 *>(up[v] + 16 * (c0 + k));
            w[v][4 * k + 0] = q.x;
            w[v][4 * k + 1] = q.y;
            w[v][4 * k + 2] = q.z;
            w[v][4 * k + 3] = q.w;
        }
    const uint32_t *ws[NR];
#pragma unroll
    for (int v = 0; v < NR; ++v) ws[v] = w[v];
    float s[NR][R], d[NR];
    block_sum_at<QT, NR, R, B, off - 16 * c0>(ws, xv, s, d);
#pragma unroll
    for (int v = 0; v < NR; ++v)
#pragma unroll
        for (int r = 0; r < R; ++r) c[v][r] = __fmaf_rn(d[v], s[v][r], c[v][r]);
}

template <int QT, int NR, int R, class XS>
__device__ __forceinline__ void unit_dot_rows(const uint8_t *const (&up)[NR], const XS &xs, int e0,
                                              float (&c)[NR][R]) {
    if constexpr (QT == QT_Q4_K) {
        q4k_unit_rows<NR, R>(up, xs, e0, c);
        return;
    }
#pragma unroll
    for (int v = 0; v < NR; ++v)
#pragma unroll
        for (int r = 0; r < R; ++r) c[v][r] = -0.0f;
    const auto xv = xs.at(e0);
    rows_block<QT, NR, R, 0>(up, xv, c);
    rows_block<QT, NR, R, 1>(up, xv, c);
    rows_block<QT, NR, R, 2>(up, xv, c);
    rows_block<QT, NR, R, 3>(up, xv, c);
    rows_block<QT, NR, R, 4>(up, xv, c);
    rows_block<QT, NR, R, 5>(up, xv, c);
    rows_block<QT, NR, R, 6>(up, xv, c);
    rows_block<QT, NR, R, 7>(up, xv, c);
}

// load a full unit from shared memory (16-byte aligned)
template <int QT>
__device__ __forceinline__ void load_unit_smem(uint32_t *w, const uint8_t *p) {
    constexpr int n16 = Fmt<QT>::unit_bytes / 16;
#pragma unroll
    for (int i = 0; i < n16; ++i) {
        const uint4 v = *reinterpret_cast<const uint4 *>(p + 16 * i);
        w[4 * i + 0] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
}

// load nbk blocks of a unit from global memory (2-byte aligned); bytes past
// the unit's blocks are zero
template <int QT>
__device__ __forceinline__ void load_unit_global(uint32_t *w, const uint8_t *p, int nbk) {
    constexpr int nw = Fmt<QT>::unit_words;
    const int nhalf = nbk * Fmt<QT>::block_bytes / 2;
    const unsigned short *h = reinterpret_cast<const unsigned short *>(p);
#pragma unroll
    for (int i = 0; i < nw; ++i) {
        const uint32_t lo = (2 * i < nhalf) ? (uint32_t)__ldg(h + 2 * i) : 0u;
        const uint32_t hi = (2 * i + 1 < nhalf) ? (uint32_t)__ldg(h + 2 * i + 1) : 0u;
        w[i] = lo | (hi << 16);
    }
}

// fold lane partials of a G-lane group (G a power of two <= 32)
__device__ __forceinline__ float fold_lanes(float v, int G) {
    for (int o = G >> 1; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
// One block (34 or 18 bytes) at a 2-byte-aligned shared-memory address,
// realigned into words so that the block's scale starts at byte 0.  Reads up
// to 4 bytes past the block; shared-memory rings keep that slack at their end.
template <int QT>
__device__ __forceinline__ void load_block_realigned(uint32_t *w, const uint8_t *p) {
    constexpr int nw = (Fmt<QT>::block_bytes + 3) / 4;
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t *q = reinterpret_cast<const uint32_t *>(a & ~(uintptr_t)3);
    const uint32_t sh = (uint32_t)(a & 3) * 8;  // 0 or 16
    uint32_t lo = q[0];
#pragma unroll
    for (int i = 0; i < nw; ++i) {
        const uint32_t hi = q[i + 1];
        w[i] = __funnelshift_r(lo, hi, sh);
        lo = hi;
    }
}

// One row of nsc full units at `rowp` (shared memory), evaluated by a whole
// warp block-parallel: in each round, lane 8j+b takes block b of unit 4r+j,
// the 8 block sums of a unit are chained in block order (c = d_b * s_b + c)
// with shuffles, and each unit's c is added to virtual lane u mod G in unit
// order.  That is exactly the tree of unit_dot + the G-lane partial sums, so
// the result (returned in lane 0 after fold_lanes) is bit-identical to the
// unit-per-lane evaluation; the latency is that of nsc/4 blocks instead of
// nsc/G units.
// Q4_K rows block-parallel: lane 8j+b takes sub-block b of unit 4r+j (its
// scale and offset, its 32 nibbles and its x block sum); the unit's two chains
// cq and cm run over the 8 lanes in sub-block order with shuffles and
// c = cq - cm, exactly q4k_unit's tree.
template <class XS>
__device__ __forceinline__ float row_dot_blockpar_q4k(const uint8_t *rowp, int nsc, int G,
                                                      const XS &xs, int lane) {
    const int j = lane >> 3, b = lane & 7;
    float p = -0.0f;
    for (int r4 = 0; r4 < nsc; r4 += 4) {
        const int u = r4 + j;
        float s[1][1] = {{0.0f}}, D = 0.0f, Mn = 0.0f, sx = 0.0f;
        if (u < nsc) {
            const uint8_t *sb = rowp + u * Fmt<QT_Q4_K>::unit_bytes;
            q4k_scale_of(*reinterpret_cast<const uint4 *>(sb), b, D, Mn);
            const uint4 a = *reinterpret_cast<const uint4 *>(sb + 16 + 32 * (b >> 1));
            const uint4 c = *reinterpret_cast<const uint4 *>(sb + 32 + 32 * (b >> 1));
            const uint32_t wq[1][8] = {{a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w}};
            const auto xv = xs.at(256 * u + 32 * b);
            q4k_sub_sum<1, 1>(wq, b & 1, xv, 0, s);
            sx = xv.bsum(0, 0);
        }
        float cq = -0.0f, cm = -0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int src = (j << 3) + k;
            cq = __fmaf_rn(__shfl_sync(0xffffffffu, D, src), __shfl_sync(0xffffffffu, s[0][0], src), cq);
            cm = __fmaf_rn(__shfl_sync(0xffffffffu, Mn, src), __shfl_sync(0xffffffffu, sx, src), cm);
        }
        const float c = __fsub_rn(cq, cm);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const float cj = __shfl_sync(0xffffffffu, c, jj << 3);
            const int uu = r4 + jj;
            if (uu < nsc && lane < G && (uu & (G - 1)) == lane) p = __fadd_rn(p, cj);
        }
    }
    return fold_lanes(p, G);
}

template <int QT, class XS>
__device__ __forceinline__ float row_dot_blockpar(const uint8_t *rowp, int nsc, int G,
                                                  const XS &xs, int lane) {
    if constexpr (QT == QT_Q4_K) return row_dot_blockpar_q4k(rowp, nsc, G, xs, lane);
    constexpr int UB = Fmt<QT>::unit_bytes, BB = Fmt<QT>::block_bytes;
    const int j = lane >> 3, b = lane & 7;
    float p = -0.0f;
    for (int r4 = 0; r4 < nsc; r4 += 4) {
        const int u = r4 + j;
        float s[1][1] = {{0.0f}}, d[1] = {0.0f};
        if (u < nsc) {
            uint32_t w[(BB + 3) / 4];
            load_block_realigned<QT>(w, rowp + u * UB + b * BB);
            const uint32_t *const ws[1] = {w};
            block_sum<QT, 1, 1, 0>(ws, xs.at(256 * u + 32 * b), s, d);
        }
        float c = -0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float dk = __shfl_sync(0xffffffffu, d[0], (j << 3) + k);
            const float sk = __shfl_sync(0xffffffffu, s[0][0], (j << 3) + k);
            c = __fmaf_rn(dk, sk, c);
        }
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            const float cj = __shfl_sync(0xffffffffu, c, jj << 3);
            const int uu = r4 + jj;
            if (uu < nsc && lane < G && (uu & (G - 1)) == lane) p = __fadd_rn(p, cj);
        }
    }
    return fold_lanes(p, G);
}


// silu(g) * u in fp32
__device__ __forceinline__ float silu_mul(float g, float u) {
    const float s = __fdiv_rn(g, __fadd_rn(1.0f, expf(-g)));
    return __fmul_rn(s, u);
}

// RMSNorm scale 1/sqrt(mean(x^2) + eps) with a summation order that does not
// depend on the number of threads: 256 virtual lanes v each sum x[v],
// x[v+256], ... in order; the 256 lane sums are folded by a fixed tree.
// Called by `nthr` threads (thread index tid) sharing `red` (>= 257 floats);
// `sync` is a barrier over exactly those threads; `xat(k)` returns x[k].
template <class XAt, class Sync>
__device__ float rms_scale_at(XAt xat, int K, float eps, float *red, int tid, int nthr, Sync sync) {
    for (int v = tid; v < 256; v += nthr) {
        float s = 0.0f;
        for (int k = v; k < K; k += 256) {
            const float t = xat(k);
            s = __fmaf_rn(t, t, s);
        }
        red[v] = s;
    }
    sync();
    if (tid < 32) {
        const float *q = red + 8 * tid;
        float v = __fadd_rn(__fadd_rn(__fadd_rn(q[0], q[1]), __fadd_rn(q[2], q[3])),
                            __fadd_rn(__fadd_rn(q[4], q[5]), __fadd_rn(q[6], q[7])));
        for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (tid == 0) red[256] = v;
    }
    sync();
    const float ms = __fdiv_rn(red[256], (float)K);
    return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, eps)));
}

template <class Sync>
__device__ float rms_scale(const float *x, int K, float eps, float *red, int tid, int nthr,
                           Sync sync) {
    return rms_scale_at([x](int k) { return x[k]; }, K, eps, red, tid, nthr, sync);
}

}  // namespace bq
