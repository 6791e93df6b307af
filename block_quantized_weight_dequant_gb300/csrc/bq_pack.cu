// bq_pack.cu -- fp32 weights -> packed Q8_0 / Q4_0 blocks and Q4_K
// super-blocks on the GPU.
//
// One warp per 32-weight block: lane j owns weight j.  The scale and codes
// follow the block definitions exactly, with IEEE fp32 operations only:
//   Q8_0: d = fp16_rne(max|w| / 127); q = clamp(round(w / d), -127, 127)
//   Q4_0: d = fp16_rne(max|w| / 8);   n = clamp(round(w / d) + 8, 0, 15)
// (round = half away from zero; the division is by the stored fp16 scale;
// d == 0 gives q = 0 / n = 8).  The byte layout is the GGUF-style block the
// RunIT README's quantization table prices at 1.06 / 0.56 B per weight.  This
// is load-time work, the counterpart of the pages' converters ("We Wrote Our
// Own Inference Engine", "The recipe rule").
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "bq_internal.h"

namespace {

template <int QT>
__global__ void __launch_bounds__(256) pack_kernel(const float *__restrict__ W, long long M,
                                                   long long K, uint8_t *__restrict__ out) {
    constexpr int BB = QT == 8 ? 34 : 18;
    const long long nb = K / 32;
    const long long total = M * nb;
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long blk = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
         blk < total; blk += warps) {
        const long long m = blk / nb, b = blk % nb;
        const float w = W[m * K + 32 * b + lane];
        float amax = fabsf(w);
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const float d32 = __fdiv_rn(amax, QT == 8 ? 127.0f : 8.0f);
        const __half dh = __float2half_rn(d32);
        const float df = __half2float(dh);
        uint8_t *dst = out + blk * BB;
        if (lane == 0) {
            const unsigned short bits = __half_as_ushort(dh);
            dst[0] = (uint8_t)(bits & 0xFFu);
            dst[1] = (uint8_t)(bits >> 8);
        }
        if (QT == 8) {
            int q = 0;
            if (df != 0.0f) q = (int)fminf(fmaxf(roundf(__fdiv_rn(w, df)), -127.0f), 127.0f);
            dst[2 + lane] = (uint8_t)(int8_t)q;
        } else {
            float r = 8.0f;
            if (df != 0.0f) r = __fadd_rn(roundf(__fdiv_rn(w, df)), 8.0f);
            const int n = (int)fminf(fmaxf(r, 0.0f), 15.0f);
            const int hi = __shfl_down_sync(0xffffffffu, n, 16);
            if (lane < 16) dst[2 + lane] = (uint8_t)(n | (hi << 4));
        }
    }
}

// Q4_K: one warp per super-block of 256 weights, lane L holding element L of
// each of the 8 sub-blocks.  The reading of the GGUF Q4_K packer (the pages
// name Q4_K_M without defining it), fp32 IEEE operations only:
//   sub-block j: lo = min(0, min w), hi = max w, scale_j = (hi - lo) / 15,
//                min_j = -lo
//   d = fp16_rne(max_j scale_j / 63), dmin = fp16_rne(max_j min_j / 63), both
//       +0 when every term is zero
//   sc_j = clamp(round(scale_j / d), 0, 63), m_j = clamp(round(min_j / dmin), 0, 63)
//       (0 when the divisor is 0)
//   q = clamp(round((w + dmin*m_j) / (d*sc_j)), 0, 15)  (0 when d*sc_j is 0)
// round = half away from zero.  The sign of a zero lo, hi or scale never
// reaches the bytes: the super-block maxima keep +0 unless a term is positive.
__global__ void __launch_bounds__(256) pack_q4k_kernel(const float *__restrict__ W, long long M,
                                                       long long K, uint8_t *__restrict__ out) {
    const long long ns = K / 256;
    const long long total = M * ns;
    const int lane = threadIdx.x & 31;
    const long long warps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long sbi = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); sbi < total;
         sbi += warps) {
        const long long m = sbi / ns, b = sbi % ns;
        const float *src = W + m * K + 256 * b;
        float w[8], scale[8], mins[8];
        float smax = 0.0f, mmax = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            w[j] = src[32 * j + lane];
            float lo = w[j], hi = w[j];
            for (int o = 16; o > 0; o >>= 1) {
                lo = fminf(lo, __shfl_xor_sync(0xffffffffu, lo, o));
                hi = fmaxf(hi, __shfl_xor_sync(0xffffffffu, hi, o));
            }
            lo = fminf(lo, 0.0f);
            scale[j] = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
            mins[j] = -lo;
            if (scale[j] > smax) smax = scale[j];
            if (mins[j] > mmax) mmax = mins[j];
        }
        const __half dh = __float2half_rn(__fdiv_rn(smax, 63.0f));
        const __half mh = __float2half_rn(__fdiv_rn(mmax, 63.0f));
        const float d = __half2float(dh), dmin = __half2float(mh);
        int sc[8], mn[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            sc[j] = d != 0.0f ? (int)fminf(fmaxf(roundf(__fdiv_rn(scale[j], d)), 0.0f), 63.0f) : 0;
            mn[j] = dmin != 0.0f ? (int)fminf(fmaxf(roundf(__fdiv_rn(mins[j], dmin)), 0.0f), 63.0f) : 0;
        }
        uint8_t *dst = out + sbi * 144;
        if (lane < 16) {
            // lane k writes header byte k
            uint32_t v;
            if (lane < 4) {
                const unsigned short bits = __half_as_ushort(lane < 2 ? dh : mh);
                v = (lane & 1) ? bits >> 8 : bits & 0xFFu;
            } else if (lane < 8) {
                const int j = lane - 4;
                v = (uint32_t)(sc[j] | ((sc[j + 4] >> 4) << 6));
            } else if (lane < 12) {
                const int j = lane - 8;
                v = (uint32_t)(mn[j] | ((mn[j + 4] >> 4) << 6));
            } else {
                const int j = lane - 12;
                v = (uint32_t)((sc[j + 4] & 15) | ((mn[j + 4] & 15) << 4));
            }
            dst[lane] = (uint8_t)v;
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            int q[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int j = 2 * g + h;
                const float D = __fmul_rn(d, (float)sc[j]), Mf = __fmul_rn(dmin, (float)mn[j]);
                q[h] = D != 0.0f
                           ? (int)fminf(fmaxf(roundf(__fdiv_rn(__fadd_rn(w[j], Mf), D)), 0.0f), 15.0f)
                           : 0;
            }
            dst[16 + 32 * g + lane] = (uint8_t)(q[0] | (q[1] << 4));
        }
    }
}

}  // namespace

int bq_internal_pack(int qtype, const float *W, long long M, long long K, void *Wq, void *stream) {
    if (qtype == 12) {
        const long long sbs = M * (K / 256);
        if (sbs == 0) return 0;
        int dev = 0, sms = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return (int)e;
        long long grid = (sbs + 7) / 8;
        if (grid > (long long)sms * 16) grid = (long long)sms * 16;
        pack_q4k_kernel<<<(unsigned)grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
            W, M, K, static_cast<uint8_t *>(Wq));
        return (int)cudaGetLastError();
    }
    const long long blocks = M * (K / 32);
    if (blocks == 0) return 0;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return (int)e;
    long long grid = (blocks + 7) / 8;  // 8 warps per CTA, one block per warp
    if (grid > (long long)sms * 16) grid = (long long)sms * 16;
    auto s = static_cast<cudaStream_t>(stream);
    if (qtype == 8)
        pack_kernel<8><<<(unsigned)grid, 256, 0, s>>>(W, M, K, static_cast<uint8_t *>(Wq));
    else
        pack_kernel<2><<<(unsigned)grid, 256, 0, s>>>(W, M, K, static_cast<uint8_t *>(Wq));
    return (int)cudaGetLastError();
}
