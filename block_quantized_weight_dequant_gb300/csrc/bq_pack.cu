// bq_pack.cu -- fp32 weights -> packed Q8_0 / Q4_0 blocks on the GPU.
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

}  // namespace

int bq_internal_pack(int qtype, const float *W, long long M, long long K, void *Wq, void *stream) {
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
