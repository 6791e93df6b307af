// bq_f16.cu -- the unquantized fp16-weight GEMV y = W x: W fp16 [M, K]
// row-major, x and y fp32 ("We Wrote Our Own Inference Engine", "What
// actually moved it" #4: a GEMV for the unquantized fp16 matrices; RunIT
// README, kernel table, gemv_f16w_f32in_f32out, vectorized half4 loads).
//
// The weights are read straight from HBM with 16-byte loads, each warp's
// loads covering 512 contiguous bytes of one row, so no shared-memory staging
// is needed: one warp evaluates one row at a time (rows grid-strided over the
// warps), and x comes through L1 (every warp reads all of it).  The 16-byte
// chunking that serves the block formats' shared-memory slots does not fit
// fp16 (a 256-weight unit is 32 chunks, 0 mod 8, so lanes reading different
// units of a row would share one bank group).
//
// The fixed summation tree of a row, a function of K alone:
//   segment s = elements 256 s .. 256 s + 255; lane l takes elements
//     256 s + 8 l + i, i = 0..7 (one 16-byte load);
//   chains c_i (i = 0..7): c_i = fma(w, x, c_i) over the segments of a group
//     of 16, in segment order, from -0;
//   group sum g = ((c_0 + c_1) + (c_2 + c_3)) + ((c_4 + c_5) + (c_6 + c_7));
//   lane sum p_l = g_0 + g_1 + ... in group order;
//   row = xor-butterfly fold of the 32 lane sums (offsets 16, 8, 4, 2, 1).
// Every step is an explicit _rn operation.  The longest rounding chain at the
// largest K (2^18: 64 groups) is 16 + 3 + 63 + 5 roundings, about 5e-6 of
// sum |w x|, inside the 1e-5 bound.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "bq_internal.h"

namespace bq {
namespace {

constexpr int F16_WARPS = 8;   // warps per CTA
constexpr int F16_SEG = 256;   // elements per warp step (32 lanes x 8)
constexpr int F16_GROUP = 16;  // segments per group: the per-lane chains restart every group

__device__ __forceinline__ float2 half2_at(uint32_t word) {
    __half2 h;
    *reinterpret_cast<uint32_t *>(&h) = word;
    return __half22float2(h);
}

__global__ void __launch_bounds__(F16_WARPS * 32)
    f16_gemv_kernel(const __half *__restrict__ W, const float *__restrict__ x, float *__restrict__ y,
                    int M, int K) {
    const int lane = threadIdx.x & 31;
    const int nseg = (K + F16_SEG - 1) / F16_SEG;
    const int stride = gridDim.x * F16_WARPS;
    for (int row = blockIdx.x * F16_WARPS + (threadIdx.x >> 5); row < M; row += stride) {
        const __half *wr = W + (size_t)row * K;
        float p = -0.0f;
        for (int g0 = 0; g0 < nseg; g0 += F16_GROUP) {
            const int g1 = min(nseg, g0 + F16_GROUP);
            float2 c0 = make_float2(-0.0f, -0.0f), c1 = c0, c2 = c0, c3 = c0;
            // one segment's arithmetic (K % 8 == 0: a lane's 8 elements are
            // all in the row or all past it)
            auto segment = [&](const uint4 &wv, int e) {
                if (e >= K) return;
                const float4 xa = __ldg(reinterpret_cast<const float4 *>(x + e));
                const float4 xb = __ldg(reinterpret_cast<const float4 *>(x + e + 4));
                c0 = __ffma2_rn(half2_at(wv.x), make_float2(xa.x, xa.y), c0);
                c1 = __ffma2_rn(half2_at(wv.y), make_float2(xa.z, xa.w), c1);
                c2 = __ffma2_rn(half2_at(wv.z), make_float2(xb.x, xb.y), c2);
                c3 = __ffma2_rn(half2_at(wv.w), make_float2(xb.z, xb.w), c3);
            };
            // four segments' weight loads in flight per lane before their
            // arithmetic, which then runs in segment order
            int s = g0;
            for (; s + 4 <= g1; s += 4) {
                uint4 wv[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int e = (s + u) * F16_SEG + 8 * lane;
                    wv[u] = e < K ? __ldg(reinterpret_cast<const uint4 *>(wr + e)) : make_uint4(0, 0, 0, 0);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) segment(wv[u], (s + u) * F16_SEG + 8 * lane);
            }
            for (; s < g1; ++s) {
                const int e = s * F16_SEG + 8 * lane;
                const uint4 wv = e < K ? __ldg(reinterpret_cast<const uint4 *>(wr + e)) : make_uint4(0, 0, 0, 0);
                segment(wv, e);
            }
            const float g = __fadd_rn(__fadd_rn(__fadd_rn(c0.x, c0.y), __fadd_rn(c1.x, c1.y)),
                                      __fadd_rn(__fadd_rn(c2.x, c2.y), __fadd_rn(c3.x, c3.y)));
            p = g0 == 0 ? g : __fadd_rn(p, g);
        }
        for (int o = 16; o > 0; o >>= 1) p = __fadd_rn(p, __shfl_xor_sync(0xffffffffu, p, o));
        if (lane == 0) y[row] = p;
    }
}

}  // namespace
}  // namespace bq

// One fp16-weight GEMV on `stream` (arguments validated by the caller): a
// grid of at most one wave of resident CTAs, rows grid-strided over the warps.
int bq_internal_f16_launch(const void *W, const float *x, float *y, long long M, long long K,
                           void *stream) {
    int dev = 0, nsm = 0, occ = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, bq::f16_gemv_kernel,
                                                          bq::F16_WARPS * 32, 0);
    if (e != cudaSuccess) return (int)e;
    const long long want = (M + bq::F16_WARPS - 1) / bq::F16_WARPS;
    const long long cap = (long long)nsm * (occ > 0 ? occ : 1);
    const int grid = (int)(want < cap ? want : cap);
    bq::f16_gemv_kernel<<<grid, bq::F16_WARPS * 32, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const __half *>(W), x, y, (int)M, (int)K);
    return (int)cudaGetLastError();
}
