// bq_f16.cu -- the unquantized fp16-weight GEMV y = W x: W fp16 [M, K]
// row-major, x fp32, y fp32 or fp16 ("We Wrote Our Own Inference Engine",
// "What actually moved it" #4: a split-K GEMV for the unquantized fp16
// matrices, and #5: fp16-output GEMVs; RunIT README, kernel table,
// gemv_f16w_f32in_f32out, vectorized half4 loads).
//
// The weights are read straight from HBM with 16-byte loads, each warp's
// loads covering 512 contiguous bytes of one row, so no shared-memory staging
// is needed, and x comes through L1 (every warp reads all of it).  The
// 16-byte chunking that serves the block formats' shared-memory slots does not
// fit fp16 (a 256-weight unit is 32 chunks, 0 mod 8, so lanes reading
// different units of a row would share one bank group).
//
// The fixed summation tree of a row, a function of K alone:
//   segment s = elements 256 s .. 256 s + 255; lane l takes elements
//     256 s + 8 l + i, i = 0..7 (one 16-byte load);
//   group j = segments 16 j .. 16 j + 15;
//   chains c_i (i = 0..7): c_i = fma(w, x, c_i) over the segments of a group,
//     in segment order, from -0;
//   lane group sum g_j = ((c_0 + c_1) + (c_2 + c_3)) + ((c_4 + c_5) + (c_6 + c_7));
//   lane sum p_l = g_0 + g_1 + ... in group order;
//   row = xor-butterfly fold of the 32 lane sums (offsets 16, 8, 4, 2, 1);
//   fp16 output: the fp32 row value rounded to nearest, ties to even.
// Every step is an explicit _rn operation.  The longest rounding chain at the
// largest K (2^18: 64 groups) is 16 + 3 + 63 + 5 roundings, about 5e-6 of
// sum |w x|, inside the 1e-5 bound.
//
// Two kernels evaluate that tree.  With many rows, one warp takes a whole row
// (rows grid-strided over the warps).  With few rows and two or more groups,
// the K dimension is split: one CTA per row, its warps taking the row's groups
// and leaving their lane group sums in shared memory, which one warp then adds
// in group order and folds.  Only the assignment of groups to warps differs,
// so both give the same bits.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "bq_internal.h"

namespace bq {
namespace {

constexpr int F16_WARPS = 8;        // warps per CTA, warp-per-row kernel
constexpr int F16_SEG = 256;        // elements per warp step (32 lanes x 8)
constexpr int F16_GROUP = 16;       // segments per group: the per-lane chains restart every group
constexpr long long F16_K_MAX = 1LL << 18;
constexpr long long F16_M_MAX = (1LL << 31) - 1;
constexpr int F16_MAX_GROUPS = (int)(F16_K_MAX / (F16_SEG * F16_GROUP));  // 64
constexpr int F16_SPLIT_WARPS = 8;  // most warps per CTA, split-K kernel
// split K when there are fewer rows than this many per SM: the warp-per-row
// kernel would then keep too few loads in flight to cover HBM latency
constexpr int F16_SPLIT_ROWS_PER_SM = 16;
constexpr long long F16_ROW_CHUNK = 1LL << 30;  // most rows per warp-per-row launch

__device__ __forceinline__ float2 half2_at(uint32_t word) {
    __half2 h;
    *reinterpret_cast<uint32_t *>(&h) = word;
    return __half22float2(h);
}

// Lane `lane`'s group sum over segments s0 .. s1 - 1 of row wr (one group:
// s1 - s0 <= 16).
__device__ __forceinline__ float lane_group_sum(const __half *__restrict__ wr,
                                                const float *__restrict__ x, int s0, int s1,
                                                int lane, int K) {
    float2 c0 = make_float2(-0.0f, -0.0f), c1 = c0, c2 = c0, c3 = c0;
    // one segment's arithmetic (K % 8 == 0: a lane's 8 elements are all in
    // the row or all past it)
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
    int s = s0;
    for (; s + 4 <= s1; s += 4) {
        uint4 wv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = (s + u) * F16_SEG + 8 * lane;
            wv[u] = e < K ? __ldg(reinterpret_cast<const uint4 *>(wr + e)) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) segment(wv[u], (s + u) * F16_SEG + 8 * lane);
    }
    for (; s < s1; ++s) {
        const int e = s * F16_SEG + 8 * lane;
        const uint4 wv = e < K ? __ldg(reinterpret_cast<const uint4 *>(wr + e)) : make_uint4(0, 0, 0, 0);
        segment(wv, e);
    }
    return __fadd_rn(__fadd_rn(__fadd_rn(c0.x, c0.y), __fadd_rn(c1.x, c1.y)),
                     __fadd_rn(__fadd_rn(c2.x, c2.y), __fadd_rn(c3.x, c3.y)));
}

__device__ __forceinline__ float to_out(float v, float *) { return v; }
__device__ __forceinline__ __half to_out(float v, __half *) { return __float2half_rn(v); }

// the 32-lane fold of the lane sums, then lane 0 stores the row
template <typename T>
__device__ __forceinline__ void fold_store(float p, int lane, T *__restrict__ y, int row) {
    for (int o = 16; o > 0; o >>= 1) p = __fadd_rn(p, __shfl_xor_sync(0xffffffffu, p, o));
    if (lane == 0) y[row] = to_out(p, y);
}

// T: float, or __half for the fp16 output.  A warp's work is a sequence of
// batches, each four segments of one row; the loads of the next batch (in
// this row, or the first of the warp's next row) are issued before the
// arithmetic of the current one, so a warp keeps loads in flight while it
// adds, folds and stores.  The arithmetic is lane_group_sum's, in the same
// order.
template <typename T>
__global__ void __launch_bounds__(F16_WARPS * 32)
    f16_gemv_kernel(const __half *__restrict__ W, const float *__restrict__ x, T *__restrict__ y,
                    int M, int K) {
    const int lane = threadIdx.x & 31;
    const int nseg = (K + F16_SEG - 1) / F16_SEG;
    // M <= 2^30 (the launcher's row chunks), so row + stride never overflows
    const int stride = gridDim.x * F16_WARPS;
    // the four segments s .. s + 3 of a row (lanes past K, and segments past
    // the row, load nothing)
    auto load = [&](uint4(&wv)[4], int row, int s) {
        const __half *wr = W + (size_t)row * K;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = (s + u) * F16_SEG + 8 * lane;
            wv[u] = e < K ? __ldg(reinterpret_cast<const uint4 *>(wr + e)) : make_uint4(0, 0, 0, 0);
        }
    };
    int row = blockIdx.x * F16_WARPS + (threadIdx.x >> 5), s = 0;
    if (row >= M) return;
    uint4 wv[4];
    load(wv, row, 0);
    float p = -0.0f;
    float2 c0 = make_float2(-0.0f, -0.0f), c1 = c0, c2 = c0, c3 = c0;
    for (;;) {
        // the next batch: a group is 16 segments, so batches never straddle one
        int nrow = row, ns = s + 4;
        if (ns >= nseg) ns = 0, nrow = row + stride;
        uint4 nx[4];
        if (nrow < M) load(nx, nrow, ns);
        if (s % F16_GROUP == 0) c0 = c1 = c2 = c3 = make_float2(-0.0f, -0.0f);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int e = (s + u) * F16_SEG + 8 * lane;
            if (e >= K) continue;
            const float4 xa = __ldg(reinterpret_cast<const float4 *>(x + e));
            const float4 xb = __ldg(reinterpret_cast<const float4 *>(x + e + 4));
            c0 = __ffma2_rn(half2_at(wv[u].x), make_float2(xa.x, xa.y), c0);
            c1 = __ffma2_rn(half2_at(wv[u].y), make_float2(xa.z, xa.w), c1);
            c2 = __ffma2_rn(half2_at(wv[u].z), make_float2(xb.x, xb.y), c2);
            c3 = __ffma2_rn(half2_at(wv[u].w), make_float2(xb.z, xb.w), c3);
        }
        if ((s + 4) % F16_GROUP == 0 || s + 4 >= nseg) {
            const float g = __fadd_rn(__fadd_rn(__fadd_rn(c0.x, c0.y), __fadd_rn(c1.x, c1.y)),
                                      __fadd_rn(__fadd_rn(c2.x, c2.y), __fadd_rn(c3.x, c3.y)));
            p = s < F16_GROUP ? g : __fadd_rn(p, g);
        }
        if (ns == 0) {
            fold_store(p, lane, y, row);
            p = -0.0f;
        }
        if (nrow >= M) break;
        row = nrow, s = ns;
#pragma unroll
        for (int u = 0; u < 4; ++u) wv[u] = nx[u];
    }
}

// Split-K: CTA b evaluates row b, warp w taking groups w, w + nw, ...
// (nw = blockDim.x / 32).  K <= 2^18, so a row has at most 64 groups.
template <typename T>
__global__ void __launch_bounds__(F16_SPLIT_WARPS * 32)
    f16_gemv_split_kernel(const __half *__restrict__ W, const float *__restrict__ x,
                          T *__restrict__ y, int K) {
    __shared__ float gsum[F16_MAX_GROUPS][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int nseg = (K + F16_SEG - 1) / F16_SEG;
    const int ngroups = (nseg + F16_GROUP - 1) / F16_GROUP;
    const __half *wr = W + (size_t)blockIdx.x * K;
    for (int j = warp; j < ngroups; j += nw)
        gsum[j][lane] = lane_group_sum(wr, x, j * F16_GROUP, min(nseg, (j + 1) * F16_GROUP), lane, K);
    __syncthreads();
    if (warp != 0) return;
    float p = gsum[0][lane];
    for (int j = 1; j < ngroups; ++j) p = __fadd_rn(p, gsum[j][lane]);
    fold_store(p, lane, y, blockIdx.x);
}

// One fp16-weight GEMV on `stream` (arguments validated by the caller).
template <typename T>
int f16_launch(const void *W, const float *x, T *y, long long M, long long K, void *stream) {
    const auto s = static_cast<cudaStream_t>(stream);
    const auto *w = static_cast<const __half *>(W);
    int dev = 0, nsm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return (int)e;
    const long long nseg = (K + F16_SEG - 1) / F16_SEG;
    const int ngroups = (int)((nseg + F16_GROUP - 1) / F16_GROUP);
    if (ngroups >= 2 && M < (long long)nsm * F16_SPLIT_ROWS_PER_SM) {
        const int nw = ngroups < F16_SPLIT_WARPS ? ngroups : F16_SPLIT_WARPS;
        f16_gemv_split_kernel<T><<<(unsigned)M, nw * 32, 0, s>>>(w, x, y, (int)K);
        return (int)cudaGetLastError();
    }
    // at most one wave of resident CTAs, rows grid-strided over the warps, in
    // launches of at most 2^30 rows
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, f16_gemv_kernel<T>,
                                                      F16_WARPS * 32, 0);
    if (e != cudaSuccess) return (int)e;
    for (long long r0 = 0; r0 < M; r0 += F16_ROW_CHUNK) {
        const long long m = M - r0 < F16_ROW_CHUNK ? M - r0 : F16_ROW_CHUNK;
        const long long want = (m + F16_WARPS - 1) / F16_WARPS;
        const long long cap = (long long)nsm * (occ > 0 ? occ : 1);
        const int grid = (int)(want < cap ? want : cap);
        f16_gemv_kernel<T><<<grid, F16_WARPS * 32, 0, s>>>(w + r0 * K, x, y + r0, (int)m, (int)K);
        e = cudaGetLastError();
        if (e != cudaSuccess) return (int)e;
    }
    return 0;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace
}  // namespace bq

int bq_internal_f16_launch(const void *W, const float *x, float *y, long long M, long long K,
                           void *stream) {
    return bq::f16_launch(W, x, y, M, K, stream);
}

// The fp16-output entry point (include/bqgemv.h).  Its checks are those of
// bq_gemv_f16 in bq_api.cu, with y 2-byte aligned instead of 4.
extern "C" bq_status bq_gemv_f16_f16out(const void *W, const float *x, void *y, int64_t M,
                                        int64_t K, void *stream) {
    if (M < 0 || M > bq::F16_M_MAX || K < 8 || K > bq::F16_K_MAX || K % 8) return BQ_ERR_SHAPE;
    if (M == 0) return BQ_OK;
    if (!W || !x || !y) return BQ_ERR_NULL;
    if (!bq::aligned(W, 16) || !bq::aligned(x, 16) || !bq::aligned(y, 2)) return BQ_ERR_ALIGN;
    return bq::f16_launch(W, x, static_cast<__half *>(y), M, K, stream) == 0 ? BQ_OK : BQ_ERR_CUDA;
}
