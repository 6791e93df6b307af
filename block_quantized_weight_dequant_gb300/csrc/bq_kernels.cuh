// bq_kernels.cuh -- the generic GEMV kernel over block-quantized weights for
// sm_103a: any K % 32 == 0 (rows that are not a whole number of 8-block
// units), reading weights straight from global memory.  Calls with
// K % 256 == 0 take the streaming kernel of bq_multi.cuh instead.  Same
// arithmetic (bq_dot.cuh), so the same bits as the streaming path on any row
// both can evaluate.
//
// MODE_PLAIN with R input rows covers the single-row GEMV (R = 1) and the
// multi-row verify GEMV (R = 2..6, weights read once for all rows).
// MODE_GATE_UP reads two matrices with one x (optionally RMSNorm-ed) and
// writes silu(g) * u.
#pragma once

#include <cuda_runtime.h>

#include "bq_device.cuh"
#include "bq_dot.cuh"
#include "bq_internal.h"

namespace bq {

template <int MODE, int R> struct NOut {
    static constexpr int n = MODE == MODE_GATE_UP ? 2 : R;
};

struct GenericArgs {
    const uint8_t *W0;
    const uint8_t *W1;
    const float *x;
    const float *gamma;
    float eps;
    float *y;
    const float *bias;  // R = 1 plain: added to y, or null
    int M, K, G;
    long long rb;
};

constexpr int GENERIC_WARPS = 4;

template <int QT, int R, int MODE>
__global__ void __launch_bounds__(GENERIC_WARPS * 32) generic_kernel(const GenericArgs a) {
    __shared__ float red[260];
    constexpr int NO = NOut<MODE, R>::n;
    constexpr int UB = Fmt<QT>::unit_bytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = a.G, rpw = 32 / G;
    // 64-bit: M may be up to 2^31 - 1 rows
    const long long row = ((long long)blockIdx.x * GENERIC_WARPS + warp) * rpw + lane / G;
    const int l = lane & (G - 1);
    const int nb = a.K / 32, nsc = (nb + 7) / 8;

    float rs = 1.0f;
    const bool norm = MODE == MODE_GATE_UP && a.gamma != nullptr;
    if (norm) rs = rms_scale(a.x, a.K, a.eps, red, threadIdx.x, GENERIC_WARPS * 32,
                             []() { __syncthreads(); });

    auto run = [&](const auto &xs) {
        float p[NO];
#pragma unroll
        for (int o = 0; o < NO; ++o) p[o] = -0.0f;
        if (row < a.M) {
            for (int u = l; u < nsc; u += G) {
                const int nbk = min(8, nb - 8 * u);
                const size_t off = (size_t)row * a.rb + (size_t)u * UB;
                if constexpr (QT == QT_Q4_K) {
                    // super-blocks are 16-byte aligned: read them in place
                    // (header, then one byte pair group at a time)
                    if constexpr (MODE == MODE_GATE_UP) {
                        const uint8_t *const up[2] = {a.W0 + off, a.W1 + off};
                        float cc[2][1];
                        unit_dot_rows<QT, 2, 1>(up, xs, 256 * u, cc);
                        p[0] = __fadd_rn(p[0], cc[0][0]);
                        p[1] = __fadd_rn(p[1], cc[1][0]);
                    } else {
                        const uint8_t *const up[1] = {a.W0 + off};
                        float cc[1][R];
                        unit_dot_rows<QT, 1, R>(up, xs, 256 * u, cc);
#pragma unroll
                        for (int r = 0; r < R; ++r) p[r] = __fadd_rn(p[r], cc[0][r]);
                    }
                } else if constexpr (MODE == MODE_GATE_UP) {
                    uint32_t wg[Fmt<QT>::unit_words], wu[Fmt<QT>::unit_words];
                    load_unit_global<QT>(wg, a.W0 + off, nbk);
                    load_unit_global<QT>(wu, a.W1 + off, nbk);
                    const uint32_t *const ws[2] = {wg, wu};
                    float cc[2][1];
                    unit_dot<QT, 2, 1>(ws, nbk, xs, 256 * u, cc);
                    p[0] = __fadd_rn(p[0], cc[0][0]);
                    p[1] = __fadd_rn(p[1], cc[1][0]);
                } else {
                    uint32_t w[Fmt<QT>::unit_words];
                    load_unit_global<QT>(w, a.W0 + off, nbk);
                    const uint32_t *const ws[1] = {w};
                    float cc[1][R];
                    unit_dot<QT, 1, R>(ws, nbk, xs, 256 * u, cc);
#pragma unroll
                    for (int r = 0; r < R; ++r) p[r] = __fadd_rn(p[r], cc[0][r]);
                }
            }
        }
#pragma unroll
        for (int o = 0; o < NO; ++o) p[o] = fold_lanes(p[o], G);
        if (row < a.M && l == 0) {
            if constexpr (MODE == MODE_GATE_UP) {
                a.y[row] = silu_mul(p[0], p[1]);
            } else {
#pragma unroll
                for (int r = 0; r < R; ++r)
                    a.y[(size_t)r * a.M + (size_t)row] =
                        R == 1 && a.bias ? __fadd_rn(p[r], a.bias[row]) : p[r];
            }
        }
    };
    if (norm) run(XGlobalNorm{a.x, a.gamma, rs});
    else run(XGlobal{a.x, a.K});
}

// ---------------------------------------------------------------------------
// host side: launch one planned generic GEMV call
// ---------------------------------------------------------------------------
template <int QT, int R, int MODE>
cudaError_t launch_generic_t(const GemvCall &c, const LaunchPlan &p) {
    GenericArgs a;
    a.W0 = static_cast<const uint8_t *>(c.W0);
    a.W1 = static_cast<const uint8_t *>(c.W1);
    a.x = c.x;
    a.gamma = c.gamma;
    a.eps = c.eps;
    a.y = c.y;
    a.bias = c.bias;
    a.M = (int)c.M;
    a.K = (int)c.K;
    a.G = p.G;
    a.rb = p.rb;
    const int rows_per_cta = GENERIC_WARPS * (32 / p.G);
    const long long grid = (c.M + rows_per_cta - 1) / rows_per_cta;
    generic_kernel<QT, R, MODE>
        <<<(unsigned)grid, GENERIC_WARPS * 32, 0, (cudaStream_t)c.stream>>>(a);
    return cudaGetLastError();
}

template <int QT>
cudaError_t launch_gemv(const GemvCall &c, const LaunchPlan &p) {
    if (c.mode == MODE_GATE_UP) return launch_generic_t<QT, 1, MODE_GATE_UP>(c, p);
    switch (c.R) {
        case 1: return launch_generic_t<QT, 1, MODE_PLAIN>(c, p);
        case 2: return launch_generic_t<QT, 2, MODE_PLAIN>(c, p);
        case 3: return launch_generic_t<QT, 3, MODE_PLAIN>(c, p);
        case 4: return launch_generic_t<QT, 4, MODE_PLAIN>(c, p);
        case 5: return launch_generic_t<QT, 5, MODE_PLAIN>(c, p);
        case 6: return launch_generic_t<QT, 6, MODE_PLAIN>(c, p);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace bq
