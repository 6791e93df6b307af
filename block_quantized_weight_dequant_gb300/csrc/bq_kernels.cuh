// bq_kernels.cuh -- GEMV kernels over block-quantized weights for sm_103a.
//
// stream_kernel: the fast path (K % 256 == 0).  A CTA owns tiles of TR
// consecutive rows.  One producer warp streams each tile's packed bytes from
// HBM into a ring of shared-memory stages with 1-D bulk copies (TMA,
// cp.async.bulk, completion counted on an mbarrier per stage, L2 evict-first
// because the weights are read once); NWC consumer warps decode the stages
// straight from shared memory.  Weights never exist as fp32 anywhere ("no
// float32 materialization", EdgeRunner blog post, "What worked" #2).  Every
// wait is bounded.  No CTA depends on another CTA: tiles are independent and
// nothing is handed off between CTAs inside a launch ("We Wrote Our Own
// Inference Engine", "One hardware finding": cross-threadgroup handoff inside
// one dispatch is not ordered).
//
// generic_kernel: any K % 32 == 0, reading weights straight from global
// memory.  Same arithmetic (bq_dot.cuh), so the same bits.
//
// MODE_PLAIN with R input rows covers the single-row GEMV (R = 1) and the
// multi-row verify GEMV (R = 2..6, weights streamed once for all rows).
// MODE_GATE_UP streams two matrices with one x (optionally RMSNorm-ed) and
// writes silu(g) * u.
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "bq_device.cuh"
#include "bq_dot.cuh"
#include "bq_internal.h"

namespace bq {

constexpr int MAX_STAGES = 8;

struct StreamArgs {
    const uint8_t *W0;
    const uint8_t *W1;
    const float *x;
    const float *gamma;
    float eps;
    float *y;
    int M, K, nsc, G;
    long long rb;  // packed row bytes
    int TR, KCU, NS, nchunks, ntiles;
    int row_stride, mat_stride, stage_bytes, single_copy;
    int x_off, x_rstride, stage_off;
};

template <int MODE, int R> struct NOut {
    static constexpr int n = MODE == MODE_GATE_UP ? 2 : R;
};

template <int QT, int R, int MODE, bool XRES>
__global__ void __launch_bounds__(288) stream_kernel(const StreamArgs a, unsigned int *status) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + MAX_STAGES;
    volatile int *flags = reinterpret_cast<volatile int *>(smem + 128);  // [0] abort [1] issued
    float *red = reinterpret_cast<float *>(smem + 256);
    uint8_t *stages = smem + a.stage_off;

    constexpr int UB = Fmt<QT>::unit_bytes;
    constexpr int NMAT = MODE == MODE_GATE_UP ? 2 : 1;
    constexpr int NO = NOut<MODE, R>::n;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NWC = (blockDim.x >> 5) - 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.NS; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, NWC);
        }
        flags[0] = 0;
        flags[1] = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NWC) {
        // ------------------------------ producer ------------------------------
        const uint64_t pol = l2_policy_evict_first();
        int it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < a.ntiles; tile += gridDim.x) {
            const int row0 = tile * a.TR;
            const int rows = min(a.TR, a.M - row0);
            for (int c = 0; c < a.nchunks; ++c) {
                const int slot = it % a.NS;
                if (it >= a.NS) {
                    if (lane == 0 && !mbar_wait_bounded(empty + slot, ((it / a.NS) - 1) & 1)) {
                        flags[0] = 1;
                        atomicOr(status, BQ_DEVERR_EMPTY_WAIT);
                    }
                    __syncwarp();
                }
                if (flags[0]) {
                    ok = false;
                    break;
                }
                const int u0 = c * a.KCU;
                const int cnt = min(a.KCU, a.nsc - u0);
                const uint32_t rowb = (uint32_t)cnt * UB;
                uint8_t *st = stages + (size_t)slot * a.stage_bytes;
                if (lane == 0) mbar_arrive_expect_tx(full + slot, rowb * rows * NMAT);
                __syncwarp();
                if (a.single_copy) {
                    if (lane == 0) {
                        const size_t off = (size_t)row0 * a.rb;
                        bulk_g2s(st, a.W0 + off, rowb * rows, full + slot, pol);
                        if (NMAT == 2)
                            bulk_g2s(st + a.mat_stride, a.W1 + off, rowb * rows, full + slot, pol);
                    }
                } else {
                    for (int r = lane; r < rows; r += 32) {
                        const size_t off = (size_t)(row0 + r) * a.rb + (size_t)u0 * UB;
                        bulk_g2s(st + r * a.row_stride, a.W0 + off, rowb, full + slot, pol);
                        if (NMAT == 2)
                            bulk_g2s(st + a.mat_stride + r * a.row_stride, a.W1 + off, rowb,
                                     full + slot, pol);
                    }
                }
                ++it;
            }
        }
        if (lane == 0) flags[1] = it;
    } else {
        // ------------------------------ consumers -----------------------------
        const int G = a.G;
        const int rpw = 32 / G;
        const int rho = warp * rpw + lane / G;  // row slot within the tile
        const int l = lane & (G - 1);
        const int nthr = NWC * 32;
        auto csync = [nthr]() { named_bar_sync(1, nthr); };

        float rs = 1.0f;
        const bool norm = MODE == MODE_GATE_UP && a.gamma != nullptr;
        if (norm) rs = rms_scale(a.x, a.K, a.eps, red, threadIdx.x, nthr, csync);

        float *xsm = reinterpret_cast<float *>(smem + a.x_off);
        if constexpr (XRES) {
            for (int r = 0; r < R; ++r)
                for (int e = 4 * threadIdx.x; e < a.K; e += 4 * nthr) {
                    float4 v = __ldg(reinterpret_cast<const float4 *>(a.x + (size_t)r * a.K + e));
                    if (norm) {
                        const float4 g = __ldg(reinterpret_cast<const float4 *>(a.gamma + e));
                        v = make_float4(__fmul_rn(__fmul_rn(v.x, rs), g.x),
                                        __fmul_rn(__fmul_rn(v.y, rs), g.y),
                                        __fmul_rn(__fmul_rn(v.z, rs), g.z),
                                        __fmul_rn(__fmul_rn(v.w, rs), g.w));
                    }
                    *reinterpret_cast<float4 *>(xsm + r * a.x_rstride + 4 * x_chunk_pos(e >> 2)) = v;
                }
            csync();
        }

        auto run = [&](const auto &xs) {
            int it = 0;
            for (int tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x) {
                const int row0 = tile * a.TR;
                const int rows = min(a.TR, a.M - row0);
                float p[NO];
#pragma unroll
                for (int o = 0; o < NO; ++o) p[o] = -0.0f;
                for (int c = 0; c < a.nchunks; ++c, ++it) {
                    const int slot = it % a.NS;
                    const bool landed = mbar_wait_bounded(full + slot, (it / a.NS) & 1);
                    if (!__all_sync(0xffffffffu, landed)) {
                        if (lane == 0) {
                            flags[0] = 1;
                            atomicOr(status, BQ_DEVERR_FULL_WAIT);
                        }
                        return;
                    }
                    const int u0 = c * a.KCU;
                    const int cnt = min(a.KCU, a.nsc - u0);
                    const uint8_t *st = stages + (size_t)slot * a.stage_bytes + rho * a.row_stride;
                    if (rho < rows) {
                        for (int ul = l; ul < cnt; ul += G) {
                            const int e0 = (u0 + ul) * 256;
                            if constexpr (MODE == MODE_GATE_UP) {
                                uint32_t wg[Fmt<QT>::unit_words], wu[Fmt<QT>::unit_words];
                                load_unit_smem<QT>(wg, st + ul * UB);
                                load_unit_smem<QT>(wu, st + a.mat_stride + ul * UB);
                                const uint32_t *const ws[2] = {wg, wu};
                                float cc[2][1];
                                unit_dot<QT, 2, 1>(ws, 8, xs, e0, cc);
                                p[0] = __fadd_rn(p[0], cc[0][0]);
                                p[1] = __fadd_rn(p[1], cc[1][0]);
                            } else {
                                uint32_t w[Fmt<QT>::unit_words];
                                load_unit_smem<QT>(w, st + ul * UB);
                                const uint32_t *const ws[1] = {w};
                                float cc[1][R];
                                unit_dot<QT, 1, R>(ws, 8, xs, e0, cc);
#pragma unroll
                                for (int r = 0; r < R; ++r) p[r] = __fadd_rn(p[r], cc[0][r]);
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(empty + slot);
                }
#pragma unroll
                for (int o = 0; o < NO; ++o) p[o] = fold_lanes(p[o], G);
                if (rho < rows && l == 0) {
                    const int row = row0 + rho;
                    if constexpr (MODE == MODE_GATE_UP) {
                        a.y[row] = silu_mul(p[0], p[1]);
                    } else {
#pragma unroll
                        for (int r = 0; r < R; ++r) a.y[(size_t)r * a.M + row] = p[r];
                    }
                }
            }
        };
        if constexpr (XRES) {
            run(XSmem{xsm, a.x_rstride});
        } else if (MODE == MODE_GATE_UP) {
            if (norm) run(XGlobalNorm{a.x, a.gamma, rs});
            else run(XGlobal{a.x, a.K});
        } else {
            run(XGlobal{a.x, a.K});
        }
    }

    __syncthreads();
    if (flags[0] && threadIdx.x == 0) {
        // an error unwound the pipeline: let every copy still in flight land
        // before the CTA (and its shared memory) goes away
        const int issued = flags[1];
        for (int it = issued > a.NS ? issued - a.NS : 0; it < issued; ++it)
            if (!mbar_wait_bounded(full + it % a.NS, (it / a.NS) & 1))
                atomicOr(status, BQ_DEVERR_DRAIN_WAIT);
    }
}

struct GenericArgs {
    const uint8_t *W0;
    const uint8_t *W1;
    const float *x;
    const float *gamma;
    float eps;
    float *y;
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
    const int row = (blockIdx.x * GENERIC_WARPS + warp) * rpw + lane / G;
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
                if constexpr (MODE == MODE_GATE_UP) {
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
                for (int r = 0; r < R; ++r) a.y[(size_t)r * a.M + row] = p[r];
            }
        }
    };
    if (norm) run(XGlobalNorm{a.x, a.gamma, rs});
    else run(XGlobal{a.x, a.K});
}

// ---------------------------------------------------------------------------
// host side: launch one planned GEMV call
// ---------------------------------------------------------------------------
template <int QT, int R, int MODE, bool XRES>
cudaError_t launch_stream_t(const GemvCall &c, const LaunchPlan &p, unsigned int *status) {
    auto kern = stream_kernel<QT, R, MODE, XRES>;
    // per device: the dynamic shared memory granted so far, and the last
    // occupancy answer keyed by (shared memory, threads)
    static std::atomic<int> granted[64];
    static std::atomic<long long> occ_key[64];
    static std::atomic<int> occ_val[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (granted[dev].load() < (int)p.smem) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)p.smem);
        if (e != cudaSuccess) return e;
        granted[dev].store((int)p.smem);
    }
    const int threads = (p.NWC + 1) * 32;
    const long long key = ((long long)p.smem << 16) | threads;
    int occ = 0;
    if (occ_key[dev].load() == key) {
        occ = occ_val[dev].load();
    } else {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, threads, p.smem);
        if (e != cudaSuccess) return e;
        occ_val[dev].store(occ);
        occ_key[dev].store(key);
    }
    if (occ < 1) return cudaErrorInvalidConfiguration;
    int grid = p.num_sms * occ;
    if (grid > p.ntiles) grid = p.ntiles;
    StreamArgs a;
    a.W0 = static_cast<const uint8_t *>(c.W0);
    a.W1 = static_cast<const uint8_t *>(c.W1);
    a.x = c.x;
    a.gamma = c.gamma;
    a.eps = c.eps;
    a.y = c.y;
    a.M = (int)c.M;
    a.K = (int)c.K;
    a.nsc = p.nsc;
    a.G = p.G;
    a.rb = p.rb;
    a.TR = p.TR;
    a.KCU = p.KCU;
    a.NS = p.NS;
    a.nchunks = p.nchunks;
    a.ntiles = p.ntiles;
    a.row_stride = p.row_stride;
    a.mat_stride = p.mat_stride;
    a.stage_bytes = p.stage_bytes;
    a.single_copy = p.single_copy;
    a.x_off = p.x_off;
    a.x_rstride = p.x_rstride;
    a.stage_off = p.stage_off;
    kern<<<grid, threads, p.smem, (cudaStream_t)c.stream>>>(a, status);
    return cudaGetLastError();
}

template <int QT, int R, int MODE>
cudaError_t launch_generic_t(const GemvCall &c, const LaunchPlan &p) {
    GenericArgs a;
    a.W0 = static_cast<const uint8_t *>(c.W0);
    a.W1 = static_cast<const uint8_t *>(c.W1);
    a.x = c.x;
    a.gamma = c.gamma;
    a.eps = c.eps;
    a.y = c.y;
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

template <int QT, int R>
cudaError_t launch_r(const GemvCall &c, const LaunchPlan &p, unsigned int *status) {
    if (p.kind == PLAN_GENERIC) return launch_generic_t<QT, R, MODE_PLAIN>(c, p);
    return p.xres ? launch_stream_t<QT, R, MODE_PLAIN, true>(c, p, status)
                  : launch_stream_t<QT, R, MODE_PLAIN, false>(c, p, status);
}

template <int QT>
cudaError_t launch_gemv(const GemvCall &c, const LaunchPlan &p, unsigned int *status) {
    if (c.mode == MODE_GATE_UP) {
        if (p.kind == PLAN_GENERIC) return launch_generic_t<QT, 1, MODE_GATE_UP>(c, p);
        return p.xres ? launch_stream_t<QT, 1, MODE_GATE_UP, true>(c, p, status)
                      : launch_stream_t<QT, 1, MODE_GATE_UP, false>(c, p, status);
    }
    switch (c.R) {
        case 1: return launch_r<QT, 1>(c, p, status);
        case 2: return launch_r<QT, 2>(c, p, status);
        case 3: return launch_r<QT, 3>(c, p, status);
        case 4: return launch_r<QT, 4>(c, p, status);
        case 5: return launch_r<QT, 5>(c, p, status);
        case 6: return launch_r<QT, 6>(c, p, status);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace bq
