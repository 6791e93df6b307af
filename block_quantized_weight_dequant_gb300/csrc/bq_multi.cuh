// bq_multi.cuh -- one launch for a list of INDEPENDENT GEMVs (a per-token
// weight stream whose ops read no output of another op of the list).
//
// Without dependences there is no reason to spread every op over every SM:
// the tiles of all ops are concatenated in list order and each CTA streams a
// contiguous, byte-balanced range of them, so a CTA meets only the few ops its
// range crosses.  Inside a CTA this is the pipeline of stream_kernel: one
// producer warp streams tile chunks from HBM into a ring of shared-memory
// stages with 1-D bulk copies (TMA), and the consumer warps decode them
// straight from shared memory.  The consumer warps form NG groups; tile k of
// the CTA goes to group k mod NG, so a stage only has to hold one group's
// rows and the ring can be deep (many bytes in flight per SM) while all
// consumer warps stay busy.  A tile's chunks and matrices (gate, up) go to the
// same group, so its partial sums stay in registers.  Each group has a ring
// of its own (NS / NG slots): an mbarrier wait only tells a phase from the one
// before it, so every waiter must see every phase of the slots it waits on.  The x of an op is staged
// into shared memory (and RMSNorm-ed) when the CTA's range enters the op.
// Arithmetic is bq_dot.cuh's fixed tree: every output is bit-identical to the
// single-op kernels.
#pragma once

#include <cuda_runtime.h>

#include "bq_device.cuh"
#include "bq_dot.cuh"
#include "bq_internal.h"

namespace bq {

struct MultiOp {
    const uint8_t *W[2];
    const float *x;
    const float *gamma;
    float *y;
    float eps;
    int M, K, rb, nsc;
    int G, rpw, TR;          // lanes per row, rows per warp, rows per tile
    int KCU, nchunks, nmat;  // units per stage row, stages per tile and matrix, 1 or 2
    int ntiles, tile_base;   // tiles of this op; its first tile in the whole list
    int row_stride, single;  // shared-memory bytes per tile row; rows copied as one block
};

struct MultiArgs {
    const MultiOp *ops;
    const int *cta_tiles;  // [grid + 1]: CTA c streams tiles [cta_tiles[c], cta_tiles[c+1])
    int nops;
    int NS, stage_bytes, NG;  // NS: slots in all (NS / NG per group)
    int x_off, stage_off;
};

#ifndef BQ_MULTI_NWC
#define BQ_MULTI_NWC 8
#endif
constexpr int MULTI_NWC = BQ_MULTI_NWC;  // consumer warps; + 1 producer warp

template <int QT>
__global__ void __launch_bounds__((MULTI_NWC + 1) * 32, 1)
    multi_kernel(const MultiArgs a, unsigned int *status) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + 16;
    volatile int *flags = reinterpret_cast<volatile int *>(smem + 256);  // [0] abort [2+g] issued
    float *red = reinterpret_cast<float *>(smem + 512);
    float *xsm = reinterpret_cast<float *>(smem + a.x_off);
    uint8_t *stages = smem + a.stage_off;
    constexpr int UB = Fmt<QT>::unit_bytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NWG = MULTI_NWC / a.NG;  // warps per consumer group
    const int t_begin = a.cta_tiles[blockIdx.x], t_end = a.cta_tiles[blockIdx.x + 1];

    if (threadIdx.x == 0) {
        for (int s = 0; s < a.NS; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, NWG);
        }
        for (int i = 0; i < 2 + 8; ++i) flags[i] = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (t_begin >= t_end) return;

    // the op holding tile t, walking forward from op index `op`
    auto op_of = [&](int t, int op) {
        while (op + 1 < a.nops && __ldg(&a.ops[op + 1].tile_base) <= t) ++op;
        return op;
    };
    int op0 = 0;
    {
        int lo = 0, hi = a.nops - 1;  // last op with tile_base <= t_begin
        while (lo < hi) {
            const int mid = (lo + hi + 1) / 2;
            if (__ldg(&a.ops[mid].tile_base) <= t_begin) lo = mid;
            else hi = mid - 1;
        }
        op0 = lo;
    }

    if (warp == MULTI_NWC) {
        // ------------------------------ producer ------------------------------
        const uint64_t pol = l2_policy_evict_first();
        const int NSG = a.NS / a.NG;
        int cnt_g[8] = {};  // items issued per group (NG <= 8)
        int op = op0;
        bool ok = true;
        for (int t = t_begin; ok && t < t_end; ++t) {
            op = op_of(t, op);
            const MultiOp &o = a.ops[op];
            const int row0 = (t - o.tile_base) * o.TR;
            const int rows = min(o.TR, o.M - row0);
            const int g = (t - t_begin) % a.NG;
            for (int m = 0; ok && m < o.nmat; ++m)
                for (int c = 0; c < o.nchunks; ++c) {
                    const int it = cnt_g[g];
                    const int slot = g * NSG + it % NSG;
                    if (it >= NSG) {
                        if (lane == 0 && !mbar_wait_bounded(empty + slot, ((it / NSG) - 1) & 1)) {
                            flags[0] = 1;
                            atomicOr(status, BQ_DEVERR_EMPTY_WAIT);
                        }
                        __syncwarp();
                    }
                    if (flags[0]) {
                        ok = false;
                        break;
                    }
                    const int u0 = c * o.KCU;
                    const int cnt = min(o.KCU, o.nsc - u0);
                    const uint32_t rowb = (uint32_t)cnt * UB;
                    uint8_t *st = stages + (size_t)slot * a.stage_bytes;
                    if (lane == 0) mbar_arrive_expect_tx(full + slot, rowb * rows);
                    __syncwarp();
                    if (o.single) {
                        if (lane == 0)
                            bulk_g2s(st, o.W[m] + (size_t)row0 * o.rb, rowb * rows, full + slot, pol);
                    } else {
                        for (int r = lane; r < rows; r += 32)
                            bulk_g2s(st + r * o.row_stride,
                                     o.W[m] + (size_t)(row0 + r) * o.rb + (size_t)u0 * UB, rowb,
                                     full + slot, pol);
                    }
                    ++cnt_g[g];
                }
        }
        if (lane == 0)
            for (int g = 0; g < a.NG; ++g) flags[2 + g] = cnt_g[g];
    } else {
        // ------------------------------ consumers -----------------------------
        // After an error a consumer keeps walking its tiles without waiting or
        // computing, so that every consumer still reaches every op-boundary
        // barrier (those have no timeout of their own).
        const int group = warp / NWG, wg = warp % NWG;
        const int nthr = MULTI_NWC * 32;
        auto csync = [nthr]() { named_bar_sync(1, nthr); };
        const int NSG = a.NS / a.NG;
        int it = 0, op = -1;  // it: this group's items so far
        bool ok = true;
        for (int t = t_begin; t < t_end; ++t) {
            const int nop = op_of(t, op < 0 ? op0 : op);
            const MultiOp &o = a.ops[nop];
            if (nop != op) {
                // entering a new op: every consumer is done with the previous
                // op's x; stage this op's (RMSNorm-ed) x
                op = nop;
                csync();
                float rs = 1.0f;
                if (o.gamma) rs = rms_scale(o.x, o.K, o.eps, red, threadIdx.x, nthr, csync);
                for (int e = 4 * threadIdx.x; e < o.K; e += 4 * nthr) {
                    float4 v = __ldg(reinterpret_cast<const float4 *>(o.x + e));
                    if (o.gamma) {
                        const float4 g = __ldg(reinterpret_cast<const float4 *>(o.gamma + e));
                        v = make_float4(__fmul_rn(__fmul_rn(v.x, rs), g.x),
                                        __fmul_rn(__fmul_rn(v.y, rs), g.y),
                                        __fmul_rn(__fmul_rn(v.z, rs), g.z),
                                        __fmul_rn(__fmul_rn(v.w, rs), g.w));
                    }
                    *reinterpret_cast<float4 *>(xsm + 4 * x_chunk_pos(e >> 2)) = v;
                }
                csync();
            }
            if (((t - t_begin) % a.NG) != group) continue;
            const int G = o.G;
            const int rho = wg * o.rpw + lane / G;  // row within the tile
            const int l = lane & (G - 1);
            const int row0 = (t - o.tile_base) * o.TR;
            const int rows = min(o.TR, o.M - row0);
            const XSmem xs{xsm, 0};
            float p[2] = {-0.0f, -0.0f};
            for (int m = 0; m < o.nmat; ++m)
                for (int c = 0; c < o.nchunks; ++c, ++it) {
                    const int slot = group * NSG + it % NSG;
                    if (ok && !__all_sync(0xffffffffu, mbar_wait_bounded(full + slot, (it / NSG) & 1))) {
                        if (lane == 0) {
                            flags[0] = 1;
                            atomicOr(status, BQ_DEVERR_FULL_WAIT);
                        }
                        ok = false;
                    }
                    if (ok) {
                        const int u0 = c * o.KCU;
                        const int cnt = min(o.KCU, o.nsc - u0);
                        const uint8_t *stp = stages + (size_t)slot * a.stage_bytes + rho * o.row_stride;
                        if (rho < rows) {
                            for (int ul = l; ul < cnt; ul += G) {
                                uint32_t w[Fmt<QT>::unit_words];
                                load_unit_smem<QT>(w, stp + ul * UB);
                                const uint32_t *const ws[1] = {w};
                                float cc[1][1];
                                unit_dot<QT, 1, 1>(ws, 8, xs, (u0 + ul) * 256, cc);
                                p[m] = __fadd_rn(p[m], cc[0][0]);
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(empty + slot);
                }
            if (!ok) continue;
            const float g = fold_lanes(p[0], G);
            if (o.nmat == 2) {
                const float u = fold_lanes(p[1], G);
                if (rho < rows && l == 0) o.y[row0 + rho] = silu_mul(g, u);
            } else if (rho < rows && l == 0) {
                o.y[row0 + rho] = g;
            }
        }
    }

    __syncthreads();
    if (flags[0] && threadIdx.x == 0) {
        // an error unwound the pipeline: let every copy still in flight land
        const int NSG = a.NS / a.NG;
        for (int g = 0; g < a.NG; ++g) {
            const int issued = flags[2 + g];
            for (int i = issued > NSG ? issued - NSG : 0; i < issued; ++i)
                if (!mbar_wait_bounded(full + g * NSG + i % NSG, (i / NSG) & 1))
                    atomicOr(status, BQ_DEVERR_DRAIN_WAIT);
        }
    }
}

}  // namespace bq
