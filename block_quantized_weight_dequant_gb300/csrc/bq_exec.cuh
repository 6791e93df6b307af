// bq_exec.cuh -- one persistent launch for a whole per-token weight stream.
//
// A decode step is a chain of dependent GEMV stages (per layer: q|k|v, o,
// gate+up, down; then the LM head).  The pages run it as one command buffer
// per token because per-dispatch cost dominates small GEMVs (EdgeRunner blog
// post, "What worked" #1: 420+ dispatches in one command buffer, ~6 us each
// to encode; "We Wrote Our Own Inference Engine", "What actually moved it":
// 770 dispatches per token).  On GB300 a launch costs microseconds while a
// 0.5 MB GEMV streams in under 0.1 us, so this kernel runs the whole stream
// in ONE cooperative launch:
//
//  - every warp owns a ring of shared-memory slots and streams its own warp
//    tiles (32/G rows x a chunk of units) of packed weights into them with
//    1-D bulk copies (TMA), running ahead of its compute -- across stage
//    boundaries too, because weights never depend on earlier stages;
//  - only x depends on the previous stage, so x is read after a grid-wide
//    stage barrier: each CTA's thread 0 adds one release-arrival per stage
//    and waits (bounded) for all CTAs with acquire loads; the CTA then loads
//    the stage's distinct x vectors into shared memory at once with plain
//    coherent loads (never the read-only path), applies RMSNorm there, and
//    every warp reads x from shared memory;
//  - arithmetic is bq_dot.cuh's fixed tree, so every output is bit-identical
//    to the standalone single-row kernels on the same inputs.
// The barrier is an explicit, ordered, device-scope handoff between CTAs of a
// cooperative launch (co-residency guaranteed), unlike the unordered
// last-arrival handoff that failed on the pages ("We Wrote Our Own Inference
// Engine", "One hardware finding").
#pragma once

#include <cuda_runtime.h>

#include "bq_device.cuh"
#include "bq_dot.cuh"
#include "bq_internal.h"

namespace bq {

#define BQ_DEVERR_BARRIER_WAIT 0x8u  // a CTA gave up waiting at a stage barrier

struct ExecOp {
    const uint8_t *W[2];
    float *y;
    long long rb;
    int mode, M, K, nsc, G, rpw;
    int KCU, nchunks, ntiles, row_stride, single, nmat;
    int tile_base;  // first tile of this op within its stage
    int xoff;       // float offset of this op's (normalised) x in the stage's x area
};

// one distinct input vector of a stage, staged into shared memory after the
// stage barrier (and RMSNorm-ed there when gamma is set)
struct ExecX {
    const float *x;
    const float *gamma;
    float eps;
    int K, off;  // off: float offset in the x area
};

struct ExecStage {
    int op_begin, op_end, tiles;
    int x_begin, x_end;  // range in the ExecX table
};

struct ExecArgs {
    const ExecOp *ops;
    const ExecStage *stages;
    const ExecX *xs;
    unsigned int *counters;  // one per stage, zero at launch
    int nstages;
    int NSW;         // ring slots per warp
    int slot_bytes;  // bytes per slot (a multiple of 128)
    int x_off;       // shared-memory offset of the stage's x area
    int ring_off;    // shared-memory offset of the rings
};

// launch geometry of a planned executor run (host side)
struct ExecGeometry {
    int n_stages, n_x, slot, nsw, x_off, ring_off, threads, grid;
    size_t smem;
};

// x read with plain (coherent) loads: x may have been written by another CTA
// before the stage barrier, so the read-only path is not allowed
__device__ __forceinline__ float4 ld_coherent4(const float *p) {
    float4 v;
    asm volatile("ld.global.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}

// Stage the x vectors of stage s into shared memory (padded layout of XSmem),
// RMSNorm-ing those with a gain: every thread of the CTA takes part; ends with
// the x area complete and visible to all warps.  The RMS scale uses the same
// fixed tree as rms_scale(), so xn matches the single-op kernels bit for bit.
__device__ __forceinline__ void exec_stage_x(const ExecArgs &a, int s, float *xa, float *red) {
    const ExecStage st = a.stages[s];
    const int nthr = blockDim.x;
    auto sync = [nthr]() { named_bar_sync(1, nthr); };
    bool any_norm = false;
    for (int j = st.x_begin; j < st.x_end; ++j) {
        const ExecX xd = a.xs[j];
        for (int e = 4 * threadIdx.x; e < xd.K; e += 4 * nthr)
            *reinterpret_cast<float4 *>(xa + xd.off + e + ((e >> 8) << 2)) = ld_coherent4(xd.x + e);
        any_norm |= xd.gamma != nullptr;
    }
    sync();
    if (!any_norm) return;
    for (int j = st.x_begin; j < st.x_end; ++j) {
        const ExecX xd = a.xs[j];
        if (!xd.gamma) continue;
        float *xv = xa + xd.off;
        for (int v = threadIdx.x; v < 256; v += nthr) {
            float acc = 0.0f;
            for (int k = v; k < xd.K; k += 256) {
                const float t = xv[k + ((k >> 8) << 2)];
                acc = __fmaf_rn(t, t, acc);
            }
            red[v] = acc;
        }
        sync();
        if (threadIdx.x < 32) {
            const float *q = red + 8 * threadIdx.x;
            float v = __fadd_rn(__fadd_rn(__fadd_rn(q[0], q[1]), __fadd_rn(q[2], q[3])),
                                __fadd_rn(__fadd_rn(q[4], q[5]), __fadd_rn(q[6], q[7])));
            for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
            if (threadIdx.x == 0) red[256] = v;
        }
        sync();
        const float ms = __fdiv_rn(red[256], (float)xd.K);
        const float rs = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, xd.eps)));
        for (int e = 4 * threadIdx.x; e < xd.K; e += 4 * nthr) {
            float4 *p = reinterpret_cast<float4 *>(xv + e + ((e >> 8) << 2));
            const float4 v = *p;
            const float4 g = __ldg(reinterpret_cast<const float4 *>(xd.gamma + e));
            *p = make_float4(__fmul_rn(__fmul_rn(v.x, rs), g.x), __fmul_rn(__fmul_rn(v.y, rs), g.y),
                             __fmul_rn(__fmul_rn(v.z, rs), g.z), __fmul_rn(__fmul_rn(v.w, rs), g.w));
        }
        sync();  // also protects red[] before the next gain's reduction
    }
}

// position of a warp in the item sequence: stage, tile index in the stage
// (this warp takes tiles gw, gw + nwarps, ...), op, matrix, chunk
struct ExecItem {
    int s, t, op, mat, chunk;
};

__device__ __forceinline__ bool exec_locate(const ExecArgs &a, ExecItem &it) {
    // find the op of tile t in stage s; false if t is past the stage's tiles
    const ExecStage st = a.stages[it.s];
    if (it.t >= st.tiles) return false;
    int op = st.op_begin;
    while (op + 1 < st.op_end && a.ops[op + 1].tile_base <= it.t) ++op;
    it.op = op;
    return true;
}

// first item of stage s at or after tile t0 (t0 = this warp's first tile); -1 op if none
__device__ __forceinline__ void exec_first_in_stage(const ExecArgs &a, ExecItem &it, int s,
                                                    int gw) {
    it.s = s;
    it.t = gw;
    it.mat = 0;
    it.chunk = 0;
    if (!exec_locate(a, it)) it.op = -1;
}

// advance within the current stage; returns false when the warp has no more
// items in this stage
__device__ __forceinline__ bool exec_next_in_stage(const ExecArgs &a, ExecItem &it, int nwarps) {
    const ExecOp &op = a.ops[it.op];
    if (++it.chunk < op.nchunks) return true;
    it.chunk = 0;
    if (++it.mat < op.nmat) return true;
    it.mat = 0;
    it.t += nwarps;
    return exec_locate(a, it);
}

// the producer side walks across stages
__device__ __forceinline__ bool exec_next_any(const ExecArgs &a, ExecItem &it, int nwarps,
                                              int gw) {
    if (it.op >= 0 && exec_next_in_stage(a, it, nwarps)) return true;
    for (int s = it.s + 1; s < a.nstages; ++s) {
        exec_first_in_stage(a, it, s, gw);
        if (it.op >= 0) return true;
    }
    it.s = a.nstages;
    it.op = -1;
    return false;
}

template <int QT>
__device__ __forceinline__ void exec_issue(const ExecArgs &a, const ExecItem &it, uint8_t *slot,
                                           uint64_t *full, uint64_t pol, int lane) {
    constexpr int UB = Fmt<QT>::unit_bytes;
    const ExecOp &op = a.ops[it.op];
    const int tile = it.t - op.tile_base;
    const int row0 = tile * op.rpw;
    const int rows = min(op.rpw, op.M - row0);
    const int u0 = it.chunk * op.KCU;
    const int cnt = min(op.KCU, op.nsc - u0);
    const uint32_t rowb = (uint32_t)cnt * UB;
    const uint8_t *W = op.W[it.mat];
    if (lane == 0) mbar_arrive_expect_tx(full, rowb * rows);
    __syncwarp();
    if (op.single) {
        if (lane == 0) bulk_g2s(slot, W + (size_t)row0 * op.rb, rowb * rows, full, pol);
    } else if (lane < rows) {
        bulk_g2s(slot + lane * op.row_stride, W + (size_t)(row0 + lane) * op.rb + (size_t)u0 * UB,
                 rowb, full, pol);
    }
}

template <int QT>
__global__ void __launch_bounds__(256, 1) exec_kernel(const ExecArgs a, unsigned int *status) {
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int UB = Fmt<QT>::unit_bytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nw = blockDim.x >> 5;
    const int nwarps = nw * gridDim.x;
    const int gw = warp * gridDim.x + blockIdx.x;  // warp-major: consecutive tiles on different SMs
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem);
    float *red = reinterpret_cast<float *>(smem + 64);                         // 260 floats
    uint64_t *fulls = reinterpret_cast<uint64_t *>(smem + 64 + 4 * 264);      // nw * NSW
    float *xa = reinterpret_cast<float *>(smem + a.x_off);
    uint8_t *ring = smem + a.ring_off + (size_t)warp * a.NSW * a.slot_bytes;
    uint64_t *full = fulls + warp * a.NSW;

    if (threadIdx.x == 0) *abort_flag = 0;
    if (lane == 0)
        for (int i = 0; i < a.NSW; ++i) mbar_init(full + i, 1);
    if (lane == 0) fence_mbar_init();
    __syncthreads();

    const uint64_t pol = l2_policy_evict_first();
    // producer cursor: prefetch the first NSW items of this warp
    ExecItem pit;
    pit.s = -1;
    pit.op = -1;
    int issued = 0, consumed = 0;
    auto issue_next = [&]() {
        if (!exec_next_any(a, pit, nwarps, gw)) return;
        exec_issue<QT>(a, pit, ring + (size_t)(issued % a.NSW) * a.slot_bytes,
                       full + issued % a.NSW, pol, lane);
        ++issued;
    };
    {
        // start the producer cursor before stage 0
        pit.s = -1;
        pit.op = -1;
        for (int i = 0; i < a.NSW; ++i) issue_next();
    }

    for (int s = 0; s < a.nstages; ++s) {
        if (s > 0) {
            // ---- grid-wide barrier: every CTA has finished stage s-1 ----
            named_bar_sync(1, blockDim.x);
            if (threadIdx.x == 0) {
                __threadfence();
                atomicAdd(a.counters + (s - 1), 1u);
                if (!*abort_flag) {
                    const uint64_t t0 = globaltimer();
                    unsigned int n = 0;
                    for (uint32_t i = 0;; ++i) {
                        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];"
                                     : "=r"(n)
                                     : "l"(a.counters + (s - 1))
                                     : "memory");
                        if (n >= gridDim.x) break;
                        if ((i & 63u) == 63u && globaltimer() - t0 > BQ_WAIT_LIMIT_NS) {
                            *abort_flag = 1;
                            atomicOr(status, BQ_DEVERR_BARRIER_WAIT);
                            break;
                        }
                    }
                }
            }
            named_bar_sync(1, blockDim.x);
        }
        if (*abort_flag) continue;  // keep every barrier's arrival, skip the work
        exec_stage_x(a, s, xa, red);

        ExecItem it;
        exec_first_in_stage(a, it, s, gw);
        if (it.op < 0) continue;
        float p0 = -0.0f, p1 = -0.0f;
        for (;;) {
            const ExecOp &op = a.ops[it.op];
            const int slot = consumed % a.NSW;
            const bool landed = mbar_wait_bounded(full + slot, (consumed / a.NSW) & 1);
            if (!__all_sync(0xffffffffu, landed)) {
                if (lane == 0) {
                    *abort_flag = 1;
                    atomicOr(status, BQ_DEVERR_FULL_WAIT);
                }
                break;
            }
            const int G = op.G;
            const int rho = lane / G, l = lane & (G - 1);
            const int tile = it.t - op.tile_base;
            const int row0 = tile * op.rpw;
            const int rows = min(op.rpw, op.M - row0);
            const int u0 = it.chunk * op.KCU;
            const int cnt = min(op.KCU, op.nsc - u0);
            if (it.mat == 0 && it.chunk == 0) {
                p0 = -0.0f;
                p1 = -0.0f;
            }
            const uint8_t *st = ring + (size_t)slot * a.slot_bytes + rho * op.row_stride;
            const XSmem xs{xa + op.xoff, 0};
            float acc = it.mat == 0 ? p0 : p1;
            if (rho < rows) {
                for (int ul = l; ul < cnt; ul += G) {
                    uint32_t w[Fmt<QT>::unit_words];
                    load_unit_smem<QT>(w, st + ul * UB);
                    const uint32_t *const ws[1] = {w};
                    float cc[1][1];
                    unit_dot<QT, 1, 1>(ws, 8, xs, (u0 + ul) * 256, cc);
                    acc = __fadd_rn(acc, cc[0][0]);
                }
            }
            if (it.mat == 0) p0 = acc;
            else p1 = acc;
            __syncwarp();
            ++consumed;
            const bool last_chunk = it.chunk + 1 == op.nchunks;
            const bool last_mat = it.mat + 1 == op.nmat;
            if (last_chunk && last_mat) {
                const float g = fold_lanes(p0, G);
                if (op.nmat == 2) {
                    const float u = fold_lanes(p1, G);
                    if (rho < rows && l == 0) op.y[row0 + rho] = silu_mul(g, u);
                } else if (rho < rows && l == 0) {
                    op.y[row0 + rho] = g;
                }
            }
            issue_next();  // refill the slot just consumed
            if (!exec_next_in_stage(a, it, nwarps)) break;
        }
    }

    // make sure no copy into this warp's ring is still in flight at exit
    if (*abort_flag) {
        for (int i = consumed; i < issued; ++i)
            if (!mbar_wait_bounded(full + i % a.NSW, (i / a.NSW) & 1) && lane == 0)
                atomicOr(status, BQ_DEVERR_DRAIN_WAIT);
    }
}

}  // namespace bq
