// bq_exec.cuh -- one persistent launch for a whole per-token weight stream.
//
// A decode step is a chain of GEMV stages (per layer: q|k|v, o, gate+up,
// down; then the LM head).  The pages run it as one command buffer per token
// because per-dispatch cost dominates small GEMVs (EdgeRunner blog post,
// "What worked" #1: 420+ dispatches in one command buffer, ~6 us each to
// encode; "We Wrote Our Own Inference Engine", "What actually moved it": 770
// dispatches per token).  On GB300 a launch costs microseconds while a 0.5 MB
// GEMV streams in under 0.1 us, so this kernel runs a whole stream in ONE
// cooperative launch:
//
//  - the descriptor tables are copied into shared memory once, so nothing on
//    a stage's critical path waits on a global-memory descriptor read;
//  - every warp owns a ring of shared-memory slots and streams its own warp
//    tiles of packed weights into them with 1-D bulk copies (TMA), running
//    ahead of its compute across stage boundaries: weights never depend on
//    earlier stages (the planner rejects outputs that overlap weights).  A
//    tile is 32/G rows x a chunk of units, one unit per lane ("tile mode"),
//    or, for ops with only a few rows per warp, a few whole rows that the
//    warp evaluates one by one block-parallel ("row mode", same tree, 8x
//    shorter latency per row); the tiles of consecutive stages are dealt out
//    to the warps round-robin across the whole stream;
//  - each stage's distinct inputs x are staged into a shared-memory x area
//    (RMSNorm applied there) and every warp reads x from shared memory; the
//    x area is double-buffered, and a stage whose inputs do not depend on
//    earlier stages has its x prefetched with cp.async during the previous
//    stage;
//  - a stage that reads (or overwrites) data of an earlier stage starts with
//    a grid-wide barrier: each CTA's thread 0 adds one release-arrival and
//    waits (bounded) for all CTAs with acquire loads; the planner marks those
//    stages by comparing address ranges, so independent GEMVs never wait;
//  - arithmetic is bq_dot.cuh's fixed tree, so every output is bit-identical
//    to the standalone single-op kernels on the same inputs.
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

#define BQ_DEVERR_BARRIER_WAIT 0x8u   // a CTA gave up waiting at a stage barrier
#define BQ_DEVERR_XFULL_WAIT 0x10u    // a warp gave up waiting for a stage's x copies
#define BQ_DEVERR_XREADY_WAIT 0x20u   // a warp gave up waiting for a stage's normalised x

// one GEMV (or gate+up pair) of the stream; 80 bytes
struct ExecOp {
    const uint8_t *W[2];
    float *y;
    const float *bias;        // GEMV: fp32[M] added to y, or null
    int M, rb;                // rows, packed bytes per row
    int ntiles, tile_base;    // warp tiles; first tile of this op within its stage
    int row_stride, xoff;     // shared-memory bytes per tile row; float offset of x
    short KCU, nchunks;       // units per row per ring slot; slots per tile and matrix
    unsigned char G, rpw, nmat, single;  // rpw: rows per tile
    int nsc;
    int rowmode;              // 1: a tile is rpw whole rows, each evaluated by the whole warp
    int soff;                 // Q4_K: float offset of x's block sums in the x area
    int pad;                  // to a multiple of 16 bytes (see below)
};

// one distinct input vector of a stage (RMSNorm-ed when gamma is set); 48 bytes
struct ExecX {
    const float *x;
    const float *gamma;
    float eps;
    int K, off;  // off: float offset in the x area
    int goff;    // float offset of the gain's staged copy (gamma set), else -1
    int soff;    // Q4_K: float offset of the 32-element block sums, else -1
    int pad[3];
};

// 32 bytes
struct ExecStage {
    int op_begin, op_end, tiles;
    int x_begin, x_end;  // range in the ExecX table
    int barrier;         // 1: wait for every CTA to finish all earlier stages first
    int tile_off;        // tiles of all earlier stages, mod the number of warps: stage s's
                         // tile t goes to warp (tile_off + t) mod nwarps, so work rotates
    int pad;
};

struct ExecArgs {
    const ExecOp *ops;
    const ExecStage *stages;
    const ExecX *xs;
    unsigned int *counters;  // one per stage, zero at launch
    int nops, nstages, nxs;
    int NSW;          // ring slots per warp
    int slot_bytes;   // bytes per slot (a multiple of 128)
    int xbar_off;     // shared-memory offset of the x-buffer mbarriers
    int tab_off;      // shared-memory offset of the descriptor tables
    int x_off;        // shared-memory offset of the x buffers
    int x_floats;     // floats per x buffer
    int x_buffers;    // x buffers in the ring (1..EXEC_MAX_XBUF)
    int ring_off;     // shared-memory offset of the weight rings
    int prefetch;     // items per warp prefetched into L2 beyond the ring
    unsigned long long wait_ns;  // limit of every bounded wait
    unsigned int barrier_extra;  // arrivals a stage barrier waits for beyond the grid's CTAs:
                                 // 0; a test sets 1 so that the wait runs out
};

constexpr int EXEC_MAX_XBUF = 8;

// The kernel copies the three tables into shared memory back to back with
// 16-byte vector loads and stores, so every entry must be a multiple of 16
// bytes: then each table starts 16-byte aligned and is copied whole.
static_assert(sizeof(ExecOp) % 16 == 0, "ExecOp: a multiple of 16 bytes");
static_assert(sizeof(ExecX) % 16 == 0, "ExecX: a multiple of 16 bytes");
static_assert(sizeof(ExecStage) % 16 == 0, "ExecStage: a multiple of 16 bytes");

// launch geometry of a planned executor run (host side)
struct ExecGeometry {
    int n_stages, n_x, slot, nsw, xbar_off, tab_off, x_off, x_floats, x_buffers, ring_off,
        threads, grid, prefetch;
    size_t smem;
};

// shared-memory bytes of the descriptor tables
__host__ __device__ inline int exec_table_bytes(int nops, int nxs, int nstages) {
    return ((nops * (int)sizeof(ExecOp) + nxs * (int)sizeof(ExecX) +
             nstages * (int)sizeof(ExecStage)) + 127) / 128 * 128;
}

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)), "l"(gsrc)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// One warp starts the copies of stage st's inputs (and the RMSNorm gains)
// into x buffer `xa` (x in the permuted layout of XSmem) with cp.async (16 bytes per lane and copy,
// through L2, so data written by other CTAs before a stage barrier is seen),
// then every lane arrives on `xfull` once its copies have landed (the
// barrier expects 32 arrivals).
// EXEC_LOAD_ALL: the inputs and gains, then the arrival; EXEC_LOAD_GAINS:
// only the RMSNorm gains (constant, so they are copied before a stage barrier
// passes; the arrival after the later EXEC_LOAD_X covers them, as an arrival
// waits for all of the thread's earlier cp.async); EXEC_LOAD_X: only the
// inputs, then the arrival.
constexpr int EXEC_LOAD_ALL = 0, EXEC_LOAD_GAINS = 1, EXEC_LOAD_X = 2;
__device__ __forceinline__ void exec_load_x(const ExecStage &st, const ExecX *xs, float *xa,
                                            uint64_t *xfull, int lane, int what = EXEC_LOAD_ALL) {
    for (int j = st.x_begin; j < st.x_end; ++j) {
        const ExecX &xd = xs[j];
        if (what != EXEC_LOAD_GAINS)
            for (int c = lane; c < xd.K / 4; c += 32)
                cp_async16(xa + xd.off + 4 * x_chunk_pos(c), xd.x + 4 * c);
        // the gain rides along (linear layout), so the RMSNorm reads it from
        // shared memory instead of waiting on global loads one by one
        if (xd.goff >= 0 && what != EXEC_LOAD_X)
            for (int c = lane; c < xd.K / 4; c += 32) cp_async16(xa + xd.goff + 4 * c, xd.gamma + 4 * c);
    }
    if (what != EXEC_LOAD_GAINS)
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(xfull))
                     : "memory");
}

// One warp RMSNorms the stage's inputs that have a gain, in place.  The RMS
// scale uses the fixed tree of rms_scale() (lane L holds the 256-virtual-lane
// sums 8L..8L+7), so xn matches the single-op kernels bit for bit.  Q4_K:
// then the 32-element block sums of every input (xblock_sum's order).
template <int QT>
__device__ __forceinline__ void exec_norm_x_warp(const ExecStage &st, const ExecX *xs, float *xa,
                                                 int lane) {
    for (int j = st.x_begin; j < st.x_end; ++j) {
        const ExecX &xd = xs[j];
        if (!xd.gamma) continue;
        float *xv = xa + xd.off;
        float q[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float acc = 0.0f;
            for (int k = 8 * lane + i; k < xd.K; k += 256) {
                const float t = xv[x_pos(k)];
                acc = __fmaf_rn(t, t, acc);
            }
            q[i] = acc;
        }
        float v = __fadd_rn(__fadd_rn(__fadd_rn(q[0], q[1]), __fadd_rn(q[2], q[3])),
                            __fadd_rn(__fadd_rn(q[4], q[5]), __fadd_rn(q[6], q[7])));
        for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
        const float ms = __fdiv_rn(v, (float)xd.K);
        const float rs = __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(ms, xd.eps)));
        __syncwarp();
        for (int c = lane; c < xd.K / 4; c += 32) {
            float4 *p = reinterpret_cast<float4 *>(xv + 4 * x_chunk_pos(c));
            const float4 x4 = *p;
            const float4 g = *reinterpret_cast<const float4 *>(xa + xd.goff + 4 * c);
            *p = make_float4(__fmul_rn(__fmul_rn(x4.x, rs), g.x), __fmul_rn(__fmul_rn(x4.y, rs), g.y),
                             __fmul_rn(__fmul_rn(x4.z, rs), g.z), __fmul_rn(__fmul_rn(x4.w, rs), g.w));
        }
        __syncwarp();
    }
    if constexpr (QT == QT_Q4_K) {
        for (int j = st.x_begin; j < st.x_end; ++j) {
            const ExecX &xd = xs[j];
            const XSmem x0{xa + xd.off, 0};
            for (int b = lane; b < xd.K / 32; b += 32) xa[xd.soff + b] = xblock_sum(x0.at(32 * b), 0, 0);
        }
        __syncwarp();
    }
}

// position of a warp in the item sequence: stage, tile index in the stage
// (this warp takes tiles gw, gw + nwarps, ...), op, matrix, chunk
struct ExecItem {
    int s, t, op, mat, chunk;
};

struct ExecTables {
    const ExecOp *ops;
    const ExecStage *stages;
    const ExecX *xs;
    int nstages;
};

__device__ __forceinline__ bool exec_locate(const ExecTables &T, ExecItem &it) {
    // find the op of tile t in stage s; false if t is past the stage's tiles
    const ExecStage &st = T.stages[it.s];
    if (it.t >= st.tiles) return false;
    int op = st.op_begin;
    while (op + 1 < st.op_end && T.ops[op + 1].tile_base <= it.t) ++op;
    it.op = op;
    return true;
}

__device__ __forceinline__ void exec_first_in_stage(const ExecTables &T, ExecItem &it, int s,
                                                    int gw, int nwarps) {
    it.s = s;
    const int t0 = gw - T.stages[s].tile_off;
    it.t = t0 < 0 ? t0 + nwarps : t0;
    it.mat = 0;
    it.chunk = 0;
    if (!exec_locate(T, it)) it.op = -1;
}

// advance within the current stage; false when the warp has no more items in it
__device__ __forceinline__ bool exec_next_in_stage(const ExecTables &T, ExecItem &it,
                                                   int nwarps) {
    const ExecOp &op = T.ops[it.op];
    if (++it.chunk < op.nchunks) return true;
    it.chunk = 0;
    if (++it.mat < op.nmat) return true;
    it.mat = 0;
    it.t += nwarps;
    return exec_locate(T, it);
}

// the producer side walks across stages
__device__ __forceinline__ bool exec_next_any(const ExecTables &T, ExecItem &it, int nwarps,
                                              int gw) {
    if (it.op >= 0 && exec_next_in_stage(T, it, nwarps)) return true;
    for (int s = it.s + 1; s < T.nstages; ++s) {
        exec_first_in_stage(T, it, s, gw, nwarps);
        if (it.op >= 0) return true;
    }
    it.s = T.nstages;
    it.op = -1;
    return false;
}

// bounded mbarrier wait that also returns (false) once the CTA is aborting
__device__ __forceinline__ bool exec_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity)) return true;
        if (*abort_flag || globaltimer() - t0 > limit_ns) return false;
    }
}

template <int QT>
__device__ __forceinline__ void exec_issue(const ExecTables &T, const ExecItem &it, uint8_t *slot,
                                           uint64_t *full, uint64_t pol, int lane) {
    constexpr int UB = Fmt<QT>::unit_bytes;
    const ExecOp &op = T.ops[it.op];
    const int tile = it.t - op.tile_base;
    const int row0 = tile * op.rpw;
    const int rows = min((int)op.rpw, op.M - row0);
    const int u0 = it.chunk * op.KCU;
    const int cnt = min((int)op.KCU, op.nsc - u0);
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

// Prefetch item `it`'s weight bytes into L2 (the same ranges exec_issue will
// copy later): more HBM requests in flight than the shared-memory ring holds.
template <int QT>
__device__ __forceinline__ void exec_prefetch(const ExecTables &T, const ExecItem &it, int lane) {
    constexpr int UB = Fmt<QT>::unit_bytes;
    const ExecOp &op = T.ops[it.op];
    const int tile = it.t - op.tile_base;
    const int row0 = tile * op.rpw;
    const int rows = min((int)op.rpw, op.M - row0);
    const int u0 = it.chunk * op.KCU;
    const int cnt = min((int)op.KCU, op.nsc - u0);
    const uint32_t rowb = (uint32_t)cnt * UB;
    const uint8_t *W = op.W[it.mat];
    if (op.single) {
        if (lane == 0) bulk_prefetch_l2(W + (size_t)row0 * op.rb, rowb * rows);
    } else if (lane < rows) {
        bulk_prefetch_l2(W + (size_t)(row0 + lane) * op.rb + (size_t)u0 * UB, rowb);
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
    const int XB = a.x_buffers;
    // control block: abort flag; per x buffer, warps done with its stage and
    // warps that entered its stage (per phase parity)
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem);
    int *done = reinterpret_cast<int *>(smem + 16);       // [EXEC_MAX_XBUF]
    int *entered = reinterpret_cast<int *>(smem + 64);    // [EXEC_MAX_XBUF][2]
    uint64_t *fulls = reinterpret_cast<uint64_t *>(smem + 256);  // nw * NSW weight slots
    uint64_t *xfull = reinterpret_cast<uint64_t *>(smem + a.xbar_off);  // [XB]: x copies landed
    uint64_t *xready = xfull + XB;                                       // [XB]: x normalised
    uint8_t *ring = smem + a.ring_off + (size_t)warp * a.NSW * a.slot_bytes;
    uint64_t *full = fulls + warp * a.NSW;

    // descriptor tables -> shared memory
    ExecTables T;
    {
        uint8_t *tab = smem + a.tab_off;
        const int ob = a.nops * (int)sizeof(ExecOp), xb = a.nxs * (int)sizeof(ExecX),
                  sb = a.nstages * (int)sizeof(ExecStage);
        for (int i = threadIdx.x; i < ob / 16; i += blockDim.x)
            reinterpret_cast<int4 *>(tab)[i] = __ldg(reinterpret_cast<const int4 *>(a.ops) + i);
        for (int i = threadIdx.x; i < xb / 16; i += blockDim.x)
            reinterpret_cast<int4 *>(tab + ob)[i] = __ldg(reinterpret_cast<const int4 *>(a.xs) + i);
        for (int i = threadIdx.x; i < sb / 16; i += blockDim.x)
            reinterpret_cast<int4 *>(tab + ob + xb)[i] =
                __ldg(reinterpret_cast<const int4 *>(a.stages) + i);
        T.ops = reinterpret_cast<const ExecOp *>(tab);
        T.xs = reinterpret_cast<const ExecX *>(tab + ob);
        T.stages = reinterpret_cast<const ExecStage *>(tab + ob + xb);
        T.nstages = a.nstages;
    }
    if (threadIdx.x == 0) {
        *abort_flag = 0;
        for (int b = 0; b < EXEC_MAX_XBUF; ++b) {
            done[b] = 0;
            entered[2 * b] = entered[2 * b + 1] = 0;
        }
        for (int b = 0; b < XB; ++b) {
            mbar_init(xfull + b, 32);
            mbar_init(xready + b, 1);
        }
    }
    if (lane == 0)
        for (int i = 0; i < a.NSW; ++i) mbar_init(full + i, 1);
    if (lane == 0) fence_mbar_init();
    __syncthreads();

    const uint64_t pol = l2_policy_evict_first();
    // weight ring: prefetch the first NSW items of this warp
    ExecItem pit;
    pit.s = -1;
    pit.op = -1;
    int issued = 0, consumed = 0;
    // L2 prefetch cursor, a.prefetch items ahead of the ring's copies
    ExecItem fit;
    fit.s = -1;
    fit.op = -1;
    bool fit_more = true;
    auto prefetch_next = [&]() {
        if (fit_more && (fit_more = exec_next_any(T, fit, nwarps, gw))) exec_prefetch<QT>(T, fit, lane);
    };
    auto issue_next = [&]() {
        if (!exec_next_any(T, pit, nwarps, gw)) return;
        exec_issue<QT>(T, pit, ring + (size_t)(issued % a.NSW) * a.slot_bytes,
                       full + issued % a.NSW, pol, lane);
        ++issued;
        prefetch_next();
    };
    for (int i = 0; i < a.NSW + a.prefetch; ++i) prefetch_next();
    for (int i = 0; i < a.NSW; ++i) issue_next();

    auto xbuf = [&](int s) {
        return reinterpret_cast<float *>(smem + a.x_off) + (size_t)(s % XB) * a.x_floats;
    };
    // the first XB stages' inputs (stage 0 never waits at a barrier; later
    // barrier stages are loaded after their barrier)
    if (warp == 0)
        for (int s = 0; s < XB && s < a.nstages; ++s)
            if (s == 0 || !T.stages[s].barrier)
                exec_load_x(T.stages[s], T.xs, xbuf(s), xfull + s % XB, lane);

    bool ok = true;
    for (int s = 0; s < a.nstages && ok; ++s) {
        const ExecStage &st = T.stages[s];
        const int b = s % XB;
        const uint32_t ph = (uint32_t)(s / XB) & 1u;
        // ---- enter stage s: the first warp in normalises x(s) and publishes it ----
        int first = 0;
        if (lane == 0) first = atomicAdd(entered + 2 * b + ph, 1) == 0;
        first = __shfl_sync(0xffffffffu, first, 0);
        if (first) {
            if (!__all_sync(0xffffffffu, exec_wait(xfull + b, ph, abort_flag, a.wait_ns))) {
                if (lane == 0) atomicOr(status, BQ_DEVERR_XFULL_WAIT);
                ok = false;
                break;
            }
            exec_norm_x_warp<QT>(st, T.xs, xbuf(s), lane);
            if (lane == 0) mbar_arrive(xready + b);
        }
        const float *xa = xbuf(s);

        // Every warp waits for x(s), even one without items in stage s: an
        // mbarrier wait only tells the current phase from the one before it,
        // so no warp may run ahead to a later phase of a buffer whose earlier
        // phase it has not seen complete.  Waiting here in stage order keeps
        // the warps of a CTA within XB stages of each other.
        if (!__all_sync(0xffffffffu, exec_wait(xready + b, ph, abort_flag, a.wait_ns))) {
            if (lane == 0) atomicOr(status, BQ_DEVERR_XREADY_WAIT);
            ok = false;
            break;
        }

        // ---- this warp's items of stage s ----
        ExecItem it;
        exec_first_in_stage(T, it, s, gw, nwarps);
        float p0 = -0.0f, p1 = -0.0f;
        while (it.op >= 0) {
            const ExecOp &op = T.ops[it.op];
            const int slot = consumed % a.NSW;
            if (!__all_sync(0xffffffffu, exec_wait(full + slot, (consumed / a.NSW) & 1, abort_flag, a.wait_ns))) {
                if (lane == 0) atomicOr(status, BQ_DEVERR_FULL_WAIT);
                ok = false;
                break;
            }
            const int G = op.G;
            const int rho = lane / G, l = lane & (G - 1);
            const int tile = it.t - op.tile_base;
            const int row0 = tile * op.rpw;
            const int rows = min((int)op.rpw, op.M - row0);
            const int u0 = it.chunk * op.KCU;
            const int cnt = min((int)op.KCU, op.nsc - u0);
            if (it.mat == 0 && it.chunk == 0) {
                p0 = -0.0f;
                p1 = -0.0f;
            }
            const XSmem xs{xa + op.xoff, 0, xa + op.soff, 0};
            if (op.rowmode) {
                // rows of this tile one by one, each by the whole warp; lane r
                // keeps row r's gate value between the two matrices of gate+up
                const uint8_t *base = ring + (size_t)slot * a.slot_bytes;
                for (int r = 0; r < rows; ++r) {
                    const float v = __shfl_sync(
                        0xffffffffu, row_dot_blockpar<QT>(base + (size_t)r * op.rb, op.nsc, G, xs, lane), 0);
                    if (op.nmat == 1) {
                        if (lane == 0) op.y[row0 + r] = op.bias ? __fadd_rn(v, op.bias[row0 + r]) : v;
                    } else if (it.mat == 0) {
                        if (lane == r) p0 = v;
                    } else {
                        const float gr = __shfl_sync(0xffffffffu, p0, r);
                        if (lane == 0) op.y[row0 + r] = silu_mul(gr, v);
                    }
                }
            } else {
                const uint8_t *stp = ring + (size_t)slot * a.slot_bytes + rho * op.row_stride;
                float acc = it.mat == 0 ? p0 : p1;
                if (rho < rows) {
                    for (int ul = l; ul < cnt; ul += G) {
                        uint32_t w[Fmt<QT>::unit_words];
                        load_unit_smem<QT>(w, stp + ul * UB);
                        const uint32_t *const ws[1] = {w};
                        float cc[1][1];
                        unit_dot<QT, 1, 1>(ws, 8, xs, (u0 + ul) * 256, cc);
                        acc = __fadd_rn(acc, cc[0][0]);
                    }
                }
                if (it.mat == 0) p0 = acc;
                else p1 = acc;
                if (it.chunk + 1 == op.nchunks && it.mat + 1 == op.nmat) {
                    const float g = fold_lanes(p0, G);
                    if (op.nmat == 2) {
                        const float u = fold_lanes(p1, G);
                        if (rho < rows && l == 0) op.y[row0 + rho] = silu_mul(g, u);
                    } else if (rho < rows && l == 0) {
                        op.y[row0 + rho] = op.bias ? __fadd_rn(g, op.bias[row0 + rho]) : g;
                    }
                }
            }
            __syncwarp();
            ++consumed;
            issue_next();  // refill the slot just consumed
            if (!exec_next_in_stage(T, it, nwarps)) break;
        }
        if (!ok) break;

        // ---- leave stage s: the last warp out starts the next loads ----
        __syncwarp();  // this warp's y stores of stage s precede its arrival
        int last = 0;
        if (lane == 0) {
            __threadfence_block();
            last = atomicAdd(done + b, 1) == nw - 1;
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (!last) continue;
        if (lane == 0) {
            done[b] = 0;             // next use: stage s + XB
            entered[2 * b + ph] = 0;  // next use: stage s + 2 XB
            __threadfence_block();
        }
        if (s + 1 < a.nstages && T.stages[s + 1].barrier) {
            // stage s+1 reads or overwrites earlier stages' data: every CTA must
            // be done with stages <= s before anyone loads its inputs
            int failed = 0;
            if (lane == 0) {
                __threadfence();  // this CTA's y stores (ordered by the done counter)
                asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(a.counters + s + 1)
                             : "memory");
            }
            __syncwarp();
            // the gains do not depend on earlier stages: their copies go out
            // once this CTA has arrived and land while the barrier propagates.
            // Buffer (s+1) % XB is free: this CTA is done with every stage <= s.
            exec_load_x(T.stages[s + 1], T.xs, xbuf(s + 1), xfull + (s + 1) % XB, lane, EXEC_LOAD_GAINS);
            if (lane == 0) {
                const uint64_t t0 = globaltimer();
                unsigned int n = 0;
                for (uint32_t i = 0;; ++i) {
                    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];"
                                 : "=r"(n)
                                 : "l"(a.counters + s + 1)
                                 : "memory");
                    if (n >= gridDim.x + a.barrier_extra) break;
                    if ((i & 63u) == 63u && (*abort_flag || globaltimer() - t0 > a.wait_ns)) {
                        failed = 1;
                        break;
                    }
                }
            }
            __syncwarp();  // the other lanes' copies below follow lane 0's acquire
            if (__shfl_sync(0xffffffffu, failed, 0)) {
                if (lane == 0) atomicOr(status, BQ_DEVERR_BARRIER_WAIT);
                ok = false;
                break;
            }
            // buffer (s+1) % XB is free: its previous stage (s+1-XB <= s) is done
            exec_load_x(T.stages[s + 1], T.xs, xbuf(s + 1), xfull + (s + 1) % XB, lane, EXEC_LOAD_X);
        }
        if (XB > 1 && s + XB < a.nstages && !T.stages[s + XB].barrier)
            exec_load_x(T.stages[s + XB], T.xs, xbuf(s + XB), xfull + b, lane);
        else if (XB == 1 && s + 1 < a.nstages && !T.stages[s + 1].barrier)
            exec_load_x(T.stages[s + 1], T.xs, xbuf(s + 1), xfull + b, lane);
    }

    if (!ok) {
        if (lane == 0) *abort_flag = 1;
        // no weight copy into this warp's ring may still be in flight at exit
        for (int i = consumed; i < issued; ++i)
            if (!mbar_wait_bounded(full + i % a.NSW, (i / a.NSW) & 1, a.wait_ns) && lane == 0)
                atomicOr(status, BQ_DEVERR_DRAIN_WAIT);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // nor any x copy
}

}  // namespace bq
