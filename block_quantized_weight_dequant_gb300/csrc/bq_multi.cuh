// bq_multi.cuh -- the streaming GEMV kernel: one launch for a list of
// INDEPENDENT GEMVs (a per-token weight stream whose ops read no output of
// another op of the list), or for one single call (decode GEMV, gate+up+SiLU,
// or the R-row verify GEMV).
//
// The tiles of all ops are concatenated in list order; a tile is the rows one
// warp evaluates at once (NR * 32/G rows, G lanes per row).  Each CTA takes a
// contiguous, byte-balanced range of tiles and its warps take the range's
// tiles round-robin.  Every warp feeds itself: it owns a ring of D shared-
// memory slots, issues the 1-D bulk copies (TMA) of its own next items into
// them and waits on each slot's mbarrier, sleeping in the wait (suspend-time
// hint) rather than spinning.  There is no producer warp and no hand-off
// between warps, so each warp keeps D - 1 items in flight while it decodes
// one.  An item is one K-chunk (KCU units) of one matrix of a tile.
//
// x phases.  All warps meet at the start of each op (or, in panel mode, each
// K-panel of the single op) to stage its x -- R input rows, RMSNorm-ed for
// gate+up -- into shared memory with 16-byte cp.async copies; the weight
// copies of the new op are already in flight by then.  With two x buffers the
// next phase's x is copied while the current phase computes.  Panel mode
// serves a verify call whose R x K input does not fit in shared memory: the
// op's K range is cut into panels of whole chunks, each warp holds at most one
// tile (its partial sums persist across panels), and the panels are staged in
// order.
//
// Single calls carry their one op in the kernel parameters ("inline"), so no
// descriptor table is needed; they are launched with programmatic dependent
// launch allowed: the kernel lets its dependents start at once, prefetches
// its first weight items into L2, and only then waits for the kernel before it
// in the stream (griddepcontrol.wait) before reading any input.  A prefetch is
// a hint that binds no value, so this is safe even if the kernel before wrote
// the weights.  But only this kernel lets its dependents start early, and it
// writes nothing but its outputs (and the error word): any other kernel
// before it completes before it starts.  So single calls, whose contract
// excludes packed weights written by an earlier GEMV call, and the stages of
// a staged plan after the first (the planner rejects outputs overlapping
// weights) copy their first weight items into the ring before the wait
// (early_ring) and compute as soon as their input is staged; the first
// stage of a plan falls under the single calls' contract.
//
// Arithmetic is bq_dot.cuh's fixed tree: every output is bit-identical to the
// single-op kernels and across R.
#pragma once

#include <cuda_runtime.h>

#include "bq_device.cuh"
#include "bq_dot.cuh"
#include "bq_internal.h"

namespace bq {

struct MultiOp {
    const uint8_t *W[2];
    const float *x;          // [R][K]
    const float *gamma;      // gate+up RMSNorm gain, or null
    float *y;                // [R][M]
    const float *bias;       // R = 1 plain GEMV: fp32[M] added to y, or null
    float eps;
    int M, K, rb, nsc;
    int G, rpw;              // lanes per row, rows per tile (NR * 32 / G)
    int KCU, nchunks, nmat;  // units per item row, items per tile and matrix, matrices (1 or 2)
    int ntiles, tile_base;   // tiles of this op; its first tile in the whole list
    int row_stride, single;  // slot bytes per tile row; rows copied as one block
    int rowmode;             // 1: a tile is rpw whole rows, each evaluated by the whole warp
    int umask;               // lane bits that form the unit column l (the rest form the row)
};

struct MultiArgs {
    const MultiOp *ops;    // op table in global memory (not used with an inline op)
    const int *cta_tiles;  // [grid + 1]: CTA c takes tiles [cta_tiles[c], cta_tiles[c+1])
    int nops;
    int nwarps, D, slot_bytes;  // warps per CTA, ring slots per warp, bytes per slot
    int x_off, ring_off;        // shared-memory offsets of the x buffers and the rings
    int nr, R;                  // weight rows per lane; input rows (1, or 2..6 for verify)
    int x_rstride;              // floats between staged input rows
    int x_floats;               // floats per x buffer
    int x_buffers;              // 1 or 2
    int panel_units;            // 0: an op's whole x is staged; else units of K per panel
    int gain_staged;            // 1: the buffers have room for the op's RMSNorm gain, which
                                // is staged with x (single gate+up calls); 0: read from L2
    int inline_op;              // 1: `op` is the only op; CTA c takes tiles [cT/grid, (c+1)T/grid)
    unsigned long long *cta_ns; // list mode: each CTA's duration in ns (plan tuning), or null
    unsigned long long wait_ns; // limit of every bounded wait
    int early_ring;             // 1: fill the weight rings before waiting for the kernel
                                // before (it is known to write no weights: an earlier
                                // stage of the same plan); 0: only prefetch the first
                                // items into L2 before the wait
    MultiOp op;
};

constexpr int MULTI_MAX_WARPS = 16;
// Warps per CTA at most, per instance: verify instances (R > 1) hold R partial
// sums per row and run at most 8 warps; Q8_0 decode runs at most 12 (its
// items are large, so shared memory allows about 12 anyway, and the bound
// leaves registers for the unrolled dot product); Q4_0 decode up to 16.
__host__ __device__ constexpr int multi_max_warps(int QT, int R) {
    return R > 1 ? 8 : QT == 8 ? 12 : MULTI_MAX_WARPS;
}
// floats after the R input rows of an x buffer that hold the rows' 32-element
// block sums (Q4_K; none for the other formats), rounded to 128 bytes
__host__ __device__ constexpr int multi_sum_floats(int QT, int R, int rstride) {
    return QT == QT_Q4_K ? (R * (rstride / 32) + 31) / 32 * 32 : 0;
}
// float offset in an x buffer of the staged RMSNorm gain (R = 1 gate+up: a
// plain copy after the input row and its block sums, when the planner sized
// the buffer for it)
__host__ __device__ constexpr int multi_gain_off(int QT, int R, int rstride) {
    return R * rstride + multi_sum_floats(QT, R, rstride);
}
static_assert(MULTI_MAX_WARPS * 32 <= 1024, "one CTA");
constexpr int MULTI_MAX_D = 4;
// shared memory header: mbarriers [0, 512), inline op [512, 768), reduction
// scratch [768, 1796), per-warp issuing state of the current op
// [MULTI_CUR_OFF, +64 per warp), abort flag at MULTI_ABORT_OFF, x buffers from
// MULTI_X_OFF
constexpr int MULTI_CUR_OFF = 1808;
constexpr int MULTI_ABORT_OFF = MULTI_CUR_OFF + 64 * MULTI_MAX_WARPS;
constexpr int MULTI_X_OFF = 2944;
static_assert(MULTI_ABORT_OFF + 4 <= MULTI_X_OFF && MULTI_X_OFF % 128 == 0, "header layout");
static_assert(sizeof(MultiOp) <= 256, "the inline op fits its header slot");

// One warp's position in its item sequence (tiles t = first, first + nwarps,
// ...; per tile its matrices, per matrix its K-chunks).  The fields of its op
// that issuing needs sit in a MultiCurOp, read from the op table only when
// the cursor enters a new op: the warp's own cursor keeps it in shared memory
// (one 64-byte slot per warp), which holds it out of the registers the dot
// product needs and lets gate+up items switch matrices without a global read.
struct MultiCursor {
    int t, op, m, c;
    const uint8_t *W;  // the current matrix (W[m] of the op)
};
struct MultiCurOp {
    const uint8_t *W[2];
    int rpw, tile_base, tile_end, M, KCU, rb, nchunks, nmat;
    int row_stride;  // slot bytes per tile row; negative: rows copied as one block
    int pad_[3];
};
static_assert(sizeof(MultiCurOp) == 64, "one 64-byte slot per warp");

// the op holding tile t, walking forward from op index `op`
__device__ __forceinline__ int multi_op_of(const MultiOp *ops, int nops, int t, int op) {
    while (op + 1 < nops && ops[op + 1].tile_base <= t) ++op;
    return op;
}

__device__ __forceinline__ void multi_load_op(const MultiOp *ops, MultiCursor &q, MultiCurOp &co) {
    const MultiOp &o = ops[q.op];
    q.W = o.W[0];
    co.W[0] = o.W[0];
    co.W[1] = o.W[1];
    co.rpw = o.rpw;
    co.tile_base = o.tile_base;
    co.tile_end = o.tile_base + o.ntiles;
    co.M = o.M;
    co.KCU = o.KCU;
    co.rb = o.rb;
    co.nchunks = o.nchunks;
    co.nmat = o.nmat;
    co.row_stride = o.single ? -1 : o.row_stride;
}

// the rows and byte range of the item under the cursor
struct MultiItem {
    const uint8_t *src;
    int rows;
    uint32_t rowb;
};
template <int QT>
__device__ __forceinline__ MultiItem multi_item(const MultiCursor &q, const MultiCurOp &co) {
    constexpr int UB = Fmt<QT>::unit_bytes;
    const int row0 = (q.t - co.tile_base) * co.rpw;
    const int b0 = q.c * co.KCU * UB;
    MultiItem it;
    it.rows = min(co.rpw, co.M - row0);
    it.rowb = (uint32_t)min(co.KCU * UB, co.rb - b0);
    it.src = q.W + (size_t)row0 * co.rb + b0;
    return it;
}

template <int QT>
__device__ __forceinline__ void multi_issue(const MultiCursor &q, const MultiCurOp &co, uint8_t *st,
                                            uint64_t *bar, uint64_t pol, int lane) {
    const MultiItem it = multi_item<QT>(q, co);
    const int row_stride = co.row_stride, rb = co.rb;
    // the slot's previous contents were read by this warp's generic loads
    __syncwarp();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (lane == 0) mbar_arrive_expect_tx(bar, it.rowb * it.rows);
    __syncwarp();
    if (row_stride < 0) {
        if (lane == 0) bulk_g2s(st, it.src, it.rowb * it.rows, bar, pol);
    } else {
        for (int r = lane; r < it.rows; r += 32)
            bulk_g2s(st + r * row_stride, it.src + (size_t)r * rb, it.rowb, bar, pol);
    }
}

// the same bytes into L2 only (a hint: no completion, no value bound)
template <int QT>
__device__ __forceinline__ void multi_prefetch(const MultiCursor &q, const MultiCurOp &co, int lane) {
    const MultiItem it = multi_item<QT>(q, co);
    if (co.row_stride < 0) {
        if (lane == 0) bulk_prefetch_l2(it.src, it.rowb * it.rows);
    } else {
        for (int r = lane; r < it.rows; r += 32) bulk_prefetch_l2(it.src + (size_t)r * co.rb, it.rowb);
    }
}

// The cursor walks a tile matrix by matrix, each matrix chunk by chunk;
// PAIR (the paired gate+up instance) walks it chunk by chunk, each chunk
// gate then up, so that the two items of a chunk land in consecutive slots.
template <bool PAIR>
__device__ __forceinline__ void multi_advance(const MultiOp *ops, int nops, int nwarps,
                                              MultiCursor &q, MultiCurOp &co) {
    if (PAIR) {
        if (++q.m < co.nmat) {
            q.W = co.W[1];
            return;
        }
        q.m = 0;
        q.W = co.W[0];
        if (++q.c < co.nchunks) return;
        q.c = 0;
    } else {
        if (++q.c < co.nchunks) return;
        q.c = 0;
        if (++q.m < co.nmat) {
            q.W = co.W[1];  // matrix 0 -> 1 (nmat is 1 or 2)
            return;
        }
        q.m = 0;
    }
    q.t += nwarps;
    if (q.t >= co.tile_end && q.op + 1 < nops) {
        q.op = multi_op_of(ops, nops, q.t, q.op);
        multi_load_op(ops, q, co);
    } else if (co.nmat > 1) {
        q.W = co.W[0];
    }
}

// bounded mbarrier wait that also gives up once another warp of the CTA has
// set the abort flag; the flag is read only when the data has not landed yet
__device__ __forceinline__ bool multi_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                           uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity)) return true;
        if (*abort_flag || globaltimer() - t0 > limit_ns) return false;
    }
}

// The row fold when virtual lane l of the group sits in hardware lane
// rho + stride * l (stride a power of two, stride * G <= 32): step o adds the
// partial of virtual lane l ^ o, exactly as fold_lanes does.
__device__ __forceinline__ float fold_lanes_strided(float v, int G, int stride) {
    for (int o = G >> 1; o > 0; o >>= 1)
        v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o * stride));
    return v;
}

// the bits of `lane` selected by `mask`, packed from bit 0 up
__device__ __forceinline__ int lane_bits(int lane, int mask) {
    int v = 0, k = 0;
#pragma unroll
    for (int b = 0; b < 5; ++b)
        if (mask >> b & 1) v |= (lane >> b & 1) << k++;
    return v;
}

// The row fold of fold_lanes when the G partials of a row sit in the lanes
// whose unit bits (umask) vary: the butterfly takes the unit bits from the
// highest to the lowest, i.e. virtual-lane offsets G/2, ..., 1, exactly as
// fold_lanes does (fp32 addition is commutative, so every lane of the row ends
// with the same bits).
__device__ __forceinline__ float fold_unit_lanes(float v, int umask) {
#pragma unroll
    for (int b = 4; b >= 0; --b)
        if (umask >> b & 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, 1 << b));
    return v;
}

__device__ __forceinline__ void cp_async_16(void *smem_dst, const void *gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)), "l"(gsrc)
                 : "memory");
}

// All threads: start the copies of elements [k0, k1) of every input row into
// an x buffer (permuted chunk layout of XSmem, relative to k0), and of the
// op's RMSNorm gain (plain layout at goff), in one group: both fetches are in
// flight together.
__device__ __forceinline__ void multi_stage_x(const MultiOp &o, int R, int k0, int k1, float *dst,
                                              int rstride, int goff, int tid, int nthr) {
    const int n4 = (k1 - k0) >> 2;
    for (int i = tid; i < R * n4; i += nthr) {
        const int r = i / n4, c = i - r * n4;
        cp_async_16(dst + r * rstride + 4 * x_chunk_pos(c), o.x + (size_t)r * o.K + k0 + 4 * c);
    }
    if (o.gamma && goff >= 0)  // gate+up: R = 1, whole K
        for (int c = tid; c < n4; c += nthr) cp_async_16(dst + goff + 4 * c, o.gamma + 4 * c);
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// NR: weight rows per lane; R: input rows.  A tile is NR * 32/G rows; lane
// (rho, l) of a warp takes rows rho, rho + 32/G, ... of the tile and units
// l, l + G, ... of each, so every x value it reads from shared memory serves
// NR weight rows.  Which lane bits form l and which form rho is the op's
// `umask`, chosen on the host per op: lanes of one unit column read the same
// x chunk, and a 16-byte shared-memory load whose lane quads read at most two
// distinct chunks takes half the cycles of one whose quads read four
// (measured on GB300); the slot's row stride keeps the weight reads of every
// quarter-warp on distinct bank groups.  NR = 0 is row mode (R = 1): a tile is rpw whole rows, each
// evaluated block-parallel by the whole warp (row_dot_blockpar: the same tree
// with one block per lane), for calls too small to keep every lane busy.
template <int QT, int NR, int R>
__global__ void __launch_bounds__(multi_max_warps(QT, R) * 32, 1)
    multi_kernel(const __grid_constant__ MultiArgs a, unsigned int *status) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);  // [nwarps][D]
    MultiOp *op_inline = reinterpret_cast<MultiOp *>(smem + 512);
    float *red = reinterpret_cast<float *>(smem + 768);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + MULTI_ABORT_OFF);
    constexpr int UB = Fmt<QT>::unit_bytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nthr = blockDim.x;
    // NR = 3 tags the paired gate+up instance: one weight row per lane of each
    // matrix, the gate and up items of a chunk evaluated in one pass over x
    constexpr bool PAIR = NR == 3;
    static_assert(!PAIR || R == 1, "gate+up pairs are single-row");

    // dependents may start now; they wait for this grid before reading
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (threadIdx.x == 0) {
        for (int i = 0; i < a.nwarps * a.D; ++i) mbar_init(full + i, 1);
        *abort_flag = 0;
        if (a.inline_op) *op_inline = a.op;
        fence_mbar_init();
    }
    __syncthreads();
    const MultiOp *ops = a.inline_op ? op_inline : a.ops;
    const int nops = a.inline_op ? 1 : a.nops;
    int t_begin, t_end;
    if (a.inline_op) {
        const long long T = op_inline->ntiles;
        t_begin = (int)(T * blockIdx.x / gridDim.x);
        t_end = (int)(T * (blockIdx.x + 1) / gridDim.x);
    } else {
        t_begin = a.cta_tiles[blockIdx.x];
        t_end = a.cta_tiles[blockIdx.x + 1];
    }
    if (t_begin >= t_end) return;

    uint64_t *wfull = full + warp * a.D;
    uint8_t *ring = smem + a.ring_off + (size_t)warp * a.D * a.slot_bytes;
    const uint64_t pol = l2_policy_evict_first();
    int op0 = 0;
    {
        int lo = 0, hi = nops - 1;  // last op with tile_base <= t_begin
        while (lo < hi) {
            const int mid = (lo + hi + 1) / 2;
            if (ops[mid].tile_base <= t_begin) lo = mid;
            else hi = mid - 1;
        }
        op0 = lo;
    }
    const int op_last = multi_op_of(ops, nops, t_end - 1, op0);

    MultiCurOp &co = reinterpret_cast<MultiCurOp *>(smem + MULTI_CUR_OFF)[warp];
    MultiCursor q;
    q.t = t_begin + warp;
    q.m = q.c = 0;
    q.op = multi_op_of(ops, nops, q.t, op0);
    multi_load_op(ops, q, co);
    // fill the ring with this warp's first D items: before the wait when the
    // kernel before writes no weights, else after it
    int issued = 0;
    auto fill_ring = [&]() {
        for (; issued < a.D && q.t < t_end; ++issued) {
            multi_issue<QT>(q, co, ring + (size_t)issued * a.slot_bytes, wfull + issued, pol, lane);
            multi_advance<PAIR>(ops, nops, a.nwarps, q, co);
        }
    };
    if (a.early_ring) {
        fill_ring();
    } else {
        // this warp's first items into L2 while the kernel before may still
        // run (a copy of the cursor with its own op state in registers)
        MultiCursor f = q;
        MultiCurOp fo = co;
        for (int i = 0; i < a.D && f.t < t_end; ++i) {
            multi_prefetch<QT>(f, fo, lane);
            multi_advance<PAIR>(ops, nops, a.nwarps, f, fo);
        }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint64_t t_start = a.cta_ns ? globaltimer() : 0;
    fill_ring();

    auto sync = []() { __syncthreads(); };
    auto xbuf = [&](int i) {
        return reinterpret_cast<float *>(smem + a.x_off) + (size_t)(i % a.x_buffers) * a.x_floats;
    };
    // the staged gain's offset in an x buffer (-1: not staged)
    const int goff = a.gain_staged ? multi_gain_off(QT, R, a.x_rstride) : -1;
    // panel mode exists only in the verify instances (R > 1)
    const int PU = R > 1 ? a.panel_units : 0;
    auto n_panels = [&](const MultiOp &o) { return PU ? (o.nsc + PU - 1) / PU : 1; };
    // x phase i = (op, panel); the first phase's copies start now
    {
        const MultiOp &o = ops[op0];
        multi_stage_x(o, R, 0, PU ? min(o.K, PU * 256) : o.K, xbuf(0), a.x_rstride, goff, threadIdx.x,
                      nthr);
    }

    int e = 0, landed = 0;  // items consumed (or skipped after an error); items seen landed
    int slot = 0;           // e mod D
    uint32_t par = 0;       // (e / D) mod 2: the phase parity of slot's next completion
    bool ok = true;
    int phase = 0;
    for (int op = op0; op <= op_last; ++op) {
        const MultiOp &o = ops[op];
        const float *gamma = o.gamma;
        const float *bias = o.bias;
        float *y = o.y;
        const int M = o.M, K = o.K, nsc = o.nsc, G = o.G, rpw = o.rpw, KCU = o.KCU;
        const int nchunks = o.nchunks, nmat = o.nmat, tile_base = o.tile_base, ntiles = o.ntiles;
        const int row_stride = o.row_stride;
        const int np = n_panels(o);
        const int lo = max(t_begin, tile_base), hi = min(t_end, tile_base + ntiles);
        // this warp's first tile in [lo, hi): (t - t_begin) mod nwarps == warp
        const int t_first = lo + ((warp - (lo - t_begin) % a.nwarps) + a.nwarps) % a.nwarps;
        // Q4_0 decode (R = 1) always takes the order with the row in the low
        // lane bits (its instance runs 16 warps at the 128-register cap, where
        // the general order measured slower); the others take the op's order
        constexpr bool ROWS_LOW = QT == QT_Q4_0 && R == 1;
        const int rg = 32 / G;
        const int umask = ROWS_LOW ? 0 : o.umask;
        const int rho = ROWS_LOW ? lane & (rg - 1) : lane_bits(lane, ~umask & 31);
        const int l = ROWS_LOW ? lane / rg : lane_bits(lane, umask);
        constexpr int NRA = PAIR ? 1 : NR ? NR : 1;
        float p0[NRA][R], p1[NRA];
        for (int pn = 0; pn < np; ++pn, ++phase) {
            // ---- x of this phase: landed, visible to all, and the other buffer free ----
            float *xa = xbuf(phase);
            asm volatile("cp.async.wait_all;" ::: "memory");
            sync();
            // the next phase's copies: at once into the other buffer, or, with
            // one buffer, after every warp is done with this phase (below)
            int nop = op, npn = pn + 1;
            if (npn == np) {
                nop = op + 1;
                npn = 0;
            }
            const bool has_next = nop <= op_last;
            auto stage_next = [&](float *dst) {
                const MultiOp &n = ops[nop];
                const int k0 = npn * PU * 256;
                const int k1 = PU ? min(n.K, k0 + PU * 256) : n.K;
                multi_stage_x(n, R, k0, k1, dst, a.x_rstride, goff, threadIdx.x, nthr);
            };
            if (has_next && a.x_buffers == 2) stage_next(xbuf(phase + 1));
            if (gamma) {
                // RMSNorm in place (R == 1, whole K): the fixed tree of rms_scale
                const float rs = rms_scale_at([xa](int k) { return xa[x_pos(k)]; }, K, o.eps, red,
                                              threadIdx.x, nthr, sync);
                for (int c = threadIdx.x; c < K / 4; c += nthr) {
                    float4 *p = reinterpret_cast<float4 *>(xa + 4 * x_chunk_pos(c));
                    const float4 v = *p;
                    const float4 g = goff >= 0 ? reinterpret_cast<const float4 *>(xa + goff)[c]
                                               : __ldg(reinterpret_cast<const float4 *>(gamma) + c);
                    *p = make_float4(__fmul_rn(__fmul_rn(v.x, rs), g.x), __fmul_rn(__fmul_rn(v.y, rs), g.y),
                                     __fmul_rn(__fmul_rn(v.z, rs), g.z), __fmul_rn(__fmul_rn(v.w, rs), g.w));
                }
                sync();
            }
            // Q4_K: the phase's 32-element x block sums, once per CTA, after
            // the input rows in the buffer (the planner sized it for them)
            float *xsums = xa + R * a.x_rstride;
            const int sstride = a.x_rstride / 32;
            if constexpr (QT == QT_Q4_K) {
                const int kcount = PU ? min(K - pn * PU * 256, PU * 256) : K;
                const int nblk = kcount / 32;
                const XSmem x0{xa, a.x_rstride};
                for (int i = threadIdx.x; i < R * nblk; i += nthr) {
                    const int r = i / nblk, b = i - r * nblk;
                    xsums[r * sstride + b] = xblock_sum(x0.at(32 * b), r, 0);
                }
                sync();
            }
            const XSmem xs{xa, a.x_rstride, xsums, sstride};
            const int k0u = pn * PU;  // first unit of the panel
            const int c_lo = PU ? k0u / KCU : 0;
            const int c_hi = PU ? min(nchunks, (k0u + PU) / KCU) : nchunks;

            for (int t = t_first; t < hi; t += a.nwarps) {
                const int row0 = (t - tile_base) * rpw;
                const int rows = min(rpw, M - row0);
                if (pn == 0) {
#pragma unroll
                    for (int v = 0; v < NRA; ++v) {
                        p1[v] = -0.0f;
#pragma unroll
                        for (int r = 0; r < R; ++r) p0[v][r] = -0.0f;
                    }
                }
                if constexpr (PAIR) {
                    // chunk c of the gate matrix and of the up matrix, in two
                    // consecutive slots; one pass over x gives both unit sums
                    // (each matrix's own tree, as unit_dot_rows promises)
                    auto wait_item = [&](int s, uint32_t p) {
                        if (!ok) return;
                        if (!__all_sync(0xffffffffu, multi_wait(wfull + s, p, abort_flag, a.wait_ns))) {
                            if (lane == 0) {
                                if (!*abort_flag) atomicOr(status, BQ_DEVERR_FULL_WAIT);
                                *abort_flag = 1;
                            }
                            ok = false;
                        } else {
                            ++landed;
                        }
                    };
                    auto next_slot = [&]() {
                        ++e;
                        slot = slot + 1 == a.D ? 0 : slot + 1;
                        par ^= slot == 0;
                    };
                    for (int c = c_lo; c < c_hi; ++c) {
                        const int sg = slot;
                        wait_item(slot, par);
                        next_slot();
                        const int su = slot;
                        wait_item(slot, par);
                        next_slot();
                        if (!ok) continue;
                        const int u0 = c * KCU;
                        const int cnt = min(KCU, nsc - u0);
                        const uint8_t *stg = ring + (size_t)sg * a.slot_bytes + rho * row_stride;
                        const uint8_t *stu = ring + (size_t)su * a.slot_bytes + rho * row_stride;
                        if (rho < rows) {
                            for (int ul = l; ul < cnt; ul += G) {
                                const uint8_t *up2[2] = {stg + ul * UB, stu + ul * UB};
                                float cc[2][1];
                                unit_dot_rows<QT, 2, 1>(up2, xs, (u0 + ul - k0u) * 256, cc);
                                p0[0][0] = __fadd_rn(p0[0][0], cc[0][0]);
                                p1[0] = __fadd_rn(p1[0], cc[1][0]);
                            }
                        }
                        // refill both slots, in the cursor's order
                        for (int k = 0; k < 2 && q.t < t_end; ++k) {
                            const int s = k == 0 ? sg : su;
                            multi_issue<QT>(q, co, ring + (size_t)s * a.slot_bytes, wfull + s, pol, lane);
                            multi_advance<PAIR>(ops, nops, a.nwarps, q, co);
                            ++issued;
                        }
                    }
                } else {
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    if (m >= nmat) break;
                    for (int c = c_lo; c < c_hi;
                         ++c, ++e, slot = slot + 1 == a.D ? 0 : slot + 1, par ^= slot == 0) {
                        if (ok) {
                            if (!__all_sync(0xffffffffu, multi_wait(wfull + slot, par, abort_flag, a.wait_ns))) {
                                if (lane == 0) {
                                    if (!*abort_flag) atomicOr(status, BQ_DEVERR_FULL_WAIT);
                                    *abort_flag = 1;
                                }
                                ok = false;
                            } else {
                                ++landed;
                            }
                        }
                        if (!ok) continue;
                        if constexpr (NR == 0) {
                            {
                                // whole rows, one by one, each block-parallel over the
                                // warp (same tree); lane r keeps row r's gate value
                                // between the two matrices of gate+up
                                const uint8_t *base = ring + (size_t)slot * a.slot_bytes;
                                for (int r = 0; r < rows; ++r) {
                                    const float v = __shfl_sync(
                                        0xffffffffu,
                                        row_dot_blockpar<QT>(base + (size_t)r * row_stride, nsc, G, xs,
                                                             lane),
                                        0);
                                    if (nmat == 1) {
                                        if (lane == 0) y[row0 + r] = bias ? __fadd_rn(v, bias[row0 + r]) : v;
                                    } else if (m == 0) {
                                        if (lane == r) p1[0] = v;
                                    } else {
                                        const float gr = __shfl_sync(0xffffffffu, p1[0], r);
                                        if (lane == 0) y[row0 + r] = silu_mul(gr, v);
                                    }
                                }
                                if (q.t < t_end) {
                                    multi_issue<QT>(q, co, ring + (size_t)slot * a.slot_bytes,
                                                    wfull + slot, pol, lane);
                                    multi_advance<PAIR>(ops, nops, a.nwarps, q, co);
                                    ++issued;
                                }
                                continue;
                            }
                        }
                        const int u0 = c * KCU;
                        const int cnt = min(KCU, nsc - u0);
                        const uint8_t *stp = ring + (size_t)slot * a.slot_bytes + rho * row_stride;
                        // rows past the tile's end read stale slot bytes; their
                        // results are dropped below
                        if (NR > 0 && rho < rows) {
                            for (int ul = l; ul < cnt; ul += G) {
                                const uint8_t *up[NRA];
#pragma unroll
                                for (int v = 0; v < NRA; ++v) up[v] = stp + v * rg * row_stride + ul * UB;
                                float cc[NRA][R];
                                unit_dot_rows<QT, NRA, R>(up, xs, (u0 + ul - k0u) * 256, cc);
#pragma unroll
                                for (int v = 0; v < NRA; ++v) {
                                    if (m == 0) {
#pragma unroll
                                        for (int r = 0; r < R; ++r) p0[v][r] = __fadd_rn(p0[v][r], cc[v][r]);
                                    } else {
                                        p1[v] = __fadd_rn(p1[v], cc[v][0]);
                                    }
                                }
                            }
                        }
                        // refill the slot just read with the item D places ahead
                        if (q.t < t_end) {
                            multi_issue<QT>(q, co, ring + (size_t)slot * a.slot_bytes, wfull + slot, pol,
                                            lane);
                            multi_advance<PAIR>(ops, nops, a.nwarps, q, co);
                            ++issued;
                        }
                    }
                }
                }
                if (!ok || pn + 1 < np || NR == 0) continue;
#pragma unroll
                for (int v = 0; v < NRA; ++v) {
                    const int row = rho + v * rg;
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        auto fold = [&](float x) {
                            return ROWS_LOW ? fold_lanes_strided(x, G, rg) : fold_unit_lanes(x, umask);
                        };
                        const float g = fold(p0[v][r]);
                        if (nmat == 2) {
                            const float u = fold(p1[v]);
                            if (row < rows && l == 0) y[row0 + row] = silu_mul(g, u);
                        } else if (row < rows && l == 0) {
                            y[(size_t)r * M + row0 + row] =
                                R == 1 && bias ? __fadd_rn(g, bias[row0 + row]) : g;
                        }
                    }
                }
            }
            if (has_next && a.x_buffers == 1) {
                sync();  // every warp is done reading this phase's x
                stage_next(xa);
            }
        }
    }

    // after an error: let this warp's copies still in flight land before exit
    if (!ok && lane == 0)
        for (int i = landed; i < issued; ++i)
            if (!mbar_wait_bounded(wfull + i % a.D, (i / a.D) & 1, a.wait_ns))
                atomicOr(status, BQ_DEVERR_DRAIN_WAIT);
    asm volatile("cp.async.wait_all;" ::: "memory");  // nor any x copy
    if (a.cta_ns) {
        __syncthreads();
        if (threadIdx.x == 0) a.cta_ns[blockIdx.x] = globaltimer() - t_start;
    }
}

}  // namespace bq
