// bq_multi.cuh -- one launch for a list of INDEPENDENT GEMVs (a per-token
// weight stream whose ops read no output of another op of the list).
//
// The tiles of all ops are concatenated in list order; a tile is the rows one
// warp evaluates at once (32 / G rows, G lanes per row).  Each CTA takes a
// contiguous, byte-balanced range of tiles and its warps take the range's
// tiles round-robin.  Every warp feeds itself: it owns a ring of D shared-
// memory slots, issues the 1-D bulk copies (TMA) of its own next items into
// them and waits on each slot's mbarrier.  There is no producer warp and no
// hand-off between warps, so each warp keeps D - 1 items in flight while it
// decodes one.  An item is one K-chunk (KCU units) of one matrix of a tile.
// When the range enters a new op, all warps meet at a barrier and stage the
// op's (RMSNorm-ed) x into shared memory; the copies of the new op's weights
// are already in flight by then.  Arithmetic is bq_dot.cuh's fixed tree:
// every output is bit-identical to the single-op kernels.
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
    int G, rpw;              // lanes per row, rows per tile (NR * 32 / G)
    int KCU, nchunks, nmat;  // units per item row, items per tile and matrix, matrices (1 or 2)
    int ntiles, tile_base;   // tiles of this op; its first tile in the whole list
    int row_stride, single;  // slot bytes per tile row; rows copied as one block
};

struct MultiArgs {
    const MultiOp *ops;
    const int *cta_tiles;  // [grid + 1]: CTA c takes tiles [cta_tiles[c], cta_tiles[c+1])
    int nops;
    int nwarps, D, slot_bytes;  // warps per CTA, ring slots per warp, bytes per slot
    int x_off, ring_off;
    int nr;                     // weight rows per lane (the kernel's NR)
};

constexpr int MULTI_MAX_WARPS = 16;
constexpr int MULTI_MAX_D = 4;
// shared memory header: mbarriers [0, 512), reduction scratch [768, 1796),
// abort flag at 2040, x from MULTI_X_OFF
constexpr int MULTI_X_OFF = 2048;

// One warp's position in its item sequence (tiles t = first, first + nwarps,
// ...; per tile its matrices, per matrix its K-chunks) together with the
// fields of its op that issuing needs, read from the table only when the
// cursor enters a new op.
struct MultiCursor {
    int t, op, m, c;
    const uint8_t *W0, *W1;
    int rpw, tile_base, tile_end, M, KCU, nsc, rb, nchunks, nmat, single, row_stride;
};

// the op holding tile t, walking forward from op index `op`
__device__ __forceinline__ int multi_op_of(const MultiArgs &a, int t, int op) {
    while (op + 1 < a.nops && __ldg(&a.ops[op + 1].tile_base) <= t) ++op;
    return op;
}

__device__ __forceinline__ void multi_load_op(const MultiArgs &a, MultiCursor &q) {
    const MultiOp &o = a.ops[q.op];
    q.W0 = reinterpret_cast<const uint8_t *>(__ldg(reinterpret_cast<const unsigned long long *>(&o.W[0])));
    q.W1 = reinterpret_cast<const uint8_t *>(__ldg(reinterpret_cast<const unsigned long long *>(&o.W[1])));
    q.rpw = __ldg(&o.rpw);
    q.tile_base = __ldg(&o.tile_base);
    q.tile_end = q.tile_base + __ldg(&o.ntiles);
    q.M = __ldg(&o.M);
    q.KCU = __ldg(&o.KCU);
    q.nsc = __ldg(&o.nsc);
    q.rb = __ldg(&o.rb);
    q.nchunks = __ldg(&o.nchunks);
    q.nmat = __ldg(&o.nmat);
    q.single = __ldg(&o.single);
    q.row_stride = __ldg(&o.row_stride);
}

template <int QT>
__device__ __forceinline__ void multi_issue(const MultiCursor &q, uint8_t *st, uint64_t *bar,
                                            uint64_t pol, int lane) {
    constexpr int UB = Fmt<QT>::unit_bytes;
    const int row0 = (q.t - q.tile_base) * q.rpw;
    const int rows = min(q.rpw, q.M - row0);
    const int u0 = q.c * q.KCU;
    const uint32_t rowb = (uint32_t)min(q.KCU, q.nsc - u0) * UB;
    const uint8_t *W = q.m ? q.W1 : q.W0;
    // the slot's previous contents were read by this warp's generic loads
    __syncwarp();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (lane == 0) mbar_arrive_expect_tx(bar, rowb * rows);
    __syncwarp();
    if (q.single) {
        if (lane == 0) bulk_g2s(st, W + (size_t)row0 * q.rb, rowb * rows, bar, pol);
    } else {
        for (int r = lane; r < rows; r += 32)
            bulk_g2s(st + r * q.row_stride, W + (size_t)(row0 + r) * q.rb + (size_t)u0 * UB, rowb,
                     bar, pol);
    }
}

__device__ __forceinline__ void multi_advance(const MultiArgs &a, MultiCursor &q) {
    if (++q.c < q.nchunks) return;
    q.c = 0;
    if (++q.m < q.nmat) return;
    q.m = 0;
    q.t += a.nwarps;
    if (q.t >= q.tile_end && q.op + 1 < a.nops) {
        q.op = multi_op_of(a, q.t, q.op);
        multi_load_op(a, q);
    }
}

// NR: weight rows per lane.  A tile is NR * 32/G rows; lane (rho, l) of a
// warp takes rows rho, rho + 32/G, ... of the tile and units l, l + G, ... of
// each, so every x value it reads from shared memory serves NR rows.
template <int QT, int NR>
__global__ void __launch_bounds__(MULTI_MAX_WARPS * 32, 1)
    multi_kernel(const MultiArgs a, unsigned int *status) {
    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);  // [nwarps][D]
    float *red = reinterpret_cast<float *>(smem + 768);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + 2040);
    float *xsm = reinterpret_cast<float *>(smem + a.x_off);
    constexpr int UB = Fmt<QT>::unit_bytes;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nthr = blockDim.x;
    const int t_begin = a.cta_tiles[blockIdx.x], t_end = a.cta_tiles[blockIdx.x + 1];

    if (threadIdx.x == 0) {
        for (int i = 0; i < a.nwarps * a.D; ++i) mbar_init(full + i, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (t_begin >= t_end) return;

    uint64_t *wfull = full + warp * a.D;
    uint8_t *ring = smem + a.ring_off + (size_t)warp * a.D * a.slot_bytes;
    const uint64_t pol = l2_policy_evict_first();
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
    const int op_last = multi_op_of(a, t_end - 1, op0);

    // fill the ring with this warp's first D items
    MultiCursor q;
    q.t = t_begin + warp;
    q.m = q.c = 0;
    q.op = multi_op_of(a, q.t, op0);
    multi_load_op(a, q);
    int issued = 0;
    for (; issued < a.D && q.t < t_end; ++issued) {
        multi_issue<QT>(q, ring + (size_t)issued * a.slot_bytes, wfull + issued, pol, lane);
        multi_advance(a, q);
    }

    int e = 0, landed = 0;  // items consumed (or skipped after an error); items seen landed
    bool ok = true;
    auto sync = []() { __syncthreads(); };
    for (int op = op0; op <= op_last; ++op) {
        const MultiOp &o = a.ops[op];
        const float *x = o.x, *gamma = o.gamma;
        float *y = o.y;
        const int M = o.M, K = o.K, nsc = o.nsc, G = o.G, rpw = o.rpw, KCU = o.KCU;
        const int nchunks = o.nchunks, nmat = o.nmat, tile_base = o.tile_base, ntiles = o.ntiles;
        const int row_stride = o.row_stride;
        // every warp is done with the previous op's x: stage this op's
        sync();
        float rs = 1.0f;
        if (gamma) rs = rms_scale(x, K, o.eps, red, threadIdx.x, nthr, sync);
        for (int k = 4 * threadIdx.x; k < K; k += 4 * nthr) {
            float4 v = __ldg(reinterpret_cast<const float4 *>(x + k));
            if (gamma) {
                const float4 g = __ldg(reinterpret_cast<const float4 *>(gamma + k));
                v = make_float4(__fmul_rn(__fmul_rn(v.x, rs), g.x), __fmul_rn(__fmul_rn(v.y, rs), g.y),
                                __fmul_rn(__fmul_rn(v.z, rs), g.z), __fmul_rn(__fmul_rn(v.w, rs), g.w));
            }
            *reinterpret_cast<float4 *>(xsm + 4 * x_chunk_pos(k >> 2)) = v;
        }
        sync();

        const int lo = max(t_begin, tile_base), hi = min(t_end, tile_base + ntiles);
        // this warp's first tile in [lo, hi): (t - t_begin) mod nwarps == warp
        int t = lo + ((warp - (lo - t_begin) % a.nwarps) + a.nwarps) % a.nwarps;
        const int rho = lane / G, l = lane & (G - 1), rg = 32 / G;
        const XSmem xs{xsm, 0};
        for (; t < hi; t += a.nwarps) {
            const int row0 = (t - tile_base) * rpw;
            const int rows = min(rpw, M - row0);
            float p0[NR], p1[NR];
#pragma unroll
            for (int r = 0; r < NR; ++r) p0[r] = p1[r] = -0.0f;
#pragma unroll
            for (int m = 0; m < 2; ++m) {
                if (m >= nmat) break;
                for (int c = 0; c < nchunks; ++c, ++e) {
                    const int slot = e % a.D;
                    if (ok) {
                        if (*abort_flag) {
                            ok = false;
                        } else if (!__all_sync(0xffffffffu,
                                               mbar_wait_bounded(wfull + slot, (e / a.D) & 1))) {
                            if (lane == 0) {
                                *abort_flag = 1;
                                atomicOr(status, BQ_DEVERR_FULL_WAIT);
                            }
                            ok = false;
                        } else {
                            ++landed;
                        }
                    }
                    if (!ok) continue;
                    const int u0 = c * KCU;
                    const int cnt = min(KCU, nsc - u0);
                    const uint8_t *stp = ring + (size_t)slot * a.slot_bytes + rho * row_stride;
                    // rows past the tile's end read stale slot bytes; their
                    // results are dropped below
                    if (rho < rows) {
                        for (int ul = l; ul < cnt; ul += G) {
                            const uint8_t *up[NR];
#pragma unroll
                            for (int r = 0; r < NR; ++r) up[r] = stp + r * rg * row_stride + ul * UB;
                            float cc[NR];
                            unit_dot_rows<QT, NR>(up, xs, (u0 + ul) * 256, cc);
#pragma unroll
                            for (int r = 0; r < NR; ++r) {
                                if (m == 0) p0[r] = __fadd_rn(p0[r], cc[r]);
                                else p1[r] = __fadd_rn(p1[r], cc[r]);
                            }
                        }
                    }
                    // refill the slot just read with the item D places ahead
                    if (q.t < t_end) {
                        multi_issue<QT>(q, ring + (size_t)slot * a.slot_bytes, wfull + slot, pol,
                                        lane);
                        multi_advance(a, q);
                        ++issued;
                    }
                }
            }
            if (!ok) continue;
#pragma unroll
            for (int r = 0; r < NR; ++r) {
                const float g = fold_lanes(p0[r], G);
                const int row = rho + r * rg;
                if (nmat == 2) {
                    const float u = fold_lanes(p1[r], G);
                    if (row < rows && l == 0) y[row0 + row] = silu_mul(g, u);
                } else if (row < rows && l == 0) {
                    y[row0 + row] = g;
                }
            }
        }
    }

    // after an error: let this warp's copies still in flight land before exit
    if (!ok && lane == 0)
        for (int i = landed; i < issued; ++i)
            if (!mbar_wait_bounded(wfull + i % a.D, (i / a.D) & 1))
                atomicOr(status, BQ_DEVERR_DRAIN_WAIT);
}

}  // namespace bq
