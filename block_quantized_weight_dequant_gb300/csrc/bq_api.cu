// bq_api.cu -- the extern "C" entry points of libbqgemv.so (include/bqgemv.h):
// argument validation, launch planning and dispatch to the per-format
// kernels.  Validation runs entirely on the host before any CUDA call, so a
// rejected call touches no device state.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>
#include <algorithm>
#include <vector>

#include "../../include/bqgemv.h"
#include "bq_dot.cuh"
#include "bq_exec.cuh"
#include "bq_multi.cuh"
#include "bq_internal.h"

namespace bq {

namespace {

constexpr long long K_MAX = 1LL << 18;
constexpr long long M_MAX = (1LL << 31) - 1;

// limit of the kernels' bounded waits (passed with every launch); a hook for
// the tests can shorten it
std::atomic<unsigned long long> g_wait_ns{BQ_WAIT_LIMIT_NS};
// how plans of dependent stages run, for plans created from now on: -1 by
// the tunable, 0 the cooperative executor, 1 one launch per stage (a hook
// for the tests, which cover both)
std::atomic<int> g_plan_kind{-1};

// launch-geometry defaults; BQ_PLAN="md=3,mw=8,pdl=0"
// overrides them for tuning sweeps (read once)
struct Tunables {
    int exec_slot = 0;     // stream executor: bytes per ring slot (0 = one warp tile of 32 units)
    int exec_nsw = 0;      // stream executor: slots per warp (0 = as many as fit, <= 4)
    int exec_warps = 8;    // stream executor: warps per CTA
    int exec_rowmode_rows = 4;  // stream executor: row mode up to this many rows per warp (0: off)
    int exec_rowmode_nsc = 12;  // ... for rows of at most this many units (measured on GB300: the
                                // chained Q8_0 token, K <= 3072, 657 GB/s in row mode against 591
                                // without; the chained 7B Q4_0 token, K = 3584 and 18944, 1278
                                // with unit-per-lane tiles against 1170 in row mode)
    int exec_prefetch = 0;      // stream executor: L2 prefetch distance beyond the ring, in items (measured: no gain)
    int multi = 1;              // independent op lists: multi-op streaming kernel (0: executor)
    int multi_warps = 0;        // multi-op kernel: warps per CTA (0: as many as fit, <= 16)
    int multi_d = 2;            // multi-op kernel: ring slots per warp
    int multi_nr = 1;           // multi-op kernel: weight rows per lane (1 or 2)
    int multi_x2_max = 32 * 1024;    // op lists: two x buffers when together at most this
    int single_x_max = 128 * 1024;   // single calls: largest staged R x K input (else panels)
    int single_pdl = 1;              // single calls: allow programmatic dependent launch
    int gu_pair = 1;                 // single gate+up calls: the paired instance (1: Q8_0, 2: Q8_0
                                     // and Q4_0, 0: off; measured on GB300, 3072x1024 Q8_0 calls
                                     // 1039 -> 1160 GB/s)
    int single_early = 1;            // single calls: fill the weight rings before waiting for
                                     // the kernel before (only this library's streaming kernel
                                     // starts its dependents early, and it writes no weights;
                                     // measured on GB300: 3072x1024 Q8_0 GEMV 781 -> 827 GB/s,
                                     // gate+up 962 -> 1015, verify R = 1 2481 -> 2557)
    int single_rowmode = 2;          // single calls: row mode up to this many unit tiles per SM (0: off;
                                     // measured on GB300 with the early ring fill: 3072x1024 Q8_0
                                     // GEMV 824 GB/s at 4, 947 at 2 or less; chained Qwen3-0.6B
                                     // token 1014 at 4 or 2, 999 at 1 or 0)
    int verify_nr = 0;               // verify calls (R > 1): weight rows per lane (1 or 2; 0: by R)
    int plan_pdl = 0;                // op-list plans: allow programmatic dependent launch
    int plan_early = 1;              // staged plans: stages after the first fill their weight
                                     // rings before waiting for the stage before (measured on
                                     // GB300, chained tokens: Qwen3-0.6B-shaped Q8_0 950 ->
                                     // 1013 GB/s, 7B-shaped Q4_0 2476 -> 2539; with an L2
                                     // prefetch of the next items as well: 1011 and 2444)
    int plan_staged = 1;             // dependent op lists: one streaming-kernel launch per stage,
                                     // chained by programmatic dependent launch (0: the cooperative
                                     // executor, one launch with grid-wide barriers)
    int tree_waste = 8;              // the tree's lanes G leave at most 1/tree_waste of slots idle
    int verify_wave = 1;             // verify panels: two rows per lane when one needs two waves
    int short_lists = 1;             // op lists with few tiles per SM: only the warps they need
    int split_by_op = 1;             // op lists with at most half as many ops as CTAs: CTAs of
                                     // each op's own (no CTA meets an op boundary)
};

const Tunables &tunables() {
    static Tunables t = [] {
        Tunables v;
        const char *s = std::getenv("BQ_PLAN");
        if (!s) return v;
        char buf[256];
        std::strncpy(buf, s, sizeof buf - 1);
        buf[sizeof buf - 1] = 0;
        for (char *tok = std::strtok(buf, ","); tok; tok = std::strtok(nullptr, ",")) {
            char *eq = std::strchr(tok, '=');
            if (!eq) continue;
            *eq = 0;
            const int val = std::atoi(eq + 1);
            if (!std::strcmp(tok, "slot") && val >= 4096) v.exec_slot = val;
            else if (!std::strcmp(tok, "nsw") && val >= 2 && val <= 8) v.exec_nsw = val;
            else if (!std::strcmp(tok, "ewarps") && val >= 1 && val <= 8) v.exec_warps = val;
            else if (!std::strcmp(tok, "rowmode") && val >= 0 && val <= 32) v.exec_rowmode_rows = val;
            else if (!std::strcmp(tok, "rownsc") && val >= 1) v.exec_rowmode_nsc = val;
            else if (!std::strcmp(tok, "pf") && val >= 0 && val <= 16) v.exec_prefetch = val;
            else if (!std::strcmp(tok, "multi") && val >= 0 && val <= 1) v.multi = val;
            else if (!std::strcmp(tok, "mw") && val >= 1 && val <= 16) v.multi_warps = val;
            else if (!std::strcmp(tok, "md") && val >= 2 && val <= 4) v.multi_d = val;
            else if (!std::strcmp(tok, "mnr") && (val == 1 || val == 2)) v.multi_nr = val;
            else if (!std::strcmp(tok, "x2") && val >= 0) v.multi_x2_max = val;
            else if (!std::strcmp(tok, "sx") && val >= 16384) v.single_x_max = val;
            else if (!std::strcmp(tok, "pdl") && val >= 0 && val <= 1) v.single_pdl = val;
            else if (!std::strcmp(tok, "searly") && val >= 0 && val <= 1) v.single_early = val;
            else if (!std::strcmp(tok, "gupair") && val >= 0 && val <= 2) v.gu_pair = val;
            else if (!std::strcmp(tok, "srow") && val >= 0 && val <= 64) v.single_rowmode = val;
            else if (!std::strcmp(tok, "vnr") && (val == 1 || val == 2)) v.verify_nr = val;
            else if (!std::strcmp(tok, "waste") && val >= 2 && val <= 64) v.tree_waste = val;
            else if (!std::strcmp(tok, "vwave") && val >= 0 && val <= 1) v.verify_wave = val;
            else if (!std::strcmp(tok, "opsplit") && val >= 0 && val <= 1) v.split_by_op = val;
            else if (!std::strcmp(tok, "short") && val >= 0 && val <= 1) v.short_lists = val;
            else if (!std::strcmp(tok, "ppdl") && val >= 0 && val <= 1) v.plan_pdl = val;
            else if (!std::strcmp(tok, "staged") && val >= 0 && val <= 1) v.plan_staged = val;
            else if (!std::strcmp(tok, "early") && val >= 0 && val <= 1) v.plan_early = val;
        }
        return v;
    }();
    return t;
}

int num_sms_current() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int n = cache[dev].load();
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev].store(n);
    }
    return n;
}

int max_smem_optin() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    int n = cache[dev].load();
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return 0;
        cache[dev].store(n);
    }
    return n;
}

// bytes per 32 weights (a Q4_K super-block is 144 bytes per 256 weights)
int block_bytes(int qtype) {
    return qtype == BQ_Q8_0 ? 34 : qtype == BQ_Q4_0 || qtype == BQ_Q4_K ? 18 : -1;
}
bool known_qtype(int qtype) { return block_bytes(qtype) > 0; }
// K granularity of a format: 32 weights per block, 256 per Q4_K super-block
int k_step(int qtype) { return qtype == BQ_Q4_K ? 256 : 32; }

}  // namespace

int tree_lanes_for_units(long long nsc) {
    const int den = tunables().tree_waste;
    for (int G = 32; G > 1; G >>= 1) {
        const long long slots = G * ((nsc + G - 1) / G);
        if ((slots - nsc) * den <= slots) return G;
    }
    return 1;
}

void plan_gemv(const GemvCall &c, LaunchPlan *p) {
    const long long nb = c.K / 32;
    p->G = tree_lanes_for_units((nb + 7) / 8);
    p->rb = nb * block_bytes(c.qtype);
}

// padded shared-memory row stride for `bytes` of units: conflict-free LDS.128
// when fewer than 8 lanes share a row (the stream executor's lane order, lane
// = rho * G + l)
int padded_stride(int bytes, int G) {
    int s16 = bytes / 16;
    if (G < 8)
        while (s16 % 8 != G % 8) ++s16;
    return s16 * 16;
}

// Lane order of the multi-op kernel (see bq_multi.cuh): bit b of `umask` set
// means bit b of the lane index is a bit of the lane's unit column l (the
// set bits, low to high, are l's bits); the other lane bits give the row rho.
// Two conditions, both for 16-byte shared-memory loads on GB300:
//  - x reads: the lanes of one unit column read the same x chunk, and a load
//    takes 2 cycles when every lane quad reads at most two distinct chunks
//    (4 when a quad reads four), so at most one of lane bits 0, 1 is a unit bit;
//  - weight reads: lane (rho, l) reads chunk rho*S + l*U + k of the slot (S the
//    row stride and U the unit, in 16-byte chunks); the 8 lanes of each
//    quarter-warp must hit 8 distinct bank groups (chunk mod 8).
static int pext5(int v, int m) {
    int r = 0, k = 0;
    for (int b = 0; b < 5; ++b)
        if (m >> b & 1) r |= (v >> b & 1) << k++;
    return r;
}
static bool lane_order_ok(int m, int G, int S, int U) {
    int ub = 0;
    while ((1 << ub) < G) ++ub;
    if (__builtin_popcount((unsigned)m) != ub) return false;
    for (int q = 0; q < 4; ++q) {
        int seen = 0;
        for (int ln = 8 * q; ln < 8 * q + 8; ++ln)
            seen |= 1 << ((pext5(ln, ~m & 31) * S + pext5(ln, m) * U) % 8);
        if (seen != 0xFF) return false;
    }
    for (int q = 0; q < 8; ++q) {
        int ls = 0;
        for (int ln = 4 * q; ln < 4 * q + 4; ++ln) ls |= 1 << pext5(ln, m);
        if (__builtin_popcount((unsigned)ls) > 2) return false;
    }
    return true;
}
// Choose the slot row stride S >= S0 (chunks) and a lane order for G unit
// columns that meets both conditions: S = S0 only when `pad` is false.  The
// candidates put rows in lane bits 0..2 (S odd), row/unit/row (S = 2 mod 4)
// or row/unit/unit (S = 4 mod 8).  Q4_0 (`rows_low`) has the single order with
// the row in the low lane bits, which its kernel instance computes by shifts.
// False when none fits.
bool lane_order(int G, int S0, int U, bool pad, int *S, int *umask, bool rows_low) {
    int ub = 0;
    while ((1 << ub) < G) ++ub;
    const int rb = 5 - ub;
    int cand[3], nc = 0;
    if (rows_low) {
        cand[nc++] = ((G - 1) << rb) & 31;
    } else {
        if (rb >= 3) cand[nc++] = ((G - 1) << rb) & 31;
        if (ub >= 1 && rb >= 2) cand[nc++] = 0x2 | (((1 << (ub - 1)) - 1) << 3);
        if (ub >= 2 && rb >= 1) cand[nc++] = (G - 1) << 1;
    }
    for (int s = S0; s < S0 + (pad ? 8 : 1); ++s)
        for (int i = 0; i < nc; ++i)
            if (lane_order_ok(cand[i], G, s, U)) {
                *S = s;
                *umask = cand[i];
                return true;
            }
    return false;
}
// The same, falling back (one row per tile, G = 32) to the unit column in the
// low lane bits: every quarter-warp then reads 8 units of one row, which is
// conflict-free for any S, and x loads take 4 cycles.
void lane_order_any(int G, int S0, int U, int *S, int *umask, bool rows_low) {
    if (lane_order(G, S0, U, true, S, umask, rows_low)) return;
    *S = S0;
    *umask = G - 1;
}

namespace {
struct Range {
    uintptr_t lo, hi;  // [lo, hi)
};
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }
Range range(const void *p, int64_t bytes) {
    const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
    return Range{lo, lo + (uintptr_t)bytes};
}
}  // namespace

bq_status plan_exec_tables(int qtype, const bq_op *ops, int n_ops, ExecOp *eo, ExecX *ex,
                           ExecStage *es, ExecGeometry *geo) {
    const Tunables &t = tunables();
    const int bb = block_bytes(qtype), ub = 8 * bb;
    if (bb < 0) return BQ_ERR_QTYPE;
    // a slot holds at least one warp tile of one unit per lane (32 units; the
    // row stride of KCU = G units needs no bank padding, as 17 and 9 are 1 mod 8)
    const int slot = (std::max(t.exec_slot, 32 * ub) + 127) / 128 * 128;
    // ---- pass 1: validate; stages and their distinct inputs ----
    int n_stages = 0, n_x = 0;
    int x_area = 0, stage_x = 0;  // floats: largest stage, current stage
    for (int i = 0; i < n_ops; ++i) {
        const bq_op &o = ops[i];
        if (o.kind != BQ_OP_GEMV && o.kind != BQ_OP_GATE_UP_SILU) return BQ_ERR_SHAPE;
        if (i == 0 ? o.stage != 0 : (o.stage != ops[i - 1].stage && o.stage != ops[i - 1].stage + 1))
            return BQ_ERR_SHAPE;
        if (o.M < 1 || o.M > M_MAX || o.K < 256 || o.K > K_MAX || o.K % 256) return BQ_ERR_SHAPE;
        const bool gu = o.kind == BQ_OP_GATE_UP_SILU;
        if (!o.W || !o.x || !o.y || (gu && !o.W_up)) return BQ_ERR_NULL;
        auto al = [](const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; };
        if (!al(o.W, 16) || !al(o.x, 16) || !al(o.y, 4) || (gu && !al(o.W_up, 16)) ||
            (gu && o.gamma && !al(o.gamma, 16)))
            return BQ_ERR_ALIGN;
        if (gu && o.gamma && !(std::isfinite(o.eps) && o.eps >= 0.0f)) return BQ_ERR_SHAPE;
        if (gu && o.bias) return BQ_ERR_SHAPE;  // gate+up takes no bias
        if (o.bias && !al(o.bias, 4)) return BQ_ERR_ALIGN;
        ExecOp &e = eo[i];
        std::memset(&e, 0, sizeof e);
        e.W[0] = static_cast<const uint8_t *>(o.W);
        e.W[1] = gu ? static_cast<const uint8_t *>(o.W_up) : nullptr;
        e.y = o.y;
        e.bias = gu ? nullptr : o.bias;
        e.nmat = gu ? 2 : 1;
        e.M = (int)o.M;
        e.nsc = (int)(o.K / 256);
        e.G = (unsigned char)tree_lanes_for_units(e.nsc);
        e.rb = e.nsc * ub;
        if (i == 0 || o.stage != ops[i - 1].stage) {
            es[n_stages++] = ExecStage{i, i + 1, 0, n_x, n_x, 0, 0, 0};
            stage_x = 0;
        }
        ExecStage &st = es[n_stages - 1];
        st.op_end = i + 1;
        // the stage's distinct inputs: ops sharing x (and its norm) share one copy
        const float *g = gu ? o.gamma : nullptr;
        const float eps = g ? o.eps : 0.0f;
        const int K = (int)o.K;
        int found = -1;
        for (int j = st.x_begin; j < st.x_end; ++j)
            if (ex[j].x == o.x && ex[j].gamma == g && ex[j].eps == eps && ex[j].K == K) found = j;
        if (found < 0) {
            ExecX &xd = ex[n_x];
            std::memset(&xd, 0, sizeof xd);
            xd.x = o.x;
            xd.gamma = g;
            xd.eps = eps;
            xd.K = K;
            xd.off = stage_x;
            stage_x += x_padded_floats(K);
            xd.goff = g ? stage_x : -1;
            if (g) stage_x += x_padded_floats(K);
            // Q4_K: the x's 32-element block sums, 16-byte aligned
            xd.soff = qtype == BQ_Q4_K ? stage_x : -1;
            if (qtype == BQ_Q4_K) stage_x += (K / 32 + 3) / 4 * 4;
            found = n_x++;
            st.x_end = n_x;
        }
        e.xoff = ex[found].off;
        e.soff = ex[found].soff;
        x_area = std::max(x_area, stage_x);
    }
    // ---- memory dependences between ops, from their address ranges ----
    // Weights are streamed ahead across stages, so no output may overlap any
    // weights; within a stage no output may overlap an input or another
    // output.  A stage that reads an earlier stage's output, or writes what an
    // earlier stage reads or writes, waits at a grid-wide barrier.
    auto in_ranges = [&](int i, Range *r) {
        const bq_op &o = ops[i];
        int n = 0;
        r[n++] = range(o.x, 4 * o.K);
        if (o.kind == BQ_OP_GATE_UP_SILU && o.gamma) r[n++] = range(o.gamma, 4 * o.K);
        if (o.kind == BQ_OP_GEMV && o.bias) r[n++] = range(o.bias, 4 * o.M);
        return n;
    };
    auto w_ranges = [&](int i, Range *r) {
        const bq_op &o = ops[i];
        int n = 0;
        r[n++] = range(o.W, (int64_t)o.M * eo[i].rb);
        if (o.kind == BQ_OP_GATE_UP_SILU) r[n++] = range(o.W_up, (int64_t)o.M * eo[i].rb);
        return n;
    };
    for (int i = 0; i < n_ops; ++i) {
        const Range yi = range(ops[i].y, 4 * ops[i].M);
        Range r[2];
        for (int j = 0; j < n_ops; ++j) {
            const int nw = w_ranges(j, r);
            for (int k = 0; k < nw; ++k)
                if (overlap(yi, r[k])) return BQ_ERR_SHAPE;
        }
    }
    for (int s = 0; s < n_stages; ++s) {
        const ExecStage &st = es[s];
        for (int i = st.op_begin; i < st.op_end; ++i) {
            const Range yi = range(ops[i].y, 4 * ops[i].M);
            Range ri[3];
            const int ni = in_ranges(i, ri);
            for (int j = 0; j < st.op_end; ++j) {
                const Range yj = range(ops[j].y, 4 * ops[j].M);
                Range rj[3];
                const int nj = in_ranges(j, rj);
                bool hit = false;
                for (int k = 0; k < nj; ++k) hit |= overlap(yi, rj[k]);
                if (j != i) hit |= overlap(yi, yj);
                for (int k = 0; k < ni; ++k) hit |= overlap(ri[k], yj);
                if (!hit) continue;
                if (j >= st.op_begin) return BQ_ERR_SHAPE;  // within one stage
                es[s].barrier = 1;
            }
        }
    }
    // ---- launch geometry ----
    // shared memory: control block + weight-slot mbarriers + x mbarriers |
    // descriptor tables | x buffers | weight rings (+ slack for realigned block
    // loads past the last slot).  Grow the x ring to 4 buffers first (stages
    // run ahead of each other), then the weight rings to 4 slots per warp,
    // then the x ring up to its maximum.
    const int warps = t.exec_warps, threads = 32 * warps;
    const int cap = max_smem_optin();
    const int tab_bytes = exec_table_bytes(n_ops, n_x, n_stages);
    const int x_bytes = (x_area * 4 + 127) / 128 * 128;
    auto xbar_offset = [warps](int nsw) { return 256 + 8 * warps * nsw; };
    auto tab_offset = [&](int nsw, int xb) { return (xbar_offset(nsw) + 16 * xb + 127) / 128 * 128; };
    auto total = [&](int nsw, int xb) {
        return (size_t)tab_offset(nsw, xb) + tab_bytes + (size_t)xb * x_bytes +
               (size_t)warps * nsw * slot + 128;
    };
    int nsw = t.exec_nsw ? t.exec_nsw : 2, xbuf = 1;
    if (total(nsw, xbuf) > (size_t)cap) return BQ_ERR_SHAPE;
    while (xbuf < 4 && total(nsw, xbuf + 1) <= (size_t)cap) ++xbuf;
    while (!t.exec_nsw && nsw < 4 && total(nsw + 1, xbuf) <= (size_t)cap) ++nsw;
    while (xbuf < EXEC_MAX_XBUF && total(nsw, xbuf + 1) <= (size_t)cap) ++xbuf;
    const size_t smem = total(nsw, xbuf);
    int occ = 0;
    const int err = fmt_exec_occupancy(qtype, threads, smem, &occ);
    if (err != 0 || occ < 1) return BQ_ERR_CUDA;
    const int grid = num_sms_current() * occ;
    const int nwarps = grid * warps;
    // ---- pass 2: tiling of every op, and the stage tile tables ----
    long long tiles_before = 0;
    for (int s = 0; s < n_stages; ++s) {
        ExecStage &st = es[s];
        st.tiles = 0;
        st.tile_off = (int)(tiles_before % nwarps);
        for (int i = st.op_begin; i < st.op_end; ++i) {
            ExecOp &e = eo[i];
            const int G = e.G, nsc = e.nsc, rb = e.rb;
            const int rows_per_warp = (int)((e.M + (long long)nwarps - 1) / nwarps);
            if (rb <= slot && rows_per_warp <= t.exec_rowmode_rows && nsc <= t.exec_rowmode_nsc) {
                // row mode: a few whole rows per tile, contiguous in memory
                e.rowmode = 1;
                e.rpw = (unsigned char)std::max(1, std::min({rows_per_warp, slot / rb, 32}));
                e.KCU = (short)nsc;
                e.row_stride = rb;
                e.single = 1;
            } else {
                // tile mode: 32/G rows, whole rows per slot when they fit, else
                // chunks of a multiple of G units
                const int rpw = 32 / G;
                int KCU = nsc, stride = 0, single = 0;
                if ((long long)rpw * rb <= slot) {
                    single = G >= 8 || (rb / 16) % 8 == G % 8;
                    stride = single ? rb : padded_stride(rb, G);
                    if ((long long)rpw * stride > slot) single = 0, stride = 0;
                }
                if (!stride) {
                    single = 0;
                    for (int m = (nsc + G - 1) / G; m >= 1; --m) {
                        KCU = std::min(nsc, G * m);
                        stride = padded_stride(KCU * ub, G);
                        if ((long long)rpw * stride <= slot) break;
                    }
                }
                e.rowmode = 0;
                e.rpw = (unsigned char)rpw;
                e.KCU = (short)KCU;
                e.row_stride = stride;
                e.single = (unsigned char)single;
            }
            e.nchunks = (short)((nsc + e.KCU - 1) / e.KCU);
            e.ntiles = (e.M + e.rpw - 1) / e.rpw;
            e.tile_base = st.tiles;
            st.tiles += e.ntiles;
        }
        tiles_before += st.tiles;
    }
    geo->n_stages = n_stages;
    geo->n_x = n_x;
    geo->slot = slot;
    geo->nsw = nsw;
    geo->xbar_off = xbar_offset(nsw);
    geo->tab_off = tab_offset(nsw, xbuf);
    geo->x_off = geo->tab_off + tab_bytes;
    geo->x_floats = x_bytes / 4;
    geo->x_buffers = xbuf;
    geo->ring_off = geo->x_off + xbuf * x_bytes;
    geo->threads = threads;
    geo->smem = smem;
    geo->grid = grid;
    geo->prefetch = t.exec_prefetch;
    return BQ_OK;
}

bool multi_chunking(MultiOp &m, int ub, int slot_cap, bool rows_low);

// CTA split of a list of n <= grid ops in which every op has CTAs of its own:
// op i gets k_i >= 1 CTAs, the grid shared by bytes (largest remainder), and
// its tiles (ntiles[i], the ops' tiles concatenated in order) split evenly
// among them.  out[c] is CTA c's first tile, out[grid] the total.
void split_by_op(const long long *bytes, const int *ntiles, int n, int grid, int *out) {
    long long total = 0;
    for (int i = 0; i < n; ++i) total += bytes[i];
    std::vector<int> k((size_t)n, 1);
    std::vector<double> rem((size_t)n, 0.0);
    int used = n;
    for (int i = 0; i < n; ++i) {
        const double q = total > 0 ? (double)grid * (double)bytes[i] / (double)total : 0.0;
        const int f = std::max(1, (int)q);
        rem[(size_t)i] = q - f;
        k[(size_t)i] = f;
        used += f - 1;
    }
    // too many (the at-least-one rule): take from the ops with the smallest remainder
    while (used > grid) {
        int j = -1;
        for (int i = 0; i < n; ++i)
            if (k[(size_t)i] > 1 && (j < 0 || rem[(size_t)i] < rem[(size_t)j])) j = i;
        if (j < 0) break;
        --k[(size_t)j];
        rem[(size_t)j] += 1.0;
        --used;
    }
    // too few: give to the ops with the largest remainder
    while (used < grid) {
        int j = 0;
        for (int i = 1; i < n; ++i)
            if (rem[(size_t)i] > rem[(size_t)j]) j = i;
        ++k[(size_t)j];
        rem[(size_t)j] -= 1.0;
        ++used;
    }
    int c = 0;
    long long base = 0;
    for (int i = 0; i < n; ++i) {
        for (int j = 0; j < k[(size_t)i]; ++j) out[c++] = (int)(base + (long long)ntiles[i] * j / k[(size_t)i]);
        base += ntiles[i];
    }
    while (c <= grid) out[c++] = (int)base;
}

bq_status plan_multi_tables(int qtype, const bq_op *ops, int n_ops, MultiOp *mo, int *cta_tiles,
                            MultiGeometry *geo) {
    const Tunables &t = tunables();
    const int bb = block_bytes(qtype), ub = 8 * bb;
    const int D = std::min(t.multi_d, MULTI_MAX_D);
    const int NR = t.multi_nr;
    // pass 1: per-op tiling that does not depend on the slot size
    int maxK = 0, slot_min = 0;
    long long tiles = 0;
    for (int i = 0; i < n_ops; ++i) {
        const bq_op &o = ops[i];
        MultiOp &m = mo[i];
        std::memset(&m, 0, sizeof m);
        const bool gu = o.kind == BQ_OP_GATE_UP_SILU;
        m.W[0] = static_cast<const uint8_t *>(o.W);
        m.W[1] = gu ? static_cast<const uint8_t *>(o.W_up) : nullptr;
        m.x = o.x;
        m.gamma = gu ? o.gamma : nullptr;
        m.eps = o.eps;
        m.y = o.y;
        m.bias = gu ? nullptr : o.bias;
        m.nmat = gu ? 2 : 1;
        m.M = (int)o.M;
        m.K = (int)o.K;
        m.nsc = m.K / 256;
        m.G = tree_lanes_for_units(m.nsc);
        m.rpw = NR * (32 / m.G);
        m.rb = m.nsc * ub;
        m.ntiles = (m.M + m.rpw - 1) / m.rpw;
        m.tile_base = (int)tiles;
        tiles += m.ntiles;
        maxK = std::max(maxK, m.K);
        // the smallest item: one unit per lane
        const int k1 = std::min(m.nsc, m.G);
        int S1 = 0, um = 0;
        lane_order_any(m.G, k1 * ub / 16, ub / 16, &S1, &um, qtype == BQ_Q4_0);
        slot_min = std::max(slot_min, m.rpw * S1 * 16);
    }
    if (tiles > (1LL << 30)) return BQ_ERR_SHAPE;
    // shared memory: header | x buffers | nwarps rings of D slots.  Two x
    // buffers (the next op's x copied while this op computes) when they are
    // small beside the rings and cost no warp: the streaming rate follows the
    // warp count (measured on GB300: 10, 11, 12 warps of the Q8_0 token stream
    // ran at 4.86, 5.20, 5.32 TB/s), while a CTA meets an op boundary only a
    // few times per launch.
    const int cap = max_smem_optin();
    const int x_off = MULTI_X_OFF;
    const int x_rstride = x_padded_floats(maxK);
    const int x_floats = x_rstride + multi_sum_floats(qtype, 1, x_rstride);
    auto warps_for = [&](int xb) {
        const int ro = (x_off + xb * x_floats * 4 + 127) / 128 * 128;
        const long long b = (long long)cap - ro;
        if (b < (long long)D * slot_min) return 0;
        int w = (int)std::min<long long>(multi_max_warps(qtype, 1), b / ((long long)D * slot_min));
        if (t.multi_warps) w = std::min(w, t.multi_warps);
        return w;
    };
    int x_buffers = 1;
    if (2 * x_floats * 4 <= t.multi_x2_max && warps_for(2) >= warps_for(1)) x_buffers = 2;
    const int ring_off = (x_off + x_buffers * x_floats * 4 + 127) / 128 * 128;
    const long long budget = (long long)cap - ring_off;
    int nwarps = warps_for(x_buffers);
    if (nwarps < 1) return BQ_ERR_SHAPE;
    // A short list (fewer tiles per SM than warps fit): one CTA per SM with the
    // warps its tiles need, so that the launch leaves shared memory to the next
    // launch's CTAs (a staged plan's next stage then starts, fills its rings
    // and waits beside this one instead of after it).
    const int nsms = num_sms_current();
    bool short_list = false;
    if (t.short_lists && nsms > 0) {
        const long long per_sm = (tiles + nsms - 1) / nsms;
        if (per_sm < nwarps) {
            nwarps = (int)std::max<long long>(1, per_sm);
            short_list = true;
        }
    }
    const int slot_cap = (int)(budget / ((long long)nwarps * D)) / 128 * 128;
    // pass 2: per op, whole rows in a slot when they fit, else the largest
    // chunk of a multiple of G units
    int slot_bytes = 0;
    for (int i = 0; i < n_ops; ++i) {
        MultiOp &m = mo[i];
        if (!multi_chunking(m, ub, slot_cap, qtype == BQ_Q4_0)) return BQ_ERR_SHAPE;
        slot_bytes = std::max(slot_bytes, m.rpw * m.row_stride);
    }
    slot_bytes = (slot_bytes + 127) / 128 * 128;
    const size_t smem = (size_t)ring_off + (size_t)nwarps * D * slot_bytes;
    if (smem > (size_t)cap) return BQ_ERR_SHAPE;
    const int threads = nwarps * 32;
    int occ = 0;
    const int err = fmt_multi_occupancy(qtype, NR, 1, threads, smem, &occ);
    if (err != 0 || occ < 1) return BQ_ERR_CUDA;
    const int grid = short_list ? nsms : std::min(MULTI_MAX_CTAS, nsms * occ);
    if (t.split_by_op && 2LL * n_ops <= grid) {
        // few ops (a stage's q, k, v): every op gets CTAs of its own, so that no
        // CTA meets an op boundary (where all its warps wait and x is staged again)
        std::vector<long long> ob((size_t)n_ops);
        std::vector<int> ot((size_t)n_ops);
        for (int i = 0; i < n_ops; ++i) {
            ob[(size_t)i] = (long long)mo[i].M * mo[i].rb * mo[i].nmat;
            ot[(size_t)i] = mo[i].ntiles;
        }
        split_by_op(ob.data(), ot.data(), n_ops, grid, cta_tiles);
    } else {
        // byte-balanced contiguous tile ranges
        long long total = 0;
        for (int i = 0; i < n_ops; ++i)
            for (int k = 0; k < mo[i].ntiles; ++k)
                total += (long long)std::min(mo[i].rpw, mo[i].M - k * mo[i].rpw) * mo[i].rb * mo[i].nmat;
        cta_tiles[0] = 0;
        int c = 1;
        long long acc = 0;
        for (int i = 0; i < n_ops && c < grid; ++i)
            for (int k = 0; k < mo[i].ntiles && c < grid; ++k) {
                acc += (long long)std::min(mo[i].rpw, mo[i].M - k * mo[i].rpw) * mo[i].rb * mo[i].nmat;
                while (c < grid && acc * grid >= total * c) cta_tiles[c++] = mo[i].tile_base + k + 1;
            }
        while (c <= grid) cta_tiles[c++] = (int)tiles;
    }
    geo->grid = grid;
    geo->threads = threads;
    geo->nwarps = nwarps;
    geo->D = D;
    geo->slot_bytes = slot_bytes;
    geo->x_off = x_off;
    geo->ring_off = ring_off;
    geo->smem = smem;
    geo->nr = NR;
    geo->R = 1;
    geo->x_rstride = x_rstride;
    geo->x_floats = x_floats;
    geo->x_buffers = x_buffers;
    geo->panel_units = 0;
    return BQ_OK;
}

// One warp-tile item layout for op m: whole rows in a slot of slot_cap bytes
// when they fit (copied as one block when their natural stride admits a lane
// order), else chunks of a multiple of G units with a padded row stride.
// rows_low: the kernel instance uses the rows-low lane order (Q4_0 decode)
bool multi_chunking(MultiOp &m, int ub, int slot_cap, bool rows_low) {
    const int U = ub / 16;
    int KCU = m.nsc, S = 0, umask = 0, single = 0;
    if ((long long)m.rpw * m.rb <= slot_cap) {
        // one copy per item; else padded rows (one copy per row); else, with
        // G >= 8, one copy in the fallback order (conflict-free for any
        // stride; for Q4_0 only where it is the rows-low order, G = 32)
        int Sp = 0, up = 0;
        if (lane_order(m.G, m.rb / 16, U, false, &Sp, &up, rows_low)) {
            S = Sp, umask = up, single = 1;
        } else if (lane_order(m.G, m.rb / 16, U, true, &Sp, &up, rows_low) &&
                   (long long)m.rpw * Sp * 16 <= slot_cap) {
            S = Sp, umask = up, single = 0;
        } else if (rows_low ? m.G == 32 : m.G >= 8) {
            S = m.rb / 16, umask = m.G - 1, single = 1;
        }
    }
    if (!S) {
        single = 0;
        for (int k = (m.nsc + m.G - 1) / m.G; k >= 1; --k) {
            KCU = std::min(m.nsc, m.G * k);
            lane_order_any(m.G, KCU * U, U, &S, &umask, rows_low);
            if ((long long)m.rpw * S * 16 <= slot_cap) break;
        }
        if ((long long)m.rpw * S * 16 > slot_cap) return false;
    }
    m.KCU = KCU;
    m.row_stride = S * 16;
    m.single = single;
    m.umask = umask;
    m.nchunks = (m.nsc + KCU - 1) / KCU;
    return true;
}

bool plan_multi_single(const GemvCall &c, MultiArgs *a, MultiGeometry *geo, bool pair) {
    const Tunables &t = tunables();
    const int bb = block_bytes(c.qtype), ub = 8 * bb;
    int D = std::min(t.multi_d, MULTI_MAX_D);
    const int R = c.R;
    // verify: two weight rows per lane share each x read up to R = 4; from
    // R = 5 on the R partial sums per row fill the registers and one row per
    // lane measured faster on GB300 (R = 6: 687 against 576 GB/s)
    int NR = R == 1 ? 1 : t.verify_nr ? t.verify_nr : R <= 4 ? 2 : 1;
    if (c.qtype == BQ_Q4_K) NR = 1;  // its verify instances hold one weight row per lane
    const int nsms = num_sms_current();
    const int cap = max_smem_optin();
    if (nsms <= 0 || cap <= 0) return false;
    std::memset(a, 0, sizeof *a);
    MultiOp &m = a->op;
    const bool gu = c.mode == MODE_GATE_UP;
    m.W[0] = static_cast<const uint8_t *>(c.W0);
    m.W[1] = gu ? static_cast<const uint8_t *>(c.W1) : nullptr;
    m.x = c.x;
    m.gamma = gu ? c.gamma : nullptr;
    m.y = c.y;
    m.bias = gu || R > 1 ? nullptr : c.bias;
    m.eps = c.eps;
    m.M = (int)c.M;
    m.K = (int)c.K;
    m.nsc = m.K / 256;
    m.G = tree_lanes_for_units(m.nsc);
    m.rpw = NR * (32 / m.G);
    m.rb = m.nsc * ub;
    m.nmat = gu ? 2 : 1;
    m.ntiles = (int)((c.M + m.rpw - 1) / m.rpw);
    m.tile_base = 0;
    // x: the whole R x K input, or (verify with a large input) double-buffered
    // panels of a multiple of G units
    const int xpad = x_padded_floats(m.K);
    int PU = 0, x_floats = R * xpad, x_rstride = xpad, x_buffers = 1;
    if ((long long)R * xpad * 4 > t.single_x_max) {
        if (gu || R == 1) return false;
        // panel mode gives each warp one tile for the whole call (its R x NR
        // partial sums stay in registers): with one weight row per lane a
        // large M can need more warps than one wave of CTAs holds (8 per SM
        // at these register counts), so take two rows per lane then
        if (NR == 1 && c.qtype != BQ_Q4_K && t.verify_wave &&
            (c.M + m.rpw - 1) / m.rpw > (long long)nsms * multi_max_warps(c.qtype, R)) {
            NR = 2;
            m.rpw = NR * (32 / m.G);
            m.ntiles = (int)((c.M + m.rpw - 1) / m.rpw);
        }
        PU = (int)(t.single_x_max / 2 / ((long long)R * 256 * 4)) / m.G * m.G;
        if (PU < m.G) return false;
        x_rstride = PU * 256;
        x_floats = R * x_rstride;
        x_buffers = 2;
    }
    x_floats += multi_sum_floats(c.qtype, R, x_rstride);
    if (m.gamma) x_floats += x_rstride;  // gate+up (R = 1, whole K): room for the staged gain
    const int ring_off = (MULTI_X_OFF + x_buffers * x_floats * 4 + 127) / 128 * 128;
    const long long budget = (long long)cap - ring_off;
    const int maxw = multi_max_warps(c.qtype, R);
    // Row mode for ops too small to give every warp a few tiles: a tile is a
    // few whole rows and each row is evaluated block-parallel by the whole
    // warp (same tree, about 8x shorter per-lane chains).  Latency-bound
    // calls gain; large calls keep one unit per lane.
    const bool rowmode = R == 1 && !PU && t.single_rowmode && m.nsc <= 16 &&
                         m.ntiles <= (long long)t.single_rowmode * nsms &&
                         D * (long long)m.rb <= budget;
    if (rowmode) {
        const long long per = (long long)nsms * maxw;
        int rows = (int)std::min<long long>(32, std::max<long long>(1, (c.M + per - 1) / per));
        while (rows > 1 && (long long)D * rows * m.rb > budget) --rows;
        m.rowmode = 1;
        m.rpw = rows;
        m.ntiles = (int)((c.M + rows - 1) / rows);
        NR = 0;
    }
    // gate+up in unit mode: the paired instance (NR = 3 tag), which takes the
    // gate and up items of a chunk together, with four ring slots (two pairs)
    // when they fit
    if (pair && gu && !rowmode && !PU &&
        ((t.gu_pair >= 1 && c.qtype == BQ_Q8_0) || (t.gu_pair >= 2 && c.qtype == BQ_Q4_0))) {
        NR = 3;
        D = MULTI_MAX_D;
    }
    // warps: enough for the tiles of one CTA per SM, at most what fits
    const int k1 = std::min(m.nsc, m.G);
    int S1 = 0, um1 = 0;
    lane_order_any(m.G, k1 * ub / 16, ub / 16, &S1, &um1, c.qtype == BQ_Q4_0 && R == 1);
    const int slot_min = rowmode ? m.rpw * m.rb : m.rpw * S1 * 16;
    if (NR == 3 && budget < (long long)D * slot_min) D = 2;
    if (budget < (long long)D * slot_min) return false;
    const int fit = (int)std::min<long long>(maxw, budget / ((long long)D * slot_min));
    const int want = (int)std::min<long long>(fit, (m.ntiles + nsms - 1) / nsms);
    int nwarps = std::max(1, want);
    const int slot_cap = (int)(budget / ((long long)nwarps * D)) / 128 * 128;
    if (rowmode) {
        m.KCU = m.nsc;
        m.row_stride = m.rb;
        m.single = 1;
        m.nchunks = 1;
    } else if (PU) {
        // one unit per lane per item, so chunks never straddle a panel
        m.KCU = m.G;
        int S = 0, um = 0;
        lane_order_any(m.G, m.G * ub / 16, ub / 16, &S, &um, c.qtype == BQ_Q4_0 && R == 1);
        m.row_stride = S * 16;
        m.umask = um;
        m.single = 0;
        m.nchunks = (m.nsc + m.G - 1) / m.G;
        if ((long long)m.rpw * m.row_stride > slot_cap) return false;
    } else if (!multi_chunking(m, ub, slot_cap, c.qtype == BQ_Q4_0 && R == 1)) {
        return false;
    }
    const int slot_bytes = (m.rpw * m.row_stride + 127) / 128 * 128;
    // + slack: block-parallel rows read up to 4 bytes past a slot's last block
    const size_t smem = (size_t)ring_off + (size_t)nwarps * D * slot_bytes + 128;
    if (smem > (size_t)cap) return false;
    const int threads = nwarps * 32;
    int occ = 0;
    const int err = fmt_multi_occupancy(c.qtype, NR, R, threads, smem, &occ);
    if (err != 0 || occ < 1) return false;
    // panel mode: every CTA holds at most nwarps tiles (one per warp); else a
    // CTA's warps take its tiles round-robin, at most one CTA wave
    long long grid = (m.ntiles + nwarps - 1) / nwarps;
    if (!PU) grid = std::min<long long>(grid, (long long)nsms * occ);
    a->ops = nullptr;
    a->cta_tiles = nullptr;
    a->nops = 1;
    a->nwarps = nwarps;
    a->D = D;
    a->slot_bytes = slot_bytes;
    a->x_off = MULTI_X_OFF;
    a->ring_off = ring_off;
    a->nr = NR;
    a->R = R;
    a->x_rstride = x_rstride;
    a->x_floats = x_floats;
    a->x_buffers = x_buffers;
    a->panel_units = PU;
    a->gain_staged = m.gamma != nullptr;
    a->inline_op = 1;
    a->wait_ns = g_wait_ns.load();
    a->early_ring = t.single_early;
    geo->grid = (int)grid;
    geo->threads = threads;
    geo->nwarps = nwarps;
    geo->D = D;
    geo->slot_bytes = slot_bytes;
    geo->x_off = MULTI_X_OFF;
    geo->ring_off = ring_off;
    geo->smem = smem;
    geo->nr = NR;
    geo->R = R;
    geo->x_rstride = x_rstride;
    geo->x_floats = x_floats;
    geo->x_buffers = x_buffers;
    geo->panel_units = PU;
    return true;
}

bool tunables_multi() { return tunables().multi != 0; }

void fill_multi_args(const MultiGeometry &geo, int n_ops, const MultiOp *ops,
                     const int *cta_tiles, MultiArgs *a) {
    a->ops = ops;
    a->cta_tiles = cta_tiles;
    a->nops = n_ops;
    a->nwarps = geo.nwarps;
    a->D = geo.D;
    a->slot_bytes = geo.slot_bytes;
    a->x_off = geo.x_off;
    a->ring_off = geo.ring_off;
    a->nr = geo.nr;
    a->R = geo.R;
    a->x_rstride = geo.x_rstride;
    a->x_floats = geo.x_floats;
    a->x_buffers = geo.x_buffers;
    a->panel_units = geo.panel_units;
    a->gain_staged = 0;
    a->inline_op = 0;
    a->cta_ns = nullptr;
    a->wait_ns = g_wait_ns.load();
    a->early_ring = 0;
}

void fill_exec_args(const ExecGeometry &geo, int n_ops, const ExecOp *ops, const ExecX *xs,
                    const ExecStage *stages, unsigned int *counters, ExecArgs *a) {
    a->ops = ops;
    a->xs = xs;
    a->stages = stages;
    a->counters = counters;
    a->nops = n_ops;
    a->nxs = geo.n_x;
    a->nstages = geo.n_stages;
    a->NSW = geo.nsw;
    a->slot_bytes = geo.slot;
    a->xbar_off = geo.xbar_off;
    a->tab_off = geo.tab_off;
    a->x_off = geo.x_off;
    a->x_floats = geo.x_floats;
    a->x_buffers = geo.x_buffers;
    a->ring_off = geo.ring_off;
    a->prefetch = geo.prefetch;
    a->wait_ns = g_wait_ns.load();
    a->barrier_extra = 0;
}

}  // namespace bq

// the opaque plan handle of include/bqgemv.h
namespace bq {
// one launch of a staged plan: the streaming kernel over one stage's ops
struct StageLaunch {
    MultiArgs args;
    int grid, threads, pdl;
    size_t smem;
};
}  // namespace bq

struct bq_stream_plan {
    int qtype, n_ops, n_stages, device;
    int multi;  // 1: independent ops, multi-op streaming kernel; 0: stream executor
    // staged plans (dependent stages, multi == 0): one streaming-kernel launch
    // per stage, in stage order; null for the executor
    bq::StageLaunch *stages;
    int grid, threads;
    size_t smem;
    bq::ExecArgs args;
    bq::MultiArgs margs;
    unsigned int *counters;
    // multi-op plans: host copies of the op table and of the CTA tile split,
    // the split's device copy, and the per-CTA timing array (plan tuning)
    bq::MultiOp *mo_host;
    int *ct_host;
    int *ct_dev;
    unsigned long long *cta_ns;
};

using bq::GemvCall;
using bq::LaunchPlan;

namespace {

bool aligned_ok(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bq_status from_cuda(int e) { return e == 0 ? BQ_OK : BQ_ERR_CUDA; }

bq_status check_shape(int qtype, long long M, long long K) {
    if (M < 0 || M > bq::M_MAX) return BQ_ERR_SHAPE;
    const int ks = bq::k_step(qtype);
    if (K < ks || K > bq::K_MAX || K % ks) return BQ_ERR_SHAPE;
    return BQ_OK;
}

bq_status run_gemv(const GemvCall &c) {
    if (c.K % 256 == 0) {
        bq::MultiArgs a;
        bq::MultiGeometry g;
        if (bq::plan_multi_single(c, &a, &g)) {
            const int pdl = bq::tunables().single_pdl;
            const int e = bq::fmt_multi_launch(c.qtype, a, g.grid, g.threads, g.smem, c.stream, pdl);
            return from_cuda(e);
        }
        // The streaming kernel stages the whole input in shared memory for a
        // single row and for gate+up (only verify cuts it into K-panels), so
        // an input beyond the staging limit (K > 32768 fp32) cannot be
        // planned there: the generic kernel, which reads x through L1 with the
        // same arithmetic tree, takes the call.
    }
    LaunchPlan p;
    bq::plan_gemv(c, &p);
    const int e = bq::fmt_generic_launch(c, p);
    return from_cuda(e);
}

bq_status gemv_common(int qtype, const void *Wq, const float *x, float *y, int R, int64_t M,
                      int64_t K, void *stream, const float *bias = nullptr) {
    if (!bq::known_qtype(qtype)) return BQ_ERR_QTYPE;
    if (R < 1 || R > BQ_VERIFY_MAX_ROWS) return BQ_ERR_SHAPE;
    bq_status s = check_shape(qtype, M, K);
    if (s != BQ_OK) return s;
    if (M == 0) return BQ_OK;  // empty product: nothing is read or written
    if (!Wq || !x || !y) return BQ_ERR_NULL;
    if (!aligned_ok(Wq, 16) || !aligned_ok(x, 16) || !aligned_ok(y, 4) ||
        (bias && !aligned_ok(bias, 4)))
        return BQ_ERR_ALIGN;
    GemvCall c{qtype, bq::MODE_PLAIN, R, Wq, nullptr, x, nullptr, 0.0f, y, M, K, stream, bias};
    return run_gemv(c);
}

// A plan of dependent stages as one streaming-kernel launch per stage.  A
// stage of one op takes the single-call geometry (row mode for small ops, as
// bq_gemv); a stage of several independent ops takes the op-list geometry,
// its op table and CTA split in the workspace.  Every launch allows
// programmatic dependent launch: a stage's kernel starts while the previous
// stage's kernel drains, prefetches its first weight items into L2, and waits
// for the previous grid (griddepcontrol.wait) before it reads any input, so
// an op may read an output of the stage before.  Outputs are bit-identical to
// the executor's and to one call per op: the same fixed tree everywhere.
// Returns BQ_ERR_SHAPE when some stage does not fit the streaming kernel.
bq_status plan_staged(int qtype, const bq_op *ops, int n_ops, const bq::ExecStage *es,
                      int n_stages, uint8_t *ws, bq_stream_plan **out) {
    const bq::Tunables &t = bq::tunables();
    std::vector<bq::StageLaunch> sl((size_t)n_stages);
    std::vector<bq::MultiOp> mo((size_t)n_ops);
    std::memset(mo.data(), 0, mo.size() * sizeof(bq::MultiOp));
    const int64_t off_ct = ((int64_t)n_ops * (int64_t)sizeof(bq::MultiOp) + 255) / 256 * 256;
    std::vector<int> ct;  // the CTA splits of the list-mode stages, back to back
    std::vector<int> ct_stage((size_t)bq::MULTI_MAX_CTAS + 1);
    auto *mo_dev = reinterpret_cast<const bq::MultiOp *>(ws);
    auto *ct_dev = reinterpret_cast<int *>(ws + off_ct);
    for (int s = 0; s < n_stages; ++s) {
        const int b = es[s].op_begin, n = es[s].op_end - es[s].op_begin;
        bq::StageLaunch &l = sl[(size_t)s];
        l.pdl = t.single_pdl;
        // the first stage follows the caller's earlier work: early only under
        // the single calls' contract (weights not written by an earlier GEMV call)
        const int early = t.plan_early && (s > 0 || t.single_early);
        if (n == 1) {
            const bq_op &o = ops[b];
            const bool gu = o.kind == BQ_OP_GATE_UP_SILU;
            GemvCall c{qtype, gu ? bq::MODE_GATE_UP : bq::MODE_PLAIN, 1, o.W,
                       gu ? o.W_up : nullptr, o.x, gu ? o.gamma : nullptr, o.eps, o.y,
                       (long long)o.M, (long long)o.K, nullptr, gu ? nullptr : o.bias};
            bq::MultiGeometry g;
            // (a paired gate+up stage measured slower in the chained Qwen3-0.6B-shaped
            // token: 895 against 1115 GB/s)
            if (!bq::plan_multi_single(c, &l.args, &g, false)) return BQ_ERR_SHAPE;
            l.args.early_ring = early;
            l.grid = g.grid;
            l.threads = g.threads;
            l.smem = g.smem;
        } else {
            bq::MultiGeometry g;
            const bq_status st = bq::plan_multi_tables(qtype, ops + b, n, mo.data() + b,
                                                       ct_stage.data(), &g);
            if (st != BQ_OK) return st == BQ_ERR_CUDA ? st : BQ_ERR_SHAPE;
            const size_t at = ct.size();
            ct.insert(ct.end(), ct_stage.begin(), ct_stage.begin() + g.grid + 1);
            bq::fill_multi_args(g, n, mo_dev + b, ct_dev + at, &l.args);
            l.args.early_ring = early;
            l.grid = g.grid;
            l.threads = g.threads;
            l.smem = g.smem;
        }
    }
    if (cudaMemcpy(ws, mo.data(), (size_t)n_ops * sizeof(bq::MultiOp), cudaMemcpyHostToDevice) !=
            cudaSuccess ||
        (!ct.empty() && cudaMemcpy(ws + off_ct, ct.data(), ct.size() * sizeof(int),
                                   cudaMemcpyHostToDevice) != cudaSuccess))
        return BQ_ERR_CUDA;
    auto *p = new (std::nothrow) bq_stream_plan;
    if (!p) return BQ_ERR_CUDA;
    std::memset(p, 0, sizeof *p);
    p->stages = new (std::nothrow) bq::StageLaunch[(size_t)n_stages];
    if (!p->stages) {
        delete p;
        return BQ_ERR_CUDA;
    }
    std::memcpy(p->stages, sl.data(), (size_t)n_stages * sizeof(bq::StageLaunch));
    p->qtype = qtype;
    p->n_ops = n_ops;
    p->n_stages = n_stages;
    p->multi = 0;
    cudaGetDevice(&p->device);
    *out = p;
    return BQ_OK;
}

}  // namespace

extern "C" {

int bq_version(void) { return 100; }

const char *bq_status_str(int status) {
    switch (status) {
        case BQ_OK: return "ok";
        case BQ_ERR_NULL: return "a required pointer is NULL";
        case BQ_ERR_SHAPE: return "shape outside the supported range (M >= 0, K % 32 == 0 (Q4_K: K % 256 == 0), 32 <= K <= 2^18, 1 <= R <= 6)";
        case BQ_ERR_ALIGN: return "pointer misaligned (packed weights and fp32 inputs need 16 bytes, outputs 4)";
        case BQ_ERR_QTYPE: return "unknown quantization type (BQ_Q8_0 = 8, BQ_Q4_0 = 2, BQ_Q4_K = 12)";
        case BQ_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
        case BQ_ERR_DEVICE: return "a kernel recorded a device-side error (bounded wait ran out)";
        default: return "unknown status";
    }
}

int64_t bq_packed_bytes(int qtype, int64_t M, int64_t K) {
    const int bb = bq::block_bytes(qtype);
    if (bb < 0 || M < 0 || K < 0 || K % bq::k_step(qtype)) return -1;
    return M * (K / 32) * bb;
}

int bq_tree_lanes(int64_t K) {
    if (K <= 0 || K % 32) return -1;
    return bq::tree_lanes_for_units((K / 32 + 7) / 8);
}

bq_status bq_quantize_pack(int qtype, const float *W, int64_t M, int64_t K, void *Wq, void *stream) {
    if (!bq::known_qtype(qtype)) return BQ_ERR_QTYPE;
    bq_status s = check_shape(qtype, M, K);
    if (s != BQ_OK) return s;
    if (M == 0) return BQ_OK;
    if (!W || !Wq) return BQ_ERR_NULL;
    if (!aligned_ok(W, 4) || !aligned_ok(Wq, 16)) return BQ_ERR_ALIGN;
    return from_cuda(bq_internal_pack(qtype, W, M, K, Wq, stream));
}

bq_status bq_gemv_q8_0(const void *Wq, const float *x, float *y, int64_t M, int64_t K, void *stream) {
    return gemv_common(BQ_Q8_0, Wq, x, y, 1, M, K, stream);
}

bq_status bq_gemv_q4_0(const void *Wq, const float *x, float *y, int64_t M, int64_t K, void *stream) {
    return gemv_common(BQ_Q4_0, Wq, x, y, 1, M, K, stream);
}

bq_status bq_gemv_q4_k(const void *Wq, const float *x, float *y, int64_t M, int64_t K, void *stream) {
    return gemv_common(BQ_Q4_K, Wq, x, y, 1, M, K, stream);
}

bq_status bq_gemv_qkv_bias(int qtype, const void *Wqkv, const float *x, const float *bias, float *y,
                           int64_t M, int64_t K, void *stream) {
    return gemv_common(qtype, Wqkv, x, y, 1, M, K, stream, bias);
}

bq_status bq_gemv_f16(const void *W, const float *x, float *y, int64_t M, int64_t K, void *stream) {
    if (M < 0 || M > bq::M_MAX || K < 8 || K > bq::K_MAX || K % 8) return BQ_ERR_SHAPE;
    if (M == 0) return BQ_OK;
    if (!W || !x || !y) return BQ_ERR_NULL;
    if (!aligned_ok(W, 16) || !aligned_ok(x, 16) || !aligned_ok(y, 4)) return BQ_ERR_ALIGN;
    return from_cuda(bq_internal_f16_launch(W, x, y, M, K, stream));
}

bq_status bq_gemv_verify(int qtype, const void *Wq, const float *X, float *Y, int R, int64_t M,
                         int64_t K, void *stream) {
    return gemv_common(qtype, Wq, X, Y, R, M, K, stream);
}

bq_status bq_gemv_gate_up_silu(int qtype, const void *Wg, const void *Wu, const float *x,
                               const float *gamma, float eps, float *y, int64_t M, int64_t K,
                               void *stream) {
    if (!bq::known_qtype(qtype)) return BQ_ERR_QTYPE;
    bq_status s = check_shape(qtype, M, K);
    if (s != BQ_OK) return s;
    if (gamma && !(std::isfinite(eps) && eps >= 0.0f)) return BQ_ERR_SHAPE;
    if (M == 0) return BQ_OK;
    if (!Wg || !Wu || !x || !y) return BQ_ERR_NULL;
    if (!aligned_ok(Wg, 16) || !aligned_ok(Wu, 16) || !aligned_ok(x, 16) || !aligned_ok(y, 4) ||
        (gamma && !aligned_ok(gamma, 16)))
        return BQ_ERR_ALIGN;
    GemvCall c{qtype, bq::MODE_GATE_UP, 1, Wg, Wu, x, gamma, eps, y, M, K, stream};
    return run_gemv(c);
}

static int64_t align256(int64_t v) { return (v + 255) / 256 * 256; }

int64_t bq_stream_workspace_bytes(int n_ops, int n_stages) {
    if (n_ops < 1 || n_stages < 1 || n_stages > n_ops) return -1;
    const int64_t exec = align256((int64_t)n_ops * sizeof(bq::ExecOp)) +
                         align256((int64_t)n_ops * sizeof(bq::ExecX)) +
                         align256((int64_t)n_stages * sizeof(bq::ExecStage)) +
                         align256((int64_t)n_stages * 4);
    const int64_t multi = align256((int64_t)n_ops * sizeof(bq::MultiOp)) +
                          align256((int64_t)(bq::MULTI_MAX_CTAS + 1) * 4) +
                          align256((int64_t)bq::MULTI_MAX_CTAS * 8);
    // staged: the op table and one CTA split per stage
    const int64_t staged = align256((int64_t)n_ops * sizeof(bq::MultiOp)) +
                           align256((int64_t)n_stages * (bq::MULTI_MAX_CTAS + 1) * 4);
    return std::max({exec, multi, staged});
}

bq_status bq_stream_plan_create(int qtype, const bq_op *ops, int n_ops, void *workspace,
                                int64_t workspace_bytes, bq_stream_plan **plan) {
    if (!plan) return BQ_ERR_NULL;
    *plan = nullptr;
    if (!bq::known_qtype(qtype)) return BQ_ERR_QTYPE;
    if (!ops || !workspace) return BQ_ERR_NULL;
    if (n_ops < 1) return BQ_ERR_SHAPE;
    if (!aligned_ok(workspace, 256)) return BQ_ERR_ALIGN;
    std::vector<bq::ExecOp> eo((size_t)n_ops);
    std::vector<bq::ExecX> ex((size_t)n_ops);
    std::vector<bq::ExecStage> es((size_t)n_ops);
    bq::ExecGeometry geo;
    const bq_status st = bq::plan_exec_tables(qtype, ops, n_ops, eo.data(), ex.data(), es.data(), &geo);
    if (st != BQ_OK) return st;
    const int n_stages = geo.n_stages;
    const int64_t need = bq_stream_workspace_bytes(n_ops, n_stages);
    if (workspace_bytes < need) return BQ_ERR_SHAPE;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    bool independent = bq::tunables().multi != 0;
    for (int s = 0; s < n_stages; ++s) independent &= !es[(size_t)s].barrier;
    if (independent) {
        std::vector<bq::MultiOp> mo((size_t)n_ops);
        std::vector<int> ct(bq::MULTI_MAX_CTAS + 1);
        bq::MultiGeometry mg;
        const bq_status ms = bq::plan_multi_tables(qtype, ops, n_ops, mo.data(), ct.data(), &mg);
        if (ms == BQ_OK) {
            const int64_t off_ct = align256((int64_t)n_ops * sizeof(bq::MultiOp));
            if (cudaMemcpy(ws, mo.data(), (size_t)n_ops * sizeof(bq::MultiOp),
                           cudaMemcpyHostToDevice) != cudaSuccess ||
                cudaMemcpy(ws + off_ct, ct.data(), (size_t)(mg.grid + 1) * sizeof(int),
                           cudaMemcpyHostToDevice) != cudaSuccess)
                return BQ_ERR_CUDA;
            auto *p = new (std::nothrow) bq_stream_plan;
            if (!p) return BQ_ERR_CUDA;
            std::memset(p, 0, sizeof *p);
            p->mo_host = new (std::nothrow) bq::MultiOp[(size_t)n_ops];
            p->ct_host = new (std::nothrow) int[(size_t)mg.grid + 1];
            if (!p->mo_host || !p->ct_host) {
                delete[] p->mo_host;
                delete[] p->ct_host;
                delete p;
                return BQ_ERR_CUDA;
            }
            std::memcpy(p->mo_host, mo.data(), (size_t)n_ops * sizeof(bq::MultiOp));
            std::memcpy(p->ct_host, ct.data(), (size_t)(mg.grid + 1) * sizeof(int));
            p->qtype = qtype;
            p->n_ops = n_ops;
            p->n_stages = n_stages;
            p->multi = 1;
            cudaGetDevice(&p->device);
            p->grid = mg.grid;
            p->threads = mg.threads;
            p->smem = mg.smem;
            p->ct_dev = reinterpret_cast<int *>(ws + off_ct);
            p->cta_ns = reinterpret_cast<unsigned long long *>(
                ws + off_ct + align256((int64_t)(bq::MULTI_MAX_CTAS + 1) * 4));
            bq::fill_multi_args(mg, n_ops, reinterpret_cast<const bq::MultiOp *>(ws), p->ct_dev,
                                &p->margs);
            *plan = p;
            return BQ_OK;
        }
        // a list the multi-op kernel cannot hold falls back to the executor
    }
    const int kind = bq::g_plan_kind.load();
    if (!independent && (kind >= 0 ? kind == 1 : bq::tunables().plan_staged != 0)) {
        bq_stream_plan *p = nullptr;
        const bq_status ss = plan_staged(qtype, ops, n_ops, es.data(), n_stages, ws, &p);
        if (ss == BQ_OK) {
            *plan = p;
            return BQ_OK;
        }
        if (ss == BQ_ERR_CUDA) return ss;
        // a stage the streaming kernel cannot hold: the executor runs the list
    }
    const int64_t off_x = align256((int64_t)n_ops * sizeof(bq::ExecOp));
    const int64_t off_st = off_x + align256((int64_t)n_ops * sizeof(bq::ExecX));
    const int64_t off_cnt = off_st + align256((int64_t)n_stages * sizeof(bq::ExecStage));
    if (cudaMemcpy(ws, eo.data(), (size_t)n_ops * sizeof(bq::ExecOp), cudaMemcpyHostToDevice) !=
            cudaSuccess ||
        cudaMemcpy(ws + off_x, ex.data(), (size_t)geo.n_x * sizeof(bq::ExecX),
                   cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemcpy(ws + off_st, es.data(), (size_t)n_stages * sizeof(bq::ExecStage),
                   cudaMemcpyHostToDevice) != cudaSuccess)
        return BQ_ERR_CUDA;
    auto *p = new (std::nothrow) bq_stream_plan;
    if (!p) return BQ_ERR_CUDA;
    std::memset(p, 0, sizeof *p);
    p->qtype = qtype;
    p->n_ops = n_ops;
    p->n_stages = n_stages;
    p->multi = 0;
    cudaGetDevice(&p->device);
    p->grid = geo.grid;
    p->threads = geo.threads;
    p->smem = geo.smem;
    p->counters = reinterpret_cast<unsigned int *>(ws + off_cnt);
    bq::fill_exec_args(geo, n_ops, reinterpret_cast<const bq::ExecOp *>(ws),
                       reinterpret_cast<const bq::ExecX *>(ws + off_x),
                       reinterpret_cast<const bq::ExecStage *>(ws + off_st), p->counters, &p->args);
    *plan = p;
    return BQ_OK;
}

bq_status bq_stream_plan_launch(const bq_stream_plan *plan, void *stream) {
    if (!plan) return BQ_ERR_NULL;
    if (plan->stages) {
        for (int s = 0; s < plan->n_stages; ++s) {
            const bq::StageLaunch &l = plan->stages[s];
            const int e = bq::fmt_multi_launch(plan->qtype, l.args, l.grid, l.threads, l.smem,
                                               stream, l.pdl);
            if (e != 0) return BQ_ERR_CUDA;
        }
        return BQ_OK;
    }
    if (plan->multi) {
        const int pdl = bq::tunables().plan_pdl;
        const int e = bq::fmt_multi_launch(plan->qtype, plan->margs, plan->grid, plan->threads,
                                           plan->smem, stream, pdl);
        return from_cuda(e);
    }
    auto s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(plan->counters, 0, (size_t)plan->n_stages * 4, s) != cudaSuccess)
        return BQ_ERR_CUDA;
    const int e = bq::fmt_exec_launch(plan->qtype, plan->args, plan->grid, plan->threads,
                                      plan->smem, stream);
    return from_cuda(e);
}

bq_status bq_stream_plan_destroy(bq_stream_plan *plan) {
    if (plan) {
        delete[] plan->mo_host;
        delete[] plan->ct_host;
        delete[] plan->stages;
    }
    delete plan;
    return BQ_OK;
}

namespace {
// packed bytes of tile k of op o (rows of the tile times row bytes, per matrix)
long long tile_bytes(const bq::MultiOp &o, int k) {
    return (long long)std::min(o.rpw, o.M - k * o.rpw) * o.rb * o.nmat;
}
// Split n tiles (tile t has tb[t] bytes) into `grid` contiguous ranges of
// equal estimated time: tile t costs its bytes times the measured time per
// byte of the CTA that ran it in split `ct` (d[c] over the bytes of range c;
// a CTA that ran nothing, or has no measurement, takes the mean).  Op
// boundaries, idle lanes and per-tile work make the time per byte differ
// between op shapes and between ranges.  out[0] = 0, out[grid] = n.
void rebalance(const double *tb, long long n, int grid, const int *ct, const double *d, int *out) {
    std::vector<double> bytes((size_t)grid, 0.0), dens((size_t)grid, 0.0);
    auto owner_walk = [&](auto f) {  // f(tile, owner CTA in ct)
        int c = 0;
        for (long long t = 0; t < n; ++t) {
            while (c + 1 < grid && t >= ct[c + 1]) ++c;
            f(t, c);
        }
    };
    owner_walk([&](long long t, int c) { bytes[(size_t)c] += tb[t]; });
    double sb = 0.0, sd = 0.0;
    for (int c = 0; c < grid; ++c)
        if (bytes[(size_t)c] > 0 && d[c] > 0) sb += bytes[(size_t)c], sd += d[c];
    const double mean = sb > 0 ? sd / sb : 1.0;
    for (int c = 0; c < grid; ++c)
        dens[(size_t)c] = bytes[(size_t)c] > 0 && d[c] > 0 ? d[c] / bytes[(size_t)c] : mean;
    double total = 0.0;
    owner_walk([&](long long t, int c) { total += tb[t] * dens[(size_t)c]; });
    out[0] = 0;
    int o = 1;
    double acc = 0.0;
    // (a relative slack of 1e-12 closes a range at an exact tie despite the
    // rounding of the running sum)
    owner_walk([&](long long t, int c) {
        acc += tb[t] * dens[(size_t)c];
        while (o < grid && acc * grid >= total * o * (1.0 - 1e-12)) out[o++] = (int)t + 1;
    });
    while (o <= grid) out[o++] = (int)n;
}
}  // namespace

// Test hooks (not declared in include/bqgemv.h).  Failure detection: the
// limit of the kernels' bounded waits for launches planned from now on, and
// extra arrivals that a plan's stage barriers wait for, so that a test can
// make a barrier wait run out and read the device error word -- the kernel
// gives up after the limit and returns; nothing faults or hangs.
extern "C" void bq_internal_set_wait_limit_ns(unsigned long long ns) {
    bq::g_wait_ns.store(ns < 1000 ? 1000 : ns);
}
// how plans of dependent stages created from now on run: -1 by the
// BQ_PLAN tunable, 0 the cooperative executor, 1 one launch per stage
extern "C" void bq_internal_set_plan_kind(int kind) {
    bq::g_plan_kind.store(kind < 0 ? -1 : kind > 0 ? 1 : 0);
}
extern "C" int bq_internal_plan_barrier_extra(bq_stream_plan *plan, unsigned int extra,
                                              unsigned long long wait_ns) {
    if (!plan || plan->multi || plan->stages) return -1;  // only the executor has stage barriers
    plan->args.barrier_extra = extra;
    plan->args.wait_ns = wait_ns < 1000 ? 1000 : wait_ns;
    return 0;
}

// Host-logic hooks for the CPU test suite (not declared in include/bqgemv.h):
// the planner's lane-order search and the time-balanced tile split.
int bq_internal_lane_order(int G, int S0, int U, int pad, int rows_low, int *S, int *umask) {
    return bq::lane_order(G, S0, U, pad != 0, S, umask, rows_low != 0) ? 1 : 0;
}
void bq_internal_rebalance(const double *tile_bytes, long long n, int grid, const int *ct,
                           const double *cta_time, int *out) {
    rebalance(tile_bytes, n, grid, ct, cta_time, out);
}
void bq_internal_split_by_op(const long long *op_bytes, const int *op_tiles, int n, int grid, int *out) {
    bq::split_by_op(op_bytes, op_tiles, n, grid, out);
}

int bq_stream_plan_launches(const bq_stream_plan *plan) {
    if (!plan) return -1;
    return plan->stages ? plan->n_stages : 1;
}

bq_status bq_stream_plan_tune(bq_stream_plan *plan, int rounds, void *stream) {
    if (!plan) return BQ_ERR_NULL;
    if (rounds < 1 || rounds > 16) return BQ_ERR_SHAPE;
    if (!plan->multi) return BQ_OK;  // dependent stages: left as planned
    auto s = static_cast<cudaStream_t>(stream);
    const int grid = plan->grid;
    constexpr int REPS = 3;  // launches averaged per measurement
    std::vector<unsigned long long> ns((size_t)grid);
    std::vector<double> d((size_t)grid);
    std::vector<int> best((size_t)grid + 1), next((size_t)grid + 1);
    std::memcpy(best.data(), plan->ct_host, (size_t)(grid + 1) * sizeof(int));
    double best_max = -1.0;
    bq::MultiArgs a = plan->margs;
    a.cta_ns = plan->cta_ns;
    std::vector<double> tb;
    for (int i = 0; i < plan->n_ops; ++i)
        for (int k = 0; k < plan->mo_host[i].ntiles; ++k) tb.push_back((double)tile_bytes(plan->mo_host[i], k));
    for (int r = 0; r <= rounds; ++r) {
        std::fill(d.begin(), d.end(), 0.0);
        for (int k = 0; k < REPS; ++k) {
            if (cudaMemsetAsync(plan->cta_ns, 0, (size_t)grid * 8, s) != cudaSuccess) return BQ_ERR_CUDA;
            const int e = bq::fmt_multi_launch(plan->qtype, a, grid, plan->threads, plan->smem,
                                               stream, 0);
            if (e != 0) return BQ_ERR_CUDA;
            if (cudaMemcpyAsync(ns.data(), plan->cta_ns, (size_t)grid * 8, cudaMemcpyDeviceToHost, s) !=
                    cudaSuccess ||
                cudaStreamSynchronize(s) != cudaSuccess)
                return BQ_ERR_CUDA;
            for (int c = 0; c < grid; ++c) d[(size_t)c] += (double)ns[(size_t)c] / REPS;
        }
        const double mx = *std::max_element(d.begin(), d.end());
        if (best_max < 0 || mx < best_max) {
            best_max = mx;
            std::memcpy(best.data(), plan->ct_host, (size_t)(grid + 1) * sizeof(int));
        }
        if (r == rounds) break;
        rebalance(tb.data(), (long long)tb.size(), grid, plan->ct_host, d.data(), next.data());
        std::memcpy(plan->ct_host, next.data(), (size_t)(grid + 1) * sizeof(int));
        if (cudaMemcpyAsync(plan->ct_dev, plan->ct_host, (size_t)(grid + 1) * sizeof(int),
                            cudaMemcpyHostToDevice, s) != cudaSuccess)
            return BQ_ERR_CUDA;
    }
    // keep the split whose slowest CTA was fastest
    std::memcpy(plan->ct_host, best.data(), (size_t)(grid + 1) * sizeof(int));
    if (cudaMemcpyAsync(plan->ct_dev, plan->ct_host, (size_t)(grid + 1) * sizeof(int),
                        cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return BQ_ERR_CUDA;
    return BQ_OK;
}

bq_status bq_device_status(unsigned int *flags, int clear) {
    if (!flags) return BQ_ERR_NULL;
    if (cudaDeviceSynchronize() != cudaSuccess) return BQ_ERR_CUDA;
    unsigned int a = 0, b = 0, c = 0;
    if (bq_internal_status_q8_0(&a, clear) != 0) return BQ_ERR_CUDA;
    if (bq_internal_status_q4_0(&b, clear) != 0) return BQ_ERR_CUDA;
    if (bq_internal_status_q4_k(&c, clear) != 0) return BQ_ERR_CUDA;
    *flags = a | b | c;
    return *flags ? BQ_ERR_DEVICE : BQ_OK;
}

}  // extern "C"
