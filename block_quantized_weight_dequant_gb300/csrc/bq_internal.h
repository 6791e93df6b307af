// bq_internal.h -- host-side types shared by the C-ABI layer (bq_api.cu) and
// the per-format kernel translation units.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>

namespace bq {

constexpr int MODE_PLAIN = 0;    // y = W x  (R input rows: R = 1 decode, R > 1 verify)
constexpr int MODE_GATE_UP = 1;  // y = silu(Wg xn) * (Wu xn)

struct GemvCall {
    int qtype, mode, R;
    const void *W0, *W1;
    const float *x, *gamma;
    float eps;
    float *y;
    long long M, K;
    void *stream;
    const float *bias;  // MODE_PLAIN with R = 1: added to every output row, or null
};

// generic-kernel geometry (K % 256 != 0).  G fixes the row's summation tree.
struct LaunchPlan {
    int G;           // lanes per row
    long long rb;    // packed bytes per row
};

// lanes per row for a row of nsc units: the largest power of two G <= 32 whose
// padding to a multiple of G wastes at most 1/8 of the lane slots
int tree_lanes_for_units(long long nsc);

// plan a generic-kernel GEMV call
void plan_gemv(const GemvCall &c, LaunchPlan *p);

}  // namespace bq

// per-format generic launchers (one translation unit each) and their device status words
int bq_internal_launch_q8_0(const bq::GemvCall &c, const bq::LaunchPlan &p);
int bq_internal_launch_q4_0(const bq::GemvCall &c, const bq::LaunchPlan &p);
int bq_internal_launch_q4_k(const bq::GemvCall &c, const bq::LaunchPlan &p);
int bq_internal_status_q8_0(unsigned int *flags, int clear);
int bq_internal_status_q4_0(unsigned int *flags, int clear);
int bq_internal_status_q4_k(unsigned int *flags, int clear);
int bq_internal_pack(int qtype, const float *W, long long M, long long K, void *Wq, void *stream);
// the fp16-weight GEMV (bq_f16.cu), arguments validated by the caller
int bq_internal_f16_launch(const void *W, const float *x, float *y, long long M, long long K,
                           void *stream);

#include "../../include/bqgemv.h"

namespace bq {
struct ExecArgs;
struct ExecOp;
struct ExecX;
struct ExecStage;
struct ExecGeometry;
// Validate a stream executor op list and plan it into caller-provided tables
// (each with room for n_ops entries) and a launch geometry for the current
// device.  Touches no device memory.
bq_status plan_exec_tables(int qtype, const bq_op *ops, int n_ops, ExecOp *eo, ExecX *ex,
                           ExecStage *es, ExecGeometry *geo);
// kernel arguments for planned tables at the given device addresses
void fill_exec_args(const ExecGeometry &geo, int n_ops, const ExecOp *ops, const ExecX *xs,
                    const ExecStage *stages, unsigned int *counters, ExecArgs *a);

struct MultiOp;
struct MultiArgs;
constexpr int MULTI_MAX_CTAS = 1024;
// launch geometry of a multi-op kernel run
struct MultiGeometry {
    int grid, threads, nwarps, D, slot_bytes, x_off, ring_off, nr, R;
    int x_rstride, x_floats, x_buffers, panel_units;
    size_t smem;
};
// Plan a list of ops none of which depends on another (validated by
// plan_exec_tables) for the multi-op streaming kernel: per-op tiles and a
// byte-balanced contiguous tile range per CTA (cta_tiles: room for
// MULTI_MAX_CTAS + 1 entries).  Touches no device memory.
bq_status plan_multi_tables(int qtype, const bq_op *ops, int n_ops, MultiOp *mo, int *cta_tiles,
                            MultiGeometry *geo);
void fill_multi_args(const MultiGeometry &geo, int n_ops, const MultiOp *ops,
                     const int *cta_tiles, MultiArgs *a);
// Plan one GEMV, gate+up or verify call (K % 256 == 0) as an inline op of the
// multi-op kernel; false if it cannot be planned.
// pair: gate+up calls may take the paired instance (single calls; the stages
// of a staged plan keep the sequential one, which measured faster there)
bool plan_multi_single(const GemvCall &c, MultiArgs *a, MultiGeometry *geo, bool pair = true);
// whether independent op lists use the multi-op kernel (tuning switch)
bool tunables_multi();
}
// per-format occupancy and launch of the multi-op kernel instance (nr, R);
// `pdl` allows programmatic dependent launch (single calls)
#define BQ_FORMAT_DECLS(FMT)                                                                       \
    int bq_internal_multi_occupancy_##FMT(int nr, int R, int threads, size_t smem, int *occ);      \
    int bq_internal_multi_launch_##FMT(const bq::MultiArgs &a, int grid, int threads, size_t smem, \
                                       void *stream, int pdl);                                     \
    int bq_internal_exec_occupancy_##FMT(int threads, size_t smem, int *occ);                      \
    int bq_internal_exec_launch_##FMT(const bq::ExecArgs &a, int grid, int threads, size_t smem,   \
                                      void *stream);
// (the persistent per-token stream executor is bq_exec.cuh, one instance per format)
BQ_FORMAT_DECLS(q8_0)
BQ_FORMAT_DECLS(q4_0)
BQ_FORMAT_DECLS(q4_k)

// dispatch on the format (qtype already validated: BQ_Q8_0, BQ_Q4_0 or BQ_Q4_K)
namespace bq {
inline int fmt_generic_launch(const GemvCall &c, const LaunchPlan &p) {
    return c.qtype == BQ_Q8_0 ? bq_internal_launch_q8_0(c, p)
           : c.qtype == BQ_Q4_0 ? bq_internal_launch_q4_0(c, p)
                                : bq_internal_launch_q4_k(c, p);
}
inline int fmt_multi_occupancy(int qt, int nr, int R, int threads, size_t smem, int *occ) {
    return qt == BQ_Q8_0 ? bq_internal_multi_occupancy_q8_0(nr, R, threads, smem, occ)
           : qt == BQ_Q4_0 ? bq_internal_multi_occupancy_q4_0(nr, R, threads, smem, occ)
                           : bq_internal_multi_occupancy_q4_k(nr, R, threads, smem, occ);
}
inline int fmt_multi_launch(int qt, const MultiArgs &a, int grid, int threads, size_t smem,
                            void *stream, int pdl) {
    return qt == BQ_Q8_0 ? bq_internal_multi_launch_q8_0(a, grid, threads, smem, stream, pdl)
           : qt == BQ_Q4_0 ? bq_internal_multi_launch_q4_0(a, grid, threads, smem, stream, pdl)
                           : bq_internal_multi_launch_q4_k(a, grid, threads, smem, stream, pdl);
}
inline int fmt_exec_occupancy(int qt, int threads, size_t smem, int *occ) {
    return qt == BQ_Q8_0 ? bq_internal_exec_occupancy_q8_0(threads, smem, occ)
           : qt == BQ_Q4_0 ? bq_internal_exec_occupancy_q4_0(threads, smem, occ)
                           : bq_internal_exec_occupancy_q4_k(threads, smem, occ);
}
inline int fmt_exec_launch(int qt, const ExecArgs &a, int grid, int threads, size_t smem,
                           void *stream) {
    return qt == BQ_Q8_0 ? bq_internal_exec_launch_q8_0(a, grid, threads, smem, stream)
           : qt == BQ_Q4_0 ? bq_internal_exec_launch_q4_0(a, grid, threads, smem, stream)
                           : bq_internal_exec_launch_q4_k(a, grid, threads, smem, stream);
}
}  // namespace bq
