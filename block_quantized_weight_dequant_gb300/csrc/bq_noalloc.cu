// bq_noalloc.cu -- the per-token stream executor for callers that cannot
// allocate device memory (bq_stream_run_noalloc in include/bqgemv.h).
//
// The regular executor keeps its descriptor tables and stage-barrier counters
// in a workspace the caller allocates.  This entry point keeps them instead in
// one file-scope device array of fixed size, which every GPU that loads the
// library holds until the process exits.  Nothing is allocated per call: the
// host side plans into static arrays, copies the tables into the device array
// on the caller's stream, clears the counters, and launches: the multi-op
// streaming kernel for independent ops, as the workspace path does, and the
// cooperative executor for dependent stages (the workspace path runs those as
// one launch per stage, whose per-stage tables would not fit the array).
//
// The copies read the static host arrays asynchronously: CUDA does not promise
// that a copy from pageable memory has read its source when cudaMemcpyAsync
// returns.  So after the copies each call records a per-device event, and the
// next call waits for that event before it refills the arrays.  (Events are
// created once per device at set-up; they hold no device memory.)
#include <cuda_runtime.h>

#include <mutex>

#include "bq_exec.cuh"
#include "bq_multi.cuh"
#include "bq_internal.h"

namespace {

constexpr size_t al256(size_t v) { return (v + 255) / 256 * 256; }

constexpr int MAX_OPS = BQ_NOALLOC_MAX_OPS;  // also the most stages and inputs
constexpr size_t OFF_X = al256((size_t)MAX_OPS * sizeof(bq::ExecOp));
constexpr size_t OFF_ST = OFF_X + al256((size_t)MAX_OPS * sizeof(bq::ExecX));
constexpr size_t OFF_CNT = OFF_ST + al256((size_t)MAX_OPS * sizeof(bq::ExecStage));
constexpr size_t SCRATCH_BYTES = OFF_CNT + al256((size_t)MAX_OPS * sizeof(unsigned int));

// The scratch: descriptor tables, then one barrier counter per stage.  In host
// code this name is only a stand-in for the symbol; the kernel gets the
// device address fetched by scratch_address().
static __device__ __align__(256) unsigned char g_noalloc_scratch[SCRATCH_BYTES];
static_assert(SCRATCH_BYTES == 82 * 1024, "the documented size of the scratch array");
// the same array holds the multi-op kernel's tables for independent op lists
constexpr size_t OFF_CT = al256((size_t)MAX_OPS * sizeof(bq::MultiOp));
static_assert(OFF_CT + (bq::MULTI_MAX_CTAS + 1) * sizeof(int) <= SCRATCH_BYTES,
              "multi-op tables fit the scratch array");

// host staging for the tables: static storage, one call at a time (under
// g_host_mutex, which also guards the per-device set-up below)
std::mutex g_host_mutex;
bq::ExecOp g_eo[MAX_OPS];
bq::ExecX g_ex[MAX_OPS];
bq::ExecStage g_es[MAX_OPS];
bq::MultiOp g_mo[MAX_OPS];
int g_ct[bq::MULTI_MAX_CTAS + 1];

// per device: the scratch's device address and the event recorded after the
// last call's table copies on that device
unsigned char *g_scratch_addr[64];
cudaEvent_t g_copied[64];
// the event of the last call (any device): its copies read the host arrays
cudaEvent_t g_pending = nullptr;

// Set-up of the current device on its first call (make that first call before
// any stream capture): the device address of the scratch array and the event.
// Caller holds g_host_mutex.
cudaError_t device_setup(int *dev_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!g_scratch_addr[dev]) {
        unsigned char *p = nullptr;
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&p), g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        cudaEvent_t ev = nullptr;
        e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
        if (e != cudaSuccess) return e;
        g_copied[dev] = ev;
        g_scratch_addr[dev] = p;
    }
    *dev_out = dev;
    return cudaSuccess;
}

}  // namespace

extern "C" bq_status bq_stream_run_noalloc(int qtype, const bq_op *ops, int n_ops, void *stream) {
    if (qtype != BQ_Q8_0 && qtype != BQ_Q4_0 && qtype != BQ_Q4_K) return BQ_ERR_QTYPE;
    if (!ops) return BQ_ERR_NULL;
    if (n_ops < 1 || n_ops > MAX_OPS) return BQ_ERR_SHAPE;
    auto s = static_cast<cudaStream_t>(stream);
    std::lock_guard<std::mutex> lock(g_host_mutex);
    int dev = 0;
    if (device_setup(&dev) != cudaSuccess) return BQ_ERR_CUDA;
    unsigned char *scratch = g_scratch_addr[dev];
    // the previous call's copies must have read the host arrays before they
    // are refilled
    if (g_pending && cudaEventSynchronize(g_pending) != cudaSuccess) return BQ_ERR_CUDA;
    g_pending = nullptr;
    auto copies_queued = [&]() {
        if (cudaEventRecord(g_copied[dev], s) != cudaSuccess) return false;
        g_pending = g_copied[dev];
        return true;
    };
    bq::ExecGeometry geo;
    const bq_status st = bq::plan_exec_tables(qtype, ops, n_ops, g_eo, g_ex, g_es, &geo);
    if (st != BQ_OK) return st;
    // independent ops run on the multi-op streaming kernel, as in a plan
    bool independent = bq::tunables_multi();
    for (int i = 0; i < geo.n_stages; ++i) independent &= !g_es[i].barrier;
    bq::MultiGeometry mg;
    if (independent && bq::plan_multi_tables(qtype, ops, n_ops, g_mo, g_ct, &mg) == BQ_OK) {
        const bool copied =
            cudaMemcpyAsync(scratch, g_mo, (size_t)n_ops * sizeof(bq::MultiOp),
                            cudaMemcpyHostToDevice, s) == cudaSuccess &&
            cudaMemcpyAsync(scratch + OFF_CT, g_ct, (size_t)(mg.grid + 1) * sizeof(int),
                            cudaMemcpyHostToDevice, s) == cudaSuccess;
        // recorded even after a failed copy: an earlier one may be in flight
        if (!copies_queued() || !copied) return BQ_ERR_CUDA;
        bq::MultiArgs ma;
        bq::fill_multi_args(mg, n_ops, reinterpret_cast<const bq::MultiOp *>(scratch),
                            reinterpret_cast<const int *>(scratch + OFF_CT), &ma);
        const int e = bq::fmt_multi_launch(qtype, ma, mg.grid, mg.threads, mg.smem, stream, 0);
        return e == 0 ? BQ_OK : BQ_ERR_CUDA;
    }
    const bool copied =
        cudaMemcpyAsync(scratch, g_eo, (size_t)n_ops * sizeof(bq::ExecOp), cudaMemcpyHostToDevice,
                        s) == cudaSuccess &&
        cudaMemcpyAsync(scratch + OFF_X, g_ex, (size_t)geo.n_x * sizeof(bq::ExecX),
                        cudaMemcpyHostToDevice, s) == cudaSuccess &&
        cudaMemcpyAsync(scratch + OFF_ST, g_es, (size_t)geo.n_stages * sizeof(bq::ExecStage),
                        cudaMemcpyHostToDevice, s) == cudaSuccess;
    if (!copies_queued() || !copied) return BQ_ERR_CUDA;
    // the counters keep the previous call's values: clear them
    if (cudaMemsetAsync(scratch + OFF_CNT, 0, (size_t)geo.n_stages * sizeof(unsigned int), s) !=
        cudaSuccess)
        return BQ_ERR_CUDA;
    bq::ExecArgs a;
    bq::fill_exec_args(geo, n_ops, reinterpret_cast<const bq::ExecOp *>(scratch),
                       reinterpret_cast<const bq::ExecX *>(scratch + OFF_X),
                       reinterpret_cast<const bq::ExecStage *>(scratch + OFF_ST),
                       reinterpret_cast<unsigned int *>(scratch + OFF_CNT), &a);
    const int e = bq::fmt_exec_launch(qtype, a, geo.grid, geo.threads, geo.smem, stream);
    return e == 0 ? BQ_OK : BQ_ERR_CUDA;
}
