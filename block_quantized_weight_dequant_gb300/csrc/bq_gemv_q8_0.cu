// bq_gemv_q8_0.cu -- the Q8_0 instantiations of the generic GEMV kernel and the stream
// executor, the dispatch among the multi-op kernel instances, and this
// format's device-side error word.
#include <atomic>

#include "bq_exec.cuh"
#include "bq_multi.cuh"
#include "bq_kernels.cuh"

namespace {
__device__ unsigned int g_status_q8_0 = 0;
}

namespace {
// the status word's device address, looked up once per device
cudaError_t status_addr(unsigned int **out) {
    static std::atomic<unsigned int *> addr[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    unsigned int *status = addr[dev].load();
    if (!status) {
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_status_q8_0);
        if (e != cudaSuccess) return e;
        addr[dev].store(status);
    }
    *out = status;
    return cudaSuccess;
}
}  // namespace

int bq_internal_launch_q8_0(const bq::GemvCall &c, const bq::LaunchPlan &p) {
    unsigned int *status = nullptr;
    cudaError_t e = status_addr(&status);
    if (e != cudaSuccess) return (int)e;
    (void)status;
    return (int)bq::launch_gemv<bq::QT_Q8_0>(c, p);
}

int bq_internal_exec_occupancy_q8_0(int threads, size_t smem, int *occ) {
    auto kern = bq::exec_kernel<bq::QT_Q8_0>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    return (int)cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, kern, threads, smem);
}

int bq_internal_exec_launch_q8_0(const bq::ExecArgs &a, int grid, int threads, size_t smem,
                               void *stream) {
    unsigned int *status = nullptr;
    cudaError_t e = status_addr(&status);
    if (e != cudaSuccess) return (int)e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return (int)cudaLaunchKernelEx(&cfg, bq::exec_kernel<bq::QT_Q8_0>, a, status);
}

int bq_internal_status_q8_0(unsigned int *flags, int clear) {
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_status_q8_0, sizeof(unsigned int));
    if (e != cudaSuccess) return (int)e;
    if (clear) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_status_q8_0, &zero, sizeof(unsigned int));
    }
    return (int)e;
}

// the multi-op kernel instances live in bq_multi_q8_0_*.cu
int bq_internal_multi_occupancy_r1_q8_0(int nr, int R, int threads, size_t smem, int *occ);
int bq_internal_multi_launch_r1_q8_0(const bq::MultiArgs &a, int grid, int threads, size_t smem,
                                  void *stream, int pdl, unsigned int *status);
int bq_internal_multi_occupancy_r234_q8_0(int nr, int R, int threads, size_t smem, int *occ);
int bq_internal_multi_launch_r234_q8_0(const bq::MultiArgs &a, int grid, int threads, size_t smem,
                                  void *stream, int pdl, unsigned int *status);
int bq_internal_multi_occupancy_r56_q8_0(int nr, int R, int threads, size_t smem, int *occ);
int bq_internal_multi_launch_r56_q8_0(const bq::MultiArgs &a, int grid, int threads, size_t smem,
                                  void *stream, int pdl, unsigned int *status);

int bq_internal_multi_occupancy_q8_0(int nr, int R, int threads, size_t smem, int *occ) {
    int e;
    if ((e = bq_internal_multi_occupancy_r1_q8_0(nr, R, threads, smem, occ)) != -1) return e;
    if ((e = bq_internal_multi_occupancy_r234_q8_0(nr, R, threads, smem, occ)) != -1) return e;
    if ((e = bq_internal_multi_occupancy_r56_q8_0(nr, R, threads, smem, occ)) != -1) return e;
    return (int)cudaErrorInvalidValue;
}

int bq_internal_multi_launch_q8_0(const bq::MultiArgs &a, int grid, int threads, size_t smem,
                                void *stream, int pdl) {
    unsigned int *status = nullptr;
    cudaError_t e = status_addr(&status);
    if (e != cudaSuccess) return (int)e;
    int r;
    if ((r = bq_internal_multi_launch_r1_q8_0(a, grid, threads, smem, stream, pdl, status)) != -1) return r;
    if ((r = bq_internal_multi_launch_r234_q8_0(a, grid, threads, smem, stream, pdl, status)) != -1) return r;
    if ((r = bq_internal_multi_launch_r56_q8_0(a, grid, threads, smem, stream, pdl, status)) != -1) return r;
    return (int)cudaErrorInvalidValue;
}
