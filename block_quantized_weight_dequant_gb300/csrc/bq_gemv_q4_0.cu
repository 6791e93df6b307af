// bq_gemv_q4_0.cu -- the Q4_0 instantiations of the GEMV kernels (one
// translation unit per format so the two compile in parallel) and this
// unit's device-side error word.
#include <atomic>

#include "bq_exec.cuh"
#include "bq_multi.cuh"
#include "bq_kernels.cuh"

namespace {
__device__ unsigned int g_status_q4_0 = 0;
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
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_status_q4_0);
        if (e != cudaSuccess) return e;
        addr[dev].store(status);
    }
    *out = status;
    return cudaSuccess;
}
}  // namespace

int bq_internal_launch_q4_0(const bq::GemvCall &c, const bq::LaunchPlan &p) {
    unsigned int *status = nullptr;
    cudaError_t e = status_addr(&status);
    if (e != cudaSuccess) return (int)e;
    (void)status;
    return (int)bq::launch_gemv<bq::QT_Q4_0>(c, p);
}

int bq_internal_exec_occupancy_q4_0(int threads, size_t smem, int *occ) {
    auto kern = bq::exec_kernel<bq::QT_Q4_0>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    return (int)cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, kern, threads, smem);
}

int bq_internal_exec_launch_q4_0(const bq::ExecArgs &a, int grid, int threads, size_t smem,
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
    return (int)cudaLaunchKernelEx(&cfg, bq::exec_kernel<bq::QT_Q4_0>, a, status);
}

int bq_internal_status_q4_0(unsigned int *flags, int clear) {
    cudaError_t e = cudaMemcpyFromSymbol(flags, g_status_q4_0, sizeof(unsigned int));
    if (e != cudaSuccess) return (int)e;
    if (clear) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_status_q4_0, &zero, sizeof(unsigned int));
    }
    return (int)e;
}

namespace {
template <int NR, int R>
int multi_occupancy(int threads, size_t smem, int *occ) {
    auto kern = bq::multi_kernel<bq::QT_Q4_0, NR, R>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return (int)e;
    return (int)cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, kern, threads, smem);
}

template <int NR, int R>
int multi_launch(const bq::MultiArgs &a, int grid, int threads, size_t smem, void *stream, int pdl,
                 unsigned int *status) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return (int)cudaLaunchKernelEx(&cfg, bq::multi_kernel<bq::QT_Q4_0, NR, R>, a, status);
}
}  // namespace

// instances: NR = 1 for R = 1..6 (decode, gate+up, verify); NR = 2 and row mode
// (NR = 0) for R = 1
int bq_internal_multi_occupancy_q4_0(int nr, int R, int threads, size_t smem, int *occ) {
    if (nr == 2 && R == 1) return multi_occupancy<2, 1>(threads, smem, occ);
    if (nr == 0 && R == 1) return multi_occupancy<0, 1>(threads, smem, occ);
    if (nr != 1) return (int)cudaErrorInvalidValue;
    switch (R) {
        case 1: return multi_occupancy<1, 1>(threads, smem, occ);
        case 2: return multi_occupancy<1, 2>(threads, smem, occ);
        case 3: return multi_occupancy<1, 3>(threads, smem, occ);
        case 4: return multi_occupancy<1, 4>(threads, smem, occ);
        case 5: return multi_occupancy<1, 5>(threads, smem, occ);
        case 6: return multi_occupancy<1, 6>(threads, smem, occ);
        default: return (int)cudaErrorInvalidValue;
    }
}

int bq_internal_multi_launch_q4_0(const bq::MultiArgs &a, int grid, int threads, size_t smem,
                                void *stream, int pdl) {
    unsigned int *status = nullptr;
    cudaError_t e = status_addr(&status);
    if (e != cudaSuccess) return (int)e;
    if (a.nr == 2 && a.R == 1) return multi_launch<2, 1>(a, grid, threads, smem, stream, pdl, status);
    if (a.nr == 0 && a.R == 1) return multi_launch<0, 1>(a, grid, threads, smem, stream, pdl, status);
    if (a.nr != 1) return (int)cudaErrorInvalidValue;
    switch (a.R) {
        case 1: return multi_launch<1, 1>(a, grid, threads, smem, stream, pdl, status);
        case 2: return multi_launch<1, 2>(a, grid, threads, smem, stream, pdl, status);
        case 3: return multi_launch<1, 3>(a, grid, threads, smem, stream, pdl, status);
        case 4: return multi_launch<1, 4>(a, grid, threads, smem, stream, pdl, status);
        case 5: return multi_launch<1, 5>(a, grid, threads, smem, stream, pdl, status);
        case 6: return multi_launch<1, 6>(a, grid, threads, smem, stream, pdl, status);
        default: return (int)cudaErrorInvalidValue;
    }
}
