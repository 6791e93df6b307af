// bq_format_unit.cuh -- everything one block format's translation unit defines
// besides its multi-op kernel instances: the generic GEMV kernel and the stream
// executor instantiated for the format, their launchers, the dispatch among the
// multi-op kernel instances (which live in bq_multi_<format>_*.cu so that nvcc
// compiles them in parallel), and the format's device-side error word.
//
// BQ_FORMAT_UNIT(q8_0, bq::QT_Q8_0) in bq_gemv_q8_0.cu defines the
// bq_internal_*_q8_0 functions declared in bq_internal.h, and so on per format.
#pragma once

#include <atomic>

#include "bq_exec.cuh"
#include "bq_kernels.cuh"
#include "bq_multi.cuh"
#include "bq_occupancy.cuh"

namespace bq {
// the device address of a format's status word, looked up once per device
template <unsigned int *Sym>
cudaError_t status_addr_of(const void *symbol, unsigned int **out) {
    static std::atomic<unsigned int *> addr[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    unsigned int *status = addr[dev].load();
    if (!status) {
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&status), symbol);
        if (e != cudaSuccess) return e;
        addr[dev].store(status);
    }
    *out = status;
    return cudaSuccess;
}

inline cudaError_t exec_launch_coop(void (*kern)(ExecArgs, unsigned int *), const ExecArgs &a,
                                    int grid, int threads, size_t smem, void *stream,
                                    unsigned int *status) {
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
    return cudaLaunchKernelEx(&cfg, kern, a, status);
}
}  // namespace bq

#define BQ_MULTI_DECL(NAME, FMT)                                                                   \
    int bq_internal_multi_occupancy_##NAME##_##FMT(int nr, int R, int threads, size_t smem,        \
                                                   int *occ);                                      \
    int bq_internal_multi_launch_##NAME##_##FMT(const bq::MultiArgs &a, int grid, int threads,     \
                                                size_t smem, void *stream, int pdl,                \
                                                unsigned int *status);

#define BQ_FORMAT_UNIT(FMT, QT)                                                                    \
    __device__ unsigned int g_status_##FMT = 0;                                                    \
    namespace {                                                                                    \
    cudaError_t status_addr(unsigned int **out) {                                                  \
        return bq::status_addr_of<&g_status_##FMT>(&g_status_##FMT, out);                          \
    }                                                                                              \
    }                                                                                              \
    int bq_internal_launch_##FMT(const bq::GemvCall &c, const bq::LaunchPlan &p) {                 \
        return (int)bq::launch_gemv<QT>(c, p);                                                     \
    }                                                                                              \
    int bq_internal_exec_occupancy_##FMT(int threads, size_t smem, int *occ) {                     \
        return bq::occupancy_cached<bq::exec_kernel<QT>>(threads, smem, occ);                      \
    }                                                                                              \
    int bq_internal_exec_launch_##FMT(const bq::ExecArgs &a, int grid, int threads, size_t smem,   \
                                      void *stream) {                                              \
        unsigned int *status = nullptr;                                                            \
        cudaError_t e = status_addr(&status);                                                      \
        if (e != cudaSuccess) return (int)e;                                                       \
        return (int)bq::exec_launch_coop(bq::exec_kernel<QT>, a, grid, threads, smem, stream,      \
                                         status);                                                  \
    }                                                                                              \
    int bq_internal_status_##FMT(unsigned int *flags, int clear) {                                 \
        cudaError_t e = cudaMemcpyFromSymbol(flags, g_status_##FMT, sizeof(unsigned int));         \
        if (e != cudaSuccess) return (int)e;                                                       \
        if (clear) {                                                                               \
            const unsigned int zero = 0;                                                           \
            e = cudaMemcpyToSymbol(g_status_##FMT, &zero, sizeof(unsigned int));                   \
        }                                                                                          \
        return (int)e;                                                                             \
    }                                                                                              \
    BQ_MULTI_DECL(r1, FMT)                                                                         \
    BQ_MULTI_DECL(r234, FMT)                                                                       \
    BQ_MULTI_DECL(r56, FMT)                                                                        \
    int bq_internal_multi_occupancy_##FMT(int nr, int R, int threads, size_t smem, int *occ) {     \
        int e;                                                                                     \
        if ((e = bq_internal_multi_occupancy_r1_##FMT(nr, R, threads, smem, occ)) != -1) return e; \
        if ((e = bq_internal_multi_occupancy_r234_##FMT(nr, R, threads, smem, occ)) != -1)         \
            return e;                                                                              \
        if ((e = bq_internal_multi_occupancy_r56_##FMT(nr, R, threads, smem, occ)) != -1)          \
            return e;                                                                              \
        return (int)cudaErrorInvalidValue;                                                         \
    }                                                                                              \
    int bq_internal_multi_launch_##FMT(const bq::MultiArgs &a, int grid, int threads, size_t smem, \
                                       void *stream, int pdl) {                                    \
        unsigned int *status = nullptr;                                                            \
        cudaError_t e = status_addr(&status);                                                      \
        if (e != cudaSuccess) return (int)e;                                                       \
        int r;                                                                                     \
        if ((r = bq_internal_multi_launch_r1_##FMT(a, grid, threads, smem, stream, pdl, status)) != -1) \
            return r;                                                                              \
        if ((r = bq_internal_multi_launch_r234_##FMT(a, grid, threads, smem, stream, pdl, status)) != \
            -1)                                                                                    \
            return r;                                                                              \
        if ((r = bq_internal_multi_launch_r56_##FMT(a, grid, threads, smem, stream, pdl, status)) != \
            -1)                                                                                    \
            return r;                                                                              \
        return (int)cudaErrorInvalidValue;                                                         \
    }
