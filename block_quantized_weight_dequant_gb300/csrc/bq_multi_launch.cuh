// bq_multi_launch.cuh -- occupancy query and launch of one multi-op kernel
// instance (format QT, NR weight rows per lane, R input rows).  The instances
// are spread over several translation units (bq_multi_<format>_<rows>.cu) so
// they compile in parallel; bq_gemv_<format>.cu dispatches among them.
#pragma once

#include <cuda_runtime.h>

#include "bq_multi.cuh"
#include "bq_occupancy.cuh"

namespace bq {

template <int QT, int NR, int R>
int multi_occupancy_t(int threads, size_t smem, int *occ) {
    return occupancy_cached<multi_kernel<QT, NR, R>>(threads, smem, occ);
}

// pdl: allow programmatic dependent launch (the kernel waits for its
// predecessor with griddepcontrol.wait before reading any input)
template <int QT, int NR, int R>
int multi_launch_t(const MultiArgs &a, int grid, int threads, size_t smem, void *stream, int pdl,
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
    return (int)cudaLaunchKernelEx(&cfg, multi_kernel<QT, NR, R>, a, status);
}

}  // namespace bq

// one translation unit's instance set: a table of (NR, R) pairs
#define BQ_MULTI_UNIT(FMT, QT, NAME, ...)                                                          \
    namespace {                                                                                    \
    struct Inst {                                                                                  \
        int nr, R;                                                                                 \
        int (*occ)(int, size_t, int *);                                                            \
        int (*launch)(const bq::MultiArgs &, int, int, size_t, void *, int, unsigned int *);       \
    };                                                                                             \
    const Inst kInst[] = {__VA_ARGS__};                                                            \
    }                                                                                              \
    int bq_internal_multi_occupancy_##NAME##_##FMT(int nr, int R, int threads, size_t smem,        \
                                                   int *occ) {                                     \
        for (const Inst &i : kInst)                                                                \
            if (i.nr == nr && i.R == R) return i.occ(threads, smem, occ);                          \
        return -1;                                                                                 \
    }                                                                                              \
    int bq_internal_multi_launch_##NAME##_##FMT(const bq::MultiArgs &a, int grid, int threads,     \
                                                size_t smem, void *stream, int pdl,                \
                                                unsigned int *status) {                            \
        for (const Inst &i : kInst)                                                                \
            if (i.nr == a.nr && i.R == a.R) return i.launch(a, grid, threads, smem, stream, pdl, status); \
        return -1;                                                                                 \
    }
#define BQ_INST(QT, NR, R) {NR, R, bq::multi_occupancy_t<QT, NR, R>, bq::multi_launch_t<QT, NR, R>}
