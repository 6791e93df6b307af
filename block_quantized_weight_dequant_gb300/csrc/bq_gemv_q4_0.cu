// bq_gemv_q4_0.cu -- the Q4_0 instantiations of the GEMV kernels (one
// translation unit per format so the two compile in parallel) and this
// unit's device-side error word.
#include "bq_kernels.cuh"

namespace {
__device__ unsigned int g_status_q4_0 = 0;
}

int bq_internal_launch_q4_0(const bq::GemvCall &c, const bq::LaunchPlan &p) {
    // the status word's device address, looked up once per device
    static unsigned int *addr[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    if (dev < 0 || dev >= 64) return (int)cudaErrorInvalidDevice;
    unsigned int *status = addr[dev];
    if (!status) {
        e = cudaGetSymbolAddress(reinterpret_cast<void **>(&status), g_status_q4_0);
        if (e != cudaSuccess) return (int)e;
        addr[dev] = status;
    }
    return (int)bq::launch_gemv<bq::QT_Q4_0>(c, p, status);
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
