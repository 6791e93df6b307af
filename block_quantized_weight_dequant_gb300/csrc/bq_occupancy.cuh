// bq_occupancy.cuh -- per-device cache of a kernel's dynamic shared-memory
// limit and of its last occupancy query, so that a single GEMV call of a shape
// seen before makes no CUDA attribute or occupancy call on the host.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

namespace bq {

// Blocks of `Kern` per SM with `threads` threads and `smem` bytes of dynamic
// shared memory on the current device (0 or a cudaError_t).  The kernel's
// dynamic shared-memory limit is raised only when a call needs more than any
// earlier call on that device, under a lock so that concurrent callers never
// lower it; the last (threads, smem) query of each device is remembered.
template <auto Kern>
int occupancy_cached(int threads, size_t smem, int *occ) {
    constexpr int NDEV = 64;
    static std::atomic<int> limit[NDEV];                   // dynamic smem set so far
    static std::atomic<unsigned long long> last[NDEV];     // threads<<40 | smem<<8 | occ
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    if (dev < 0 || dev >= NDEV || threads < 1 || threads > 1024 || smem >= (1u << 30))
        return (int)cudaErrorInvalidValue;
    const unsigned long long key = (unsigned long long)threads << 40 | (unsigned long long)smem << 8;
    const unsigned long long hit = last[dev].load(std::memory_order_acquire);
    if (hit && (hit & ~0xFFull) == key) {
        *occ = (int)(hit & 0xFF);
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    if ((int)smem > limit[dev].load()) {
        e = cudaFuncSetAttribute(Kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return (int)e;
        limit[dev].store((int)smem);
    }
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, Kern, threads, smem);
    if (e != cudaSuccess) return (int)e;
    *occ = n;
    if (n >= 0 && n < 256) last[dev].store(key | (unsigned long long)n, std::memory_order_release);
    return 0;
}

}  // namespace bq
