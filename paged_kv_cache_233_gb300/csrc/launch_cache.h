// launch_cache.h -- per-device host records shared by the kernel launchers:
// the dynamic shared memory a kernel has been opened up to, and the result of
// its occupancy query for the last shared-memory size asked about. Both are
// read and written with atomics, so host threads may launch concurrently.
#pragma once

#include <atomic>

#include <cuda_runtime.h>

#include "context_id.h"

namespace pkv {

constexpr int kLaunchCacheDevices = 64;

// Raises `kernel`'s dynamic shared-memory limit to at least `smem` bytes on
// device `dev`, calling the runtime only when this record is below `smem` or
// was made in another context (a kernel attribute belongs to the context the
// kernel was loaded in; cudaDeviceReset replaces it). The record packs the low
// 32 bits of the context id with the size; the attribute call itself is
// idempotent, so two threads racing here both succeed. Devices past the
// record's range are opened on every call.
template <typename Kernel>
cudaError_t open_dynamic_smem(std::atomic<unsigned long long> *opened, int dev, Kernel kernel,
                              int smem) {
    const unsigned long long ctx = current_context_id() & 0xffffffffull;
    const bool cached = ctx != 0 && dev >= 0 && dev < kLaunchCacheDevices;
    if (cached) {
        const unsigned long long r = opened[dev].load(std::memory_order_acquire);
        if ((r >> 32) == ctx && int(r & 0xffffffffull) >= smem) return cudaSuccess;
    }
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess || !cached) return e;
    const unsigned long long want = (ctx << 32) | unsigned(smem);
    unsigned long long cur = opened[dev].load(std::memory_order_relaxed);
    // keep the larger size of the same context; a record of another context is replaced
    while (((cur >> 32) != ctx || int(cur & 0xffffffffull) < smem) &&
           !opened[dev].compare_exchange_weak(cur, want, std::memory_order_acq_rel))
    {
    }
    return cudaSuccess;
}

// Resident CTAs per SM of `kernel` at `threads` threads and `smem` bytes of
// dynamic shared memory on device `dev`. The record packs (smem, result) in
// one word, so a reader sees a matching pair; a size other than the last one
// asked about is queried again.
template <typename Kernel>
cudaError_t occupancy_per_sm(std::atomic<long long> *record, int dev, Kernel kernel, int threads,
                             int smem, int *per_sm) {
    const bool cached = dev >= 0 && dev < kLaunchCacheDevices;
    if (cached) {
        const long long r = record[dev].load(std::memory_order_acquire);
        if (r > 0 && int(r >> 32) == smem) {
            *per_sm = int(r & 0xffffffffLL);
            return cudaSuccess;
        }
    }
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem);
    if (e != cudaSuccess) return e;
    *per_sm = n;
    if (cached && n > 0)
        record[dev].store((static_cast<long long>(smem) << 32) | n, std::memory_order_release);
    return cudaSuccess;
}

}  // namespace pkv
