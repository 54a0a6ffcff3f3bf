// context_id.h -- the unique id of the calling thread's current CUDA context.
//
// The library keeps a few per-device host records (the error word's and the
// no-allocation scratch array's device addresses, the dynamic shared memory a
// kernel was opened up to). They belong to one context: cudaDeviceReset ends
// the device's primary context, and the next runtime call makes a new one in
// which the library's device code is loaded again, at other addresses and
// with default kernel attributes. Each record therefore keeps the id of the
// context it was filled in, and is filled again when the current context's id
// differs. The driver never reuses an id within a process.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

namespace pkv {

// The current context's id, or 0 when there is none yet (no runtime call has
// made one current on this thread) or the driver cannot say.
inline unsigned long long current_context_id() {
    using GetCurrentFn = CUresult (*)(CUcontext *);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long *);
    static std::atomic<GetCurrentFn> get_current{nullptr};
    static std::atomic<GetIdFn> get_id{nullptr};
    GetCurrentFn cur = get_current.load(std::memory_order_acquire);
    GetIdFn gid = get_id.load(std::memory_order_acquire);
    if (!cur || !gid) {
        void *a = nullptr, *b = nullptr;
        cudaDriverEntryPointQueryResult qa, qb;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 4000, cudaEnableDefault, &qa) !=
                cudaSuccess ||
            qa != cudaDriverEntryPointSuccess || !a)
            return 0;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) !=
                cudaSuccess ||
            qb != cudaDriverEntryPointSuccess || !b)
            return 0;
        cur = reinterpret_cast<GetCurrentFn>(a);
        gid = reinterpret_cast<GetIdFn>(b);
        get_current.store(cur, std::memory_order_release);
        get_id.store(gid, std::memory_order_release);
    }
    CUcontext ctx = nullptr;
    if (cur(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    unsigned long long id = 0;
    if (gid(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

}  // namespace pkv
