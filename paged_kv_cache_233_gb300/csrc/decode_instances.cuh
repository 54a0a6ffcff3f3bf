// decode_instances.cuh -- launch helper shared by the per-element-type
// translation units (each includes this once with its own element type).
#pragma once

#include "decode_kernel.cuh"
#include "decode_launch.h"
#include "launch_cache.h"

namespace pkv {

template <typename T, int D, int GM, bool kMma>
static cudaError_t launch_decode_instance(DecodeLaunch &a) {
    auto kernel = paged_decode_kernel<T, D, GM, kMma>;
    const int stage_bytes = decode_stage_bytes(int(sizeof(T)), D, a.p.heads_per_unit);
    const int merge = a.p.heads_per_unit < kConsumerWarps ? 1 : 0;
    const DecodeSmem lay{stage_bytes, a.p.stages, a.p.num_seqs, D, GM, merge,
                         a.p.seq_group != nullptr ? 1 : 0};
    const int smem = lay.request();
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    // per-device records of this instantiation: shared memory opened, occupancy
    static std::atomic<unsigned long long> opened[kLaunchCacheDevices];
    static std::atomic<long long> occupancy[kLaunchCacheDevices];
    e = open_dynamic_smem(opened, dev, kernel, smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = occupancy_per_sm(occupancy, dev, kernel, kDecodeThreads, smem, &per_sm);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int want = a.ctas_per_sm > 0 ? a.ctas_per_sm : 2;
    long long grid = (long long)(want < per_sm ? want : per_sm) * a.num_sms;
    if (grid > a.max_units) grid = a.max_units;
    if (grid < 1) grid = 1;
    a.grid_used = int(grid);
    // programmatic dependent launch: the set-up (barriers, per-sequence unit
    // counts) overlaps the previous kernel's tail; the producer waits for that
    // kernel (griddepcontrol.wait) before its first read of the pools
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kDecodeThreads);
    cfg.dynamicSmemBytes = size_t(smem);
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a.kmap, a.vmap, a.p);
}

template <typename T, int D>
static cudaError_t launch_simt_by_group(DecodeLaunch &a) {
    switch (a.gmax) {
        case 1: return launch_decode_instance<T, D, 1, false>(a);
        case 2: return launch_decode_instance<T, D, 2, false>(a);
        case 4: return launch_decode_instance<T, D, 4, false>(a);
        case 8: return launch_decode_instance<T, D, 8, false>(a);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
