// swap.cu -- whole-block copies between two pools (device <-> page-locked host).
//
// "Paged Attention and the Block Manager", section "Running out of memory
// becomes a scheduling decision": a preempted sequence either loses its cache
// and is recomputed, or keeps it by copying its blocks out to host memory and
// back in on re-admission. Swap costs link bandwidth each way, so the copy is
// one kernel over every pair of the call: on a Grace-Blackwell node the GPU
// reads and writes page-locked host memory in place over NVLink-C2C, and one
// launch keeps enough 16-byte accesses in flight to cover the link latency
// instead of issuing two driver copies per block.
//
// The file also holds the bounded-wait check behind pagedkv_check_bounded_wait.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pagedkv.h"
#include "ptx.cuh"

namespace pkv {

constexpr int kSwapThreads = 256;
constexpr int kSwapUnroll = 4;                              // 16-byte vectors per thread per chunk
constexpr long long kSwapChunk = kSwapThreads * kSwapUnroll; // vectors per chunk (16 KiB)

// Work item c of the flattened (pair, pool, chunk) space: chunk `part` of the K
// (pool 0) or V (pool 1) block of pair i. Every load of a chunk is issued
// before its stores, so a thread keeps kSwapUnroll reads in flight.
__global__ void __launch_bounds__(kSwapThreads)
swap_blocks_kernel(const uint4 *__restrict__ src_k, const uint4 *__restrict__ src_v,
                   uint4 *__restrict__ dst_k, uint4 *__restrict__ dst_v,
                   const int32_t *__restrict__ pairs, int num_pairs, int src_blocks,
                   int dst_blocks, long long vec_per_block, int chunks, unsigned int *err) {
    const long long per_pair = 2LL * chunks;
    const long long total = per_pair * num_pairs;
    for (long long c = blockIdx.x; c < total; c += gridDim.x) {
        const int i = int(c / per_pair);
        const int rem = int(c - (long long)i * per_pair);
        const int pool = rem >= chunks;
        const int part = rem - pool * chunks;
        const int from = __ldg(pairs + 2 * i), to = __ldg(pairs + 2 * i + 1);
        if (from < 0 || from >= src_blocks || to < 0 || to >= dst_blocks) {
            if (rem == 0 && threadIdx.x == 0) atomicOr(err, PAGEDKV_DEVERR_BLOCK_ID);
            continue;
        }
        const uint4 *s = (pool ? src_v : src_k) + (long long)from * vec_per_block;
        uint4 *d = (pool ? dst_v : dst_k) + (long long)to * vec_per_block;
        const long long e0 = part * kSwapChunk + threadIdx.x;
        uint4 r[kSwapUnroll];
#pragma unroll
        for (int u = 0; u < kSwapUnroll; ++u) {
            const long long e = e0 + u * kSwapThreads;
            if (e < vec_per_block) r[u] = __ldcs(s + e);
        }
#pragma unroll
        for (int u = 0; u < kSwapUnroll; ++u) {
            const long long e = e0 + u * kSwapThreads;
            if (e < vec_per_block) d[e] = r[u];
        }
    }
}

cudaError_t launch_swap_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                               const int32_t *pairs, int num_pairs, int src_blocks,
                               int dst_blocks, long long block_bytes, int num_sms,
                               unsigned int *err, cudaStream_t st) {
    const long long vec = block_bytes / 16;
    const long long chunks = (vec + kSwapChunk - 1) / kSwapChunk;
    const long long items = 2 * chunks * num_pairs;
    // up to 8 resident CTAs of 256 threads per SM; work items are grid-strided
    long long grid = (long long)num_sms * 8;
    if (grid > items) grid = items;
    if (grid < 1) grid = 1;
    swap_blocks_kernel<<<unsigned(grid), kSwapThreads, 0, st>>>(
        static_cast<const uint4 *>(src_k), static_cast<const uint4 *>(src_v),
        static_cast<uint4 *>(dst_k), static_cast<uint4 *>(dst_v), pairs, num_pairs, src_blocks,
        dst_blocks, vec, int(chunks), err);
    return cudaGetLastError();
}

// The bounded-wait check: one thread waits on an mbarrier that nothing ever
// arrives on. The wait gives up after its time limit, sets
// PAGEDKV_DEVERR_TIMEOUT and returns false, and the kernel exits normally,
// which is what every in-kernel wait of the library does when a peer never
// arrives.
__global__ void bounded_wait_check_kernel(unsigned int *err) {
    __shared__ __align__(8) uint64_t bar_storage;
    const uint32_t bar = smem_addr(&bar_storage);
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
        mbar_wait(bar, 0, err);
    }
}

cudaError_t launch_bounded_wait_check(unsigned int *err, cudaStream_t stream) {
    bounded_wait_check_kernel<<<1, 32, 0, stream>>>(err);
    return cudaGetLastError();
}

}  // namespace pkv
