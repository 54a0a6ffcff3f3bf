// decode_noalloc.cu -- split-K paged-attention decode that allocates nothing
// and needs no caller workspace.
//
// Some callers cannot allocate device memory on their call path: a serving
// loop with a fixed per-step latency budget (cudaMalloc may synchronise the
// device and take milliseconds), a plug-in whose host application owns all
// device memory through its own pool, or a process that has already handed
// the free memory to another allocator. For them the split-K partition
// states live in one library-owned array of fixed size,
// PAGEDKV_NOALLOC_SCRATCH_BYTES, placed in device memory when the library's
// device code is loaded; every GPU that loads it keeps the array until the
// process exits.
//
// The array's host-side name is only a stand-in: its device address is looked
// up with cudaGetSymbolAddress once per device and context (on the first call
// made with that device current, and again after cudaDeviceReset has replaced
// the device's context) and passed to the kernels like any workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/pagedkv.h"
#include "context_id.h"

static __device__ __align__(256) unsigned char g_noalloc_scratch[PAGEDKV_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
struct ScratchRecord {
    void *addr;
    unsigned long long context;   // id of the context the address belongs to
};
ScratchRecord g_scratch[kMaxDevices] = {};

// Device address of the scratch array on the current device.
int scratch_address(void **addr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PAGEDKV_ERR_CUDA;
    const unsigned long long ctx = pkv::current_context_id();
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchRecord &r = g_scratch[dev];
    if (!r.addr || ctx == 0 || r.context != ctx) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) return PAGEDKV_ERR_CUDA;
        r.addr = p;
        // the lookup above makes the device's context current if it was not yet
        r.context = ctx ? ctx : pkv::current_context_id();
    }
    *addr = r.addr;
    return PAGEDKV_OK;
}

}  // namespace

extern "C" int paged_attention_decode_noalloc(const void *q, const void *k_cache,
                                              const void *v_cache, const int32_t *block_tables,
                                              const int32_t *context_lens, float scale, void *out,
                                              int num_seqs, int n_q_heads, int n_kv_heads,
                                              int head_dim, int num_blocks, int block_size,
                                              int max_blocks_per_seq, int partition_tokens,
                                              int dtype, void *stream) {
    if (partition_tokens == 0)
        return paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                                      num_seqs, n_q_heads, n_kv_heads, head_dim, num_blocks,
                                      block_size, max_blocks_per_seq, 0, nullptr, 0, dtype, stream);
    const size_t need = paged_attention_workspace_bytes(num_seqs, n_q_heads, head_dim,
                                                        max_blocks_per_seq, block_size,
                                                        partition_tokens);
    if (need > PAGEDKV_NOALLOC_SCRATCH_BYTES) return PAGEDKV_ERR_WORKSPACE;
    void *scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != PAGEDKV_OK) return st;
    return paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                                  num_seqs, n_q_heads, n_kv_heads, head_dim, num_blocks,
                                  block_size, max_blocks_per_seq, partition_tokens, scratch,
                                  PAGEDKV_NOALLOC_SCRATCH_BYTES, dtype, stream);
}
