// api.cu -- the C ABI of libpagedkv (declared in include/pagedkv.h).
//
// Host-side argument checks, the per-device error word, TMA descriptor
// encoding for the K/V pools, decode-path selection and the launches. No
// memory is allocated here; every buffer belongs to the caller.
#include <cuda.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <stdint.h>

#include <mutex>

#include "../../include/pagedkv.h"
#include "context_id.h"
#include "decode_launch.h"
#include "prefill.h"

namespace pkv {
cudaError_t launch_slot_mapping(const int32_t *block_tables, const int32_t *token_seq,
                                const int32_t *token_pos, int64_t *slot_mapping, int num_tokens,
                                int num_seqs, int max_blocks, int block_size, int num_blocks,
                                unsigned int *err, cudaStream_t st);
cudaError_t launch_append(const void *k, const void *v, const int64_t *slots, void *k_cache,
                          void *v_cache, int num_tokens, long long row_bytes, long long num_slots,
                          int num_sms, unsigned int *err, cudaStream_t st);
cudaError_t launch_append_tokens(const void *k, const void *v, const int32_t *block_tables,
                                 const int32_t *token_seq, const int32_t *token_pos,
                                 int64_t *slot_mapping, void *k_cache, void *v_cache,
                                 int num_tokens, int num_seqs, int max_blocks, int block_size,
                                 int num_blocks, long long row_bytes, int num_sms,
                                 unsigned int *err, cudaStream_t st);
cudaError_t launch_bounded_wait_check(unsigned int *err, cudaStream_t stream);
cudaError_t launch_copy_blocks(void *k_cache, void *v_cache, const int32_t *pairs, int num_pairs,
                               int num_blocks, long long block_bytes, int num_sms,
                               unsigned int *err, cudaStream_t st);
cudaError_t launch_swap_blocks(const void *src_k, const void *src_v, void *dst_k, void *dst_v,
                               const int32_t *pairs, int num_pairs, int src_blocks,
                               int dst_blocks, long long block_bytes, int num_sms,
                               unsigned int *err, cudaStream_t st);
}  // namespace pkv

// Sticky error word, one per device that loads the library.
__device__ unsigned int g_pagedkv_errors = 0;

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxSeqs = 4096;
constexpr int kMaxCtasPerSm = 8;

std::mutex g_mu;
unsigned int *g_err_ptr[kMaxDevices] = {};
unsigned long long g_err_ctx[kMaxDevices] = {};   // context the error word's address belongs to
int g_num_sms[kMaxDevices] = {};
long long g_l2_bytes[kMaxDevices] = {};

int g_opt_path = pkv::kPathAuto;
int g_opt_ctas_per_sm = 0;
// the tensor-core consumer is the faster one at every group size measured
// (1, 2, 4, 8; 16-bit pools), so the automatic path takes it from group 1
int g_opt_mma_min_group = 1;
int g_opt_stages = 0;
int g_opt_prefill_path = 0;
int g_opt_l2_hints = 0;
int g_last_path = 0;

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int elem_bytes(int dtype) { return dtype == PAGEDKV_F32 ? 4 : 2; }

bool valid_dtype(int dtype) {
    return dtype == PAGEDKV_F32 || dtype == PAGEDKV_F16 || dtype == PAGEDKV_BF16;
}

// Error-word address and SM count of the current device (looked up once per
// device and context: again after cudaDeviceReset has replaced the context).
int device_state(unsigned int **err, int *sms, long long *l2_bytes = nullptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PAGEDKV_ERR_CUDA;
    const unsigned long long ctx = pkv::current_context_id();
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_err_ptr[dev] || ctx == 0 || g_err_ctx[dev] != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pagedkv_errors) != cudaSuccess || !p) return PAGEDKV_ERR_CUDA;
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
            return PAGEDKV_ERR_CUDA;
        int l2 = 0;
        if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess || l2 < 0)
            return PAGEDKV_ERR_CUDA;
        g_num_sms[dev] = n;
        g_l2_bytes[dev] = l2;
        g_err_ptr[dev] = static_cast<unsigned int *>(p);
        g_err_ctx[dev] = ctx ? ctx : pkv::current_context_id();
    }
    *err = g_err_ptr[dev];
    *sms = g_num_sms[dev];
    if (l2_bytes) *l2_bytes = g_l2_bytes[dev];
    return PAGEDKV_OK;
}

int encoder(EncodeTiledFn *fn) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_encode) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !p)
            return PAGEDKV_ERR_CUDA;
        g_encode = reinterpret_cast<EncodeTiledFn>(p);
    }
    *fn = g_encode;
    return PAGEDKV_OK;
}

// TMA view of one pool as a 4-D tensor (x: 128-byte column slab elements,
// token slot, slab, kv head) so that one box holds [heads][slabs][tokens][128 B]
// in shared memory; strides in bytes: token n_kv_heads*head_dim*eb, slab 128,
// head head_dim*eb. The box is every slab of `heads` heads x 16 tokens; for
// 8-token blocks it is every slab of `heads` heads x 8 tokens (one block), or,
// when `per_slab8` is set, one slab of one head x 8 tokens. 128-byte swizzle.
int encode_pool_map(CUtensorMap *map, const void *pool, int dtype, int head_dim, int n_kv_heads,
                    long long num_slots, int block_size, int heads, bool per_slab8 = false) {
    EncodeTiledFn fn = nullptr;
    int st = encoder(&fn);
    if (st != PAGEDKV_OK) return st;
    const int eb = elem_bytes(dtype);
    const int slabs = head_dim * eb / 128;
    const CUtensorMapDataType dt = dtype == PAGEDKV_F32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : dtype == PAGEDKV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                          : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint64_t dims[4] = {cuuint64_t(128 / eb), cuuint64_t(num_slots), cuuint64_t(slabs),
                                cuuint64_t(n_kv_heads)};
    const cuuint64_t strides[3] = {cuuint64_t(n_kv_heads) * head_dim * eb, 128u,
                                   cuuint64_t(head_dim) * eb};
    const bool whole = block_size >= pkv::kTile;
    const bool all = whole || !per_slab8;
    const cuuint32_t box[4] = {cuuint32_t(128 / eb), cuuint32_t(whole ? pkv::kTile : block_size),
                               cuuint32_t(all ? slabs : 1), cuuint32_t(all ? heads : 1)};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    const CUresult r = fn(map, dt, 4, const_cast<void *>(pool), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PAGEDKV_OK : PAGEDKV_ERR_CUDA;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// TMA view of one pool for the tcgen05 prefill kernel: the same 4-D tensor as
// encode_pool_map, with a box of one 128-byte column slab of one kv head x 16
// tokens (8 for 8-token blocks), so that the boxes of a tile can be placed as
// [slab][keys][128 B], the tensor core's K-major / MN-major operand layout.
int encode_pool_map_slab(CUtensorMap *map, const void *pool, int dtype, int head_dim,
                         int n_kv_heads, long long num_slots, int block_size) {
    EncodeTiledFn fn = nullptr;
    int st = encoder(&fn);
    if (st != PAGEDKV_OK) return st;
    const int eb = elem_bytes(dtype);
    const int slabs = head_dim * eb / 128;
    const CUtensorMapDataType dt = dtype == PAGEDKV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint64_t dims[4] = {cuuint64_t(128 / eb), cuuint64_t(num_slots), cuuint64_t(slabs),
                                cuuint64_t(n_kv_heads)};
    const cuuint64_t strides[3] = {cuuint64_t(n_kv_heads) * head_dim * eb, 128u,
                                   cuuint64_t(head_dim) * eb};
    const cuuint32_t box[4] = {cuuint32_t(128 / eb),
                               cuuint32_t(block_size >= pkv::kTile ? pkv::kTile : block_size), 1u, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    const CUresult r = fn(map, dt, 4, const_cast<void *>(pool), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PAGEDKV_OK : PAGEDKV_ERR_CUDA;
}

// TMA view of the queries of a prefill call for the tcgen05 kernel: q as a
// 4-D tensor (x: 128-byte column slab elements, slab, query head, token) with
// a box of one slab x `group` heads x 128 / group whole tokens, so that one box
// is a Q tile's rows (token, head of the group) of one column slab, 128-byte
// swizzle: all 128 of them when the group divides 128. Strides in bytes: slab
// 128, head head_dim*eb, token n_q_heads*head_dim*eb.
int encode_q_map(CUtensorMap *map, const void *q, int dtype, int head_dim, int n_q_heads,
                 int num_tokens, int group) {
    EncodeTiledFn fn = nullptr;
    int st = encoder(&fn);
    if (st != PAGEDKV_OK) return st;
    const int eb = elem_bytes(dtype);
    const int slabs = head_dim * eb / 128;
    const CUtensorMapDataType dt = dtype == PAGEDKV_F16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint64_t dims[4] = {cuuint64_t(128 / eb), cuuint64_t(slabs), cuuint64_t(n_q_heads),
                                cuuint64_t(num_tokens)};
    const cuuint64_t strides[3] = {128u, cuuint64_t(head_dim) * eb, cuuint64_t(n_q_heads) * head_dim * eb};
    const cuuint32_t box[4] = {cuuint32_t(128 / eb), 1u, cuuint32_t(group), cuuint32_t(128 / group)};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    const CUresult r = fn(map, dt, 4, const_cast<void *>(q), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PAGEDKV_OK : PAGEDKV_ERR_CUDA;
}

// SM count of the current device (no error word lookup).
int current_sm_count(int *sms) {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PAGEDKV_ERR_CUDA;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
        return PAGEDKV_ERR_CUDA;
    *sms = n;
    return PAGEDKV_OK;
}

// Piece rows of the balanced split: two slots per CTA of the largest grid the
// CTAs-per-SM option allows, each with up to 4 kv heads x 8 query heads.
size_t balanced_rows(int sms, int n_q_heads) {
    const size_t rows_per_piece = size_t(n_q_heads < 32 ? n_q_heads : 32);
    return 2 * size_t(kMaxCtasPerSm) * size_t(sms) * rows_per_piece;
}

long long max_parts_for(int max_blocks, int block_size, int part_tokens) {
    const long long cap = (long long)max_blocks * block_size;
    return (cap + part_tokens - 1) / part_tokens;
}

}  // namespace

extern "C" {

int pagedkv_abi_version(void) { return PAGEDKV_ABI_VERSION; }

const char *pagedkv_status_string(int status) {
    switch (status) {
        case PAGEDKV_OK: return "ok";
        case PAGEDKV_ERR_INVALID_ARG: return "invalid argument";
        case PAGEDKV_ERR_UNSUPPORTED: return "unsupported configuration";
        case PAGEDKV_ERR_CUDA: return "CUDA error";
        case PAGEDKV_ERR_BOUNDS: return "device reported an out-of-range value";
        case PAGEDKV_ERR_WORKSPACE: return "split-K workspace missing or too small";
        default: return "unknown status";
    }
}

int pagedkv_set_option(int option, int value) {
    switch (option) {
        case PAGEDKV_OPT_DECODE_PATH:
            if (value < 0 || value > 2) return PAGEDKV_ERR_INVALID_ARG;
            g_opt_path = value;
            return PAGEDKV_OK;
        case PAGEDKV_OPT_CTAS_PER_SM:
            if (value < 0 || value > kMaxCtasPerSm) return PAGEDKV_ERR_INVALID_ARG;
            g_opt_ctas_per_sm = value;
            return PAGEDKV_OK;
        case PAGEDKV_OPT_MMA_MIN_GROUP:
            if (value < 1 || value > 9) return PAGEDKV_ERR_INVALID_ARG;
            g_opt_mma_min_group = value;
            return PAGEDKV_OK;
        case PAGEDKV_OPT_STAGES:
            if (value < 0 || value == 1 || value > 16) return PAGEDKV_ERR_INVALID_ARG;
            g_opt_stages = value;
            return PAGEDKV_OK;
        case PAGEDKV_OPT_PREFILL_PATH:
            if (value < 0 || value > 2) return PAGEDKV_ERR_INVALID_ARG;
            g_opt_prefill_path = value;
            return PAGEDKV_OK;
        case PAGEDKV_OPT_L2_HINTS:
            if (value < 0 || value > 2) return PAGEDKV_ERR_INVALID_ARG;
            g_opt_l2_hints = value;
            return PAGEDKV_OK;
        default:
            return PAGEDKV_ERR_INVALID_ARG;
    }
}

int pagedkv_get_option(int option) {
    switch (option) {
        case PAGEDKV_OPT_DECODE_PATH: return g_opt_path;
        case PAGEDKV_OPT_CTAS_PER_SM: return g_opt_ctas_per_sm;
        case PAGEDKV_OPT_MMA_MIN_GROUP: return g_opt_mma_min_group;
        case PAGEDKV_OPT_STAGES: return g_opt_stages;
        case PAGEDKV_OPT_PREFILL_PATH: return g_opt_prefill_path;
        case PAGEDKV_OPT_L2_HINTS: return g_opt_l2_hints;
        default: return PAGEDKV_ERR_INVALID_ARG;
    }
}

int pagedkv_last_decode_path(void) { return g_last_path; }

int pagedkv_device_errors(unsigned int *flags, int reset) {
    if (!flags) return PAGEDKV_ERR_INVALID_ARG;
    unsigned int *err = nullptr;
    int sms = 0;
    int st = device_state(&err, &sms);
    if (st != PAGEDKV_OK) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) return PAGEDKV_ERR_CUDA;
    unsigned int h = 0;
    if (cudaMemcpy(&h, err, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess) return PAGEDKV_ERR_CUDA;
    if (reset && cudaMemset(err, 0, sizeof h) != cudaSuccess) return PAGEDKV_ERR_CUDA;
    *flags = h;
    return h ? PAGEDKV_ERR_BOUNDS : PAGEDKV_OK;
}

int pagedkv_check_bounded_wait(void *stream) {
    unsigned int *err = nullptr;
    int sms = 0;
    int st = device_state(&err, &sms);
    if (st != PAGEDKV_OK) return st;
    return pkv::launch_bounded_wait_check(err, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PAGEDKV_OK
               : PAGEDKV_ERR_CUDA;
}

int paged_kv_slot_mapping(const int32_t *block_tables, const int32_t *token_seq,
                          const int32_t *token_pos, int64_t *slot_mapping, int num_tokens,
                          int num_seqs, int max_blocks_per_seq, int block_size, int num_blocks,
                          void *stream) {
    if (num_tokens < 0 || num_seqs < 0 || max_blocks_per_seq < 1 || block_size < 1 ||
        num_blocks < 1)
        return PAGEDKV_ERR_INVALID_ARG;
    if ((long long)num_blocks * block_size > (1ll << 62)) return PAGEDKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PAGEDKV_OK;
    if (!block_tables || !token_seq || !token_pos || !slot_mapping) return PAGEDKV_ERR_INVALID_ARG;
    if (!aligned(block_tables, 4) || !aligned(token_seq, 4) || !aligned(token_pos, 4) ||
        !aligned(slot_mapping, 8))
        return PAGEDKV_ERR_INVALID_ARG;
    unsigned int *err = nullptr;
    int sms = 0;
    int st = device_state(&err, &sms);
    if (st != PAGEDKV_OK) return st;
    const cudaError_t e = pkv::launch_slot_mapping(block_tables, token_seq, token_pos, slot_mapping,
                                                   num_tokens, num_seqs, max_blocks_per_seq,
                                                   block_size, num_blocks, err,
                                                   static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PAGEDKV_OK : PAGEDKV_ERR_CUDA;
}

int paged_kv_append(const void *k, const void *v, const int64_t *slot_mapping, void *k_cache,
                    void *v_cache, int num_tokens, int num_blocks, int block_size, int n_kv_heads,
                    int head_dim, int dtype, void *stream) {
    if (num_tokens < 0 || num_blocks < 1 || block_size < 1 || n_kv_heads < 1 || head_dim < 1 ||
        !valid_dtype(dtype))
        return PAGEDKV_ERR_INVALID_ARG;
    const long long row_bytes = (long long)n_kv_heads * head_dim * elem_bytes(dtype);
    if (row_bytes % 16 != 0 || row_bytes / 16 > INT_MAX) return PAGEDKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PAGEDKV_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PAGEDKV_ERR_INVALID_ARG;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(slot_mapping, 8))
        return PAGEDKV_ERR_INVALID_ARG;
    unsigned int *err = nullptr;
    int sms = 0;
    int st = device_state(&err, &sms);
    if (st != PAGEDKV_OK) return st;
    const cudaError_t e = pkv::launch_append(k, v, slot_mapping, k_cache, v_cache, num_tokens,
                                             row_bytes, (long long)num_blocks * block_size, sms,
                                             err, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PAGEDKV_OK : PAGEDKV_ERR_CUDA;
}

int paged_kv_append_tokens(const void *k, const void *v, const int32_t *block_tables,
                           const int32_t *token_seq, const int32_t *token_pos,
                           int64_t *slot_mapping, void *k_cache, void *v_cache, int num_tokens,
                           int num_seqs, int max_blocks_per_seq, int num_blocks, int block_size,
                           int n_kv_heads, int head_dim, int dtype, void *stream) {
    if (num_tokens < 0 || num_seqs < 0 || max_blocks_per_seq < 1 || num_blocks < 1 ||
        block_size < 1 || n_kv_heads < 1 || head_dim < 1 || !valid_dtype(dtype))
        return PAGEDKV_ERR_INVALID_ARG;
    if ((long long)num_blocks * block_size > (1ll << 62)) return PAGEDKV_ERR_INVALID_ARG;
    const long long row_bytes = (long long)n_kv_heads * head_dim * elem_bytes(dtype);
    if (row_bytes % 16 != 0 || row_bytes / 16 > INT_MAX) return PAGEDKV_ERR_INVALID_ARG;
    if (num_tokens == 0) return PAGEDKV_OK;
    if (!k || !v || !block_tables || !token_seq || !token_pos || !k_cache || !v_cache)
        return PAGEDKV_ERR_INVALID_ARG;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(block_tables, 4) || !aligned(token_seq, 4) || !aligned(token_pos, 4) ||
        (slot_mapping && !aligned(slot_mapping, 8)))
        return PAGEDKV_ERR_INVALID_ARG;
    unsigned int *err = nullptr;
    int sms = 0;
    int st = device_state(&err, &sms);
    if (st != PAGEDKV_OK) return st;
    const cudaError_t e = pkv::launch_append_tokens(
        k, v, block_tables, token_seq, token_pos, slot_mapping, k_cache, v_cache, num_tokens,
        num_seqs, max_blocks_per_seq, block_size, num_blocks, row_bytes, sms, err,
        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PAGEDKV_OK : PAGEDKV_ERR_CUDA;
}

int paged_kv_copy_blocks(void *k_cache, void *v_cache, const int32_t *block_pairs, int num_pairs,
                         int num_blocks, int block_size, int n_kv_heads, int head_dim, int dtype,
                         void *stream) {
    if (num_pairs < 0 || num_blocks < 1 || block_size < 1 || n_kv_heads < 1 || head_dim < 1 ||
        !valid_dtype(dtype))
        return PAGEDKV_ERR_INVALID_ARG;
    const long long block_bytes = (long long)block_size * n_kv_heads * head_dim * elem_bytes(dtype);
    if (block_bytes % 16 != 0) return PAGEDKV_ERR_INVALID_ARG;
    if (num_pairs == 0) return PAGEDKV_OK;
    if (!k_cache || !v_cache || !block_pairs) return PAGEDKV_ERR_INVALID_ARG;
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(block_pairs, 4))
        return PAGEDKV_ERR_INVALID_ARG;
    unsigned int *err = nullptr;
    int sms = 0;
    int st = device_state(&err, &sms);
    if (st != PAGEDKV_OK) return st;
    const cudaError_t e = pkv::launch_copy_blocks(k_cache, v_cache, block_pairs, num_pairs,
                                                  num_blocks, block_bytes, sms, err,
                                                  static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PAGEDKV_OK : PAGEDKV_ERR_CUDA;
}

}  // extern "C"

namespace {

// The address through which the current device reaches `p`, or null when it
// cannot: memory of this device, managed memory, or page-locked host memory
// mapped into the device's address space. Pageable host memory and other
// devices' memory are refused.
const void *device_view(const void *p) {
    if (!p) return nullptr;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    switch (a.type) {
    case cudaMemoryTypeDevice: return a.device == dev ? p : nullptr;
    case cudaMemoryTypeManaged: return p;
    case cudaMemoryTypeHost: return a.devicePointer;
    default: return nullptr;
    }
}

}  // namespace

extern "C" {

int paged_kv_swap_blocks(const void *src_k, const void *src_v, int src_num_blocks, void *dst_k,
                         void *dst_v, int dst_num_blocks, const int32_t *block_pairs,
                         int num_pairs, int block_size, int n_kv_heads, int head_dim, int dtype,
                         void *stream) {
    if (num_pairs < 0 || src_num_blocks < 1 || dst_num_blocks < 1 || block_size < 1 ||
        n_kv_heads < 1 || head_dim < 1 || !valid_dtype(dtype))
        return PAGEDKV_ERR_INVALID_ARG;
    const long long block_bytes = (long long)block_size * n_kv_heads * head_dim * elem_bytes(dtype);
    if (block_bytes % 16 != 0) return PAGEDKV_ERR_INVALID_ARG;
    if (num_pairs == 0) return PAGEDKV_OK;
    const void *sk = device_view(src_k), *sv = device_view(src_v);
    void *dk = const_cast<void *>(device_view(dst_k));
    void *dv = const_cast<void *>(device_view(dst_v));
    const int32_t *pairs = static_cast<const int32_t *>(device_view(block_pairs));
    if (!sk || !sv || !dk || !dv || !pairs) return PAGEDKV_ERR_INVALID_ARG;
    if (!aligned(sk, 16) || !aligned(sv, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
        !aligned(pairs, 4))
        return PAGEDKV_ERR_INVALID_ARG;
    unsigned int *err = nullptr;
    int sms = 0;
    int st = device_state(&err, &sms);
    if (st != PAGEDKV_OK) return st;
    const cudaError_t e = pkv::launch_swap_blocks(sk, sv, dk, dv, pairs, num_pairs,
                                                  src_num_blocks, dst_num_blocks, block_bytes,
                                                  sms, err, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PAGEDKV_OK : PAGEDKV_ERR_CUDA;
}

namespace {

constexpr int kMaxKeyParts = pkv::kPfMaxSplitParts;

// Bytes of the key split's workspace for a grid of `ctas` CTAs: the plan (an
// int per item), then fp32 O [2 ctas][256 rows][head_dim], then m and l
// [2 ctas][256 rows], each on a 256-byte boundary.
size_t prefill_split_bytes(int head_dim, int ctas) {
    const size_t rows = size_t(2) * size_t(ctas) * 256;
    return round256(size_t(pkv::kPfMaxSplitItems) * 4) + round256(rows * size_t(head_dim) * 4) +
           2 * round256(rows * 4);
}

int prefill_impl(const void *q, const void *k_cache, const void *v_cache,
                 const int32_t *block_tables, const int32_t *query_start,
                 const int32_t *context_lens, float scale, void *out, int num_seqs, int num_tokens,
                 int max_query_len, int n_q_heads, int n_kv_heads, int head_dim, int num_blocks,
                 int block_size, int max_blocks_per_seq, int dtype, int key_parts, void *workspace,
                 size_t workspace_bytes, void *stream) {
    if (key_parts < 0 || key_parts > kMaxKeyParts) return PAGEDKV_ERR_INVALID_ARG;
    if (num_seqs < 0 || num_tokens < 0 || max_query_len < 0 || n_q_heads < 1 || n_kv_heads < 1 ||
        head_dim < 1 || num_blocks < 1 || block_size < 1 || max_blocks_per_seq < 1 ||
        !valid_dtype(dtype))
        return PAGEDKV_ERR_INVALID_ARG;
    if (n_q_heads % n_kv_heads != 0) return PAGEDKV_ERR_INVALID_ARG;
    if (!(scale == scale) || scale == INFINITY || scale == -INFINITY) return PAGEDKV_ERR_INVALID_ARG;
    if (dtype == PAGEDKV_F32) return PAGEDKV_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PAGEDKV_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PAGEDKV_ERR_UNSUPPORTED;
    const int group = n_q_heads / n_kv_heads;
    if (group > pkv::kPfRows || num_seqs > 65535 || n_kv_heads > 65535) return PAGEDKV_ERR_UNSUPPORTED;
    const long long num_slots = (long long)num_blocks * block_size;
    const long long cap = (long long)max_blocks_per_seq * block_size;
    if (num_slots > INT_MAX || cap > INT_MAX / 2) return PAGEDKV_ERR_UNSUPPORTED;
    if (num_seqs == 0 || num_tokens == 0 || max_query_len == 0) return PAGEDKV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !query_start || !context_lens || !out)
        return PAGEDKV_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(block_tables, 4) || !aligned(query_start, 4) || !aligned(context_lens, 4))
        return PAGEDKV_ERR_INVALID_ARG;
    unsigned int *err = nullptr;
    int sms = 0;
    int st = device_state(&err, &sms);
    if (st != PAGEDKV_OK) return st;
    // path: 1 warp-level MMA kernel, 2 tcgen05 kernel (auto)
    const bool tc = g_opt_prefill_path != 1;
    CUtensorMap kmap, vmap, qmap = {};
    if (tc) {
        st = encode_pool_map_slab(&kmap, k_cache, dtype, head_dim, n_kv_heads, num_slots, block_size);
        if (st != PAGEDKV_OK) return st;
        st = encode_pool_map_slab(&vmap, v_cache, dtype, head_dim, n_kv_heads, num_slots, block_size);
        if (st == PAGEDKV_OK)
            st = encode_q_map(&qmap, q, dtype, head_dim, n_q_heads, num_tokens, group);
    } else {
        st = encode_pool_map(&kmap, k_cache, dtype, head_dim, n_kv_heads, num_slots, block_size, 1,
                             true);
        if (st != PAGEDKV_OK) return st;
        st = encode_pool_map(&vmap, v_cache, dtype, head_dim, n_kv_heads, num_slots, block_size, 1,
                             true);
    }
    if (st != PAGEDKV_OK) return st;
    pkv::PrefillParams p{};
    p.q = q;
    p.out = out;
    p.block_tables = block_tables;
    p.query_start = query_start;
    p.context_lens = context_lens;
    p.err = err;
    p.scale_log2 = scale * pkv::kLog2e;
    p.num_seqs = num_seqs;
    p.num_tokens = num_tokens;
    p.n_q_heads = n_q_heads;
    p.n_kv_heads = n_kv_heads;
    p.group = group;
    // chunk tokens per item: the tcgen05 kernel's two Q tiles hold 128 / group
    // whole tokens each
    p.tile_tokens = tc ? 2 * (128 / group) : pkv::kPfRows / group;
    // key split (tcgen05 kernel only): the call's key tiles in equal ranges,
    // one per SM. 0 takes it when the items leave SMs idle and the workspace
    // holds it (no item then in more than kMaxKeyParts ranges); an explicit
    // count needs the workspace. Calls of more than kPfMaxSplitItems items,
    // or whose key tiles could pass the plan's ints, run whole items.
    const long long tiles = ((long long)max_query_len + p.tile_tokens - 1) / p.tile_tokens;
    const long long items = tiles * n_kv_heads * num_seqs;
    const long long tile_cap = (cap + 63) / 64;   // key tiles of one item at most
    const bool splittable = tc && items <= pkv::kPfMaxSplitItems && items * tile_cap <= INT_MAX / 2;
    const size_t split_bytes = prefill_split_bytes(head_dim, sms);
    int parts = splittable ? key_parts : 1;
    if (parts == 0)
        parts = items < sms && workspace && split_bytes <= workspace_bytes ? kMaxKeyParts : 1;
    if (parts > 1) {
        if (!workspace || split_bytes > workspace_bytes) return PAGEDKV_ERR_WORKSPACE;
        if (!aligned(workspace, 256)) return PAGEDKV_ERR_INVALID_ARG;
        const size_t rows = size_t(2) * size_t(sms) * 256;
        uint8_t *ws = static_cast<uint8_t *>(workspace);
        p.ws_plan = reinterpret_cast<int *>(ws);
        p.ws_o = reinterpret_cast<float *>(ws + round256(size_t(pkv::kPfMaxSplitItems) * 4));
        p.ws_m = p.ws_o + round256(rows * size_t(head_dim) * 4) / 4;
        p.ws_l = p.ws_m + round256(rows * 4) / 4;
    }
    p.key_parts = parts;
    if (tc) {
        // the persistent kernel counts its work items in ints
        const long long per_seq = tiles * n_kv_heads;
        if (per_seq > (INT_MAX / 2) / num_seqs) return PAGEDKV_ERR_UNSUPPORTED;
    }
    p.num_blocks = num_blocks;
    p.block_size = block_size;
    int log2_block = 0;
    while ((1 << log2_block) < block_size) ++log2_block;
    p.log2_block = log2_block;
    p.max_blocks = max_blocks_per_seq;
    cudaError_t e =
        tc ? pkv::launch_prefill_tc(dtype, head_dim, kmap, vmap, qmap, p, max_query_len, sms,
                                    static_cast<cudaStream_t>(stream))
           : pkv::launch_prefill(dtype, head_dim, kmap, vmap, p, max_query_len,
                                 static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess && parts > 1)
        e = pkv::launch_prefill_merge(dtype, head_dim, p, max_query_len, sms,
                                      static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PAGEDKV_OK : PAGEDKV_ERR_CUDA;
}

}  // namespace

int paged_attention_prefill(const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, const int32_t *query_start,
                            const int32_t *context_lens, float scale, void *out, int num_seqs,
                            int num_tokens, int max_query_len, int n_q_heads, int n_kv_heads,
                            int head_dim, int num_blocks, int block_size,
                            int max_blocks_per_seq, int dtype, void *stream) {
    return prefill_impl(q, k_cache, v_cache, block_tables, query_start, context_lens, scale, out,
                        num_seqs, num_tokens, max_query_len, n_q_heads, n_kv_heads, head_dim,
                        num_blocks, block_size, max_blocks_per_seq, dtype, 1, nullptr, 0, stream);
}

int paged_attention_prefill_split(const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *block_tables, const int32_t *query_start,
                                  const int32_t *context_lens, float scale, void *out, int num_seqs,
                                  int num_tokens, int max_query_len, int n_q_heads, int n_kv_heads,
                                  int head_dim, int num_blocks, int block_size,
                                  int max_blocks_per_seq, int dtype, int key_parts, void *workspace,
                                  size_t workspace_bytes, void *stream) {
    return prefill_impl(q, k_cache, v_cache, block_tables, query_start, context_lens, scale, out,
                        num_seqs, num_tokens, max_query_len, n_q_heads, n_kv_heads, head_dim,
                        num_blocks, block_size, max_blocks_per_seq, dtype, key_parts, workspace,
                        workspace_bytes, stream);
}

size_t paged_attention_prefill_workspace_bytes(int head_dim) {
    if (head_dim != 64 && head_dim != 128) return 0;
    unsigned int *err = nullptr;
    int sms = 0;
    if (device_state(&err, &sms) != PAGEDKV_OK) return 0;
    return prefill_split_bytes(head_dim, sms);
}

size_t paged_attention_workspace_bytes(int num_seqs, int n_q_heads, int head_dim,
                                       int max_blocks_per_seq, int block_size,
                                       int partition_tokens) {
    if (num_seqs < 0 || n_q_heads < 1 || head_dim < 1 || max_blocks_per_seq < 1 || block_size < 1)
        return 0;
    size_t rows = 0;
    if (partition_tokens == PAGEDKV_PARTITION_BALANCED) {
        int sms = 0;
        if (current_sm_count(&sms) != PAGEDKV_OK) return 0;
        rows = balanced_rows(sms, n_q_heads);
    } else if (partition_tokens > 0) {
        rows = size_t(num_seqs) * n_q_heads *
               size_t(max_parts_for(max_blocks_per_seq, block_size, partition_tokens));
    } else {
        return 0;
    }
    return round256(rows * head_dim * sizeof(float)) + 2 * round256(rows * sizeof(float));
}

static int decode_impl(const void *q, const void *k_cache, const void *v_cache,
                       const int32_t *block_tables, const int32_t *context_lens,
                       const int32_t *seq_group, const int32_t *group_prefix, int num_groups,
                       float scale, void *out, int num_seqs, int n_q_heads, int n_kv_heads,
                       int head_dim, int num_blocks, int block_size, int max_blocks_per_seq,
                       int partition_tokens, void *workspace, size_t workspace_bytes, int dtype,
                       void *stream) {
    // ---- shapes
    if (num_seqs < 0 || n_q_heads < 1 || n_kv_heads < 1 || head_dim < 1 || num_blocks < 1 ||
        block_size < 1 || max_blocks_per_seq < 1 || !valid_dtype(dtype) ||
        (partition_tokens < 0 && partition_tokens != PAGEDKV_PARTITION_BALANCED))
        return PAGEDKV_ERR_INVALID_ARG;
    if (n_q_heads % n_kv_heads != 0) return PAGEDKV_ERR_INVALID_ARG;
    const bool balanced = partition_tokens == PAGEDKV_PARTITION_BALANCED;
    if (!balanced && partition_tokens % pkv::kTile != 0) return PAGEDKV_ERR_INVALID_ARG;
    if (!(scale == scale) || scale == INFINITY || scale == -INFINITY) return PAGEDKV_ERR_INVALID_ARG;
    const int group = n_q_heads / n_kv_heads;
    if (head_dim != 64 && head_dim != 128) return PAGEDKV_ERR_UNSUPPORTED;
    if (block_size != 8 && block_size != 16 && block_size != 32) return PAGEDKV_ERR_UNSUPPORTED;
    if (group > 8 || num_seqs > kMaxSeqs) return PAGEDKV_ERR_UNSUPPORTED;
    const long long num_slots = (long long)num_blocks * block_size;
    const long long cap = (long long)max_blocks_per_seq * block_size;
    if (num_slots > INT_MAX || cap > INT_MAX / 2) return PAGEDKV_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PAGEDKV_OK;
    // ---- pointers
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
        return PAGEDKV_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(block_tables, 4) || !aligned(context_lens, 4))
        return PAGEDKV_ERR_INVALID_ARG;
    // ---- shared prefixes (fixed split, one consumer warp per kv head)
    const bool prefix = seq_group != nullptr;
    if (prefix) {
        if (partition_tokens <= 0 || num_groups < 1 || !group_prefix) return PAGEDKV_ERR_INVALID_ARG;
        if (!aligned(seq_group, 4) || !aligned(group_prefix, 4)) return PAGEDKV_ERR_INVALID_ARG;
        if (n_kv_heads % 4 != 0) return PAGEDKV_ERR_UNSUPPORTED;
    }
    // ---- path
    int path = g_opt_path;
    if (path == pkv::kPathAuto)
        path = (dtype != PAGEDKV_F32 && (group >= g_opt_mma_min_group || prefix)) ? pkv::kPathMma
                                                                                  : pkv::kPathSimt;
    if (path == pkv::kPathMma && dtype == PAGEDKV_F32) return PAGEDKV_ERR_UNSUPPORTED;
    int gmax = 8;
    if (path == pkv::kPathSimt) gmax = group <= 1 ? 1 : group <= 2 ? 2 : group <= 4 ? 4 : 8;
    // ---- split-K
    const bool split = partition_tokens != 0;
    const int P = partition_tokens > 0 ? partition_tokens
                                       : int((cap + pkv::kTile - 1) / pkv::kTile * pkv::kTile);
    const long long max_parts =
        partition_tokens > 0 ? max_parts_for(max_blocks_per_seq, block_size, P) : 1;
    float *ws_o = nullptr, *ws_m = nullptr, *ws_l = nullptr;
    if (split) {
        const size_t need = paged_attention_workspace_bytes(num_seqs, n_q_heads, head_dim,
                                                            max_blocks_per_seq, block_size,
                                                            partition_tokens);
        if (need == 0 || !workspace || workspace_bytes < need || !aligned(workspace, 256))
            return PAGEDKV_ERR_WORKSPACE;
        size_t rows;
        if (balanced) {
            int sms = 0;
            if (current_sm_count(&sms) != PAGEDKV_OK) return PAGEDKV_ERR_CUDA;
            rows = balanced_rows(sms, n_q_heads);
        } else {
            rows = size_t(num_seqs) * n_q_heads * size_t(max_parts);
        }
        uint8_t *w = static_cast<uint8_t *>(workspace);
        ws_o = reinterpret_cast<float *>(w);
        ws_m = reinterpret_cast<float *>(w + round256(rows * head_dim * sizeof(float)));
        ws_l = reinterpret_cast<float *>(w + round256(rows * head_dim * sizeof(float)) +
                                         round256(rows * sizeof(float)));
    }
    // ---- device
    unsigned int *err = nullptr;
    int sms = 0;
    long long l2_bytes = 0;
    int st = device_state(&err, &sms, &l2_bytes);
    if (st != PAGEDKV_OK) return st;
    // kv heads per unit: one consumer warp per head when n_kv_heads allows
    const int hpu = n_kv_heads % 4 == 0 ? 4 : (n_kv_heads % 2 == 0 ? 2 : 1);
    pkv::DecodeLaunch a;
    st = encode_pool_map(&a.kmap, k_cache, dtype, head_dim, n_kv_heads, num_slots, block_size, hpu);
    if (st != PAGEDKV_OK) return st;
    st = encode_pool_map(&a.vmap, v_cache, dtype, head_dim, n_kv_heads, num_slots, block_size, hpu);
    if (st != PAGEDKV_OK) return st;
    int log2_block = 0;
    while ((1 << log2_block) < block_size) ++log2_block;
    pkv::DecodeParams &p = a.p;
    p.q = q;
    p.out = out;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.ws_o = ws_o;
    p.ws_m = ws_m;
    p.ws_l = ws_l;
    p.err = err;
    p.scale_log2 = scale * pkv::kLog2e;
    p.num_seqs = num_seqs;
    p.n_q_heads = n_q_heads;
    p.n_kv_heads = n_kv_heads;
    p.group = group;
    p.num_blocks = num_blocks;
    p.block_size = block_size;
    p.log2_block = log2_block;
    p.max_blocks = max_blocks_per_seq;
    p.part_tokens = P;
    p.max_parts = int(max_parts);
    p.split = split ? 1 : 0;
    p.balanced = balanced ? 1 : 0;
    // Stage ring. Fixed partitions take the rule of decode_stages. The balanced
    // split sizes the ring for two stages when even the block tables' full
    // width of K/V fits in L2 (a small call: shared memory it does not use
    // costs it launch time); otherwise it holds the short-unit ring and each
    // CTA falls back to two stages when the mean context is long.
    const long long token_bytes = 2ll * n_kv_heads * head_dim * elem_bytes(dtype);
    if (g_opt_stages) {
        p.stages = p.stages_alt = g_opt_stages;
    } else if (balanced) {
        const bool small = (long long)num_seqs * cap <= l2_bytes / token_bytes;
        p.stages = small ? 2 : pkv::decode_stages(elem_bytes(dtype), head_dim, hpu, pkv::kTile);
        p.stages_alt = 2;
    } else {
        p.stages = p.stages_alt = pkv::decode_stages(elem_bytes(dtype), head_dim, hpu, P);
    }
    p.long_seq_tokens = pkv::kLongSeqTokens;
    p.heads_per_unit = hpu;
    p.log2_hpu = hpu == 4 ? 2 : (hpu == 2 ? 1 : 0);
    p.rows_per_box = block_size < pkv::kTile ? block_size : pkv::kTile;
    p.seq_group = prefix ? seq_group : nullptr;
    p.group_prefix = prefix ? group_prefix : nullptr;
    p.num_groups = prefix ? num_groups : 0;
    // a shared-prefix unit fills the tensor-core tile's 8 columns with (member, q head) pairs
    p.max_members = (prefix && path == pkv::kPathMma) ? 8 / group : 1;
    // L2 priorities once the call's K/V stream is larger than the L2 (auto)
    p.hint_min_tokens = g_opt_l2_hints == 1 ? LLONG_MAX
                      : g_opt_l2_hints == 2 ? 0 : l2_bytes / token_bytes;

    a.head_dim = head_dim;
    a.path = path;
    a.gmax = gmax;
    a.ctas_per_sm = g_opt_ctas_per_sm;
    a.num_sms = sms;
    a.max_units = balanced ? (long long)num_seqs * (n_kv_heads / hpu) * ((cap + pkv::kTile - 1) / pkv::kTile)
                           : (long long)num_seqs * (n_kv_heads / hpu) * max_parts;
    a.grid_used = 0;
    a.stream = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (dtype) {
        case PAGEDKV_F32: e = pkv::launch_decode_f32(a); break;
        case PAGEDKV_F16: e = pkv::launch_decode_f16(a); break;
        default: e = pkv::launch_decode_bf16(a); break;
    }
    if (e != cudaSuccess) return PAGEDKV_ERR_CUDA;
    if (balanced) {
        e = pkv::launch_piece_merge(dtype, head_dim, ws_o, ws_m, ws_l, context_lens, out, num_seqs,
                                    n_q_heads, n_kv_heads / hpu, hpu * group, a.grid_used,
                                    int(cap), a.stream);
        if (e != cudaSuccess) return PAGEDKV_ERR_CUDA;
    } else if (split) {
        e = pkv::launch_lse_merge(dtype, head_dim, ws_o, ws_m, ws_l, context_lens, out, num_seqs,
                                  n_q_heads, P, int(max_parts), int(cap), err, a.stream);
        if (e != cudaSuccess) return PAGEDKV_ERR_CUDA;
    }
    g_last_path = path;
    return PAGEDKV_OK;
}

int paged_attention_decode(const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *block_tables, const int32_t *context_lens, float scale,
                           void *out, int num_seqs, int n_q_heads, int n_kv_heads, int head_dim,
                           int num_blocks, int block_size, int max_blocks_per_seq,
                           int partition_tokens, void *workspace, size_t workspace_bytes,
                           int dtype, void *stream) {
    return decode_impl(q, k_cache, v_cache, block_tables, context_lens, nullptr, nullptr, 0, scale,
                       out, num_seqs, n_q_heads, n_kv_heads, head_dim, num_blocks, block_size,
                       max_blocks_per_seq, partition_tokens, workspace, workspace_bytes, dtype,
                       stream);
}

int paged_attention_decode_shared_prefix(const void *q, const void *k_cache, const void *v_cache,
                                         const int32_t *block_tables, const int32_t *context_lens,
                                         const int32_t *seq_group, const int32_t *group_prefix,
                                         int num_groups, float scale, void *out, int num_seqs,
                                         int n_q_heads, int n_kv_heads, int head_dim,
                                         int num_blocks, int block_size, int max_blocks_per_seq,
                                         int partition_tokens, void *workspace,
                                         size_t workspace_bytes, int dtype, void *stream) {
    if (num_groups < 0 || (num_groups > 0 && (!seq_group || !group_prefix)))
        return PAGEDKV_ERR_INVALID_ARG;
    if (num_groups == 0)   // nothing is shared: the ordinary decode
        return paged_attention_decode(q, k_cache, v_cache, block_tables, context_lens, scale, out,
                                      num_seqs, n_q_heads, n_kv_heads, head_dim, num_blocks,
                                      block_size, max_blocks_per_seq, partition_tokens, workspace,
                                      workspace_bytes, dtype, stream);
    return decode_impl(q, k_cache, v_cache, block_tables, context_lens, seq_group, group_prefix,
                       num_groups, scale, out, num_seqs, n_q_heads, n_kv_heads, head_dim,
                       num_blocks, block_size, max_blocks_per_seq, partition_tokens, workspace,
                       workspace_bytes, dtype, stream);
}

}  // extern "C"
