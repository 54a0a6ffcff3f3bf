// append.cu -- address translation, the paged KV append and the copy-on-write
// block copy.
//
// slot_mapping: "How a serving engine actually works", section "The one
// formula": slot = block_table[seq][pos / B] * B + pos % B.
// append_tokens: both in one launch (the slot, then the copy of the row).
// append: "Paged-KV + Continuous Batching From Scratch", section 1 (one pool
// per layer laid out [num_blocks][block_size][n_kv_heads][head_dim]): each
// new token's K and V rows are copied, 16 bytes per thread and instruction,
// to row `slot` of the pools.
// copy_blocks: "How a serving engine actually works", section "Copy-on-write,
// because you have used fork()": before a sequence writes into a block others
// still reference, its fresh private block receives the shared block's bytes.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pagedkv.h"

namespace pkv {

__global__ void __launch_bounds__(256)
slot_mapping_kernel(const int32_t *__restrict__ block_tables, const int32_t *__restrict__ token_seq,
                    const int32_t *__restrict__ token_pos, int64_t *__restrict__ slot_mapping,
                    int num_tokens, int num_seqs, int max_blocks, int block_size, int num_blocks,
                    unsigned int *err) {
    // the append that follows may start while the slots are computed: it
    // waits for this grid before reading them
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= num_tokens) return;
    const int pos = token_pos[t];
    const int seq = token_seq[t];
    int64_t slot = -1;
    if (pos >= 0) {
        const int j = pos / block_size;
        if (seq < 0 || seq >= num_seqs) {
            atomicOr(err, PAGEDKV_DEVERR_SEQ_INDEX);
        } else if (j >= max_blocks) {
            atomicOr(err, PAGEDKV_DEVERR_POSITION);
        } else {
            const int pb = block_tables[int64_t(seq) * max_blocks + j];
            if (pb < 0 || pb >= num_blocks)
                atomicOr(err, PAGEDKV_DEVERR_BLOCK_ID);
            else
                slot = int64_t(pb) * block_size + (pos - j * block_size);
        }
    }
    slot_mapping[t] = slot;
}

// `tpr` threads copy one row; a CTA works on blockDim.x / tpr rows at a time.
__global__ void __launch_bounds__(256)
append_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
              const int64_t *__restrict__ slots, uint4 *__restrict__ k_cache,
              uint4 *__restrict__ v_cache, int num_tokens, int vec_per_row, int tpr,
              long long num_slots, unsigned int *err) {
    // a decode or prefill that follows may start its set-up now; it waits for
    // this grid before reading the pools
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // the slots (and the pools) of the kernels before this one, complete and visible
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int rows_per_cta = blockDim.x / tpr;
    const int sub = threadIdx.x / tpr;
    const int c0 = threadIdx.x - sub * tpr;
    for (long long t = (long long)blockIdx.x * rows_per_cta + sub; t < num_tokens;
         t += (long long)gridDim.x * rows_per_cta) {
        const long long slot = slots[t];
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (c0 == 0) atomicOr(err, PAGEDKV_DEVERR_SLOT_RANGE);
            continue;
        }
        const uint4 *ks = k + t * vec_per_row;
        const uint4 *vs = v + t * vec_per_row;
        uint4 *kd = k_cache + slot * vec_per_row;
        uint4 *vd = v_cache + slot * vec_per_row;
        for (int c = c0; c < vec_per_row; c += tpr) {
            const uint4 a = __ldcs(ks + c);
            const uint4 b = __ldcs(vs + c);
            kd[c] = a;
            vd[c] = b;
        }
    }
}

// Slot mapping and append in one pass: the `tpr` threads of a row compute its
// slot with the formula and the checks of slot_mapping_kernel (one of them
// records an error bit and, when asked, the slot), then copy the row.
__global__ void __launch_bounds__(256)
append_tokens_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                     const int32_t *__restrict__ block_tables, const int32_t *__restrict__ token_seq,
                     const int32_t *__restrict__ token_pos, int64_t *__restrict__ slot_mapping,
                     uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache, int num_tokens,
                     int num_seqs, int max_blocks, int block_size, int num_blocks, int vec_per_row,
                     int tpr, unsigned int *err) {
    // a decode or prefill that follows may start its set-up now; it waits for
    // this grid before reading the pools
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int rows_per_cta = blockDim.x / tpr;
    const int sub = threadIdx.x / tpr;
    const int c0 = threadIdx.x - sub * tpr;
    for (long long t = (long long)blockIdx.x * rows_per_cta + sub; t < num_tokens;
         t += (long long)gridDim.x * rows_per_cta) {
        const uint4 *ks = k + t * vec_per_row;
        const uint4 *vs = v + t * vec_per_row;
        // The row's first two chunks do not depend on the slot: their loads go
        // out together with those of the position, the sequence and the table
        // entry. All of these are the caller's inputs, which no kernel of this
        // library writes, so they are read before the grid dependency wait.
        uint4 a0 = make_uint4(0u, 0u, 0u, 0u), b0 = a0, a1 = a0, b1 = a0;
        if (c0 < vec_per_row) {
            a0 = __ldcs(ks + c0);
            b0 = __ldcs(vs + c0);
        }
        if (c0 + tpr < vec_per_row) {
            a1 = __ldcs(ks + c0 + tpr);
            b1 = __ldcs(vs + c0 + tpr);
        }
        const int pos = token_pos[t];
        const int seq = token_seq[t];
        long long slot = -1;
        unsigned int bit = 0;
        if (pos >= 0) {
            const int j = pos / block_size;
            if (seq < 0 || seq >= num_seqs) {
                bit = PAGEDKV_DEVERR_SEQ_INDEX;
            } else if (j >= max_blocks) {
                bit = PAGEDKV_DEVERR_POSITION;
            } else {
                const int pb = block_tables[int64_t(seq) * max_blocks + j];
                if (pb < 0 || pb >= num_blocks)
                    bit = PAGEDKV_DEVERR_BLOCK_ID;
                else
                    slot = (long long)pb * block_size + (pos - j * block_size);
            }
        }
        // every store after the kernels before this one have completed (the
        // previous decode may still read a block this append writes, e.g. one
        // freed and handed to another sequence; the slot output may be what a
        // previous append reads); a later wait returns at once
        asm volatile("griddepcontrol.wait;" ::: "memory");
        if (c0 == 0) {
            if (bit) atomicOr(err, bit);
            if (slot_mapping) slot_mapping[t] = slot;
        }
        if (slot < 0) continue;
        uint4 *kd = k_cache + slot * vec_per_row;
        uint4 *vd = v_cache + slot * vec_per_row;
        if (c0 < vec_per_row) {
            kd[c0] = a0;
            vd[c0] = b0;
        }
        if (c0 + tpr < vec_per_row) {
            kd[c0 + tpr] = a1;
            vd[c0 + tpr] = b1;
        }
        for (int c = c0 + 2 * tpr; c < vec_per_row; c += tpr) {
            const uint4 a = __ldcs(ks + c);
            const uint4 b = __ldcs(vs + c);
            kd[c] = a;
            vd[c] = b;
        }
    }
}

// Copy-on-write: copy whole blocks (K and V) src -> dst. `tpb` threads copy
// one block pair at a time, 16 bytes per thread and instruction.
__global__ void __launch_bounds__(256)
copy_blocks_kernel(uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                   const int32_t *__restrict__ pairs, int num_pairs, int num_blocks,
                   long long vec_per_block, unsigned int *err) {
    for (int i = blockIdx.y; i < num_pairs; i += gridDim.y) {
        const int src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(err, PAGEDKV_DEVERR_BLOCK_ID);
            continue;
        }
        if (src == dst) continue;
        const uint4 *ks = k_cache + src * vec_per_block;
        const uint4 *vs = v_cache + src * vec_per_block;
        uint4 *kd = k_cache + dst * vec_per_block;
        uint4 *vd = v_cache + dst * vec_per_block;
        for (long long c = blockIdx.x * (long long)blockDim.x + threadIdx.x; c < vec_per_block;
             c += (long long)gridDim.x * blockDim.x) {
            const uint4 a = __ldcs(ks + c);
            const uint4 b = __ldcs(vs + c);
            kd[c] = a;
            vd[c] = b;
        }
    }
}

cudaError_t launch_copy_blocks(void *k_cache, void *v_cache, const int32_t *pairs, int num_pairs,
                               int num_blocks, long long block_bytes, int num_sms,
                               unsigned int *err, cudaStream_t st) {
    const long long vec = block_bytes / 16;
    // CTAs along x split one block; along y they walk the pairs
    int per_block = int((vec + 255) / 256);
    if (per_block > 8) per_block = 8;
    long long along_y = num_pairs;
    const long long cap = (long long)num_sms * 16 / per_block;
    if (along_y > cap) along_y = cap;
    if (along_y > 65535) along_y = 65535;
    if (along_y < 1) along_y = 1;
    copy_blocks_kernel<<<dim3(unsigned(per_block), unsigned(along_y)), 256, 0, st>>>(
        static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), pairs, num_pairs,
        num_blocks, vec, err);
    return cudaGetLastError();
}

cudaError_t launch_slot_mapping(const int32_t *block_tables, const int32_t *token_seq,
                                const int32_t *token_pos, int64_t *slot_mapping, int num_tokens,
                                int num_seqs, int max_blocks, int block_size, int num_blocks,
                                unsigned int *err, cudaStream_t st) {
    const int blocks = (num_tokens + 255) / 256;
    slot_mapping_kernel<<<blocks, 256, 0, st>>>(block_tables, token_seq, token_pos, slot_mapping,
                                                num_tokens, num_seqs, max_blocks, block_size,
                                                num_blocks, err);
    return cudaGetLastError();
}

cudaError_t launch_append(const void *k, const void *v, const int64_t *slots, void *k_cache,
                          void *v_cache, int num_tokens, long long row_bytes, long long num_slots,
                          int num_sms, unsigned int *err, cudaStream_t st) {
    const int vec_per_row = int(row_bytes / 16);
    int tpr = 32;
    while (tpr < vec_per_row && tpr < 256) tpr <<= 1;
    const int rows_per_cta = 256 / tpr;
    long long blocks = (num_tokens + rows_per_cta - 1) / rows_per_cta;
    const long long cap = (long long)num_sms * 16;
    if (blocks > cap) blocks = cap;
    // programmatic dependent launch: the kernel waits for the previous grid
    // itself (griddepcontrol.wait) before it reads anything that grid wrote
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, append_kernel, static_cast<const uint4 *>(k),
                              static_cast<const uint4 *>(v), slots, static_cast<uint4 *>(k_cache),
                              static_cast<uint4 *>(v_cache), num_tokens, vec_per_row, tpr,
                              num_slots, err);
}

cudaError_t launch_append_tokens(const void *k, const void *v, const int32_t *block_tables,
                                 const int32_t *token_seq, const int32_t *token_pos,
                                 int64_t *slot_mapping, void *k_cache, void *v_cache,
                                 int num_tokens, int num_seqs, int max_blocks, int block_size,
                                 int num_blocks, long long row_bytes, int num_sms,
                                 unsigned int *err, cudaStream_t st) {
    const int vec_per_row = int(row_bytes / 16);
    int tpr = 32;
    while (tpr < vec_per_row && tpr < 256) tpr <<= 1;
    const int rows_per_cta = 256 / tpr;
    long long blocks = (num_tokens + rows_per_cta - 1) / rows_per_cta;
    const long long cap = (long long)num_sms * 16;
    if (blocks > cap) blocks = cap;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(blocks));
    cfg.blockDim = dim3(256);
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, append_tokens_kernel, static_cast<const uint4 *>(k),
                              static_cast<const uint4 *>(v), block_tables, token_seq, token_pos,
                              slot_mapping, static_cast<uint4 *>(k_cache),
                              static_cast<uint4 *>(v_cache), num_tokens, num_seqs, max_blocks,
                              block_size, num_blocks, vec_per_row, tpr, err);
}

}  // namespace pkv
