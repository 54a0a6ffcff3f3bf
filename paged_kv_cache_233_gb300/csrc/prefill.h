// prefill.h -- parameters of the chunked-prefill attention kernel, shared by
// the C ABI layer and the kernel's translation unit.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pkv {

constexpr int kPfRows = 64;      // query rows (chunk token, query head) per CTA
constexpr int kPfKeys = 64;      // keys per pipeline stage
constexpr int kPfStages = 3;     // depth of the K/V ring
constexpr int kPfThreads = 160;  // one producer warp + four consumer warps of 16 rows

struct PrefillParams {
    const void *q;               // [num_tokens][n_q_heads][head_dim]
    void *out;                   // [num_tokens][n_q_heads][head_dim]
    const int32_t *block_tables; // [num_seqs][max_blocks]
    const int32_t *query_start;  // [num_seqs + 1]
    const int32_t *context_lens; // [num_seqs], the chunk included
    unsigned int *err;
    float scale_log2;            // softmax scale * log2(e)
    int num_seqs;
    int num_tokens;
    int n_q_heads;
    int n_kv_heads;
    int group;                   // n_q_heads / n_kv_heads
    int tile_tokens;             // chunk tokens per item: kPfRows / group (warp-level MMA
                                 // kernel), 2 * (128 / group) (tcgen05 kernel)
    int num_blocks;
    int block_size;
    int log2_block;
    int max_blocks;
    // tcgen05 kernel, key split (key_parts >= 2): one CTA per SM, each taking
    // an equal contiguous range of the call's key tiles (all items' end to
    // end; no item in more than key_parts ranges). An item cut by a range
    // boundary writes, per piece, its rows' unnormalised fp32 O, reference
    // maximum m (base 2, scaled) and sum l to ws_o [slot][row][D], ws_m and
    // ws_l [slot][row] (2 slots per CTA, 256 row slots each), and CTA 0 writes
    // each item's first CTA and range count to ws_plan [item], for
    // launch_prefill_merge; an item within one range writes `out` itself.
    // key_parts == 1: whole items
    int key_parts;
    int *ws_plan;
    float *ws_o;
    float *ws_m;
    float *ws_l;
};

// Bytes of dynamic shared memory the kernel asks for at this head_dim (16-bit types).
int prefill_smem_bytes(int head_dim);

// The warp-level MMA kernel: grid (query tiles of the longest chunk, kv heads,
// sequences), 64 query rows per CTA, pool maps with boxes of every column
// block. The tcgen05 kernel: one persistent CTA per SM working through items
// of two Q tiles of 128 / group whole tokens each (tile_tokens = 2 * (128 /
// group)), pool maps with boxes of one 64-column block, and a map of q with
// boxes of [128 / group tokens][group heads][one 64-column block].
cudaError_t launch_prefill(int dtype, int head_dim, const CUtensorMap &kmap,
                           const CUtensorMap &vmap, const PrefillParams &p, int max_query_len,
                           cudaStream_t stream);

cudaError_t launch_prefill_tc(int dtype, int head_dim, const CUtensorMap &kmap,
                              const CUtensorMap &vmap, const CUtensorMap &qmap,
                              const PrefillParams &p, int max_query_len, int num_sms,
                              cudaStream_t stream);
int prefill_tc_smem_bytes(int head_dim);

// Key split limits: items per call (the plan lives in the kernel's shared
// memory) and ranges per item (a merge lane each).
constexpr int kPfMaxSplitItems = 500;
constexpr int kPfMaxSplitParts = 32;

// The key split's merge: per row of every item cut into pieces, the pieces'
// states combined into `out` (rows of a flagged sequence left unwritten, as
// the kernel does).
cudaError_t launch_prefill_merge(int dtype, int head_dim, const PrefillParams &p, int max_query_len,
                                 int num_sms, cudaStream_t stream);

}  // namespace pkv
