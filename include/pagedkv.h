/*
 * pagedkv.h -- C ABI of libpagedkv: attention over a block-paged KV cache on
 * one GB300 (sm_103a).
 *
 * The cache of one layer is a pool of fixed-size blocks, one K pool and one V
 * pool, each laid out
 *
 *     [num_blocks][block_size][n_kv_heads][head_dim]      (row-major, dense)
 *
 * and indexed by physical block, not by sequence (page "Paged-KV + Continuous
 * Batching From Scratch", section 1 "Paging is really about not reserving").
 * A sequence owns a block table: the list of its physical blocks in logical
 * order. Token i of sequence s lives in slot
 *
 *     slot(s, i) = block_table[s][i / block_size] * block_size + i % block_size
 *
 * (page "How a serving engine actually works", section "The one formula").
 *
 * Conventions shared by every entry point:
 *   - All array arguments are DEVICE pointers owned by the caller. The
 *     library allocates no memory, frees nothing and keeps no pointer after a
 *     call returns. Arrays are dense, row-major, 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream). Calls only enqueue work on it and return without
 *     synchronising; results are ready when the stream reaches them.
 *   - `dtype` is a pagedkv_dtype. q, k, v, the pools and out share it.
 *   - Argument and shape checks run on the host before anything is enqueued;
 *     a failed check returns a negative pagedkv_status and enqueues nothing.
 *   - Out-of-range values found on the device (a block id outside the pool,
 *     a slot past the pool, a context length longer than the block table) are
 *     never dereferenced: the kernel skips or clamps the access and sets a bit
 *     in a sticky device error word that pagedkv_device_errors() returns.
 *   - Kernels never trap. Every wait inside a kernel is bounded in time; a
 *     wait that gives up sets PAGEDKV_DEVERR_TIMEOUT and the kernel returns.
 *   - Host threads may call the entry points concurrently, each with its own
 *     buffers and stream: the library's per-device records (error word,
 *     shared memory a kernel was opened up to, occupancy) are kept under a
 *     lock or in atomics. Two exceptions: the tuning options
 *     (pagedkv_set_option) and the library-owned scratch of
 *     paged_attention_decode_noalloc, whose calls must be ordered on one
 *     stream.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PAGEDKV_ABI_VERSION 1

typedef enum {
    PAGEDKV_F32 = 0,   /* IEEE binary32 */
    PAGEDKV_F16 = 1,   /* IEEE binary16 */
    PAGEDKV_BF16 = 2   /* bfloat16 */
} pagedkv_dtype;

typedef enum {
    PAGEDKV_OK = 0,
    PAGEDKV_ERR_INVALID_ARG = -1,  /* null pointer, bad size, misaligned pointer */
    PAGEDKV_ERR_UNSUPPORTED = -2,  /* valid but not built: e.g. head_dim 96 */
    PAGEDKV_ERR_CUDA = -3,         /* a CUDA runtime call or launch failed */
    PAGEDKV_ERR_BOUNDS = -4,       /* pagedkv_device_errors() found a set bit */
    PAGEDKV_ERR_WORKSPACE = -5     /* split-K workspace missing or too small */
} pagedkv_status;

/* Bits of the sticky device error word. */
#define PAGEDKV_DEVERR_SLOT_RANGE   0x01u  /* append: slot >= num_blocks*block_size */
#define PAGEDKV_DEVERR_BLOCK_ID     0x02u  /* a block table entry outside [0, num_blocks) */
#define PAGEDKV_DEVERR_CONTEXT_LEN  0x04u  /* context_len < 0 or > max_blocks_per_seq*block_size */
#define PAGEDKV_DEVERR_POSITION     0x08u  /* slot mapping: position past the block table */
#define PAGEDKV_DEVERR_SEQ_INDEX    0x10u  /* slot mapping: token_seq outside [0, num_seqs);
                                              shared-prefix decode: a group id outside
                                              [-1, num_groups) */
#define PAGEDKV_DEVERR_TIMEOUT      0x20u  /* a bounded in-kernel wait gave up */

/* partition_tokens value of paged_attention_decode selecting the balanced split. */
#define PAGEDKV_PARTITION_BALANCED  (-1)

/*
 * paged_kv_slot_mapping -- address translation for a batch of new tokens.
 *
 * Implements "The one formula" (page "How a serving engine actually works"):
 * token t belongs to sequence token_seq[t] at logical position token_pos[t];
 *
 *     slot_mapping[t] = block_tables[seq][pos / block_size] * block_size
 *                       + pos % block_size.
 *
 *   block_tables  int32 [num_seqs][max_blocks_per_seq], device
 *   token_seq     int32 [num_tokens], device
 *   token_pos     int32 [num_tokens], device; a negative position is padding
 *   slot_mapping  int64 [num_tokens], device, written
 *
 * Padding maps to -1. A position past the table, a sequence index outside
 * [0, num_seqs) or a block id outside [0, num_blocks) also maps to -1 and sets
 * the matching device error bit. num_tokens == 0 enqueues nothing.
 */
int paged_kv_slot_mapping(const int32_t *block_tables, const int32_t *token_seq,
                          const int32_t *token_pos, int64_t *slot_mapping, int num_tokens,
                          int num_seqs, int max_blocks_per_seq, int block_size, int num_blocks,
                          void *stream);

/*
 * paged_kv_append -- scatter new tokens' K and V rows into their pool slots.
 *
 * The write half of the paged cache (page "Paged-KV + Continuous Batching From
 * Scratch", section "What's deliberately still missing": the append is plain
 * indexing into the pool):
 *
 *     k_cache[slot / block_size][slot % block_size][:][:] = k[t][:][:]
 *     v_cache[slot / block_size][slot % block_size][:][:] = v[t][:][:]
 *
 * with slot = slot_mapping[t]. A bit copy: the pools end up bit-identical to
 * what plain indexing produces.
 *
 *   k, v          [num_tokens][n_kv_heads][head_dim] of dtype, device
 *   slot_mapping  int64 [num_tokens], device; slot < 0 is padding (skipped)
 *   k_cache,
 *   v_cache       [num_blocks][block_size][n_kv_heads][head_dim] of dtype,
 *                 device, updated in place
 *
 * A slot >= num_blocks*block_size is skipped and sets PAGEDKV_DEVERR_SLOT_RANGE.
 * Two tokens with the same slot race; the caller must not do that.
 * Requires n_kv_heads*head_dim*sizeof(dtype) to be a multiple of 16 bytes.
 */
int paged_kv_append(const void *k, const void *v, const int64_t *slot_mapping, void *k_cache,
                    void *v_cache, int num_tokens, int num_blocks, int block_size,
                    int n_kv_heads, int head_dim, int dtype, void *stream);

/*
 * paged_kv_append_tokens -- paged_kv_slot_mapping and paged_kv_append in one
 * launch.
 *
 * For each new token t, the slot of "The one formula" (page "How a serving
 * engine actually works"),
 *
 *     slot = block_tables[token_seq[t]][token_pos[t] / block_size] * block_size
 *            + token_pos[t] % block_size,
 *
 * with the checks and device error bits of paged_kv_slot_mapping, then the
 * token's K and V rows copied to that slot as paged_kv_append does. The pools
 * end up bit-identical to those two calls' result.
 *
 *   k, v          [num_tokens][n_kv_heads][head_dim] of dtype, device
 *   block_tables  int32 [num_seqs][max_blocks_per_seq], device
 *   token_seq     int32 [num_tokens], device
 *   token_pos     int32 [num_tokens], device; a negative position is padding
 *   slot_mapping  int64 [num_tokens], device, written (-1 for padding and for
 *                 tokens that fail a check); may be NULL when not wanted
 *   k_cache,
 *   v_cache       [num_blocks][block_size][n_kv_heads][head_dim] of dtype,
 *                 device, updated in place
 *
 * A token whose check fails is not copied. Two tokens with the same slot race;
 * the caller must not do that. Requires n_kv_heads*head_dim*sizeof(dtype) to
 * be a multiple of 16 bytes. num_tokens == 0 enqueues nothing.
 */
int paged_kv_append_tokens(const void *k, const void *v, const int32_t *block_tables,
                           const int32_t *token_seq, const int32_t *token_pos,
                           int64_t *slot_mapping, void *k_cache, void *v_cache, int num_tokens,
                           int num_seqs, int max_blocks_per_seq, int num_blocks, int block_size,
                           int n_kv_heads, int head_dim, int dtype, void *stream);

/*
 * paged_kv_copy_blocks -- copy whole blocks of both pools, for copy-on-write.
 *
 * Page "How a serving engine actually works", section "Copy-on-write, because
 * you have used fork()": sequences forked from one prompt share its blocks;
 * the first write into a block that others still reference goes to a fresh
 * block, which must first receive the shared block's contents. For each pair
 * i, block_pairs[2i] (source) is copied to block_pairs[2i+1] (destination), K
 * and V, all block_size * n_kv_heads * head_dim elements: a bit copy.
 *
 *   k_cache, v_cache  [num_blocks][block_size][n_kv_heads][head_dim], device, updated
 *   block_pairs       int32 [num_pairs][2] = {src, dst}, device
 *
 * A pair with an id outside [0, num_blocks) is skipped and sets
 * PAGEDKV_DEVERR_BLOCK_ID; src == dst is a no-op. Destinations must be
 * distinct and must not be the source of another pair of the same call.
 */
int paged_kv_copy_blocks(void *k_cache, void *v_cache, const int32_t *block_pairs, int num_pairs,
                         int num_blocks, int block_size, int n_kv_heads, int head_dim, int dtype,
                         void *stream);

/*
 * paged_kv_swap_blocks -- copy whole blocks from one pair of pools into another.
 *
 * Page "Paged Attention and the Block Manager", section "Running out of memory
 * becomes a scheduling decision": a preempted sequence can keep its cache by
 * having its blocks copied out to host memory, and copied back on re-admission
 * into whichever device blocks are free then. For each pair i, block
 * block_pairs[2i] of the source pools is copied to block block_pairs[2i+1] of
 * the destination pools, K and V: a bit copy. One call covers every pair.
 *
 *   src_k, src_v    [src_num_blocks][block_size][n_kv_heads][head_dim] of dtype
 *   dst_k, dst_v    [dst_num_blocks][block_size][n_kv_heads][head_dim] of dtype,
 *                   updated in place
 *   block_pairs     int32 [num_pairs][2] = {source block, destination block}
 *
 * Every pointer may be memory of the current device, managed memory, or
 * page-locked host memory (cudaHostAlloc, cudaHostRegister, a pinned torch
 * tensor), which the kernel reads or writes in place over the host link; pool
 * pointers must be 16-byte aligned. Pageable host memory or another device's
 * memory: PAGEDKV_ERR_INVALID_ARG, nothing launched. Host memory must stay
 * allocated and page-locked until the copy has completed on `stream`.
 *
 * A pair with an id outside its own pool is skipped and sets
 * PAGEDKV_DEVERR_BLOCK_ID. Destinations must be distinct; when a source and a
 * destination pool are the same memory, no block may be both a source and a
 * destination of one call (such pairs race).
 */
int paged_kv_swap_blocks(const void *src_k, const void *src_v, int src_num_blocks, void *dst_k,
                         void *dst_v, int dst_num_blocks, const int32_t *block_pairs,
                         int num_pairs, int block_size, int n_kv_heads, int head_dim, int dtype,
                         void *stream);

/*
 * paged_attention_prefill -- chunked-prefill attention over the paged cache.
 *
 * Page "How a serving engine actually works", section "Prefill and decode are
 * two different jobs": a long prompt is prefilled in chunks, one chunk per
 * iteration, so that sequences decoding beside it are not stalled behind the
 * whole prompt. The chunk's K/V rows must already be in the pools (appended
 * with paged_kv_append). Sequence s owns query rows query_start[s] ..
 * query_start[s+1]-1 (n_s rows); with L_s = context_lens[s] cached tokens, the
 * chunk included, row j is the token at position L_s - n_s + j and attends over
 * keys 0 .. L_s - n_s + j of its sequence, read through its block table:
 *
 *     out[row][qh][:] = softmax_i(scale * q[row][qh] . K[i][qh / g]) V[i][qh / g]
 *
 * Decode is the case n_s = 1. Tensor-core path: fp16 and bf16 only, fp32
 * accumulation, one rounding of `out` to the input type. Two kernels compute
 * it (PAGEDKV_OPT_PREFILL_PATH): tcgen05 MMAs with accumulators in tensor
 * memory (default), or warp-level m16n8k16 MMAs.
 *
 *   q, out         [num_tokens][n_q_heads][head_dim] of dtype, device, 16-byte aligned;
 *                  every row of q may be read (the tcgen05 kernel copies Q
 *                  tiles of 128 / group whole tokens by TMA, past a chunk's end
 *                  too), but a row outside a chunk, such as padding past
 *                  query_start[num_seqs], never reaches an output row and its
 *                  out row is not written
 *   k_cache,
 *   v_cache        [num_blocks][block_size][n_kv_heads][head_dim], device, 16-byte aligned
 *   block_tables   int32 [num_seqs][max_blocks_per_seq], device
 *   query_start    int32 [num_seqs + 1], device, non-decreasing from 0 (num_tokens
 *                  may be larger than query_start[num_seqs])
 *   context_lens   int32 [num_seqs], device
 *   max_query_len  an upper bound of every n_s (sizes the work: query tiles per
 *                  sequence; the tcgen05 kernel runs one persistent CTA per SM
 *                  over them)
 *
 * Returns PAGEDKV_ERR_UNSUPPORTED for fp32, head_dim other than 64/128, block
 * size other than 8/16/32, more than 64 query heads per kv head, or (tcgen05
 * kernel) more than 2^30 work items of (sequence, kv head, 256 query rows). On the
 * device, a sequence whose rows fall outside [0, num_tokens) or exceed the
 * grid's max_query_len sets PAGEDKV_DEVERR_POSITION; one with n_s > L_s or L_s
 * beyond its table sets PAGEDKV_DEVERR_CONTEXT_LEN; a block id outside the pool
 * sets PAGEDKV_DEVERR_BLOCK_ID (block 0 is read instead). The rows of a
 * flagged sequence are left unwritten. Asynchronous on `stream`; allocates
 * nothing.
 */
int paged_attention_prefill(const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, const int32_t *query_start,
                            const int32_t *context_lens, float scale, void *out, int num_seqs,
                            int num_tokens, int max_query_len, int n_q_heads, int n_kv_heads,
                            int head_dim, int num_blocks, int block_size,
                            int max_blocks_per_seq, int dtype, void *stream);

/*
 * paged_attention_prefill_split -- the same attention with the call's keys
 * shared out evenly over the SMs (a split-K over the key range), for calls
 * with few items over long contexts (one short chunk, few sequences). The key
 * tiles (64 keys) of every (sequence, 2 * (128 / group) chunk tokens, kv
 * head) item of the tcgen05 kernel, all items end to end, are cut into one
 * contiguous range per SM of r tiles each: r at least the total over the SMs,
 * at least min(16, the longest item's tiles), and long enough that no item
 * meets more than key_parts ranges. An item inside one range writes `out`
 * itself; an item cut by a range boundary writes, per piece, its rows'
 * unnormalised fp32 output and softmax state to `workspace`, and a merge
 * kernel on the same stream combines them into `out` (softmax's LSE identity,
 * the same one split-K decode uses). The result equals
 * paged_attention_prefill's within rounding.
 *
 *   key_parts        1 .. 32: most ranges one item meets; 1 is
 *                    paged_attention_prefill itself. 0 splits when the items
 *                    (counted from max_query_len) are fewer than the SMs and
 *                    the workspace holds the split (32 ranges at most), else
 *                    runs whole items. Calls of more than 500 items run whole
 *                    items at any key_parts.
 *   workspace        device, 256-byte aligned, caller-owned, at least
 *                    paged_attention_prefill_workspace_bytes(head_dim) bytes
 *                    (it depends on the device's SM count only); its contents
 *                    on entry do not matter and are garbage afterwards
 *   other arguments  as for paged_attention_prefill
 *
 * Returns PAGEDKV_ERR_WORKSPACE when the call splits (key_parts >= 2) and the
 * workspace is missing or too small, PAGEDKV_ERR_INVALID_ARG for key_parts
 * outside 0 .. 32 or a misaligned workspace; otherwise as
 * paged_attention_prefill (whose device errors it sets the same way). With
 * PAGEDKV_OPT_PREFILL_PATH = 1 (the warp-level MMA kernel) the keys are not
 * split. Asynchronous on `stream`; allocates nothing. Calls that share a
 * workspace must be ordered on one stream.
 */
int paged_attention_prefill_split(const void *q, const void *k_cache, const void *v_cache,
                                  const int32_t *block_tables, const int32_t *query_start,
                                  const int32_t *context_lens, float scale, void *out, int num_seqs,
                                  int num_tokens, int max_query_len, int n_q_heads, int n_kv_heads,
                                  int head_dim, int num_blocks, int block_size,
                                  int max_blocks_per_seq, int dtype, int key_parts, void *workspace,
                                  size_t workspace_bytes, void *stream);

/* Workspace bytes of paged_attention_prefill_split on the current device
 * (head_dim 64 or 128; 0 for any other, or without a device): an int per
 * item (500), then fp32 outputs [2 * SMs][256 rows][head_dim], then two fp32
 * [2 * SMs][256 rows] arrays, each on a 256-byte boundary. */
size_t paged_attention_prefill_workspace_bytes(int head_dim);

/*
 * paged_attention_decode -- fused paged-attention decode.
 *
 * The kernel the pages name as the next step and never build (page "Paged-KV +
 * Continuous Batching From Scratch", section "What's deliberately still
 * missing"; page "Paged Attention and the Block Manager", section "The
 * measurement"): attention over each sequence's cache, reading K and V
 * through the block table inside the kernel instead of gathering them into a
 * contiguous copy first. The mathematics is unchanged softmax attention:
 *
 *     for each sequence s and query head h (kv head h / (n_q_heads/n_kv_heads)):
 *         z_i   = scale * q[s][h] . K_s[i]          for i < context_lens[s]
 *         out[s][h] = sum_i softmax(z)_i V_s[i]
 *
 * with K_s[i] = k_cache at slot(s, i). Scores, the running max and sum and the
 * output accumulator are fp32; out is rounded once to dtype (round to nearest
 * even). A context length of 0 gives a zero row.
 *
 *   q             [num_seqs][n_q_heads][head_dim] of dtype, device
 *   k_cache,
 *   v_cache       [num_blocks][block_size][n_kv_heads][head_dim] of dtype, device
 *   block_tables  int32 [num_seqs][max_blocks_per_seq], device; entries past a
 *                 sequence's ceil(context_len / block_size) blocks are never read
 *   context_lens  int32 [num_seqs], device
 *   out           [num_seqs][n_q_heads][head_dim] of dtype, device, written
 *
 * partition_tokens == 0: each (sequence, kv head) is processed whole.
 * partition_tokens == PAGEDKV_PARTITION_BALANCED (-1): balanced split. The
 *   list of all 16-token tiles, ordered [sequence][kv head group][tile], is
 *   cut into equal contiguous shares, one per CTA of the (persistent) grid, so
 *   every CTA streams the same number of bytes whatever the length mix. A
 *   (sequence, kv head) that falls inside one share is written directly; one
 *   that spans shares leaves one unnormalised state per share (at most two
 *   per CTA) in the workspace, which a merge kernel combines as below. The
 *   workspace layout of this mode is internal; size it with
 *   paged_attention_workspace_bytes(..., PAGEDKV_PARTITION_BALANCED), which
 *   depends on the current device's SM count.
 * partition_tokens > 0 (a multiple of 16): split-K. Each sequence's context is
 *   cut into partitions of that many tokens; each (sequence, kv head,
 *   partition) produces an unnormalised state per query head
 *       m_p = max z_i,  l_p = sum e^(z_i - m_p),  o_p = sum e^(z_i - m_p) V_i
 *   over its tokens, and a merge kernel combines them:
 *       M = max_p m_p,  out = sum_p e^(m_p - M) o_p / sum_p e^(m_p - M) l_p.
 *   Sequences that fit in one partition skip the merge. The states live in
 *   the caller's workspace (see paged_attention_workspace_bytes), as fp32
 *       o [num_seqs][n_q_heads][P][head_dim], then m [num_seqs][n_q_heads][P],
 *       then l [num_seqs][n_q_heads][P],
 *   P = ceil(max_blocks_per_seq*block_size / partition_tokens), each array
 *   starting on a 256-byte boundary; m is in natural-log units. Entries of
 *   partitions a sequence does not have are left untouched.
 *
 * Supported: head_dim 64 or 128; block_size 8, 16 or 32; n_q_heads a multiple
 * of n_kv_heads with n_q_heads / n_kv_heads <= 8; num_seqs <= 4096.
 * workspace may be NULL when partition_tokens == 0.
 */
int paged_attention_decode(const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *block_tables, const int32_t *context_lens,
                           float scale, void *out, int num_seqs, int n_q_heads, int n_kv_heads,
                           int head_dim, int num_blocks, int block_size, int max_blocks_per_seq,
                           int partition_tokens, void *workspace, size_t workspace_bytes,
                           int dtype, void *stream);

/*
 * paged_attention_decode_shared_prefix -- decode that reads each shared
 * prefix once per group of sequences instead of once per sequence.
 *
 * Pages "Paged-KV + Continuous Batching From Scratch" (section 1: sequences
 * that share a system prompt share its physical blocks, a reference-count
 * bump instead of a copy) and "How a serving engine actually works" (sections
 * "Copy-on-write, because you have used fork()" and "Prefix caching: prefill
 * you already did"): sharing saves memory; this entry point also saves the
 * bandwidth of reading the shared blocks once per sharer.
 *
 * Same arguments and results as paged_attention_decode (within the same
 * tolerance) plus the sharing structure:
 *   seq_group     int32 [num_seqs], device: prefix group of each sequence, -1
 *                 for none. Members of a group are consecutive sequences. A
 *                 group id >= num_groups or below -1 sets
 *                 PAGEDKV_DEVERR_SEQ_INDEX and the sequence is decoded as if
 *                 it had no group (a run of the group's members that it
 *                 interrupts continues after it as a new run).
 *   group_prefix  int32 [num_groups], device: the number of leading tokens
 *                 that every member of the group holds in the SAME physical
 *                 blocks as the group's first member (the caller's
 *                 reference-counted prefix); it must not exceed any member's
 *                 context length (else PAGEDKV_DEVERR_CONTEXT_LEN).
 * The whole partitions of each prefix (floor(group_prefix / partition_tokens))
 * are computed once per chunk of up to 8 / (n_q_heads / n_kv_heads) members:
 * the chunk's (member, query head) pairs fill the columns of one tensor-core
 * tile, so the prefix's K/V are read once per chunk; the rest of each
 * sequence is computed per sequence and everything is merged as in split-K.
 * Requires partition_tokens > 0 (with its workspace) and n_kv_heads a
 * multiple of 4. The kernel trusts the sharing structure: if a member's
 * prefix blocks differ from the first member's, its result is computed
 * with the first member's.
 */
int paged_attention_decode_shared_prefix(const void *q, const void *k_cache, const void *v_cache,
                                         const int32_t *block_tables, const int32_t *context_lens,
                                         const int32_t *seq_group, const int32_t *group_prefix,
                                         int num_groups, float scale, void *out, int num_seqs,
                                         int n_q_heads, int n_kv_heads, int head_dim,
                                         int num_blocks, int block_size, int max_blocks_per_seq,
                                         int partition_tokens, void *workspace,
                                         size_t workspace_bytes, int dtype, void *stream);

/* Workspace bytes paged_attention_decode needs for these sizes (0 when
 * partition_tokens == 0). Returns 0 for invalid sizes as well, and for the
 * balanced split when no CUDA device is current. */
size_t paged_attention_workspace_bytes(int num_seqs, int n_q_heads, int head_dim,
                                       int max_blocks_per_seq, int block_size,
                                       int partition_tokens);

/*
 * paged_attention_decode_noalloc -- paged_attention_decode for callers that
 * must not allocate device memory on their call path and so cannot provide a
 * split-K workspace: a serving loop with a fixed per-step latency budget
 * (cudaMalloc may synchronise the device and take milliseconds), a plug-in
 * whose host application owns all device memory through its own pool, or a
 * process that has already handed the free memory to another allocator.
 * The pages have no counterpart to this entry point.
 *
 * Same arguments and results as paged_attention_decode, without workspace
 * and workspace_bytes: the partition states live in one library-owned device
 * array of PAGEDKV_NOALLOC_SCRATCH_BYTES, which every GPU that loads the
 * library keeps until the process exits. The call allocates nothing.
 *   - A split whose paged_attention_workspace_bytes() exceeds
 *     PAGEDKV_NOALLOC_SCRATCH_BYTES is rejected with PAGEDKV_ERR_WORKSPACE
 *     before anything is enqueued. partition_tokens == 0 needs no scratch;
 *     PAGEDKV_PARTITION_BALANCED uses it like any split.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current, and so does the first
 *     call after cudaDeviceReset has replaced the device's context; make
 *     those calls before any stream capture.
 *   - Every call on a device shares the one array, and it keeps the last
 *     call's contents. Nothing in it needs to start at zero: each call writes
 *     every partition state it later reads. Calls whose work overlaps on the
 *     GPU (for example on two streams without an ordering between them) race
 *     on the array and give wrong results; order them on one stream.
 */
#define PAGEDKV_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int paged_attention_decode_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                   const int32_t *block_tables, const int32_t *context_lens,
                                   float scale, void *out, int num_seqs, int n_q_heads,
                                   int n_kv_heads, int head_dim, int num_blocks, int block_size,
                                   int max_blocks_per_seq, int partition_tokens, int dtype,
                                   void *stream);


/*
 * pagedkv_device_errors -- read (and optionally clear) the sticky device
 * error word of the current device. Synchronises the device first, so it
 * sees every kernel enqueued before the call. *flags receives the PAGEDKV_DEVERR_*
 * bits. Returns PAGEDKV_OK when no bit is set, PAGEDKV_ERR_BOUNDS when one is,
 * PAGEDKV_ERR_CUDA when the read fails.
 */
int pagedkv_device_errors(unsigned int *flags, int reset);

/*
 * pagedkv_check_bounded_wait -- a check of the library's failure path. Enqueues
 * one small kernel on `stream` whose wait on an mbarrier that nothing arrives
 * on gives up after the in-kernel time limit (1 s), as every wait of the
 * library's kernels does when a peer never arrives: it sets
 * PAGEDKV_DEVERR_TIMEOUT in the sticky device error word and the kernel exits
 * normally, leaving the context usable. Returns PAGEDKV_OK once enqueued.
 */
int pagedkv_check_bounded_wait(void *stream);

/* Tuning knobs, process-wide and not thread-safe; for tests and benchmarks. */
#define PAGEDKV_OPT_DECODE_PATH    1  /* 0 auto, 1 CUDA-core (SIMT) path, 2 tensor-core (mma) path */
#define PAGEDKV_OPT_CTAS_PER_SM    2  /* persistent decode CTAs per SM; 0 = library default */
#define PAGEDKV_OPT_MMA_MIN_GROUP  3  /* auto path: smallest q-per-kv group that takes the mma path (default 1:
                                         every 16-bit pool; fp32 always takes the CUDA-core path) */
#define PAGEDKV_OPT_STAGES         4  /* decode stage-ring size (2..16) for every call; 0 = automatic: fixed
                                         partitions take 2 from 512 tokens up, else about 96 KB of stages; the
                                         balanced split takes 2 when the block tables' full width of K/V fits in
                                         L2, else about 96 KB of stages of which each CTA uses 2 when the mean
                                         context is 6144 tokens or more */
#define PAGEDKV_OPT_PREFILL_PATH   5  /* 0 auto (= 2), 1 warp-level MMA prefill kernel, 2 tcgen05 prefill kernel */
#define PAGEDKV_OPT_L2_HINTS       6  /* L2 priorities on the decode's K/V loads (blocks that the previous or next
                                         sequence holds at the same table index evict_last, the rest evict_first):
                                         0 auto = when the call's K/V tokens exceed what the L2 holds, 1 never,
                                         2 always. Only neighbouring sequences' blocks are compared: order the
                                         batch so that sequences sharing blocks sit next to each other (e.g. by
                                         first block id) */
int pagedkv_set_option(int option, int value);
int pagedkv_get_option(int option);

/* Library path of the last decode call, for tests: 1 SIMT, 2 mma. */
int pagedkv_last_decode_path(void);

/* Human-readable name of a pagedkv_status. Never NULL. */
const char *pagedkv_status_string(int status);

/* PAGEDKV_ABI_VERSION of the built library. */
int pagedkv_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
