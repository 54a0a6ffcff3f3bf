// decode_params.h -- parameters and shared-memory layout of the paged decode
// kernel, visible to host launch code and device code alike.
#pragma once

#include <stdint.h>

#ifndef __CUDACC__
#define __host__
#define __device__
#endif

namespace pkv {

constexpr int kTile = 16;                 // tokens per pipeline stage
constexpr int kConsumerWarps = 4;         // also the largest kv-head group of a unit
constexpr int kDecodeThreads = 32 * (1 + kConsumerWarps);
constexpr int kRowBytes128 = 128;         // width of one swizzled column slab
// Balanced split: mean context (tokens) from which a call streams long runs of
// blocks and takes the two-stage ring (measured on GB300: three stages are
// ahead up to 4K-token means, two from 8K on)
constexpr int kLongSeqTokens = 6144;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;

struct DecodeParams {
    const void *q;
    void *out;
    const int32_t *block_tables;
    const int32_t *context_lens;
    float *ws_o;
    float *ws_m;
    float *ws_l;
    unsigned int *err;
    float scale_log2;     // softmax scale * log2(e): scores are kept in base-2 units
    int num_seqs;
    int n_q_heads;
    int n_kv_heads;
    int group;            // n_q_heads / n_kv_heads
    int num_blocks;
    int block_size;
    int log2_block;
    int max_blocks;       // block table row length
    int part_tokens;      // tokens per partition (multiple of kTile)
    int max_parts;        // partitions per (seq, q head) in the workspace
    int split;            // 1: multi-partition sequences write partition states
    int balanced;         // 1: balanced split (equal tile shares per CTA, pieces merged)
    int stages;           // ring size the shared memory holds (>= 2)
    int stages_alt;       // ring size used (<= stages) when the mean context is at least
    int long_seq_tokens;  // this many tokens
    int heads_per_unit;   // kv heads per unit: 1, 2 or 4 (one consumer warp per head)
    int log2_hpu;
    int rows_per_box;     // tokens per TMA box: min(block_size, kTile)
    // shared prefixes (fixed split only): consecutive sequences of one group hold
    // their first group_prefix[g] tokens in the same physical blocks
    const int32_t *seq_group;     // [num_seqs], -1 = no group; null = feature off
    const int32_t *group_prefix;  // [num_groups] tokens
    int num_groups;
    int max_members;      // sequences whose queries one prefix unit serves
    // the K/V loads carry L2 eviction priorities when the call attends over more
    // tokens than this (0: always; LLONG_MAX: never)
    long long hint_min_tokens;
};

// Byte layout of the dynamic shared memory (host and device agree on it).
// merge == 0 when every consumer warp owns a whole head (no cross-warp merge);
// prefix == 1 adds two per-sequence arrays for shared-prefix units.
struct DecodeSmem {
    int stage_bytes, stages, seqs, head_dim, gmax, merge, prefix;
    __host__ __device__ int ring() const { return stages * stage_bytes; }
    __host__ __device__ int bars() const { return ring(); }                        // full, empty
    __host__ __device__ int flag() const { return bars() + 16 * stages; }
    __host__ __device__ int seq_base() const { return flag() + 16; }               // seqs + 1 ints
    __host__ __device__ int seq_len() const { return seq_base() + 4 * (seqs + 1); }
    __host__ __device__ int seq_p0() const { return seq_len() + 4 * seqs; }        // first own partition
    __host__ __device__ int seq_pu() const { return seq_p0() + (prefix ? 4 * seqs : 0); }  // prefix units led
    __host__ __device__ int merge_o() const { return (seq_pu() + (prefix ? 4 * seqs : 0) + 15) & ~15; }
    __host__ __device__ int row_stride() const { return head_dim + 4; }            // floats
    // two slots (double buffer) x consumer warps x gmax heads
    __host__ __device__ int merge_rows() const { return merge ? 2 * kConsumerWarps * gmax : 0; }
    __host__ __device__ int merge_m() const { return merge_o() + 4 * merge_rows() * row_stride(); }
    __host__ __device__ int merge_l() const { return merge_m() + 4 * merge_rows(); }
    __host__ __device__ int total() const { return merge_l() + 4 * merge_rows(); }
    // bytes to request: layout plus slack to align the ring to 1024 B
    __host__ __device__ int request() const { return total() + 1024; }
};

// Bytes of one stage: K and V for kTile tokens of `heads` kv heads.
__host__ __device__ inline int decode_stage_bytes(int elem_bytes, int head_dim, int heads) {
    return 2 * heads * head_dim * elem_bytes * kTile;
}

}  // namespace pkv
