// decode_launch.h -- host-side launch interface between the C ABI layer and
// the per-element-type decode translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "decode_params.h"

namespace pkv {

enum DecodePath { kPathAuto = 0, kPathSimt = 1, kPathMma = 2 };

struct DecodeLaunch {
    DecodeParams p;
    CUtensorMap kmap;
    CUtensorMap vmap;
    int head_dim;
    int path;          // kPathSimt or kPathMma
    int gmax;          // query-group capacity of the instantiation (1, 2, 4 or 8)
    int ctas_per_sm;   // wanted persistent CTAs per SM
    int num_sms;
    long long max_units;  // upper bound of the units the grid can find
    cudaStream_t stream;
    int grid_used;        // out: CTAs launched
};

// One per element type; each returns the launch's cudaError_t.
cudaError_t launch_decode_f32(DecodeLaunch &a);
cudaError_t launch_decode_f16(DecodeLaunch &a);
cudaError_t launch_decode_bf16(DecodeLaunch &a);

// Log-sum-exp merge of split-K partition states (dtype: pagedkv_dtype).
cudaError_t launch_lse_merge(int dtype, int head_dim, const float *ws_o, const float *ws_m,
                             const float *ws_l, const int32_t *context_lens, void *out,
                             int num_seqs, int n_q_heads, int part_tokens, int max_parts,
                             int max_context, unsigned int *err, cudaStream_t stream);

// Merge of balanced-split pieces (and zero rows of empty sequences).
cudaError_t launch_piece_merge(int dtype, int head_dim, const float *ws_o, const float *ws_m,
                               const float *ws_l, const int32_t *context_lens, void *out,
                               int num_seqs, int n_q_heads, int groups, int rows_per_unit,
                               int decode_grid, int max_context, cudaStream_t stream);

// Stage-ring size for an element size, head_dim and kv heads per unit.
int decode_stages(int elem_bytes, int head_dim, int heads_per_unit, int part_tokens);

}  // namespace pkv
