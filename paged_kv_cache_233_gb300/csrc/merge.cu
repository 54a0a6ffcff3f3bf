// merge.cu -- log-sum-exp merge of split-K partition states.
//
// For each (sequence, query head) whose context spans more than one
// partition: M = max_p m_p, out = sum_p e^(m_p - M) o_p / sum_p e^(m_p - M) l_p,
// the identity that recombines softmax attention computed over disjoint token
// ranges. One warp per (sequence, query head); each lane owns head_dim / 32
// contiguous output elements.
#include "decode_launch.h"
#include "ptx.cuh"

namespace pkv {

template <int E> struct Vec;
template <> struct Vec<2> { using type = float2; };
template <> struct Vec<4> { using type = float4; };

template <typename T, int D>
__global__ void __launch_bounds__(256)
lse_merge_kernel(const float *__restrict__ ws_o, const float *__restrict__ ws_m,
                 const float *__restrict__ ws_l, const int32_t *__restrict__ lens,
                 T *__restrict__ out, int num_seqs, int n_q_heads, int part_tokens,
                 int max_parts, int cap) {
    constexpr int E = D / 32;
    const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (gw >= num_seqs * n_q_heads) return;
    const int s = gw / n_q_heads;
    const int L = min(max(__ldg(lens + s), 0), cap);
    const int np = L > 0 ? (L + part_tokens - 1) / part_tokens : 1;
    if (np <= 1) return;  // written directly by the partition kernel
    const size_t row0 = size_t(gw) * max_parts;
    float M = -INFINITY;
    for (int k = lane; k < np; k += 32) M = fmaxf(M, ws_m[row0 + k]);
#pragma unroll
    for (int mask = 16; mask >= 1; mask >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, mask));
    float den = 0.f;
    for (int k = lane; k < np; k += 32)
        den = fmaf(fast_exp2((ws_m[row0 + k] - M) * kLog2e), ws_l[row0 + k], den);
#pragma unroll
    for (int mask = 16; mask >= 1; mask >>= 1) den += __shfl_xor_sync(0xffffffffu, den, mask);
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    using V = typename Vec<E>::type;
#pragma unroll 4
    for (int k = 0; k < np; ++k) {
        const float w = fast_exp2((ws_m[row0 + k] - M) * kLog2e);
        const V x = *reinterpret_cast<const V *>(ws_o + (row0 + k) * D + lane * E);
        const float *xf = reinterpret_cast<const float *>(&x);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(w, xf[e], acc[e]);
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) out[size_t(gw) * D + lane * E + e] = Elem<T>::from_float(acc[e] * inv);
}

template <typename T>
static cudaError_t launch_merge_typed(int head_dim, const float *ws_o, const float *ws_m,
                                      const float *ws_l, const int32_t *lens, void *out, int S,
                                      int Hq, int P, int max_parts, int cap, cudaStream_t st) {
    const long long warps = (long long)S * Hq;
    const int per_block = 8;
    const unsigned blocks = unsigned((warps + per_block - 1) / per_block);
    if (blocks == 0) return cudaSuccess;
    if (head_dim == 64)
        lse_merge_kernel<T, 64><<<blocks, 32 * per_block, 0, st>>>(
            ws_o, ws_m, ws_l, lens, static_cast<T *>(out), S, Hq, P, max_parts, cap);
    else
        lse_merge_kernel<T, 128><<<blocks, 32 * per_block, 0, st>>>(
            ws_o, ws_m, ws_l, lens, static_cast<T *>(out), S, Hq, P, max_parts, cap);
    return cudaGetLastError();
}

cudaError_t launch_lse_merge(int dtype, int head_dim, const float *ws_o, const float *ws_m,
                             const float *ws_l, const int32_t *context_lens, void *out,
                             int num_seqs, int n_q_heads, int part_tokens, int max_parts,
                             int max_context, unsigned int *, cudaStream_t stream) {
    switch (dtype) {
        case PAGEDKV_F32:
            return launch_merge_typed<float>(head_dim, ws_o, ws_m, ws_l, context_lens, out,
                                             num_seqs, n_q_heads, part_tokens, max_parts,
                                             max_context, stream);
        case PAGEDKV_F16:
            return launch_merge_typed<__half>(head_dim, ws_o, ws_m, ws_l, context_lens, out,
                                              num_seqs, n_q_heads, part_tokens, max_parts,
                                              max_context, stream);
        case PAGEDKV_BF16:
            return launch_merge_typed<__nv_bfloat16>(head_dim, ws_o, ws_m, ws_l, context_lens,
                                                     out, num_seqs, n_q_heads, part_tokens,
                                                     max_parts, max_context, stream);
        default:
            return cudaErrorInvalidValue;
    }
}

int decode_stages(int elem_bytes, int head_dim, int heads_per_unit) {
    // about 96 KB of K/V stages per CTA (two CTAs per SM), at least double buffered
    const int stage = decode_stage_bytes(elem_bytes, head_dim, heads_per_unit);
    int n = (96 * 1024) / stage;
    return n < 2 ? 2 : (n > 8 ? 8 : n);
}

}  // namespace pkv
