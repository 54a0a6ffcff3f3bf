// merge.cu -- log-sum-exp merge of split-K partition states.
//
// For each (sequence, query head) whose context spans more than one
// partition: M = max_p m_p, out = sum_p e^(m_p - M) o_p / sum_p e^(m_p - M) l_p,
// the identity that recombines softmax attention computed over disjoint token
// ranges.
#include "decode_launch.h"
#include "ptx.cuh"

namespace pkv {

template <int E> struct Vec;
template <> struct Vec<2> { using type = float2; };
template <> struct Vec<4> { using type = float4; };

constexpr int kMergeWarps = 8;

// Block-wide reduction helper over kMergeWarps warps (max or sum).
template <bool kMax>
__device__ __forceinline__ float block_reduce(float v, float *scratch) {
#pragma unroll
    for (int mask = 16; mask >= 1; mask >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, v, mask);
        v = kMax ? fmaxf(v, o) : v + o;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    v = scratch[0];
#pragma unroll
    for (int w = 1; w < kMergeWarps; ++w) v = kMax ? fmaxf(v, scratch[w]) : v + scratch[w];
    return v;
}

// One CTA per (sequence, query head), for rows of many partitions. Warps take
// partitions round-robin; each lane owns head_dim / 32 contiguous outputs.
template <typename T, int D>
__global__ void __launch_bounds__(32 * kMergeWarps)
lse_merge_kernel(const float *__restrict__ ws_o, const float *__restrict__ ws_m,
                 const float *__restrict__ ws_l, const int32_t *__restrict__ lens,
                 T *__restrict__ out, int n_q_heads, int part_tokens, int max_parts, int cap) {
    constexpr int E = D / 32;
    using V = typename Vec<E>::type;
    __shared__ float red[kMergeWarps];
    __shared__ float acc_s[kMergeWarps][D];
    // partition states are written by the preceding decode launch
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int row = blockIdx.x;   // s * n_q_heads + qh
    const int s = row / n_q_heads;
    const int L = min(max(__ldg(lens + s), 0), cap);
    const int np = L > 0 ? (L + part_tokens - 1) / part_tokens : 1;
    if (np <= 1) return;  // written directly by the partition kernel
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t row0 = size_t(row) * max_parts;
    float M = -INFINITY;
    for (int k = threadIdx.x; k < np; k += blockDim.x) M = fmaxf(M, ws_m[row0 + k]);
    M = block_reduce<true>(M, red);
    float den = 0.f;
    for (int k = threadIdx.x; k < np; k += blockDim.x)
        den = fmaf(fast_exp2((ws_m[row0 + k] - M) * kLog2e), ws_l[row0 + k], den);
    den = block_reduce<false>(den, red);
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll 4
    for (int k = warp; k < np; k += kMergeWarps) {
        const float w = fast_exp2((ws_m[row0 + k] - M) * kLog2e);
        const V x = *reinterpret_cast<const V *>(ws_o + (row0 + k) * D + lane * E);
        const float *xf = reinterpret_cast<const float *>(&x);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(w, xf[e], acc[e]);
    }
#pragma unroll
    for (int e = 0; e < E; ++e) acc_s[warp][lane * E + e] = acc[e];
    __syncthreads();
    const float inv = den > 0.f ? 1.f / den : 0.f;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kMergeWarps; ++w) v += acc_s[w][d];
        out[size_t(row) * D + d] = Elem<T>::from_float(v * inv);
    }
}

// One warp per (sequence, query head), for rows of at most 32 partitions:
// lane p holds partition p's (m, l); each lane owns head_dim / 32 outputs.
template <typename T, int D>
__global__ void __launch_bounds__(256)
lse_merge_rows_kernel(const float *__restrict__ ws_o, const float *__restrict__ ws_m,
                      const float *__restrict__ ws_l, const int32_t *__restrict__ lens,
                      T *__restrict__ out, int rows, int n_q_heads, int part_tokens, int max_parts,
                      int cap) {
    constexpr int E = D / 32;
    using V = typename Vec<E>::type;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int s = row / n_q_heads;
    const int L = min(max(__ldg(lens + s), 0), cap);
    const int np = L > 0 ? (L + part_tokens - 1) / part_tokens : 1;
    if (np <= 1) return;  // written directly by the partition kernel
    const size_t row0 = size_t(row) * max_parts;
    const float mp = lane < np ? ws_m[row0 + lane] : -INFINITY;
    float M = mp;
#pragma unroll
    for (int mask = 16; mask >= 1; mask >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, mask));
    const float w = lane < np ? fast_exp2((mp - M) * kLog2e) : 0.f;
    float den = lane < np ? w * ws_l[row0 + lane] : 0.f;
#pragma unroll
    for (int mask = 16; mask >= 1; mask >>= 1) den += __shfl_xor_sync(0xffffffffu, den, mask);
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll 4
    for (int k = 0; k < np; ++k) {
        const float wk = __shfl_sync(0xffffffffu, w, k);
        const V x = *reinterpret_cast<const V *>(ws_o + (row0 + k) * D + lane * E);
        const float *xf = reinterpret_cast<const float *>(&x);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = fmaf(wk, xf[e], acc[e]);
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) out[size_t(row) * D + lane * E + e] = Elem<T>::from_float(acc[e] * inv);
}

// Launched as a programmatic dependent of the decode kernel when the device
// allows it, so that its launch overlaps the decode kernel's last CTAs; the
// kernel's griddepcontrol.wait still orders it after all of the decode's writes.
template <typename T>
static cudaError_t launch_merge_typed(int head_dim, const float *ws_o, const float *ws_m,
                                      const float *ws_l, const int32_t *lens, void *out, int S,
                                      int Hq, int P, int max_parts, int cap, cudaStream_t st) {
    const long long rows = (long long)S * Hq;
    if (rows == 0) return cudaSuccess;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    T *o = static_cast<T *>(out);
    if (max_parts <= 32) {
        // few partitions per row: a warp per row, 8 rows per CTA
        cfg.gridDim = dim3(unsigned((rows + 7) / 8));
        cfg.blockDim = dim3(256);
        if (head_dim == 64)
            return cudaLaunchKernelEx(&cfg, lse_merge_rows_kernel<T, 64>, ws_o, ws_m, ws_l, lens, o,
                                      int(rows), Hq, P, max_parts, cap);
        return cudaLaunchKernelEx(&cfg, lse_merge_rows_kernel<T, 128>, ws_o, ws_m, ws_l, lens, o,
                                  int(rows), Hq, P, max_parts, cap);
    }
    cfg.gridDim = dim3(unsigned(rows));
    cfg.blockDim = dim3(32 * kMergeWarps);
    if (head_dim == 64)
        return cudaLaunchKernelEx(&cfg, lse_merge_kernel<T, 64>, ws_o, ws_m, ws_l, lens, o, Hq, P,
                                  max_parts, cap);
    return cudaLaunchKernelEx(&cfg, lse_merge_kernel<T, 128>, ws_o, ws_m, ws_l, lens, o, Hq, P,
                              max_parts, cap);
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

int decode_stages(int elem_bytes, int head_dim, int heads_per_unit, int part_tokens) {
    // About 96 KB of K/V stages per CTA (two CTAs per SM), at least double
    // buffered. Units of 512 tokens or more stream long runs of blocks and do
    // best with two stages per CTA (measured on the long-context workload);
    // shorter units take three.
    const int stage = decode_stage_bytes(elem_bytes, head_dim, heads_per_unit);
    int n = (96 * 1024) / stage;
    if (part_tokens >= 512 && n > 2) n = 2;
    return n < 2 ? 2 : (n > 8 ? 8 : n);
}

}  // namespace pkv
