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

// E consecutive outputs of a row (E = head_dim / 32, one lane's share) as one
// vector store: 8 or 16 bytes instead of E scalar stores.
template <typename T, int E>
__device__ __forceinline__ void store_outputs(T *dst, const float *v) {
    if constexpr (sizeof(T) == 4) {
        if constexpr (E == 4) *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
        else *reinterpret_cast<float2 *>(dst) = make_float2(v[0], v[1]);
    } else {
        if constexpr (E == 4)
            *reinterpret_cast<uint2 *>(dst) = make_uint2(Elem<T>::pack2(v[0], v[1]), Elem<T>::pack2(v[2], v[3]));
        else
            *reinterpret_cast<uint32_t *>(dst) = Elem<T>::pack2(v[0], v[1]);
    }
}

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

// One CTA per (sequence, query head), for rows of many partitions. Each
// thread loads the (m, l) of partitions t, t + 256, ... once; the block
// reduces M and the denominator and leaves each partition's weight
// e^(m_p - M) in shared memory; then every warp takes partitions
// round-robin and issues the loads of up to kOBatch of its o rows at once
// (lane i holds head_dim / 32 outputs), so a row costs a few round trips to
// L2 whatever its partition count. Rows of up to kMaxParts partitions keep
// their weights in shared memory; longer rows recompute them.
constexpr int kMaxParts = 1024;
constexpr int kOBatch = 8;

template <typename T, int D>
__global__ void __launch_bounds__(32 * kMergeWarps)
lse_merge_kernel(const float *__restrict__ ws_o, const float *__restrict__ ws_m,
                 const float *__restrict__ ws_l, const int32_t *__restrict__ lens,
                 T *__restrict__ out, int n_q_heads, int part_tokens, int max_parts, int cap) {
    constexpr int E = D / 32;
    using V = typename Vec<E>::type;
    __shared__ float red[kMergeWarps];
    __shared__ float wgt[kMaxParts];
    __shared__ float acc_s[kMergeWarps][D];
    // the next kernel of the stream may start its set-up now: it waits for
    // this grid before it reads or writes what this grid touches
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // the lengths are the caller's (no kernel of this library writes them), so
    // they are read while the decode may still run; its partition states only
    // after griddepcontrol.wait
    const int row = blockIdx.x;   // s * n_q_heads + qh
    const int s = row / n_q_heads;
    const int L = min(max(__ldg(lens + s), 0), cap);
    const int np = L > 0 ? (L + part_tokens - 1) / part_tokens : 1;
    if (np <= 1) return;  // written directly by the partition kernel
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t row0 = size_t(row) * max_parts;
    const bool keep = np <= kMaxParts;
    // (m, l) of this thread's partitions, loaded once
    float M = -INFINITY;
    for (int k = threadIdx.x; k < np; k += blockDim.x) {
        const float mk = __ldcg(ws_m + row0 + k);
        if (keep) wgt[k] = mk;
        M = fmaxf(M, mk);
    }
    M = block_reduce<true>(M, red);
    float den = 0.f;
    for (int k = threadIdx.x; k < np; k += blockDim.x) {
        const float mk = keep ? wgt[k] : __ldcg(ws_m + row0 + k);
        const float w = fast_exp2((mk - M) * kLog2e);
        if (keep) wgt[k] = w;
        den = fmaf(w, __ldcg(ws_l + row0 + k), den);
    }
    den = block_reduce<false>(den, red);   // its barriers also publish wgt
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    for (int k0 = warp; k0 < np; k0 += kMergeWarps * kOBatch) {
        V x[kOBatch];
#pragma unroll
        for (int b = 0; b < kOBatch; ++b) {
            const int k = k0 + b * kMergeWarps;
            if (k < np) x[b] = __ldcg(reinterpret_cast<const V *>(ws_o + (row0 + k) * D) + lane);
        }
#pragma unroll
        for (int b = 0; b < kOBatch; ++b) {
            const int k = k0 + b * kMergeWarps;
            if (k < np) {
                const float w = keep ? wgt[k] : fast_exp2((__ldcg(ws_m + row0 + k) - M) * kLog2e);
                const float *xf = reinterpret_cast<const float *>(&x[b]);
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = fmaf(w, xf[e], acc[e]);
            }
        }
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
// Every load is issued before the first reduction, so a row costs about one
// round trip to L2 (where the partition states still sit).
template <typename T, int D>
__global__ void __launch_bounds__(256)
lse_merge_rows_kernel(const float *__restrict__ ws_o, const float *__restrict__ ws_m,
                      const float *__restrict__ ws_l, const int32_t *__restrict__ lens,
                      T *__restrict__ out, int rows, int n_q_heads, int part_tokens, int max_parts,
                      int cap) {
    constexpr int E = D / 32;
    constexpr int kBatch = 8;
    using V = typename Vec<E>::type;
    // the next kernel of the stream may start its set-up now: it waits for
    // this grid before it reads or writes what this grid touches
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    // the length first (the caller's, read while the decode may still run),
    // the partition states only after griddepcontrol.wait
    const int s = row / n_q_heads;
    const int L = min(max(__ldg(lens + s), 0), cap);
    const int np = L > 0 ? (L + part_tokens - 1) / part_tokens : 1;
    if (np <= 1) return;  // written directly by the partition kernel
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const size_t row0 = size_t(row) * max_parts;
    const float mp = lane < np ? __ldcg(ws_m + row0 + lane) : -INFINITY;
    const float lp = lane < np ? __ldcg(ws_l + row0 + lane) : 0.f;
    V x[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k)
        if (k < np) x[k] = __ldcg(reinterpret_cast<const V *>(ws_o + (row0 + k) * D) + lane);
    float M = mp;
#pragma unroll
    for (int mask = 16; mask >= 1; mask >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, mask));
    const float w = lane < np ? fast_exp2((mp - M) * kLog2e) : 0.f;
    float den = w * lp;
#pragma unroll
    for (int mask = 16; mask >= 1; mask >>= 1) den += __shfl_xor_sync(0xffffffffu, den, mask);
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    for (int k0 = 0; k0 < np; k0 += kBatch) {
        if (k0 > 0) {
#pragma unroll
            for (int k = 0; k < kBatch; ++k)
                if (k0 + k < np)
                    x[k] = __ldcg(reinterpret_cast<const V *>(ws_o + (row0 + k0 + k) * D) + lane);
        }
#pragma unroll
        for (int k = 0; k < kBatch; ++k) {
            const float wk = __shfl_sync(0xffffffffu, w, (k0 + k) & 31);
            if (k0 + k < np) {
                const float *xf = reinterpret_cast<const float *>(&x[k]);
#pragma unroll
                for (int e = 0; e < E; ++e) acc[e] = fmaf(wk, xf[e], acc[e]);
            }
        }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    float v[E];
#pragma unroll
    for (int e = 0; e < E; ++e) v[e] = acc[e] * inv;
    store_outputs<T, E>(out + size_t(row) * D + lane * E, v);
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

// Balanced split: one CTA per (sequence, head group). The CTA recomputes where
// the pair's tiles fall in the global tile list [sequence][head group][tile],
// which of the decode's equal tile shares they span and, if more than one,
// combines the pieces those CTAs left in their slots (slot 0 for a share's
// first unit, slot 1 for its last). Pairs inside one share were written by the
// decode directly; empty sequences get zero rows here.
template <typename T, int D>
__global__ void __launch_bounds__(32 * kMergeWarps)
lse_merge_pieces_kernel(const float *__restrict__ ws_o, const float *__restrict__ ws_m,
                        const float *__restrict__ ws_l, const int32_t *__restrict__ lens,
                        T *__restrict__ out, int num_seqs, int n_q_heads, int groups,
                        int rows_per_unit, int decode_grid, int cap) {
    constexpr int E = D / 32;
    constexpr int kBatch = 8;
    using V = typename Vec<E>::type;
    // the next kernel of the stream may start its set-up now: it waits for
    // this grid before it reads or writes what this grid touches
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int s = blockIdx.x / groups;
    const int hg = blockIdx.x - s * groups;
    const int warps = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Tiles before this sequence, and in total (exact integer sums). The
    // lengths are the caller's (no kernel of this library writes them), so
    // this runs while the decode may still be running; the pieces are read
    // only after griddepcontrol.wait.
    __shared__ unsigned long long sums[2];
    if (threadIdx.x == 0) sums[0] = sums[1] = 0ull;
    const int L = min(max(__ldg(lens + s), 0), cap);
    unsigned long long before_t = 0, total_t = 0;
    for (int t = threadIdx.x; t < num_seqs; t += blockDim.x) {
        const int Lt = min(max(__ldg(lens + t), 0), cap);
        const unsigned long long n = (unsigned long long)((Lt + kTile - 1) / kTile) * groups;
        total_t += n;
        if (t < s) before_t += n;
    }
    // warp sums first, then one shared-memory atomic per warp and sum
#pragma unroll
    for (int mask = 16; mask >= 1; mask >>= 1) {
        before_t += __shfl_xor_sync(0xffffffffu, before_t, mask);
        total_t += __shfl_xor_sync(0xffffffffu, total_t, mask);
    }
    __syncthreads();
    if ((threadIdx.x & 31) == 0) {
        atomicAdd(&sums[0], before_t);
        atomicAdd(&sums[1], total_t);
    }
    __syncthreads();
    const unsigned long long before = sums[0], total = sums[1];
    const int nt = (L + kTile - 1) / kTile;
    const int qh0 = hg * rows_per_unit;
    const long long Tt = (long long)total;
    const long long A = (long long)before + (long long)hg * nt;   // first tile of this pair
    const long long Z = A + nt - 1;                               // last tile
    auto share_start = [=](long long c) { return Tt * c / decode_grid; };
    auto share_of = [&](long long t) {
        long long c = t * decode_grid / Tt;
        while (c + 1 < decode_grid && share_start(c + 1) <= t) ++c;
        while (c > 0 && share_start(c) > t) --c;
        return c;
    };
    const long long c0 = nt > 0 ? share_of(A) : 0, c1 = nt > 0 ? share_of(Z) : 0;
    if (nt > 0 && c0 == c1) return;   // the decode wrote this pair's rows itself
    const int np = int(c1 - c0 + 1);
    const int slot0 = nt > 0 && A != share_start(c0) ? 1 : 0;
    // piece i of a row comes from share c0 + i: the first share's piece sits in
    // slot0, every later one in slot 0; shares with no tiles (fewer tiles than
    // CTAs) hold no piece and get weight 0
    auto piece = [=](int i, int r) {
        return (size_t(c0 + i) * 2 + (i == 0 ? slot0 : 0)) * rows_per_unit + r;
    };
    auto has_piece = [&](int i) {
        return i < np && share_start(c0 + i) != share_start(c0 + i + 1);
    };
    // everything so far follows from the lengths alone
    const bool has0 = nt > 0 && has_piece(lane);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (nt == 0) {
        for (int x = threadIdx.x; x < rows_per_unit * D; x += blockDim.x)
            out[(size_t(s) * n_q_heads + qh0) * D + x] = Elem<T>::from_float(0.f);
        return;
    }
    for (int r = warp; r < rows_per_unit; r += warps) {
        // one round trip: lane i's (m, l) of the first 32 pieces and the first
        // kBatch pieces' rows
        const float m0 = has0 ? __ldcg(ws_m + piece(lane, r)) : -INFINITY;
        const float l0 = has0 ? __ldcg(ws_l + piece(lane, r)) : 0.f;
        V x[kBatch];
#pragma unroll
        for (int k = 0; k < kBatch; ++k)
            if (k < np) x[k] = __ldcg(reinterpret_cast<const V *>(ws_o + piece(k, r) * D) + lane);
        float M = m0;
        for (int b = 32; b < np; b += 32)
            if (has_piece(b + lane)) M = fmaxf(M, __ldcg(ws_m + piece(b + lane, r)));
#pragma unroll
        for (int mask = 16; mask >= 1; mask >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, mask));
        float den = 0.f;
        float acc[E];
#pragma unroll
        for (int e = 0; e < E; ++e) acc[e] = 0.f;
        for (int b = 0; b < np; b += 32) {
            float mp = m0, lp = l0;
            bool has = has0;
            if (b > 0) {
                has = has_piece(b + lane);
                mp = has ? __ldcg(ws_m + piece(b + lane, r)) : -INFINITY;
                lp = has ? __ldcg(ws_l + piece(b + lane, r)) : 0.f;
            }
            const float w = has ? fast_exp2((mp - M) * kLog2e) : 0.f;
            den = fmaf(w, lp, den);
            const int n = min(32, np - b);
            for (int k0 = 0; k0 < n; k0 += kBatch) {
                if (b > 0 || k0 > 0) {
#pragma unroll
                    for (int k = 0; k < kBatch; ++k)
                        if (k0 + k < n)
                            x[k] = __ldcg(reinterpret_cast<const V *>(ws_o + piece(b + k0 + k, r) * D) +
                                          lane);
                }
#pragma unroll
                for (int k = 0; k < kBatch; ++k) {
                    const float wk = __shfl_sync(0xffffffffu, w, (k0 + k) & 31);
                    // a share without a piece may hold anything: skip it
                    if (k0 + k < n && wk != 0.f) {
                        const float *xf = reinterpret_cast<const float *>(&x[k]);
#pragma unroll
                        for (int e = 0; e < E; ++e) acc[e] = fmaf(wk, xf[e], acc[e]);
                    }
                }
            }
        }
#pragma unroll
        for (int mask = 16; mask >= 1; mask >>= 1) den += __shfl_xor_sync(0xffffffffu, den, mask);
        const float inv = den > 0.f ? 1.f / den : 0.f;
        float v[E];
#pragma unroll
        for (int e = 0; e < E; ++e) v[e] = acc[e] * inv;
        store_outputs<T, E>(out + (size_t(s) * n_q_heads + qh0 + r) * D + lane * E, v);
    }
}

template <typename T>
static cudaError_t launch_pieces_typed(int head_dim, const float *ws_o, const float *ws_m,
                                       const float *ws_l, const int32_t *lens, void *out, int S,
                                       int Hq, int groups, int rows_per_unit, int grid, int cap,
                                       cudaStream_t st) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(S * groups));
    // a warp per row of the pair (at most kMergeWarps warps, each then taking several)
    cfg.blockDim = dim3(32 * (rows_per_unit < kMergeWarps ? rows_per_unit : kMergeWarps));
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    T *o = static_cast<T *>(out);
    if (head_dim == 64)
        return cudaLaunchKernelEx(&cfg, lse_merge_pieces_kernel<T, 64>, ws_o, ws_m, ws_l, lens, o, S,
                                  Hq, groups, rows_per_unit, grid, cap);
    return cudaLaunchKernelEx(&cfg, lse_merge_pieces_kernel<T, 128>, ws_o, ws_m, ws_l, lens, o, S,
                              Hq, groups, rows_per_unit, grid, cap);
}

cudaError_t launch_piece_merge(int dtype, int head_dim, const float *ws_o, const float *ws_m,
                               const float *ws_l, const int32_t *context_lens, void *out,
                               int num_seqs, int n_q_heads, int groups, int rows_per_unit,
                               int decode_grid, int max_context, cudaStream_t stream) {
    if (num_seqs == 0) return cudaSuccess;
    switch (dtype) {
        case PAGEDKV_F32:
            return launch_pieces_typed<float>(head_dim, ws_o, ws_m, ws_l, context_lens, out,
                                              num_seqs, n_q_heads, groups, rows_per_unit,
                                              decode_grid, max_context, stream);
        case PAGEDKV_F16:
            return launch_pieces_typed<__half>(head_dim, ws_o, ws_m, ws_l, context_lens, out,
                                               num_seqs, n_q_heads, groups, rows_per_unit,
                                               decode_grid, max_context, stream);
        case PAGEDKV_BF16:
            return launch_pieces_typed<__nv_bfloat16>(head_dim, ws_o, ws_m, ws_l, context_lens,
                                                      out, num_seqs, n_q_heads, groups,
                                                      rows_per_unit, decode_grid, max_context,
                                                      stream);
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
