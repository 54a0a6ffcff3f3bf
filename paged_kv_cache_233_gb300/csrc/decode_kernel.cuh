// decode_kernel.cuh -- fused paged-attention decode for sm_103a.
//
// What it computes (page "Paged-KV + Continuous Batching From Scratch",
// section "What's deliberately still missing"): softmax attention of each
// sequence's query heads over that sequence's cached keys and values, with
// the cache read through the block table inside the kernel ("How a serving
// engine actually works", section "The one formula") instead of being
// gathered into a contiguous copy first ("Paged Attention and the Block
// Manager", section "The measurement").
//
// Work decomposition. A unit is (sequence s, kv head h, partition p): the
// tokens [p*P, min((p+1)*P, L_s)) of one kv head, for all g = n_q_heads /
// n_kv_heads query heads that read it (so each K/V byte is fetched once per kv
// head). Without split-K, P covers the whole context and p = 0. Units are
// numbered sequence-major and dealt round-robin to a persistent grid of CTAs.
//
// Inside a CTA (5 warps):
//   warp 0      producer. Its lanes hold a window of the block table row and
//               hand each block id to lane 0 by shuffle; lane 0 issues one TMA
//               tile load per 128-byte column slab of K and of V for every
//               16-token tile into a ring of shared-memory stages
//               (mbarrier transaction counts signal arrival).
//   warps 1..4  consumers. Tile i of a unit goes to consumer i mod 4; each
//               keeps an fp32 online-softmax state (running max m, running sum
//               l, accumulator o) per query head. At the end of a unit the four
//               states are combined through shared memory and written either
//               as the normalised output or as the unnormalised partition state
//               (split-K), which a merge kernel combines.
//
// Stage layout: for each of K and V, kSlabs column slabs of 16 rows x 128 B,
// written by TMA with the 128-byte swizzle (16-byte chunk c of row r lands at
// chunk c ^ (r & 7)), so that both row-wise vector loads and the 8x8 matrix
// loads of the tensor-core path are free of bank conflicts.
//
// Two consumer flavours:
//   SIMT  CUDA-core FMAs. Lanes own 16-byte column chunks of rows; per tile a
//         lane computes partial dot products for its rows and a butterfly
//         transpose-reduction turns them into full scores.
//   MMA   tensor cores (mma.sync m16n8k16, fp32 accumulate), for 16-bit types
//         when the query group is large enough to fill a tile: tokens are the
//         M dimension (a 16-token tile is exactly M = 16) and the query group
//         is N (8, padded): S^T = K Q^T, then O^T += V^T P^T with P^T moved
//         from accumulator layout to operand layout by movmatrix.
#pragma once

#include <type_traits>

#include "decode_params.h"
#include "ptx.cuh"

namespace pkv {

constexpr uint32_t kFull = 0xffffffffu;

template <typename T, int D>
struct StageGeometry {
    static constexpr int kRowBytes = D * int(sizeof(T));
    static constexpr int kSlabs = kRowBytes / 128;
    static constexpr int kHalf = kSlabs * kSlabBytes;  // K (or V) part of a stage
    static constexpr int kStageBytes = 2 * kHalf;
    static constexpr int kBoxElems = 128 / int(sizeof(T));
    static_assert(kRowBytes % 128 == 0, "rows must be whole 128-byte slabs");
};

// Shared-memory byte offset of 16-byte chunk `chunk` (0 .. kSlabs*8-1) of row `row`.
__device__ __forceinline__ uint32_t swz(int chunk, int row) {
    return uint32_t((chunk >> 3) * kSlabBytes + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

// Butterfly transpose-reduction: N partial sums per lane across the low
// log2(2*MASK) lane bits; afterwards lane i holds the full sum of value
// index (i >> (log2 lanes - log2 N)).
template <int N, int MASK>
__device__ __forceinline__ float transpose_reduce(float *v, int i) {
    if constexpr (MASK == 0) {
        return v[0];
    } else if constexpr (N > 1) {
        const bool up = (i & MASK) != 0;
#pragma unroll
        for (int a = 0; a < N / 2; ++a) {
            const float keep = up ? v[a + N / 2] : v[a];
            const float send = up ? v[a] : v[a + N / 2];
            v[a] = keep + __shfl_xor_sync(kFull, send, MASK);
        }
        return transpose_reduce<N / 2, MASK / 2>(v, i);
    } else {
        v[0] += __shfl_xor_sync(kFull, v[0], MASK);
        return transpose_reduce<1, MASK / 2>(v, i);
    }
}

// 16 bytes of a row -> floats
template <typename T>
__device__ __forceinline__ void unpack16(const uint4 &w, float *f) {
    if constexpr (sizeof(T) == 4) {
        f[0] = __uint_as_float(w.x);
        f[1] = __uint_as_float(w.y);
        f[2] = __uint_as_float(w.z);
        f[3] = __uint_as_float(w.w);
    } else {
        float2 a = Elem<T>::unpack2(w.x), b = Elem<T>::unpack2(w.y);
        float2 c = Elem<T>::unpack2(w.z), d = Elem<T>::unpack2(w.w);
        f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
        f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
    }
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(addr));
    return r;
}

__device__ __forceinline__ void sts128_zero(uint32_t addr) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0) : "memory");
}

// ---------------------------------------------------------------------------
// CUDA-core consumer
// ---------------------------------------------------------------------------
template <typename T, int D, int GM>
struct SimtConsumer {
    using G = StageGeometry<T, D>;
    static constexpr int LPR = G::kRowBytes / 16;       // lanes per row (8, 16 or 32)
    static constexpr int TPW = 32 / LPR;                // rows per warp-wide load
    static constexpr int NT = kTile / TPW;              // rows per lane per tile
    static constexpr int EPL = 16 / int(sizeof(T));     // elements per lane per row
    static constexpr int LOG_LPR = LPR == 8 ? 3 : (LPR == 16 ? 4 : 5);
    static constexpr int LOG_NT = NT == 4 ? 2 : (NT == 8 ? 3 : 4);
    static constexpr int DUP = LPR / NT;                // lanes sharing one reduced score

    float q[GM][EPL];
    float o[GM][EPL];
    float m[GM];
    float l[GM];
    int r;   // row group of this lane
    int i;   // 16-byte chunk of the row owned by this lane

    __device__ void init(int lane) {
        r = lane / LPR;
        i = lane % LPR;
    }

    __device__ void begin_unit(const T *qrow0, int g, float scale_log2) {
#pragma unroll
        for (int j = 0; j < GM; ++j) {
            m[j] = -INFINITY;
            l[j] = 0.f;
#pragma unroll
            for (int e = 0; e < EPL; ++e) o[j][e] = 0.f;
            if (j < g) {
                const uint4 w = __ldg(reinterpret_cast<const uint4 *>(qrow0 + j * D) + i);
                unpack16<T>(w, q[j]);
#pragma unroll
                for (int e = 0; e < EPL; ++e) q[j][e] *= scale_log2;
            } else {
#pragma unroll
                for (int e = 0; e < EPL; ++e) q[j][e] = 0.f;
            }
        }
    }

    __device__ void tile(uint32_t kaddr, uint32_t vaddr, int nvalid, int g) {
        float x[NT][EPL];
#pragma unroll
        for (int k = 0; k < NT; ++k) {
            const int t = k * TPW + r;
            unpack16<T>(lds128(kaddr + swz(i, t)), x[k]);
        }
        const int my_tok = (i >> (LOG_LPR - LOG_NT)) * TPW + r;
        float p[GM], alpha[GM];
#pragma unroll
        for (int j = 0; j < GM; ++j) {
            p[j] = 0.f;
            alpha[j] = 1.f;
            if (j < g) {
                float part[NT];
#pragma unroll
                for (int k = 0; k < NT; ++k) {
                    float acc = 0.f;
#pragma unroll
                    for (int e = 0; e < EPL; ++e) acc = fmaf(q[j][e], x[k][e], acc);
                    part[k] = acc;
                }
                float sc = transpose_reduce<NT, LPR / 2>(part, i);
                sc = my_tok < nvalid ? sc : -INFINITY;
                float mx = sc;
#pragma unroll
                for (int mask = 16; mask >= DUP; mask >>= 1)
                    mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, mask));
                const float m_new = fmaxf(m[j], mx);
                alpha[j] = fast_exp2(m[j] - m_new);
                p[j] = fast_exp2(sc - m_new);
                l[j] = l[j] * alpha[j] + ((i & (DUP - 1)) == 0 ? p[j] : 0.f);
                m[j] = m_new;
            }
        }
#pragma unroll
        for (int k = 0; k < NT; ++k) {
            const int t = k * TPW + r;
            unpack16<T>(lds128(vaddr + swz(i, t)), x[k]);
            if (t >= nvalid) {
#pragma unroll
                for (int e = 0; e < EPL; ++e) x[k][e] = 0.f;
            }
        }
#pragma unroll
        for (int j = 0; j < GM; ++j) {
            if (j < g) {
#pragma unroll
                for (int e = 0; e < EPL; ++e) o[j][e] *= alpha[j];
#pragma unroll
                for (int k = 0; k < NT; ++k) {
                    const float pk = __shfl_sync(kFull, p[j], r * LPR + (k << (LOG_LPR - LOG_NT)));
#pragma unroll
                    for (int e = 0; e < EPL; ++e) o[j][e] = fmaf(pk, x[k][e], o[j][e]);
                }
            }
        }
    }

    // Fold the lane-distributed state into the merge buffer row of this warp.
    __device__ void end_unit(float *mo, float *mm, float *ml, int g, int lane, int stride) {
#pragma unroll
        for (int j = 0; j < GM; ++j) {
            if (j < g) {
#pragma unroll
                for (int mask = LPR; mask < 32; mask <<= 1)
#pragma unroll
                    for (int e = 0; e < EPL; ++e)
                        o[j][e] += __shfl_xor_sync(kFull, o[j][e], mask);
                float lj = l[j];
#pragma unroll
                for (int mask = 16; mask >= 1; mask >>= 1) lj += __shfl_xor_sync(kFull, lj, mask);
                if (r == 0) {
#pragma unroll
                    for (int e = 0; e < EPL; ++e) mo[j * stride + i * EPL + e] = o[j][e];
                }
                if (lane == 0) {
                    mm[j] = m[j];
                    ml[j] = lj;
                }
            }
        }
    }
};

// ---------------------------------------------------------------------------
// Tensor-core consumer (16-bit types, query group <= 8)
// ---------------------------------------------------------------------------
template <typename T, int D>
struct MmaConsumer {
    static constexpr int KS = D / 16;   // k-steps of S^T = K Q^T
    static constexpr int MT = D / 16;   // m-tiles of O^T = V^T P^T
    static constexpr bool kBf16 = Elem<T>::kBf16;

    uint32_t qb[KS][2];
    float o[MT][4];
    float m[2];     // running max (base 2) of heads 2c, 2c+1
    float lp[2];    // this lane's part of the running sums
    int grp, c;     // lane / 4, lane % 4
    int mi, r8;     // which 8x8 matrix this lane addresses in ldmatrix.x4, and its row

    __device__ void init(int lane) {
        grp = lane >> 2;
        c = lane & 3;
        mi = lane >> 3;
        r8 = lane & 7;
    }

    __device__ void begin_unit(const T *qrow0, int g) {
        m[0] = m[1] = -INFINITY;
        lp[0] = lp[1] = 0.f;
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[t][e] = 0.f;
        const bool live = grp < g;
        const uint32_t *row = reinterpret_cast<const uint32_t *>(qrow0 + grp * D);
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            qb[kk][0] = live ? __ldg(row + kk * 8 + c) : 0u;
            qb[kk][1] = live ? __ldg(row + kk * 8 + 4 + c) : 0u;
        }
    }

    __device__ void tile(uint32_t kaddr, uint32_t vaddr, int nvalid, float scale_log2) {
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const int tok = r8 + ((mi & 1) << 3);
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                uint32_t a[4];
                ldmatrix_x4(kaddr + swz(2 * kk + (mi >> 1), tok), a);
                mma_m16n8k16<kBf16>(s, a, qb[kk][0], qb[kk][1]);
            }
        }
        // s: [0] (token grp, head 2c) [1] (grp, 2c+1) [2] (grp+8, 2c) [3] (grp+8, 2c+1)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[e] *= scale_log2;
        if (grp >= nvalid) s[0] = s[1] = -INFINITY;
        if (grp + 8 >= nvalid) s[2] = s[3] = -INFINITY;
        float mx0 = fmaxf(s[0], s[2]), mx1 = fmaxf(s[1], s[3]);
#pragma unroll
        for (int mask = 4; mask <= 16; mask <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, mask));
            mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, mask));
        }
        const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
        const float a0 = fast_exp2(m[0] - mn0), a1 = fast_exp2(m[1] - mn1);
        const float p0 = fast_exp2(s[0] - mn0), p1 = fast_exp2(s[1] - mn1);
        const float p2 = fast_exp2(s[2] - mn0), p3 = fast_exp2(s[3] - mn1);
        lp[0] = lp[0] * a0 + (p0 + p2);
        lp[1] = lp[1] * a1 + (p1 + p3);
        m[0] = mn0;
        m[1] = mn1;
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            o[t][0] *= a0;
            o[t][1] *= a1;
            o[t][2] *= a0;
            o[t][3] *= a1;
        }
        const uint32_t b0 = movmatrix_trans(Elem<T>::pack2(p0, p1));
        const uint32_t b1 = movmatrix_trans(Elem<T>::pack2(p2, p3));
        const int tok = r8 + ((mi >> 1) << 3);
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            uint32_t a[4];
            ldmatrix_x4_trans(vaddr + swz(2 * t + (mi & 1), tok), a);
            mma_m16n8k16<kBf16>(o[t], a, b0, b1);
        }
    }

    __device__ void end_unit(float *mo, float *mm, float *ml, int g, int stride) {
        float l0 = lp[0], l1 = lp[1];
#pragma unroll
        for (int mask = 4; mask <= 16; mask <<= 1) {
            l0 += __shfl_xor_sync(kFull, l0, mask);
            l1 += __shfl_xor_sync(kFull, l1, mask);
        }
        const int h0 = 2 * c, h1 = 2 * c + 1;
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            const int d = t * 16 + grp;
            if (h0 < g) {
                mo[h0 * stride + d] = o[t][0];
                mo[h0 * stride + d + 8] = o[t][2];
            }
            if (h1 < g) {
                mo[h1 * stride + d] = o[t][1];
                mo[h1 * stride + d + 8] = o[t][3];
            }
        }
        if (grp == 0) {
            if (h0 < g) { mm[h0] = m[0]; ml[h0] = l0; }
            if (h1 < g) { mm[h1] = m[1]; ml[h1] = l1; }
        }
    }
};

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <typename T, int D, int GM, bool kMma>
__global__ void __launch_bounds__(kDecodeThreads, 2)
paged_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
    using G = StageGeometry<T, D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const sm = smem_raw + (base - raw);
    const int NS = 1 << p.log2_stages;
    const int S = p.num_seqs;
    DecodeSmem lay{G::kStageBytes, NS, S, D, GM};
    const uint32_t full0 = base + lay.bars();
    const uint32_t empty0 = full0 + 8 * NS;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + lay.flag());
    int *seq_base = reinterpret_cast<int *>(sm + lay.seq_base());
    int *seq_len = reinterpret_cast<int *>(sm + lay.seq_len());
    float *merge_o = reinterpret_cast<float *>(sm + lay.merge_o());
    float *merge_m = reinterpret_cast<float *>(sm + lay.merge_m());
    float *merge_l = reinterpret_cast<float *>(sm + lay.merge_l());
    const int stride = lay.row_stride();

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int B = p.block_size;
    const int Hkv = p.n_kv_heads;
    const int P = p.part_tokens;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_descriptor(&kmap);
            tma_prefetch_descriptor(&vmap);
        }
        // units of each sequence: max(1, ceil(L / P)) partitions x n_kv_heads, prefix-summed
        const int cap = p.max_blocks * B;
        int carry = 0;
        if (lane == 0) seq_base[0] = 0;
        for (int s0 = 0; s0 < S; s0 += 32) {
            const int s = s0 + lane;
            int cnt = 0;
            if (s < S) {
                const int L = p.context_lens[s];
                const int Lc = min(max(L, 0), cap);
                if (Lc != L) atomicOr(p.err, PAGEDKV_DEVERR_CONTEXT_LEN);
                seq_len[s] = Lc;
                cnt = (Lc > 0 ? (Lc + P - 1) / P : 1) * Hkv;
            }
            int x = cnt;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(kFull, x, off);
                if (lane >= off) x += y;
            }
            if (s < S) seq_base[s + 1] = carry + x;
            carry += __shfl_sync(kFull, x, 31);
        }
    }
    __syncthreads();
    const int total_units = seq_base[S];

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        uint32_t gt = 0;      // tiles armed so far by this CTA
        bool ok = true;
        int s = 0;
        for (int u = blockIdx.x; u < total_units && ok; u += gridDim.x) {
            while (seq_base[s + 1] <= u) ++s;
            const int rr = u - seq_base[s];
            const int part = rr / Hkv;
            const int h = rr - part * Hkv;
            const int L = seq_len[s];
            const int t0 = part * P;
            const int t1 = min(L, t0 + P);
            const int ntiles = (t1 - t0 + kTile - 1) / kTile;
            const int nblk = (L + B - 1) >> p.log2_block;    // blocks this sequence holds
            const int32_t *bt_row = p.block_tables + size_t(s) * p.max_blocks;
            int win_base = -64, win_val = -1;
            for (int i = 0; i < ntiles; ++i) {
                const int tok = t0 + i * kTile;
                const int j0 = tok >> p.log2_block;
                const bool two = (B < kTile) && (tok + B < t1);
                if (j0 < win_base || j0 + 1 >= win_base + 32) {
                    win_base = j0;
                    const int j = j0 + lane;
                    win_val = j < nblk ? __ldg(bt_row + j) : -1;
                }
                int pb0 = __shfl_sync(kFull, win_val, j0 - win_base);
                int pb1 = __shfl_sync(kFull, win_val, (j0 + 1 - win_base) & 31);
                if (lane == 0) {
                    const uint32_t stage = gt & uint32_t(NS - 1);
                    const uint32_t parity = ((gt >> p.log2_stages) & 1u) ^ 1u;
                    if (*abort_flag || !mbar_wait(empty0 + 8 * stage, parity, p.err)) {
                        ok = false;
                    } else {
                        if (pb0 < 0 || pb0 >= p.num_blocks) {
                            atomicOr(p.err, PAGEDKV_DEVERR_BLOCK_ID);
                            pb0 = 0;
                        }
                        if (two && (pb1 < 0 || pb1 >= p.num_blocks)) {
                            atomicOr(p.err, PAGEDKV_DEVERR_BLOCK_ID);
                            pb1 = 0;
                        }
                        const uint32_t box = B >= kTile ? kSlabBytes : kSlabBytes / 2;
                        const uint32_t bytes = 2u * G::kSlabs * (two ? 2u * box : box);
                        const uint32_t fb = full0 + 8 * stage;
                        mbar_arrive_expect_tx(fb, bytes);
                        const uint32_t kdst = base + stage * G::kStageBytes;
                        const uint32_t vdst = kdst + G::kHalf;
                        const int z0 = pb0 * B + (tok & (B - 1));
#pragma unroll
                        for (int sl = 0; sl < G::kSlabs; ++sl) {
                            tma_load_3d(kdst + sl * kSlabBytes, &kmap, sl * G::kBoxElems, h, z0, fb);
                            tma_load_3d(vdst + sl * kSlabBytes, &vmap, sl * G::kBoxElems, h, z0, fb);
                        }
                        if (two) {
                            const int z1 = pb1 * B;
#pragma unroll
                            for (int sl = 0; sl < G::kSlabs; ++sl) {
                                tma_load_3d(kdst + sl * kSlabBytes + box, &kmap, sl * G::kBoxElems, h, z1, fb);
                                tma_load_3d(vdst + sl * kSlabBytes + box, &vmap, sl * G::kBoxElems, h, z1, fb);
                            }
                        }
                        ++gt;
                    }
                }
                ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
            }
        }
        if (!ok && lane == 0) {
            // Stop everyone, then wait (bounded) for this CTA's copies still in flight.
            *abort_flag = 1;
            const uint32_t first = gt > uint32_t(NS) ? gt - NS : 0u;
            for (uint32_t k = first; k < gt; ++k)
                mbar_wait(full0 + 8 * (k & uint32_t(NS - 1)), (k >> p.log2_stages) & 1u, p.err);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int cw = warp - 1;
    const int g = p.group;
    const int tid_c = threadIdx.x - 32;
    constexpr int kConsumerThreads = 32 * kConsumerWarps;
    using Simt = SimtConsumer<T, D, GM>;
    using Mma = MmaConsumer<T, D>;
    typename std::conditional<kMma, Mma, Simt>::type st;
    st.init(lane);
    float *my_o = merge_o + cw * GM * stride;
    float *my_m = merge_m + cw * GM;
    float *my_l = merge_l + cw * GM;

    uint32_t gt_base = 0;
    int s = 0;
    for (int u = blockIdx.x; u < total_units; u += gridDim.x) {
        while (seq_base[s + 1] <= u) ++s;
        const int rr = u - seq_base[s];
        const int part = rr / Hkv;
        const int h = rr - part * Hkv;
        const int L = seq_len[s];
        const int t0 = part * P;
        const int t1 = min(L, t0 + P);
        const int ntiles = (t1 - t0 + kTile - 1) / kTile;
        const int nparts = L > 0 ? (L + P - 1) / P : 1;
        const T *qrow0 = reinterpret_cast<const T *>(p.q) + (size_t(s) * p.n_q_heads + h * g) * D;
        if constexpr (kMma) st.begin_unit(qrow0, g);
        else st.begin_unit(qrow0, g, p.scale_log2);

        for (int i = cw; i < ntiles; i += kConsumerWarps) {
            const uint32_t gt = gt_base + uint32_t(i);
            const uint32_t stage = gt & uint32_t(NS - 1);
            int good = !*abort_flag;
            if (good) good = mbar_wait(full0 + 8 * stage, (gt >> p.log2_stages) & 1u, p.err);
            if (!__all_sync(kFull, good)) {
                *abort_flag = 1;
                continue;
            }
            const int nvalid = min(kTile, t1 - (t0 + i * kTile));
            const uint32_t kaddr = base + stage * G::kStageBytes;
            const uint32_t vaddr = kaddr + G::kHalf;
            if constexpr (kMma) {
                if (nvalid < kTile) {
                    // rows past the context may hold anything (even NaN): zero the V rows
                    const int n16 = (kTile - nvalid) * G::kSlabs * 8;
                    for (int x = lane; x < n16; x += 32) {
                        const int row = nvalid + x / (G::kSlabs * 8);
                        const int rem = x % (G::kSlabs * 8);
                        sts128_zero(vaddr + (rem >> 3) * kSlabBytes + row * 128 + (rem & 7) * 16);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                st.tile(kaddr, vaddr, nvalid, p.scale_log2);
            } else {
                st.tile(kaddr, vaddr, nvalid, g);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * stage);
        }
        gt_base += uint32_t(ntiles);

        // ---- combine the four consumer states of this unit
        if constexpr (kMma) st.end_unit(my_o, my_m, my_l, g, stride);
        else st.end_unit(my_o, my_m, my_l, g, lane, stride);
        named_barrier(1, kConsumerThreads);
        const bool write_partial = p.split && nparts > 1;
        for (int idx = tid_c; idx < g * D; idx += kConsumerThreads) {
            const int j = idx / D;
            const int d = idx - j * D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, merge_m[w * GM + j]);
            float num = 0.f, den = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < kConsumerWarps; ++w) {
                    const float f = fast_exp2(merge_m[w * GM + j] - M);
                    num = fmaf(f, merge_o[(w * GM + j) * stride + d], num);
                    den = fmaf(f, merge_l[w * GM + j], den);
                }
            }
            const int qh = h * g + j;
            if (write_partial) {
                const size_t row = (size_t(s) * p.n_q_heads + qh) * p.max_parts + part;
                p.ws_o[row * D + d] = num;
                if (d == 0) {
                    p.ws_m[row] = M * kLn2;
                    p.ws_l[row] = den;
                }
            } else {
                const float v = den > 0.f ? num / den : 0.f;
                reinterpret_cast<T *>(p.out)[(size_t(s) * p.n_q_heads + qh) * D + d] =
                    Elem<T>::from_float(v);
            }
        }
        named_barrier(1, kConsumerThreads);
    }
}

}  // namespace pkv
