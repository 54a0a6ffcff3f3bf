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
// Work decomposition. A unit is (sequence s, group of H kv heads, partition
// p): tokens [p*P, min((p+1)*P, L_s)) of H consecutive kv heads, for all the
// query heads that read them (each K/V byte is fetched once per kv head).
// H is 4 when n_kv_heads allows, else 2 or 1. Without split-K, P covers the
// whole context and p = 0. Units are numbered sequence-major and dealt
// round-robin to a persistent grid of CTAs.
//
// Inside a CTA (5 warps):
//   warp 0      producer. Its lanes hold a window of the block table row and
//               hand each block id to lane 0 by shuffle; lane 0 issues, per
//               16-token tile, one 4-D TMA load of K and one of V covering all
//               H heads and all 128-byte column slabs of those tokens, into a
//               ring of shared-memory stages (mbarrier transaction counts
//               signal arrival; all four consumers release a stage). The ring
//               holds params.stages stages; every CTA uses stages_alt of them
//               instead when the call's mean context is long. When the call
//               streams more K/V than the L2 holds, each load carries an L2
//               priority: evict_last for blocks a neighbouring sequence
//               shares, evict_first for the rest.
//   warps 1..4  consumers. Warp w owns kv head (w mod H) of the unit and, when
//               H < 4, every (4/H)-th tile of it. Each keeps an fp32
//               online-softmax state (running max m, running sum l,
//               accumulator o) per query head of its kv head and writes its
//               result straight to the output (or, under split-K, its
//               unnormalised partition state to the workspace). Only when
//               H < 4 do warps sharing a head combine states through shared
//               memory at the end of a unit. Every consumer waits on every
//               stage in ring order, so a stage's parity is never ambiguous.
//
// Stage layout, for each of K and V: [head][slab][16 rows][128 B], written by
// TMA with the 128-byte swizzle (16-byte chunk c of row r lands at chunk
// c ^ (r & 7)), so row-wise vector loads and the 8x8 matrix loads of the
// tensor-core path are both free of bank conflicts. With 8-token blocks a
// tile is two blocks, each brought by one box per operand:
// [block][head][slab][8 rows][128 B].
//
// Two consumer flavours:
//   SIMT  CUDA-core FMAs. Lanes own 16-byte column chunks of rows; per tile a
//         lane computes partial dot products for its rows and a butterfly
//         transpose-reduction turns them into full scores.
//   MMA   tensor cores (mma.sync m16n8k16, fp32 accumulate), for 16-bit types
//         at any query-group size: tokens are the M dimension (a 16-token
//         tile is exactly M = 16) and the query group is N (8, padded with
//         zero columns): S^T = K Q^T, then O^T += V^T P^T with P^T moved from
//         accumulator layout to operand layout by movmatrix.
#pragma once

#include <type_traits>

#include "decode_params.h"
#include "ptx.cuh"

namespace pkv {

constexpr uint32_t kFull = 0xffffffffu;

template <typename T, int D>
struct StageGeometry {
    static constexpr int kRowBytes = D * int(sizeof(T));
    static constexpr int kSlabs = kRowBytes / kRowBytes128;
    static constexpr int kSlabBytes = kTile * kRowBytes128;   // 16 rows of one slab, one head
    static constexpr int kHeadBytes = kSlabs * kSlabBytes;    // all slabs of one head
    static_assert(kRowBytes % kRowBytes128 == 0, "rows must be whole 128-byte slabs");
};

// Shared-memory byte offset, within one head's part of a stage, of 16-byte
// chunk `chunk` (0 .. slabs*8-1) of token row `row` (0 .. 15). Rows 0-7 and
// rows 8-15 of a slab are each one 1024-byte swizzle atom: `hi` bytes apart
// (1024 when one box brings 16 rows; the size of one block's box when 8-token
// blocks arrive as two boxes, each every slab of every head of the unit),
// with `slab` bytes between slabs.
struct TileAddr {
    uint32_t slab, hi;
    __device__ __forceinline__ uint32_t operator()(int chunk, int row) const {
        return uint32_t((chunk >> 3) * slab + (row >> 3) * hi + (row & 7) * kRowBytes128 +
                        (((chunk & 7) ^ (row & 7)) << 4));
    }
};

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

// floats -> 16 bytes of elements
template <typename T>
__device__ __forceinline__ uint4 pack16(const float *f) {
    uint4 w;
    if constexpr (sizeof(T) == 4) {
        w.x = __float_as_uint(f[0]);
        w.y = __float_as_uint(f[1]);
        w.z = __float_as_uint(f[2]);
        w.w = __float_as_uint(f[3]);
    } else {
        w.x = Elem<T>::pack2(f[0], f[1]);
        w.y = Elem<T>::pack2(f[2], f[3]);
        w.z = Elem<T>::pack2(f[4], f[5]);
        w.w = Elem<T>::pack2(f[6], f[7]);
    }
    return w;
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

// Where a unit's result goes: the output rows (normalised) or, under split-K,
// the partition-state rows of the workspace.
struct UnitSink {
    bool partial;
    size_t out_row0;   // row (s * n_q_heads + qh0) of out, qh0 = this warp's first q head
    size_t ws_row0;    // workspace row of q head qh0 of this unit's state
    int j_stride;      // rows between consecutive q heads of the group
};

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
    uint4 qn[GM];   // next unit's query rows, prefetched
    int r;          // row group of this lane
    int i;          // 16-byte chunk of the row owned by this lane

    __device__ void init(int lane) {
        r = lane / LPR;
        i = lane % LPR;
    }

    // q rows of q heads qh0 .. qh0+g-1 of sequence s0 (one sequence per unit on this path)
    __device__ void prefetch_q(const T *qbase, size_t s0, int qh0, int g, int, int Hq) {
        const T *qrow0 = qbase + (s0 * Hq + qh0) * D;
#pragma unroll
        for (int j = 0; j < GM; ++j)
            qn[j] = j < g ? __ldg(reinterpret_cast<const uint4 *>(qrow0 + j * D) + i)
                          : make_uint4(0, 0, 0, 0);
    }

    __device__ void begin_unit(float scale_log2) {
#pragma unroll
        for (int j = 0; j < GM; ++j) {
            m[j] = -INFINITY;
            l[j] = 0.f;
            unpack16<T>(qn[j], q[j]);
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                o[j][e] = 0.f;
                q[j][e] *= scale_log2;
            }
        }
    }

    __device__ void tile(uint32_t kaddr, uint32_t vaddr, int nvalid, int g, TileAddr ta) {
        float x[NT][EPL];
#pragma unroll
        for (int k = 0; k < NT; ++k) {
            const int t = k * TPW + r;
            unpack16<T>(lds128(kaddr + ta(i, t)), x[k]);
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
            unpack16<T>(lds128(vaddr + ta(i, t)), x[k]);
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

    // Sum the lane-distributed state: afterwards lanes of row group 0 hold o
    // and every lane holds the full l.
    __device__ void reduce(int g) {
#pragma unroll
        for (int j = 0; j < GM; ++j) {
            if (j < g) {
#pragma unroll
                for (int mask = LPR; mask < 32; mask <<= 1)
#pragma unroll
                    for (int e = 0; e < EPL; ++e)
                        o[j][e] += __shfl_xor_sync(kFull, o[j][e], mask);
#pragma unroll
                for (int mask = 16; mask >= 1; mask >>= 1)
                    l[j] += __shfl_xor_sync(kFull, l[j], mask);
            }
        }
    }

    // Write the whole result of this warp's kv head (after reduce()).
    __device__ void store(const UnitSink &sink, T *out, float *ws_o, float *ws_m, float *ws_l,
                          int g, int lane) {
#pragma unroll
        for (int j = 0; j < GM; ++j) {
            if (j < g) {
                if (sink.partial) {
                    const size_t row = sink.ws_row0 + size_t(j) * sink.j_stride;
                    if (r == 0) {
                        float *dst = ws_o + row * D + i * EPL;
#pragma unroll
                        for (int e = 0; e < EPL; e += 4)
                            *reinterpret_cast<float4 *>(dst + e) =
                                make_float4(o[j][e], o[j][e + 1], o[j][e + 2], o[j][e + 3]);
                    }
                    if (lane == 0) {
                        ws_m[row] = m[j] * kLn2;
                        ws_l[row] = l[j];
                    }
                } else if (r == 0) {
                    const float inv = l[j] > 0.f ? 1.f / l[j] : 0.f;
                    float v[EPL];
#pragma unroll
                    for (int e = 0; e < EPL; ++e) v[e] = o[j][e] * inv;
                    *reinterpret_cast<uint4 *>(out + (sink.out_row0 + j) * D + i * EPL) = pack16<T>(v);
                }
            }
        }
    }

    // Stage this warp's state for a cross-warp merge (after reduce()).
    __device__ void stash(float *mo, float *mm, float *ml, int g, int lane, int stride) {
#pragma unroll
        for (int j = 0; j < GM; ++j) {
            if (j < g) {
                if (r == 0) {
#pragma unroll
                    for (int e = 0; e < EPL; ++e) mo[j * stride + i * EPL + e] = o[j][e];
                }
                if (lane == 0) {
                    mm[j] = m[j];
                    ml[j] = l[j];
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
    using G = StageGeometry<T, D>;
    static constexpr int KS = D / 16;   // k-steps of S^T = K Q^T
    static constexpr int MT = D / 16;   // m-tiles of O^T = V^T P^T
    static constexpr bool kBf16 = Elem<T>::kBf16;

    uint32_t qb[KS][2];
    uint32_t qn[KS][2];   // next unit's fragments, prefetched
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

    // Column n of the tile is query head qh0 + n % g of sequence s0 + n / g, for
    // n < members * g (members > 1 only for units of a shared prefix).
    __device__ void prefetch_q(const T *qbase, size_t s0, int qh0, int g, int members, int Hq) {
        const int m = grp / g;
        const bool live = grp < members * g;
        const uint32_t *row = reinterpret_cast<const uint32_t *>(
            qbase + ((s0 + m) * Hq + qh0 + (grp - m * g)) * D);
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            qn[kk][0] = live ? __ldg(row + kk * 8 + c) : 0u;
            qn[kk][1] = live ? __ldg(row + kk * 8 + 4 + c) : 0u;
        }
    }

    __device__ void begin_unit() {
        m[0] = m[1] = -INFINITY;
        lp[0] = lp[1] = 0.f;
#pragma unroll
        for (int t = 0; t < MT; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[t][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            qb[kk][0] = qn[kk][0];
            qb[kk][1] = qn[kk][1];
        }
    }

    __device__ void tile(uint32_t kaddr, uint32_t vaddr, int nvalid, float scale_log2,
                         TileAddr ta) {
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const int tok = r8 + ((mi & 1) << 3);
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
                uint32_t a[4];
                ldmatrix_x4(kaddr + ta(2 * kk + (mi >> 1), tok), a);
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
            ldmatrix_x4_trans(vaddr + ta(2 * t + (mi & 1), tok), a);
            mma_m16n8k16<kBf16>(o[t], a, b0, b1);
        }
    }

    // Full row sums of this lane's two heads (lanes with the same c agree).
    __device__ void reduce() {
#pragma unroll
        for (int mask = 4; mask <= 16; mask <<= 1) {
            lp[0] += __shfl_xor_sync(kFull, lp[0], mask);
            lp[1] += __shfl_xor_sync(kFull, lp[1], mask);
        }
    }

    __device__ void store(const UnitSink &sink, T *out, float *ws_o, float *ws_m, float *ws_l,
                          int g) {
#pragma unroll
        for (int hsel = 0; hsel < 2; ++hsel) {
            const int h = 2 * c + hsel;
            if (h >= g) continue;
            if (sink.partial) {
                const size_t row = sink.ws_row0 + size_t(h) * sink.j_stride;
                float *dst = ws_o + row * D;
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    dst[t * 16 + grp] = o[t][hsel];
                    dst[t * 16 + grp + 8] = o[t][2 + hsel];
                }
                if (grp == 0) {
                    ws_m[row] = m[hsel] * kLn2;
                    ws_l[row] = lp[hsel];
                }
            } else {
                const float inv = lp[hsel] > 0.f ? 1.f / lp[hsel] : 0.f;
                T *dst = out + (sink.out_row0 + h) * D;
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    dst[t * 16 + grp] = Elem<T>::from_float(o[t][hsel] * inv);
                    dst[t * 16 + grp + 8] = Elem<T>::from_float(o[t][2 + hsel] * inv);
                }
            }
        }
    }

    // Results of a shared-prefix unit: column n belongs to sequence s0 + n / g;
    // its state is partial unless that sequence fits in one partition.
    __device__ void store_members(T *out, float *ws_o, float *ws_m, float *ws_l, const int *seq_len,
                                  size_t s0, int members, int qh0, int g, int Hq, int P, int part,
                                  int max_parts) {
#pragma unroll
        for (int hsel = 0; hsel < 2; ++hsel) {
            const int h = 2 * c + hsel;
            if (h >= members * g) continue;
            const int mem = h / g;
            const size_t sm = s0 + mem;
            const int qh = qh0 + h - mem * g;
            if (seq_len[sm] > P) {
                const size_t row = (sm * Hq + qh) * max_parts + part;
                float *dst = ws_o + row * D;
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    dst[t * 16 + grp] = o[t][hsel];
                    dst[t * 16 + grp + 8] = o[t][2 + hsel];
                }
                if (grp == 0) {
                    ws_m[row] = m[hsel] * kLn2;
                    ws_l[row] = lp[hsel];
                }
            } else {
                const float inv = lp[hsel] > 0.f ? 1.f / lp[hsel] : 0.f;
                T *dst = out + (sm * Hq + qh) * D;
#pragma unroll
                for (int t = 0; t < MT; ++t) {
                    dst[t * 16 + grp] = Elem<T>::from_float(o[t][hsel] * inv);
                    dst[t * 16 + grp + 8] = Elem<T>::from_float(o[t][2 + hsel] * inv);
                }
            }
        }
    }

    __device__ void stash(float *mo, float *mm, float *ml, int g, int stride) {
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
            if (h0 < g) { mm[h0] = m[0]; ml[h0] = lp[0]; }
            if (h1 < g) { mm[h1] = m[1]; ml[h1] = lp[1]; }
        }
    }
};

// ---------------------------------------------------------------------------
// Unit walk shared by the producer and the consumers
// ---------------------------------------------------------------------------
struct Unit {
    int s, hg, L, t0, t1, ntiles;
    int part;       // fixed partitions: partition index within the sequence
    bool partial;   // the result is a partition state, not the final row
    int slot;       // balanced split: which of this CTA's two piece slots
    int members;    // sequences s .. s+members-1 whose queries the unit serves (shared prefix)
};

// This CTA's units, in order (producer and consumers walk identical copies).
//  Fixed mode: units blockIdx.x + k * gridDim.x of the sequence-major list
//    [sequence][partition][head group]; a unit is partial when split-K is on
//    and its sequence has more than one partition.
//  Balanced mode: the CTA's equal, contiguous share of the global list of
//    16-token tiles [sequence][head group][tile]; a unit is the part of one
//    (sequence, head group) inside that share, partial unless it is the whole
//    sequence. Only a share's first and last units can be partial; they go to
//    piece slots 0 and 1 of the CTA.
struct Walk {
    const int *seq_base;   // per-sequence prefix sums of units (fixed) or tiles (balanced)
    const int *seq_len;
    const int *seq_p0;     // shared prefixes: first partition a sequence reads itself
    const int *seq_pu;     // shared prefixes: prefix units the sequence leads
    const int32_t *seq_group;
    int S, max_members;
    int groups, P, split, balanced;
    int s, pos, end, stride, count;

    __device__ void init(const int *base, const int *len, int S_, int groups_, int P_, int split_,
                         int balanced_, const int *p0 = nullptr, const int *pu = nullptr,
                         const int32_t *group = nullptr, int max_members_ = 1) {
        seq_base = base;
        seq_len = len;
        seq_p0 = p0;
        seq_pu = pu;
        seq_group = group;
        S = S_;
        max_members = max_members_;
        groups = groups_;
        P = P_;
        split = split_;
        balanced = balanced_;
        s = 0;
        count = 0;
        const long long total = base[S_];
        if (balanced) {
            pos = int(total * blockIdx.x / gridDim.x);
            end = int(total * (blockIdx.x + 1) / gridDim.x);
            stride = 0;
        } else {
            pos = blockIdx.x;
            end = int(total);
            stride = gridDim.x;
        }
    }

    __device__ bool has_work() const { return pos < end; }

    // Called by all 32 lanes of a warp together (the producer warp and each
    // consumer warp walk their own copy). The sequence of the next unit is
    // found 32 candidates at a time: lane i tests whether sequence s + i ends
    // past `pos`, and the first such lane is it. Units are dealt with a stride
    // of the grid size, so the next unit is often dozens of sequences on
    // (about 30 with 256 sequences of 9 units each): one or two rounds of
    // shared-memory loads instead of one dependent load per sequence.
    __device__ bool next(Unit &x) {
        if (pos >= end) return false;
        const int lane = threadIdx.x & 31;
        for (;;) {
            const int c = s + 1 + lane;
            const bool past = c > S || seq_base[c] > pos;
            const unsigned m = __ballot_sync(kFull, past);
            if (m) {
                s += __ffs(m) - 1;
                break;
            }
            s += 32;
        }
        x.s = s;
        x.L = seq_len[s];
        const int rr = pos - seq_base[s];
        if (balanced) {
            const int nt = (x.L + kTile - 1) / kTile;     // tiles per head group (> 0 here)
            x.hg = rr / nt;
            const int tf = rr - x.hg * nt;
            const int tl = min(nt, tf + (end - pos));
            x.part = 0;
            x.t0 = tf * kTile;
            x.t1 = min(x.L, tl * kTile);
            x.ntiles = tl - tf;
            x.partial = !(tf == 0 && tl == nt);
            x.slot = count == 0 ? 0 : 1;
            x.members = 1;
            pos += tl - tf;
        } else {
            const int pu = seq_pu ? seq_pu[s] : 0;
            x.slot = 0;
            if (rr < pu) {
                // a partition of a shared prefix, for up to max_members sequences of the group
                x.part = rr / groups;
                x.hg = rr - x.part * groups;
                x.t0 = x.part * P;
                x.t1 = x.t0 + P;
                x.ntiles = P / kTile;
                int m = 1;
                const int32_t grp = __ldg(seq_group + s);
                while (m < max_members && s + m < S && __ldg(seq_group + s + m) == grp) ++m;
                x.members = m;
                // a one-member unit is an ordinary partition of that sequence
                x.partial = m > 1 || (split && x.L > P);
            } else {
                const int r2 = rr - pu;
                const int p0 = seq_p0 ? seq_p0[s] : 0;
                x.part = p0 + r2 / groups;
                x.hg = r2 - (r2 / groups) * groups;
                x.t0 = x.part * P;
                x.t1 = min(x.L, x.t0 + P);
                x.ntiles = max(0, (x.t1 - x.t0 + kTile - 1) / kTile);
                x.members = 1;
                x.partial = split && x.L > P;
            }
            pos += stride;
        }
        ++count;
        return true;
    }
};

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
// CTAs per SM the register budget is sized for: two, except for the CUDA-core
// consumer of query groups of 4 or 8, which keeps the query and output
// fragments of the whole group in registers and would spill under two CTAs'
// 168-register cap; it runs one CTA per SM with up to 255 registers.
template <int GM, bool kMma>
constexpr int decode_min_ctas() { return (!kMma && GM >= 4) ? 1 : 2; }

template <typename T, int D, int GM, bool kMma>
__global__ void __launch_bounds__(kDecodeThreads, decode_min_ctas<GM, kMma>())
paged_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                    const __grid_constant__ CUtensorMap vmap, const DecodeParams p) {
    using G = StageGeometry<T, D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const sm = smem_raw + (base - raw);
    const int NS_cap = p.stages;   // stages the shared memory holds (barriers for all)
    const int S = p.num_seqs;
    const int H = p.heads_per_unit;
    const int TL = kConsumerWarps >> p.log2_hpu;          // consumer warps per kv head
    const int half_bytes = H * G::kHeadBytes;            // K (or V) part of a stage
    const int stage_bytes = 2 * half_bytes;
    const DecodeSmem lay{stage_bytes, NS_cap, S, D, GM, TL > 1 ? 1 : 0, p.seq_group != nullptr ? 1 : 0};
    const uint32_t full0 = base + lay.bars();
    const uint32_t empty0 = full0 + 8 * NS_cap;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + lay.flag());
    int *ring_stages = reinterpret_cast<int *>(sm + lay.flag() + 4);
    int *seq_base = reinterpret_cast<int *>(sm + lay.seq_base());
    int *seq_len = reinterpret_cast<int *>(sm + lay.seq_len());
    int *seq_p0 = reinterpret_cast<int *>(sm + lay.seq_p0());
    int *seq_pu = reinterpret_cast<int *>(sm + lay.seq_pu());
    const bool prefix = p.seq_group != nullptr;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int B = p.block_size;
    const int groups = p.n_kv_heads >> p.log2_hpu;       // head groups per sequence
    const int P = p.part_tokens;

    if (threadIdx.x == 0) {
        for (int s = 0; s < NS_cap; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, kConsumerWarps);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    // Every thread: the per-sequence inputs into shared memory, four sequences
    // per thread in flight (the caller's arrays; like the rest of the set-up,
    // read before the grid dependency wait). Shared prefixes: the group id goes
    // to seq_pu until the scan below replaces it with the prefix units.
    const int cap = p.max_blocks * B;
    {
        constexpr int kIn = 4;
        for (int s0 = threadIdx.x; s0 < S; s0 += kIn * kDecodeThreads) {
            int len[kIn], grp[kIn], want[kIn];
#pragma unroll
            for (int k = 0; k < kIn; ++k) {
                const int s = s0 + k * kDecodeThreads;
                len[k] = s < S ? __ldg(p.context_lens + s) : 0;
                grp[k] = prefix && s < S ? __ldg(p.seq_group + s) : -1;
            }
#pragma unroll
            for (int k = 0; k < kIn; ++k)
                want[k] = grp[k] >= 0 && grp[k] < p.num_groups ? __ldg(p.group_prefix + grp[k]) : 0;
#pragma unroll
            for (int k = 0; k < kIn; ++k) {
                const int s = s0 + k * kDecodeThreads;
                if (s >= S) continue;
                const int Lc = min(max(len[k], 0), cap);
                if (Lc != len[k]) atomicOr(p.err, PAGEDKV_DEVERR_CONTEXT_LEN);
                seq_len[s] = Lc;
                if (prefix) {
                    int gsel = grp[k];
                    // -1 is the only "no group" value: ids past the groups and
                    // other negative ids are flagged and decoded ungrouped
                    if (gsel >= p.num_groups || gsel < -1) {
                        atomicOr(p.err, PAGEDKV_DEVERR_SEQ_INDEX);
                        gsel = -1;
                    }
                    int p0 = 0;
                    if (gsel >= 0) {
                        if (want[k] > Lc) atomicOr(p.err, PAGEDKV_DEVERR_CONTEXT_LEN);
                        p0 = min(max(want[k], 0), cap) / P;
                    }
                    seq_p0[s] = p0;
                    seq_pu[s] = gsel;
                }
            }
        }
    }
    __syncthreads();
    long long kv_tokens = 0;   // tokens attended over by the whole call (warp 0)
    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_descriptor(&kmap);
            tma_prefetch_descriptor(&vmap);
        }
        // per sequence, prefix-summed: units = max(1, ceil(L / P)) partitions x head
        // groups (fixed mode), or 16-token tiles x head groups (balanced mode)
        int carry = 0;
        int run_carry = -1;   // start of the group run in progress (shared prefixes)
        int gprev = -1;       // group of the previous chunk's last sequence
        if (lane == 0) seq_base[0] = 0;
        for (int s0 = 0; s0 < S; s0 += 32) {
            const int s = s0 + lane;
            const int Lc = s < S ? seq_len[s] : 0;
            kv_tokens += Lc;
            int cnt = s < S ? (p.balanced ? (Lc + kTile - 1) / kTile : (Lc > 0 ? (Lc + P - 1) / P : 1)) * groups
                            : 0;
            if (prefix) {
                // group runs: a run starts where the group id changes; sequence s is
                // member (s - run start) of its run; every max_members-th member leads
                // the units of the run's shared prefix partitions
                const int gsel = s < S ? seq_pu[s] : -1;
                int prev = __shfl_up_sync(kFull, gsel, 1);
                if (lane == 0) prev = gprev;
                gprev = __shfl_sync(kFull, gsel, 31);
                int f = (gsel >= 0 && prev != gsel) ? s : -1;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int y = __shfl_up_sync(kFull, f, off);
                    if (lane >= off) f = max(f, y);
                }
                const int run_start = max(f, run_carry);
                run_carry = __shfl_sync(kFull, run_start, 31);
                if (s < S) {
                    const int p0 = seq_p0[s];
                    const int pu = gsel >= 0 && (s - run_start) % p.max_members == 0 ? p0 * groups : 0;
                    const int own = Lc > 0 ? max(0, (Lc + P - 1) / P - p0) : (p0 > 0 ? 0 : 1);
                    cnt = pu + own * groups;
                    seq_pu[s] = pu;
                }
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
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) kv_tokens += __shfl_xor_sync(kFull, kv_tokens, off);
        // stages in use: the alternative ring size when the sequences are long
        // on average (long runs of blocks per unit)
        if (lane == 0)
            *ring_stages = kv_tokens >= (long long)p.long_seq_tokens * S ? p.stages_alt : NS_cap;
    }
    __syncthreads();
    const int NS = *ring_stages;
    Walk walk;
    walk.init(seq_base, seq_len, S, groups, P, p.split, p.balanced, prefix ? seq_p0 : nullptr,
              prefix ? seq_pu : nullptr, p.seq_group, p.max_members);
    if (!walk.has_work()) return;
    // a dependent merge launch may start once every CTA got here or exited;
    // it waits on this grid's completion before reading the partition states
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        uint32_t armed = 0;   // tiles armed so far by this CTA
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        // L2 priority of the K/V lines, once the call streams more K/V than the
        // L2 holds (a smaller stream is left to the default policy: the next
        // step reads it again and may find it there). A block that the previous
        // or the next sequence also holds at the same table index (a shared
        // prefix, a forked sequence) is read again soon by another unit:
        // evict_last. Every other block is read once per call: evict_first.
        const bool hint = kv_tokens > p.hint_min_tokens;
        uint64_t pol_shared = 0, pol_own = 0;
        if (hint) {
            pol_shared = l2_policy_evict_last();
            pol_own = l2_policy_evict_first();
        }
        // lane-parallel window of 32 block-table entries starting at block j0,
        // and the mask of those held by a neighbouring sequence too
        auto load_window = [&](const Unit &x, int j0, unsigned &shared) {
            const int nblk = (x.L + B - 1) >> p.log2_block;
            const int j = j0 + lane;
            const int v = j < nblk ? __ldg(p.block_tables + size_t(x.s) * p.max_blocks + j) : -1;
            bool sh = false;
            if (hint) {
                const int nprev = x.s > 0 ? (seq_len[x.s - 1] + B - 1) >> p.log2_block : 0;
                const int nnext = x.s + 1 < S ? (seq_len[x.s + 1] + B - 1) >> p.log2_block : 0;
                const int a = j < nprev ? __ldg(p.block_tables + size_t(x.s - 1) * p.max_blocks + j) : -1;
                const int b = j < nnext ? __ldg(p.block_tables + size_t(x.s + 1) * p.max_blocks + j) : -1;
                sh = v >= 0 && (v == a || v == b);
            }
            shared = __ballot_sync(kFull, sh);
            return v;
        };
        Unit cur;
        walk.next(cur);
        // the block tables are the caller's (no kernel of this library writes
        // them): the first window is in flight during the wait below
        int nxt_base = cur.t0 >> p.log2_block;
        unsigned nxt_sh;
        int nxt_val = load_window(cur, nxt_base, nxt_sh);
        // the pools as the kernels before this one left them (an append
        // launched just before may still be running: launched as its
        // programmatic dependent, this kernel set itself up meanwhile)
        grid_dependency_wait();
        while (ok) {
            int win_base = nxt_base, win_val = nxt_val;
            unsigned win_sh = nxt_sh;
            Unit nx;
            const bool has_next = walk.next(nx);
            if (has_next) {
                // prefetch the first window of this CTA's next unit
                nxt_base = nx.t0 >> p.log2_block;
                nxt_val = load_window(nx, nxt_base, nxt_sh);
            }
            const int h0 = cur.hg << p.log2_hpu;
            for (int i = 0; i < cur.ntiles; ++i) {
                const int tok = cur.t0 + i * kTile;
                const int j0 = tok >> p.log2_block;
                const bool two = (B < kTile) && (tok + B < cur.t1);
                if (j0 < win_base || j0 + 1 >= win_base + 32) {
                    win_base = j0;
                    win_val = load_window(cur, j0, win_sh);
                }
                const int i0 = j0 - win_base, i1 = (j0 + 1 - win_base) & 31;
                int pb0 = __shfl_sync(kFull, win_val, i0);
                int pb1 = __shfl_sync(kFull, win_val, i1);
                if (lane == 0) {
                    if (*abort_flag || !mbar_wait(empty0 + 8 * stage, phase ^ 1u, p.err)) {
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
                        const uint32_t fb = full0 + 8 * stage;
                        const uint32_t kdst = base + stage * stage_bytes;
                        const uint32_t vdst = kdst + half_bytes;
                        if (B >= kTile) {
                            // one box per operand: every slab of H heads x 16 tokens
                            const int z0 = pb0 * B + (tok & (B - 1));
                            mbar_arrive_expect_tx(fb, uint32_t(stage_bytes));
                            if (hint) {
                                const uint64_t pol = (win_sh >> i0) & 1u ? pol_shared : pol_own;
                                tma_load_4d_hint(kdst, &kmap, 0, z0, 0, h0, fb, pol);
                                tma_load_4d_hint(vdst, &vmap, 0, z0, 0, h0, fb, pol);
                            } else {
                                tma_load_4d(kdst, &kmap, 0, z0, 0, h0, fb);
                                tma_load_4d(vdst, &vmap, 0, z0, 0, h0, fb);
                            }
                        } else {
                            // 8-token blocks: one box per block and operand (every
                            // slab of H heads x 8 tokens); the second block's box
                            // lands half of the operand's part further on
                            const int nb = two ? 2 : 1;
                            mbar_arrive_expect_tx(fb, uint32_t(stage_bytes / 2 * nb));
                            for (int b = 0; b < nb; ++b) {
                                const int z = (b ? pb1 : pb0) * B;
                                const uint32_t off = uint32_t(b) * uint32_t(half_bytes / 2);
                                if (hint) {
                                    const uint64_t pol = (win_sh >> (b ? i1 : i0)) & 1u ? pol_shared : pol_own;
                                    tma_load_4d_hint(kdst + off, &kmap, 0, z, 0, h0, fb, pol);
                                    tma_load_4d_hint(vdst + off, &vmap, 0, z, 0, h0, fb, pol);
                                } else {
                                    tma_load_4d(kdst + off, &kmap, 0, z, 0, h0, fb);
                                    tma_load_4d(vdst + off, &vmap, 0, z, 0, h0, fb);
                                }
                            }
                        }
                        ++armed;
                    }
                }
                ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
                if (!ok) break;
                if (++stage == NS) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!has_next) break;
            cur = nx;
        }
        if (!ok && lane == 0) {
            // Stop everyone, then wait (bounded) for this CTA's copies still in flight.
            *abort_flag = 1;
            const uint32_t first = armed > uint32_t(NS) ? armed - NS : 0u;
            for (uint32_t k = first; k < armed; ++k)
                mbar_wait(full0 + 8 * (k % uint32_t(NS)), (k / uint32_t(NS)) & 1u, p.err);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int cw = warp - 1;
    const int hh = cw & (H - 1);          // kv head of the unit this warp owns
    // where a head's rows sit in a stage: 16-row boxes, or two 8-row boxes
    // (one per 8-token block) each holding every head of the unit
    const bool two_boxes = B < kTile;
    const TileAddr ta{uint32_t(two_boxes ? G::kSlabBytes / 2 : G::kSlabBytes),
                      uint32_t(two_boxes ? half_bytes / 2 : kTile / 2 * kRowBytes128)};
    const int head_bytes = two_boxes ? G::kHeadBytes / 2 : G::kHeadBytes;
    const int tw = cw >> p.log2_hpu;      // which of the TL warps sharing that head
    const int g = p.group;
    using Simt = SimtConsumer<T, D, GM>;
    using Mma = MmaConsumer<T, D>;
    typename std::conditional<kMma, Mma, Simt>::type st;
    st.init(lane);

    int stage = 0;
    uint32_t phase = 0;
    int unit_count = 0;
    const T *qbase = reinterpret_cast<const T *>(p.q);
    Unit cur;
    walk.next(cur);
    st.prefetch_q(qbase, size_t(cur.s), ((cur.hg << p.log2_hpu) + hh) * g, g, cur.members, p.n_q_heads);
    // No store to out or the workspace before the kernels ahead of this one
    // have completed: a unit with no tiles (an empty context) writes its zero
    // row without waiting on any stage, and the previous decode of the stream
    // may still be writing the same rows (it let this grid start early). The
    // q rows above are the caller's and were safe to read before.
    grid_dependency_wait();
    for (;; ++unit_count) {
        const int qh0 = ((cur.hg << p.log2_hpu) + hh) * g;   // first q head of this warp
        if constexpr (kMma) st.begin_unit();
        else st.begin_unit(p.scale_log2);
        Unit nx;
        const bool has_next = walk.next(nx);
        if (has_next)
            st.prefetch_q(qbase, size_t(nx.s), ((nx.hg << p.log2_hpu) + hh) * g, g, nx.members, p.n_q_heads);
        for (int i = 0; i < cur.ntiles; ++i) {
            int good = !*abort_flag;
            if (good) good = mbar_wait(full0 + 8 * stage, phase, p.err);
            if (!__all_sync(kFull, good)) {
                *abort_flag = 1;
            } else if ((i & (TL - 1)) == tw) {
                const int nvalid = min(kTile, cur.t1 - (cur.t0 + i * kTile));
                const uint32_t kaddr = base + stage * stage_bytes + hh * head_bytes;
                const uint32_t vaddr = kaddr + half_bytes;
                if constexpr (kMma) {
                    if (nvalid < kTile) {
                        // rows past the context may hold anything (even NaN): zero this head's V rows
                        const int n16 = (kTile - nvalid) * G::kSlabs * 8;
                        for (int x = lane; x < n16; x += 32) {
                            const int row = nvalid + x / (G::kSlabs * 8);
                            const int rem = x % (G::kSlabs * 8);
                            sts128_zero(vaddr + (rem >> 3) * ta.slab + (row >> 3) * ta.hi +
                                        (row & 7) * kRowBytes128 + (rem & 7) * 16);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                    st.tile(kaddr, vaddr, nvalid, p.scale_log2, ta);
                } else {
                    st.tile(kaddr, vaddr, nvalid, g, ta);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8 * stage);
            if (++stage == NS) {
                stage = 0;
                phase ^= 1u;
            }
        }

        // ---- result of this unit
        UnitSink sink;
        sink.partial = cur.partial;
        sink.out_row0 = size_t(cur.s) * p.n_q_heads + qh0;
        if (p.balanced) {
            // piece slot of this CTA: rows [piece][head of unit][q head of group]
            const size_t piece = size_t(blockIdx.x) * 2 + cur.slot;
            sink.ws_row0 = (piece * H + hh) * g;
            sink.j_stride = 1;
        } else {
            sink.ws_row0 = (size_t(cur.s) * p.n_q_heads + qh0) * p.max_parts + cur.part;
            sink.j_stride = p.max_parts;
        }
        if constexpr (kMma) st.reduce();
        else st.reduce(g);
        if (cur.members > 1) {
            // shared-prefix unit (tensor-core path, one consumer warp per kv head)
            if constexpr (kMma)
                st.store_members(reinterpret_cast<T *>(p.out), p.ws_o, p.ws_m, p.ws_l, seq_len,
                                 size_t(cur.s), cur.members, qh0, g, p.n_q_heads, P, cur.part,
                                 p.max_parts);
        } else if (TL == 1) {
            if constexpr (kMma) st.store(sink, reinterpret_cast<T *>(p.out), p.ws_o, p.ws_m, p.ws_l, g);
            else st.store(sink, reinterpret_cast<T *>(p.out), p.ws_o, p.ws_m, p.ws_l, g, lane);
        } else {
            // warps sharing a kv head combine their states (double-buffered slots,
            // so one barrier per unit suffices)
            const int stride = lay.row_stride();
            const int slot = unit_count & 1;
            float *mo0 = reinterpret_cast<float *>(sm + lay.merge_o()) + slot * kConsumerWarps * GM * stride;
            float *mm0 = reinterpret_cast<float *>(sm + lay.merge_m()) + slot * kConsumerWarps * GM;
            float *ml0 = reinterpret_cast<float *>(sm + lay.merge_l()) + slot * kConsumerWarps * GM;
            if constexpr (kMma) st.stash(mo0 + cw * GM * stride, mm0 + cw * GM, ml0 + cw * GM, g, stride);
            else st.stash(mo0 + cw * GM * stride, mm0 + cw * GM, ml0 + cw * GM, g, lane, stride);
            named_barrier(1, 32 * kConsumerWarps);
            const int qu0 = (cur.hg << p.log2_hpu) * g;      // first q head of the unit
            for (int idx = threadIdx.x - 32; idx < H * g * D; idx += 32 * kConsumerWarps) {
                const int h = idx / (g * D);
                const int rem = idx - h * g * D;
                const int j = rem / D;
                const int d = rem - j * D;
                float M = -INFINITY;
                for (int t = 0; t < TL; ++t) M = fmaxf(M, mm0[(t * H + h) * GM + j]);
                float num = 0.f, den = 0.f;
                if (M != -INFINITY) {
                    for (int t = 0; t < TL; ++t) {
                        const int w = t * H + h;
                        const float f = fast_exp2(mm0[w * GM + j] - M);
                        num = fmaf(f, mo0[(w * GM + j) * stride + d], num);
                        den = fmaf(f, ml0[w * GM + j], den);
                    }
                }
                const int qh = qu0 + h * g + j;
                if (sink.partial) {
                    const size_t row = p.balanced
                        ? (size_t(blockIdx.x) * 2 + cur.slot) * H * g + size_t(h) * g + j
                        : (size_t(cur.s) * p.n_q_heads + qh) * p.max_parts + cur.part;
                    p.ws_o[row * D + d] = num;
                    if (d == 0) {
                        p.ws_m[row] = M * kLn2;
                        p.ws_l[row] = den;
                    }
                } else {
                    const float v = den > 0.f ? num / den : 0.f;
                    reinterpret_cast<T *>(p.out)[(size_t(cur.s) * p.n_q_heads + qh) * D + d] =
                        Elem<T>::from_float(v);
                }
            }
        }
        if (!has_next) break;
        cur = nx;
    }
}

}  // namespace pkv
