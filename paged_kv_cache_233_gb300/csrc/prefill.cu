// prefill.cu -- chunked-prefill attention over the paged KV cache.
//
// "How a serving engine actually works", section "Prefill and decode are two
// different jobs": a long prompt is prefilled in chunks, one chunk per
// iteration, so that the sequences decoding beside it are not stalled behind
// the whole prompt. Each chunk's K/V rows are appended to the cache first;
// then every query row of the chunk attends, causally, over all of the
// sequence's cached tokens up to and including its own position, read in
// place through the block table. With L cached tokens (the chunk included)
// and a chunk of n rows, row j is the token at position L - n + j and sees
// keys 0 .. L - n + j. Decode is the case n = 1.
//
// Unlike decode, a chunk of n tokens reuses every K/V byte for n * g query
// rows (g = query heads per kv head), so the work is a dense contraction and
// runs on the tensor cores. One CTA owns (sequence, kv head, query tile): 64
// rows of (chunk token, query head of the group), so all g heads of a kv head
// share each K/V byte read. A producer warp streams 64-key tiles of K and V
// through the block table with 4-D TMA loads (128-byte swizzle) into a ring
// of three stages; four consumer warps of 16 rows each compute S = Q K^T and
// O += P V with m16n8k16 MMAs (fp32 accumulation) and a base-2 online
// softmax in registers. Every wait is bounded in time.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "launch_cache.h"
#include "prefill.h"
#include "ptx.cuh"

namespace pkv {

namespace {

constexpr unsigned kFullMask = 0xffffffffu;

template <typename T, int D>
struct PrefillGeometry {
    static constexpr int kSlabs = D * int(sizeof(T)) / 128;   // 128-byte column slabs per row
    static constexpr int kGroup16 = kSlabs * 16 * 128;        // 16 keys, every slab
    static constexpr int kHalf = (kPfKeys / 16) * kGroup16;   // K (or V) of one stage
    static constexpr int kStage = 2 * kHalf;
    static constexpr int kBarriers = kPfStages * kStage;      // offset of the barriers
    static constexpr int kFlag = kBarriers + 16 * kPfStages;
    static constexpr int kTotal = kFlag + 16;
};

// Byte offset of (key t of the stage, 16-byte chunk ch of its row) in a K or V
// half-stage: [16-key group][slab][16 rows][128 B], 128-byte swizzle.
template <int kGroup16>
__device__ __forceinline__ uint32_t kv_off(int t, int ch) {
    const int row = t & 15;
    return uint32_t((t >> 4) * kGroup16 + (ch >> 3) * 2048 + row * 128 +
                    (((ch & 7) ^ (row & 7)) << 4));
}

// Keep the 16-bit halves of a register whose keys lie before `limit`.
__device__ __forceinline__ uint32_t keep_keys(uint32_t w, int key_lo, int limit) {
    const uint32_t lo = key_lo < limit ? 0x0000ffffu : 0u;
    const uint32_t hi = key_lo + 1 < limit ? 0xffff0000u : 0u;
    return w & (lo | hi);
}

}  // namespace

template <typename T, int D>
__global__ void __launch_bounds__(kPfThreads, 2)
paged_prefill_kernel(const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
    using G = PrefillGeometry<T, D>;
    constexpr bool kBf16 = Elem<T>::kBf16;
    constexpr int KS = D / 16;    // k-steps of Q K^T
    constexpr int NT = D / 8;     // n-tiles of O
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const sm = smem_raw + (base - raw);
    const uint32_t full0 = base + G::kBarriers;
    const uint32_t empty0 = full0 + 8 * kPfStages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + G::kFlag);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int s = blockIdx.z;
    const int h = blockIdx.y;
    const int qt = int(gridDim.x) - 1 - int(blockIdx.x);   // longest-running tiles first
    const int B = p.block_size;
    const int g = p.group;

    // ---- this CTA's slice of the chunk (uniform across the CTA)
    const int q0 = __ldg(p.query_start + s);
    const int q1 = __ldg(p.query_start + s + 1);
    const int n = q1 - q0;
    const int L = __ldg(p.context_lens + s);
    const bool rows_ok = q0 >= 0 && q1 >= q0 && q1 <= p.num_tokens &&
                         n <= int(gridDim.x) * p.tile_tokens;
    const bool len_ok = L >= n && L <= p.max_blocks * B;
    if (!rows_ok || !len_ok) {
        if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0)
            atomicOr(p.err, rows_ok ? PAGEDKV_DEVERR_CONTEXT_LEN : PAGEDKV_DEVERR_POSITION);
        return;
    }
    const int j0 = qt * p.tile_tokens;        // first chunk row of the tile
    if (j0 >= n) return;
    const int tokens = min(p.tile_tokens, n - j0);
    const int rows = tokens * g;
    const int pos0 = L - n + j0;              // position of the tile's first token
    const int nkt = (pos0 + tokens - 1) / kPfKeys + 1;   // key tiles: keys 0 .. last position

    if (threadIdx.x == 0) {
        for (int k = 0; k < kPfStages; ++k) {
            mbar_init(full0 + 8 * k, 1);
            mbar_init(empty0 + 8 * k, kPfThreads / 32 - 1);
        }
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        tma_prefetch_descriptor(&kmap);
        tma_prefetch_descriptor(&vmap);
        const int32_t *table = p.block_tables + size_t(s) * p.max_blocks;
        int stage = 0;
        uint32_t phase = 0;
        uint32_t armed = 0;
        bool ok = true;
        for (int kt = 0; kt < nkt && ok; ++kt) {
            if (*abort_flag || !mbar_wait(empty0 + 8 * stage, phase ^ 1u, p.err)) {
                ok = false;
                break;
            }
            const int k0 = kt * kPfKeys;
            const int present = min(kPfKeys, L - k0);       // keys of this tile in the cache
            const uint32_t fb = full0 + 8 * stage;
            const uint32_t kdst = base + stage * G::kStage;
            const uint32_t vdst = kdst + G::kHalf;
            if (B >= 16) {
                // one box of 16 keys x every slab per 16-key group
                const int groups = (present + 15) >> 4;
                mbar_arrive_expect_tx(fb, uint32_t(groups * 2 * G::kGroup16));
                for (int i = 0; i < groups; ++i) {
                    const int t = k0 + 16 * i;
                    int pb = __ldg(table + (t >> p.log2_block));
                    if (pb < 0 || pb >= p.num_blocks) {
                        atomicOr(p.err, PAGEDKV_DEVERR_BLOCK_ID);
                        pb = 0;
                    }
                    const int z = pb * B + (t & (B - 1));
                    tma_load_4d(kdst + i * G::kGroup16, &kmap, 0, z, 0, h, fb);
                    tma_load_4d(vdst + i * G::kGroup16, &vmap, 0, z, 0, h, fb);
                }
            } else {
                // 8-token blocks: one box per (block, slab), placed as rows 0-7 or 8-15
                const int blocks = (present + 7) >> 3;
                mbar_arrive_expect_tx(fb, uint32_t(blocks * G::kSlabs * 1024 * 2));
                for (int b = 0; b < blocks; ++b) {
                    const int t = k0 + 8 * b;
                    int pb = __ldg(table + (t >> p.log2_block));
                    if (pb < 0 || pb >= p.num_blocks) {
                        atomicOr(p.err, PAGEDKV_DEVERR_BLOCK_ID);
                        pb = 0;
                    }
                    for (int sl = 0; sl < G::kSlabs; ++sl) {
                        const uint32_t off = (b >> 1) * G::kGroup16 + sl * 2048 + (b & 1) * 1024;
                        tma_load_4d(kdst + off, &kmap, 0, pb * B, sl, h, fb);
                        tma_load_4d(vdst + off, &vmap, 0, pb * B, sl, h, fb);
                    }
                }
            }
            ++armed;
            if (++stage == kPfStages) {
                stage = 0;
                phase ^= 1u;
            }
        }
        if (!ok) {
            // stop the consumers, then wait (bounded) for the copies still in flight
            *abort_flag = 1;
            const uint32_t first = armed > uint32_t(kPfStages) ? armed - kPfStages : 0u;
            for (uint32_t k = first; k < armed; ++k)
                mbar_wait(full0 + 8 * (k % kPfStages), (k / kPfStages) & 1u, p.err);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int cw = warp - 1;
    const int grp = lane >> 2, c = lane & 3;
    const int mi = lane >> 3, r8 = lane & 7;
    const int r0 = 16 * cw + grp, r1 = r0 + 8;           // this lane's two rows
    const int posA = r0 < rows ? pos0 + r0 / g : -1;
    const int posB = r1 < rows ? pos0 + r1 / g : -1;
    const bool live = 16 * cw < rows;
    const int wpos_min = pos0 + (16 * cw) / g;
    const int wpos_max = pos0 + (min(16 * cw + 15, rows - 1)) / g;

    // Q fragments of the two rows, kept in registers for the whole tile loop
    uint32_t qa[KS][4];
    {
        const uint32_t *rowA = nullptr, *rowB = nullptr;
        if (r0 < rows)
            rowA = reinterpret_cast<const uint32_t *>(
                reinterpret_cast<const T *>(p.q) +
                (size_t(q0 + j0 + r0 / g) * p.n_q_heads + h * g + r0 % g) * D);
        if (r1 < rows)
            rowB = reinterpret_cast<const uint32_t *>(
                reinterpret_cast<const T *>(p.q) +
                (size_t(q0 + j0 + r1 / g) * p.n_q_heads + h * g + r1 % g) * D);
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
            qa[kk][0] = rowA ? __ldg(rowA + 8 * kk + c) : 0u;
            qa[kk][1] = rowB ? __ldg(rowB + 8 * kk + c) : 0u;
            qa[kk][2] = rowA ? __ldg(rowA + 8 * kk + 4 + c) : 0u;
            qa[kk][3] = rowB ? __ldg(rowB + 8 * kk + 4 + c) : 0u;
        }
    }

    float o[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
    float mA = -INFINITY, mB = -INFINITY;   // running maxima (base 2)
    float lA = 0.f, lB = 0.f;               // this lane's part of the running sums

    int stage = 0;
    uint32_t phase = 0;
    for (int kt = 0; kt < nkt; ++kt) {
        int good = !*abort_flag;
        if (good) good = mbar_wait(full0 + 8 * stage, phase, p.err);
        if (!__all_sync(kFullMask, good)) {
            *abort_flag = 1;
        } else if (live && kt * kPfKeys <= wpos_max) {
            const int k0 = kt * kPfKeys;
            const uint32_t kaddr = base + stage * G::kStage;
            const uint32_t vaddr = kaddr + G::kHalf;
            // ---- S = Q K^T over the 64 keys of the stage
            float sc[8][4];
#pragma unroll
            for (int t = 0; t < 8; ++t) sc[t][0] = sc[t][1] = sc[t][2] = sc[t][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
                for (int np = 0; np < 4; ++np) {
                    uint32_t b[4];
                    ldmatrix_x4(kaddr + kv_off<G::kGroup16>(16 * np + (mi >> 1) * 8 + r8,
                                                            2 * kk + (mi & 1)), b);
                    mma_m16n8k16<kBf16>(sc[2 * np], qa[kk], b[0], b[1]);
                    mma_m16n8k16<kBf16>(sc[2 * np + 1], qa[kk], b[2], b[3]);
                }
            }
            // ---- scale, causal mask (a select: rows past the context may hold NaN)
            const bool masked = k0 + kPfKeys - 1 > wpos_min;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const int key = k0 + 8 * t + 2 * c;
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    sc[t][e] *= p.scale_log2;
                    sc[t][2 + e] *= p.scale_log2;
                    if (masked) {
                        if (key + e > posA) sc[t][e] = -INFINITY;
                        if (key + e > posB) sc[t][2 + e] = -INFINITY;
                    }
                }
            }
            // ---- online softmax, rows r0 (A) and r1 (B)
            float xA = -INFINITY, xB = -INFINITY;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                xA = fmaxf(xA, fmaxf(sc[t][0], sc[t][1]));
                xB = fmaxf(xB, fmaxf(sc[t][2], sc[t][3]));
            }
            xA = fmaxf(xA, __shfl_xor_sync(kFullMask, xA, 1));
            xA = fmaxf(xA, __shfl_xor_sync(kFullMask, xA, 2));
            xB = fmaxf(xB, __shfl_xor_sync(kFullMask, xB, 1));
            xB = fmaxf(xB, __shfl_xor_sync(kFullMask, xB, 2));
            const float nA = fmaxf(mA, xA), nB = fmaxf(mB, xB);
            const float uA = nA == -INFINITY ? 0.f : nA;   // a row with no key yet keeps zeros
            const float uB = nB == -INFINITY ? 0.f : nB;
            const float aA = fast_exp2(mA - uA), aB = fast_exp2(mB - uB);
            mA = nA;
            mB = nB;
            float sumA = 0.f, sumB = 0.f;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                sc[t][0] = fast_exp2(sc[t][0] - uA);
                sc[t][1] = fast_exp2(sc[t][1] - uA);
                sc[t][2] = fast_exp2(sc[t][2] - uB);
                sc[t][3] = fast_exp2(sc[t][3] - uB);
                sumA += sc[t][0] + sc[t][1];
                sumB += sc[t][2] + sc[t][3];
            }
            lA = lA * aA + sumA;
            lB = lB * aB + sumB;
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                o[t][0] *= aA;
                o[t][1] *= aA;
                o[t][2] *= aB;
                o[t][3] *= aB;
            }
            // ---- O += P V; P's accumulator layout is the A operand's layout
            const bool tail = k0 + kPfKeys > L;   // keys past the context: zero their V
#pragma unroll
            for (int kk = 0; kk < kPfKeys / 16; ++kk) {
                uint32_t a[4];
                a[0] = Elem<T>::pack2(sc[2 * kk][0], sc[2 * kk][1]);
                a[1] = Elem<T>::pack2(sc[2 * kk][2], sc[2 * kk][3]);
                a[2] = Elem<T>::pack2(sc[2 * kk + 1][0], sc[2 * kk + 1][1]);
                a[3] = Elem<T>::pack2(sc[2 * kk + 1][2], sc[2 * kk + 1][3]);
                const int klo = k0 + 16 * kk + 2 * c;
#pragma unroll
                for (int tp = 0; tp < NT / 2; ++tp) {
                    uint32_t b[4];
                    ldmatrix_x4_trans(vaddr + kv_off<G::kGroup16>(16 * kk + (mi & 1) * 8 + r8,
                                                                  2 * tp + (mi >> 1)), b);
                    if (tail) {
                        b[0] = keep_keys(b[0], klo, L);
                        b[1] = keep_keys(b[1], klo + 8, L);
                        b[2] = keep_keys(b[2], klo, L);
                        b[3] = keep_keys(b[3], klo + 8, L);
                    }
                    mma_m16n8k16<kBf16>(o[2 * tp], a, b[0], b[1]);
                    mma_m16n8k16<kBf16>(o[2 * tp + 1], a, b[2], b[3]);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * stage);
        if (++stage == kPfStages) {
            stage = 0;
            phase ^= 1u;
        }
    }

    // ---- normalise and store this lane's part of rows r0 and r1
    lA += __shfl_xor_sync(kFullMask, lA, 1);
    lA += __shfl_xor_sync(kFullMask, lA, 2);
    lB += __shfl_xor_sync(kFullMask, lB, 1);
    lB += __shfl_xor_sync(kFullMask, lB, 2);
    T *out = reinterpret_cast<T *>(p.out);
    if (r0 < rows) {
        const float inv = lA > 0.f ? 1.f / lA : 0.f;
        uint32_t *dst = reinterpret_cast<uint32_t *>(
            out + (size_t(q0 + j0 + r0 / g) * p.n_q_heads + h * g + r0 % g) * D);
#pragma unroll
        for (int t = 0; t < NT; ++t) dst[4 * t + c] = Elem<T>::pack2(o[t][0] * inv, o[t][1] * inv);
    }
    if (r1 < rows) {
        const float inv = lB > 0.f ? 1.f / lB : 0.f;
        uint32_t *dst = reinterpret_cast<uint32_t *>(
            out + (size_t(q0 + j0 + r1 / g) * p.n_q_heads + h * g + r1 % g) * D);
#pragma unroll
        for (int t = 0; t < NT; ++t) dst[4 * t + c] = Elem<T>::pack2(o[t][2] * inv, o[t][3] * inv);
    }
}

int prefill_smem_bytes(int head_dim) {
    const int total = head_dim == 64 ? PrefillGeometry<__half, 64>::kTotal
                                     : PrefillGeometry<__half, 128>::kTotal;
    return total + 1024;   // slack to align the ring to 1024 bytes
}

template <typename T, int D>
static cudaError_t launch_prefill_instance(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                           const PrefillParams &p, int max_query_len,
                                           cudaStream_t stream) {
    auto kernel = paged_prefill_kernel<T, D>;
    const int smem = PrefillGeometry<T, D>::kTotal + 1024;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::atomic<unsigned long long> opened[kLaunchCacheDevices];
    e = open_dynamic_smem(opened, dev, kernel, smem);
    if (e != cudaSuccess) return e;
    const unsigned tiles = unsigned((max_query_len + p.tile_tokens - 1) / p.tile_tokens);
    const dim3 grid(tiles, unsigned(p.n_kv_heads), unsigned(p.num_seqs));
    kernel<<<grid, kPfThreads, smem, stream>>>(kmap, vmap, p);
    return cudaGetLastError();
}

cudaError_t launch_prefill(int dtype, int head_dim, const CUtensorMap &kmap,
                           const CUtensorMap &vmap, const PrefillParams &p, int max_query_len,
                           cudaStream_t stream) {
    const bool bf16 = dtype == PAGEDKV_BF16;
    if (head_dim == 64)
        return bf16 ? launch_prefill_instance<__nv_bfloat16, 64>(kmap, vmap, p, max_query_len, stream)
                    : launch_prefill_instance<__half, 64>(kmap, vmap, p, max_query_len, stream);
    return bf16 ? launch_prefill_instance<__nv_bfloat16, 128>(kmap, vmap, p, max_query_len, stream)
                : launch_prefill_instance<__half, 128>(kmap, vmap, p, max_query_len, stream);
}

}  // namespace pkv
