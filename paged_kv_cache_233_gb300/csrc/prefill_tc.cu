// prefill_tc.cu -- chunked-prefill attention on the fifth-generation tensor
// cores (tcgen05): the same operation as prefill.cu ("How a serving engine
// actually works", section "Prefill and decode are two different jobs": each
// query row of a chunk attends causally over its sequence's cached tokens up
// to its own position, read through the block table), with the contractions
// moved off the warp-level MMA pipe.
//
// One CTA owns (sequence, kv head, 256 query rows of (chunk token, query head
// of the group)), held as two 128-row Q tiles that share every K/V tile.
// Eleven warps:
//   warp 0     producer: per 64-key tile, lane 0 waits for a free stage of a
//              four-stage ring and arms its barrier; then one lane per (16
//              keys, 64-column block, operand) looks up its block id and
//              issues that TMA box, so that each operand lands as [column
//              block][64 keys][128 B] with 128-byte swizzle (the canonical
//              layout the tensor core reads);
//   warps 1,10 MMA issuers, one per Q tile (warp 1 also allocates tensor
//              memory); lane 0 issues, for its tile, S = Q K^T into one of two
//              S buffers in tensor memory and, once the softmax has written P,
//              O += P V with P read from tensor memory, into the O accumulator
//              that stays in tensor memory for the whole key loop; completions
//              are tracked by tcgen05.commit on mbarriers. An issuing thread
//              runs only about two MMAs ahead of the tensor core, so each of
//              its waits leaves the tensor core idle unless the other tile's
//              issuer has MMAs to give it;
//   warps 2-9  softmax, four warps per Q tile, one thread per query row (=
//              tensor-memory lane), so that every SM sub-partition runs two
//              softmax warps whose work interleaves. A thread reads its S row,
//              applies the causal limit (a select, so K rows past the context
//              never matter), exponentiates against a reference maximum and
//              writes P (packed 16-bit pairs) over the first half of the same
//              S buffer in tensor memory, so P never touches shared memory. The
//              reference moves only when a tile's maximum exceeds it by more
//              than 2^8 (P stays below 256, sums stay in fp32); when it moves,
//              the warp rescales its rows of O in tensor memory before that
//              tile's P V may start. The result is exact softmax attention.
//              V rows past the context are zeroed in shared memory before any
//              P V reads them (the tensor core would turn 0 * NaN into NaN).
// A Q tile skips the key tiles that lie wholly past its last row. Every
// mbarrier wait is bounded in time; on a timeout the CTA stops, waits for its
// copies and MMAs in flight, frees its tensor memory and exits.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "launch_cache.h"
#include "prefill.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr unsigned kAll = 0xffffffffu;
constexpr int kTcTiles = 2;      // Q tiles per CTA
constexpr int kTcRows = 128;     // query rows per Q tile = tensor-memory lanes
constexpr int kTcKeys = 64;      // keys per pipeline stage
constexpr int kTcStages = 4;
// warp 0 producer, warp 1 MMA issuer of Q tile 0, warps 2-9 softmax, warp 10
// MMA issuer of Q tile 1
constexpr int kIssuer1Warp = 2 + kTcTiles * kTcRows / 32;
constexpr int kTcThreads = 32 * (kIssuer1Warp + 1);
constexpr int kTmemTile = 256;   // tensor-memory columns per Q tile: S, S, O
constexpr float kRescaleLog2 = 8.f;  // the reference maximum moves past 2^8

template <int D>
struct TcLayout {
    static constexpr int kSlabs = D * 2 / 128;             // 64-element column blocks per row
    static constexpr int kQSlab = kTcRows * 128;           // bytes of one Q column block
    static constexpr int kKvSlab = kTcKeys * 128;          // bytes of one K (or V) column block
    static constexpr int kQTile = kSlabs * kQSlab;
    static constexpr int kQ = 0;                           // Q tile t at kQ + t * kQTile
    static constexpr int kKv = kQ + kTcTiles * kQTile;     // stage s: K at kKv + s*kStage, V after it
    static constexpr int kHalf = kSlabs * kKvSlab;
    static constexpr int kStage = 2 * kHalf;
    static constexpr int kBars = kKv + kTcStages * kStage;
    static constexpr int kNumBars = 2 * kTcStages + 6 * kTcTiles + 3;
    static constexpr int kTmemSlot = kBars + 8 * kNumBars;
    static constexpr int kFlag = kTmemSlot + 8;
    static constexpr int kTotal = kFlag + 8;
    static_assert(2 * kTcKeys + D <= kTmemTile, "S buffers and O must fit a Q tile's columns");
};

// mbarrier indices
constexpr int kKvFull = 0;
constexpr int kKvEmpty = kTcStages;
// per Q tile t, buffer b: S full, P full, O full (P V of key tile j completes
// on O barrier j & 1, so a wait never meets a barrier two completions away)
__device__ __forceinline__ int bar_s(int t, int b) { return 2 * kTcStages + 6 * t + b; }
__device__ __forceinline__ int bar_p(int t, int b) { return 2 * kTcStages + 6 * t + 2 + b; }
__device__ __forceinline__ int bar_o(int t, int b) { return 2 * kTcStages + 6 * t + 4 + b; }
constexpr int kQFull = 2 * kTcStages + 6 * kTcTiles;
constexpr int kDone = kQFull + 1;
// the last key tile's V rows past the context are zeroed (one phase per CTA,
// so a wait on it is never ambiguous however far the Q tiles drift apart)
constexpr int kVZero = kDone + 1;

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                 ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

}  // namespace

template <typename T, int D>
__global__ void __launch_bounds__(kTcThreads, 1)
paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
    using Ly = TcLayout<D>;
    constexpr bool kBf16 = Elem<T>::kBf16;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const sm = smem_raw + (base - raw);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(sm + Ly::kFlag);
    auto bar = [&](int i) { return base + Ly::kBars + 8u * uint32_t(i); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int s = blockIdx.z;
    const int h = blockIdx.y;
    const int qt = int(gridDim.x) - 1 - int(blockIdx.x);   // tiles with the most keys first
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
    const int j0 = qt * p.tile_tokens;
    if (j0 >= n) return;
    const int rows = min(p.tile_tokens, n - j0) * g;   // rows of the CTA (both Q tiles)
    const int pos0 = L - n + j0;                       // position of the CTA's first token
    // key tiles of Q tile t: through the position of its last row
    auto key_tiles = [&](int t) {
        const int rt = min(max(rows - t * kTcRows, 0), kTcRows);
        return rt > 0 ? (pos0 + (t * kTcRows + rt - 1) / g) / kTcKeys + 1 : 0;
    };
    const int nk0 = key_tiles(0), nk1 = key_tiles(1);
    auto nkt_of = [&](int t) { return t ? nk1 : nk0; };
    const int t_last = nk1 > 0 ? 1 : 0;                // holds the CTA's last row
    const int nkt = t_last ? nk1 : nk0;
    const bool tail = nkt * kTcKeys > L;               // the last key tile runs past the context

    if (threadIdx.x == 0) {
        for (int k = 0; k < kTcStages; ++k) {
            mbar_init(bar(kKvFull + k), 1);
            mbar_init(bar(kKvEmpty + k), kTcTiles);   // one commit per issuer and key tile
        }
        for (int t = 0; t < kTcTiles; ++t)
            for (int b = 0; b < 2; ++b) {
                mbar_init(bar(bar_s(t, b)), 1);
                mbar_init(bar(bar_p(t, b)), kTcRows / 32);   // one arrival per softmax warp
                mbar_init(bar(bar_o(t, b)), 1);
            }
        mbar_init(bar(kQFull), kTcTiles * kTcRows / 32);
        mbar_init(bar(kDone), kTcTiles);
        mbar_init(bar(kVZero), kTcRows / 32);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(base + Ly::kTmemSlot, kTcTiles * kTmemTile);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + Ly::kTmemSlot);

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // Lane 0 waits for a free stage and arms its barrier with the tile's
        // bytes; then one lane per (box, column block, operand) issues that copy
        // (a single thread issuing all of a tile's copies took about 100 cycles
        // each, most of a key tile's period at D = 128).
        if (lane == 0) {
            tma_prefetch_descriptor(&kmap);
            tma_prefetch_descriptor(&vmap);
        }
        // the pools as the kernels before this one left them (launched as
        // the programmatic dependent of an append that may still be running)
        grid_dependency_wait();
        const int32_t *table = p.block_tables + size_t(s) * p.max_blocks;
        const int rows_per_box = B >= 16 ? 16 : 8;
        // this lane's copy: box i (rows_per_box keys), column block sl, operand op
        constexpr int kCopies = 2 * Ly::kSlabs;              // per box
        const int ci = lane / kCopies, csl = (lane / 2) % Ly::kSlabs, cop = lane & 1;
        int armed = 0;
        bool ok = true;
        for (int j = 0; j < nkt; ++j) {
            const int st = j % kTcStages;
            const int k0 = j * kTcKeys;
            const int present = min(kTcKeys, L - k0);
            const int boxes = (present + rows_per_box - 1) / rows_per_box;
            const bool mine = ci < boxes && ci < kTcKeys / 8;
            // the lane's block id first, while the slot may still be busy
            int pb = mine ? __ldg(table + ((k0 + rows_per_box * ci) >> p.log2_block)) : 0;
            bool got = true;
            if (lane == 0) {
                got = !*abort_flag &&
                      mbar_wait(bar(kKvEmpty + st), uint32_t((j / kTcStages) & 1) ^ 1u, p.err);
                if (got)
                    mbar_arrive_expect_tx(bar(kKvFull + st),
                                          uint32_t(boxes * Ly::kSlabs * rows_per_box * 128 * 2));
            }
            // the arming is ordered before every lane's copy by the warp barrier
            __syncwarp();
            if (!__shfl_sync(kAll, got ? 1 : 0, 0)) {
                ok = false;
                break;
            }
            if (mine) {
                if (pb < 0 || pb >= p.num_blocks) {
                    atomicOr(p.err, PAGEDKV_DEVERR_BLOCK_ID);
                    pb = 0;
                }
                const int z = pb * B + ((k0 + rows_per_box * ci) & (B - 1));
                const uint32_t dst = base + Ly::kKv + st * Ly::kStage + uint32_t(cop) * Ly::kHalf +
                                     csl * Ly::kKvSlab + ci * rows_per_box * 128;
                tma_load_4d(dst, cop ? &vmap : &kmap, 0, z, csl, h, bar(kKvFull + st));
            }
            ++armed;
        }
        if (!ok && lane == 0) {
            // stop everyone, then wait (bounded) for this CTA's copies still in flight
            *abort_flag = 1;
            const int first = armed > kTcStages ? armed - kTcStages : 0;
            for (int k = first; k < armed; ++k)
                mbar_wait(bar(kKvFull + k % kTcStages), uint32_t((k / kTcStages) & 1), p.err);
        }
        __syncwarp();
    } else if (warp == 1 || warp == kIssuer1Warp) {
        // ------------------------------------------------------- MMA issuers
        // One thread per Q tile issues that tile's MMAs. A thread that issues
        // tcgen05.mma runs only about two MMAs ahead of the tensor core, so
        // every wait of an issuing thread is idle tensor time; with one issuer
        // per tile, one tile's MMAs go in while the other's issuer waits.
        if (lane == 0) {
            const int t = warp == 1 ? 0 : 1;
            const int nk = nkt_of(t);
            constexpr uint32_t kIdS = tc_idesc_f16(kBf16, false, kTcRows, kTcKeys);
            constexpr uint32_t kIdO = tc_idesc_f16(kBf16, true, kTcRows, D);
            auto wait = [&](int i, int phase) {
                return !*abort_flag && mbar_wait(bar(i), uint32_t(phase & 1), p.err);
            };
            const uint32_t qb = base + Ly::kQ + t * Ly::kQTile;
            auto issue_s = [&](int j) {
                const uint32_t kb = base + Ly::kKv + (j % kTcStages) * Ly::kStage;
                const uint32_t d = tmem + uint32_t(t * kTmemTile + (j & 1) * kTcKeys);
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t a = tc_desc_sw128(qb + (kk >> 2) * Ly::kQSlab + (kk & 3) * 32, 16, 1024);
                    const uint64_t b = tc_desc_sw128(kb + (kk >> 2) * Ly::kKvSlab + (kk & 3) * 32, 16, 1024);
                    tc_mma_f16(d, a, b, kIdS, kk > 0 ? 1u : 0u);
                }
                tc_commit(bar(bar_s(t, j & 1)));
            };
            auto issue_pv = [&](int j) {
                const uint32_t vb = base + Ly::kKv + (j % kTcStages) * Ly::kStage + Ly::kHalf;
                // P of key tile j: the first 32 columns of S buffer j & 1 (16 keys per 8 columns)
                const uint32_t pa = tmem + uint32_t(t * kTmemTile + (j & 1) * kTcKeys);
                const uint32_t d = tmem + uint32_t(t * kTmemTile + 2 * kTcKeys);
#pragma unroll
                for (int kk = 0; kk < kTcKeys / 16; ++kk) {
                    const uint64_t b = tc_desc_sw128(vb + kk * 2048, Ly::kKvSlab, 1024);
                    tc_mma_f16_tmem_a(d, pa + uint32_t(8 * kk), b, kIdO, (j > 0 || kk > 0) ? 1u : 0u);
                }
                tc_commit(bar(bar_o(t, j & 1)));
            };
            bool ok = wait(kQFull, 0);
            for (int j = 0; ok && j < 2 && j < nk; ++j) {
                ok = wait(kKvFull + j % kTcStages, j / kTcStages);
                if (!ok) break;
                tc_fence_after_sync();
                issue_s(j);
            }
            for (int j = 0; ok && j < nkt; ++j) {
                if (j < nk) {
                    // the last key tile's V rows past the context are zeroed by the
                    // last Q tile's softmax: no P V may read that tile before
                    if (tail && j == nkt - 1) ok = wait(kVZero, 0);
                    if (ok) ok = wait(bar_p(t, j & 1), j >> 1);
                    if (!ok) break;
                    tc_fence_after_sync();
                    issue_pv(j);
                    // the stage of key tile j is free once this P V (the last MMA of
                    // this thread that reads it) completes: release it before this
                    // thread blocks on issuing the next S, so that the producer
                    // refills it a whole S earlier
                    tc_commit(bar(kKvEmpty + j % kTcStages));
                    // this tile's S two key tiles ahead (its S buffer j & 1 is free
                    // once the P V just issued has read P)
                    if (j + 2 < nk) {
                        ok = wait(kKvFull + (j + 2) % kTcStages, (j + 2) / kTcStages);
                        if (!ok) break;
                        tc_fence_after_sync();
                        issue_s(j + 2);
                    }
                } else {
                    // a key tile this Q tile skips: its stage may be released only
                    // after it landed (the arrival belongs to this phase of the slot)
                    ok = wait(kKvFull + j % kTcStages, j / kTcStages);
                    if (!ok) break;
                    tc_commit(bar(kKvEmpty + j % kTcStages));
                }
            }
            if (!ok) *abort_flag = 1;
            // every MMA of both issuers has completed before tensor memory is freed
            tc_commit(bar(kDone));
            mbar_wait(bar(kDone), 0, p.err);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int t = (warp - 2) >> 2;                 // Q tile of this warp
        const int quarter = warp & 3;                  // tensor-memory lanes this warp may read
        const int r = 32 * quarter + lane;             // row within the Q tile
        const int R = t * kTcRows + r;                 // row within the CTA
        const uint32_t trow = tmem + (uint32_t(32 * quarter) << 16) + uint32_t(t * kTmemTile);
        const uint32_t otile = trow + uint32_t(2 * kTcKeys);
        const int pos = R < rows ? pos0 + R / g : -1;
        const int nk = nkt_of(t);
        const size_t qrow = size_t(q0 + j0 + (R < rows ? R / g : 0)) * p.n_q_heads + h * g +
                            (R < rows ? R % g : 0);
        {
            const uint4 *src = reinterpret_cast<const uint4 *>(reinterpret_cast<const T *>(p.q) + qrow * D);
            const uint32_t qdst = base + Ly::kQ + t * Ly::kQTile + r * 128;
#pragma unroll
            for (int c = 0; c < D / 8; ++c) {
                const uint4 v = R < rows ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
                sts128(qdst + (c >> 3) * Ly::kQSlab + (((c & 7) ^ (r & 7)) << 4), v);
            }
            // every lane's stores are ordered for the tensor core's (async proxy)
            // reads by its own fence; after the warp barrier one lane arrives
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(kQFull));
        }
        float ref = -INFINITY;   // reference maximum (base 2) that P and O are relative to
        float l = 0.f;
        bool ok = true;

        for (int j = 0; j < nk; ++j) {
            const int b = j & 1;
            bool got = !*abort_flag && mbar_wait(bar(bar_s(t, b)), uint32_t((j >> 1) & 1), p.err);
            if (!__all_sync(kAll, got)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            float sc[kTcKeys];
            tmem_ld64(trow + uint32_t(b * kTcKeys), sc);
            const int k0 = j * kTcKeys;
            if (k0 + kTcKeys - 1 > pos) {
#pragma unroll
                for (int i = 0; i < kTcKeys; ++i) sc[i] = k0 + i <= pos ? sc[i] : -INFINITY;
            }
            float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int i = 0; i < kTcKeys; i += 8) {
                m4[0] = fmax3(m4[0], sc[i], sc[i + 1]);
                m4[1] = fmax3(m4[1], sc[i + 2], sc[i + 3]);
                m4[2] = fmax3(m4[2], sc[i + 4], sc[i + 5]);
                m4[3] = fmax3(m4[3], sc[i + 6], sc[i + 7]);
            }
            const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * p.scale_log2;
            const bool move = mx > ref + kRescaleLog2;
            const float alpha = move ? fast_exp2(ref - mx) : 1.f;   // 0 while no key was seen
            if (move) ref = mx;
            if (j > 0 && __any_sync(kAll, move)) {
                // rescale this warp's rows of O (every earlier P V has completed first)
                got = !*abort_flag &&
                      mbar_wait(bar(bar_o(t, (j - 1) & 1)), uint32_t(((j - 1) >> 1) & 1), p.err);
                if (!__all_sync(kAll, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float v[32];
                    tmem_ld32(otile + uint32_t(32 * c), v);
#pragma unroll
                    for (int x = 0; x < 32; ++x) v[x] *= alpha;
                    tmem_st32(otile + uint32_t(32 * c), v);
                }
            }
            const float nu = ref == -INFINITY ? 0.f : -ref;
            float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int i = 0; i < kTcKeys; i += 2) {
                ffma2(sc[i], sc[i + 1], p.scale_log2, nu);
                sc[i] = fast_exp2(sc[i]);
                sc[i + 1] = fast_exp2(sc[i + 1]);
                if (i & 2) fadd2(s4[2], s4[3], sc[i], sc[i + 1]);
                else fadd2(s4[0], s4[1], sc[i], sc[i + 1]);
            }
            l = l * alpha + ((s4[0] + s4[1]) + (s4[2] + s4[3]));
            if (tail && t == t_last && j == nkt - 1) {
                // keys past the context: zero their V rows once the tile has landed
                got = !*abort_flag &&
                      mbar_wait(bar(kKvFull + j % kTcStages), uint32_t((j / kTcStages) & 1), p.err);
                if (!__all_sync(kAll, got)) {
                    ok = false;
                    break;
                }
                if (r < kTcKeys && k0 + r >= L) {
                    const uint32_t vrow = base + Ly::kKv + (j % kTcStages) * Ly::kStage + Ly::kHalf + r * 128;
#pragma unroll
                    for (int sl = 0; sl < Ly::kSlabs; ++sl)
#pragma unroll
                        for (int c = 0; c < 8; ++c)
                            sts128(vrow + sl * Ly::kKvSlab + c * 16, make_uint4(0u, 0u, 0u, 0u));
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kVZero));
            }
            uint32_t pk[kTcKeys / 2];
#pragma unroll
            for (int c = 0; c < kTcKeys / 2; ++c) pk[c] = Elem<T>::pack2(sc[2 * c], sc[2 * c + 1]);
            tmem_st32u(trow + uint32_t(b * kTcKeys), pk);
            // each lane's tensor-memory store has completed (tmem_st32u waits) and is
            // ordered before the warp barrier; then one lane arrives for the warp
            tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(bar_p(t, b)));
        }
        if (ok && nk > 0) {
            // the last P V's completion covers every earlier MMA of the issuing thread
            const bool got = !*abort_flag &&
                             mbar_wait(bar(bar_o(t, (nk - 1) & 1)), uint32_t(((nk - 1) >> 1) & 1), p.err);
            ok = __all_sync(kAll, got);
        }
        if (!ok) {
            *abort_flag = 1;
        } else if (nk > 0) {
            tc_fence_after_sync();
            const float inv = l > 0.f ? 1.f / l : 0.f;
            uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<T *>(p.out) + qrow * D);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float v[32];
                tmem_ld32(otile + uint32_t(32 * c), v);
                if (R < rows) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        uint4 w;
                        w.x = Elem<T>::pack2(v[8 * e + 0] * inv, v[8 * e + 1] * inv);
                        w.y = Elem<T>::pack2(v[8 * e + 2] * inv, v[8 * e + 3] * inv);
                        w.z = Elem<T>::pack2(v[8 * e + 4] * inv, v[8 * e + 5] * inv);
                        w.w = Elem<T>::pack2(v[8 * e + 6] * inv, v[8 * e + 7] * inv);
                        dst[4 * c + e] = w;
                    }
                }
            }
        }
    }

    // ---- every role is done: release the tensor memory
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTcTiles * kTmemTile);
    }
}

int prefill_tc_smem_bytes(int head_dim) {
    return (head_dim == 64 ? TcLayout<64>::kTotal : TcLayout<128>::kTotal) + 1024;
}

template <typename T, int D>
static cudaError_t launch_tc_instance(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                      const PrefillParams &p, int max_query_len,
                                      cudaStream_t stream) {
    auto kernel = paged_prefill_tc_kernel<T, D>;
    const int smem = TcLayout<D>::kTotal + 1024;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::atomic<unsigned long long> opened[kLaunchCacheDevices];
    e = open_dynamic_smem(opened, dev, kernel, smem);
    if (e != cudaSuccess) return e;
    const unsigned tiles = unsigned((max_query_len + p.tile_tokens - 1) / p.tile_tokens);
    const dim3 grid(tiles, unsigned(p.n_kv_heads), unsigned(p.num_seqs));
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = size_t(smem);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, kmap, vmap, p);
}

cudaError_t launch_prefill_tc(int dtype, int head_dim, const CUtensorMap &kmap,
                              const CUtensorMap &vmap, const PrefillParams &p, int max_query_len,
                              cudaStream_t stream) {
    const bool bf16 = dtype == PAGEDKV_BF16;
    if (head_dim == 64)
        return bf16 ? launch_tc_instance<__nv_bfloat16, 64>(kmap, vmap, p, max_query_len, stream)
                    : launch_tc_instance<__half, 64>(kmap, vmap, p, max_query_len, stream);
    return bf16 ? launch_tc_instance<__nv_bfloat16, 128>(kmap, vmap, p, max_query_len, stream)
                : launch_tc_instance<__half, 128>(kmap, vmap, p, max_query_len, stream);
}

}  // namespace pkv
