// prefill_tc.cu -- chunked-prefill attention on the fifth-generation tensor
// cores (tcgen05): the same operation as prefill.cu ("How a serving engine
// actually works", section "Prefill and decode are two different jobs": each
// query row of a chunk attends causally over its sequence's cached tokens up
// to its own position, read through the block table), with the contractions
// moved off the warp-level MMA pipe.
//
// A work item is (sequence, kv head, 2 * tq chunk tokens), held as two Q tiles
// that share every K/V tile; a Q tile holds tq = 128 / group whole tokens, its
// rows (token, query head of the group), 128 rows when the group divides 128
// (126 for groups of 3, 6 or 7: the rows past them are masked).
// The kernel is persistent: one CTA per SM works through its share of the
// items (sequences ranked by context length, dealt in bands whose direction
// alternates), and every ring, buffer and barrier phase runs on across items,
// so that an item's Q copy, first K/V tiles and first S MMAs overlap the
// previous item's last P V and epilogue. Twelve warps:
//   warp 0     producer: per 64-key tile, lane 0 waits for a free stage of a
//              four-stage ring and arms its barrier; then one lane per (16
//              keys, 64-column block, operand) looks up its block id and
//              issues that TMA box, so that each operand lands as [column
//              block][64 keys][128 B] with 128-byte swizzle (the canonical
//              layout the tensor core reads);
//   warps 1,10 MMA issuers, one per Q tile (warp 1 also allocates tensor
//              memory): the warp runs the loop and its waits, and lane 0
//              issues, for its tile, S = Q K^T into one of two S buffers in
//              tensor memory and, once the softmax has written P, O += P V
//              with P read from tensor memory, into the O accumulator that
//              stays in tensor memory for the whole key loop; completions are
//              tracked by tcgen05.commit on mbarriers. An issuing thread runs
//              only about two MMAs ahead of the tensor core, so each of its
//              waits leaves the tensor core idle unless the other tile's
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
//              Between items a tile's warps write out the item's rows from O,
//              before their first P of the next item (so the issuer's wait for
//              that P also frees O for the item's first P V);
//   warp 11    copies each item's Q tiles by TMA as soon as every S of the
//              item before has completed (about two key tiles before the
//              softmax warps finish it), and zeroes the V rows past a context
//              (below).
// V rows past the context are zeroed in shared memory before any P V reads
// them (the tensor core would turn 0 * NaN into NaN): the V copies of a
// context's last key tile land on a per-stage barrier of their own, and a
// twelfth warp zeroes those rows and only then completes the stage.
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
// MMA issuer of Q tile 1, warp 11 copies Q tiles and zeroes the V rows past a
// context
constexpr int kIssuer1Warp = 2 + kTcTiles * kTcRows / 32;
constexpr int kZeroWarp = kIssuer1Warp + 1;
constexpr int kTcThreads = 32 * (kZeroWarp + 1);
constexpr int kTmemTile = 256;   // tensor-memory columns per Q tile: S, S, O
constexpr float kRescaleLog2 = 8.f;  // the reference maximum moves past 2^8

// mbarrier indices
constexpr int kKvFull = 0;
constexpr int kKvEmpty = kTcStages;
// per Q tile t: S full, P full and O full per buffer b (P V of key tile j
// completes on O barrier j & 1, so a wait never meets a barrier two
// completions away); Q full (an item's Q rows of the tile are in shared
// memory) and Q free (every S MMA of the item, the readers of Q, has
// completed). A softmax warp reads an item's O out of tensor memory before it
// writes the next item's first P, so the wait for that P also tells the
// issuer that O may start afresh.
constexpr int kPerTileBars = 8;
__device__ __forceinline__ int bar_s(int t, int b) { return 2 * kTcStages + kPerTileBars * t + b; }
__device__ __forceinline__ int bar_p(int t, int b) { return 2 * kTcStages + kPerTileBars * t + 2 + b; }
__device__ __forceinline__ int bar_o(int t, int b) { return 2 * kTcStages + kPerTileBars * t + 4 + b; }
__device__ __forceinline__ int bar_qfull(int t) { return 2 * kTcStages + kPerTileBars * t + 6; }
__device__ __forceinline__ int bar_qfree(int t) { return 2 * kTcStages + kPerTileBars * t + 7; }
constexpr int kDone = 2 * kTcStages + kPerTileBars * kTcTiles;
// per stage: the V copies of a context's last key tile land here first; the
// zeroing warp clears the V rows past the context, then completes the stage
// (one phase per such use of the stage: it is not reused before the stage
// completes and both issuers have released it)
constexpr int kTailV = kDone + 1;
constexpr int kNumBars = kTailV + kTcStages;
// key split: the CTAs share the call's key tiles (all items' tiles end to end)
// in equal contiguous ranges of r tiles, r at least min(kMinPartTiles, the
// longest item) so that an item is not cut into pieces shorter than that
// merely to reach every SM; a piece is an item's tiles within one range, and
// an item cut into several pieces leaves per-row states for the merge
constexpr int kMinPartTiles = 16;
constexpr int kMaxSplitParts = kPfMaxSplitParts;   // pieces of one item (a merge lane each)
// the split's plan in the item-order region: off[i] = key tiles of items
// before i (i = 0 .. items), then this CTA's range
constexpr int kMaxSplitItems = kPfMaxSplitItems;
constexpr int kPlanRange = 504;        // r, start, end, first item, piece count, parts layout
// sequences ranked by context length in shared memory (beyond this count the
// items keep the sequences' own order)
constexpr int kMaxRankedSeqs = 256;

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
    static constexpr int kTmemSlot = kBars + 8 * kNumBars;
    static constexpr int kFlag = kTmemSlot + 8;
    static constexpr int kOrder = kFlag + 8;               // ranked sequence ids, then their lengths
    // per softmax thread, the output row of its item (kept here through the key
    // loop; under a key split the item's part in bits 48-63), then the row's
    // reference maximum at the item's end (key split)
    static constexpr int kOutRow = kOrder + 8 * kMaxRankedSeqs;
    static constexpr int kRefRow = kOutRow + 8 * kTcTiles * kTcRows;
    static constexpr int kTotal = kRefRow + 4 * kTcTiles * kTcRows;
    static_assert(2 * kTcKeys + D <= kTmemTile, "S buffers and O must fit a Q tile's columns");
    static_assert(kMaxSplitItems < kPlanRange && 4 * (kPlanRange + 6) <= 8 * kMaxRankedSeqs,
                  "the key split's plan must fit the item-order region");
};

// Whether the barrier's phase of this parity has completed, without waiting.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                 ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

// Shared-memory word at a 32-bit shared address (a generic pointer would hold
// two registers through the softmax warps' loops).
__device__ __forceinline__ int lds32(uint32_t addr) {
    int v;
    asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void sts32(uint32_t addr, int v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// One work item: (sequence, kv head, query tile of tile_tokens chunk tokens =
// 256 rows of (chunk token, query head of the group)), held as two Q tiles.
struct PfItem {
    int s, h;
    int q0, j0, ntok, pos0, L;   // ntok: chunk tokens of the item
    int slot, kb;       // key split: the piece's state slot and its first key tile
    bool split;         // the item's keys are split (its rows leave states for the merge)
    int nk[kTcTiles];   // key tiles of Q tile t from kb: through the position of its last row
    int nkt;            // key tiles of the item from kb (the piece's range)
    bool tail;          // the item's last key tile runs past the context
};

// Items in one order shared by every CTA: sequences by decreasing context
// length (ranked, when there are few enough), within a sequence its query
// tiles from the last (the most keys), then kv heads, so that the items that
// read a sequence's K/V run close together in time and share it through L2.
// Item k of that order: fills `it` but for its key range and returns its key
// tiles N (through its last row's position), or 0 for an item with no rows or
// a sequence whose chunk or length is invalid (reported once per sequence
// when `report`).
__device__ __forceinline__ int pf_decode(const PrefillParams &p, uint32_t ranked, int tiles, int k,
                                         bool report, PfItem &it, int (&nk_all)[kTcTiles]) {
    const int per_seq = tiles * p.n_kv_heads;
    const int r = k / per_seq;
    const int rem = k - r * per_seq;
    const int s = ranked ? lds32(ranked + 4u * uint32_t(r)) : r;
    const int qt = tiles - 1 - rem / p.n_kv_heads;
    const int h = rem - (rem / p.n_kv_heads) * p.n_kv_heads;
    const int q0 = __ldg(p.query_start + s);
    const int q1 = __ldg(p.query_start + s + 1);
    const int n = q1 - q0;
    const int L = __ldg(p.context_lens + s);
    const bool rows_ok = q0 >= 0 && q1 >= q0 && q1 <= p.num_tokens && n <= tiles * p.tile_tokens;
    const bool len_ok = L >= n && L <= p.max_blocks * p.block_size;
    if (!rows_ok || !len_ok) {
        if (report && qt == tiles - 1 && h == 0)
            atomicOr(p.err, rows_ok ? PAGEDKV_DEVERR_CONTEXT_LEN : PAGEDKV_DEVERR_POSITION);
        return 0;
    }
    const int j0 = qt * p.tile_tokens;
    if (j0 >= n) return 0;
    it.s = s;
    it.h = h;
    it.q0 = q0;
    it.j0 = j0;
    it.L = L;
    it.ntok = min(p.tile_tokens, n - j0);
    it.pos0 = L - n + j0;
    // Q tile t holds the item's tokens t*tq .. t*tq + tq - 1, tq = 128 / group
    // whole tokens (all of a token's heads in one tile)
    const int tq = kTcRows / p.group;
#pragma unroll
    for (int t = 0; t < kTcTiles; ++t) {
        const int nt = min(max(it.ntok - t * tq, 0), tq);
        nk_all[t] = nt > 0 ? (it.pos0 + t * tq + nt - 1) / kTcKeys + 1 : 0;
    }
    return nk_all[kTcTiles - 1] > 0 ? nk_all[kTcTiles - 1] : nk_all[0];
}

// This CTA's m-th piece of work. Whole items: item k of the shared order
// (`order`: the ranked sequence ids, or 0). Key split: the m-th item that
// meets this CTA's range of key tiles (`order`: the plan), restricted to the
// range. Returns false for an item with no rows or no key tiles there.
template <bool kSplit>
__device__ __forceinline__ bool pf_item(const PrefillParams &p, uint32_t order, int tiles, int k,
                                        bool report, PfItem &it) {
    int nk_all[kTcTiles];
    if (!kSplit) {
        const int N = pf_decode(p, order, tiles, k, report, it, nk_all);
        if (N == 0) return false;
        it.slot = 0;
        it.kb = 0;
        it.split = false;
#pragma unroll
        for (int t = 0; t < kTcTiles; ++t) it.nk[t] = nk_all[t];
        it.nkt = N;
        it.tail = N * kTcKeys > it.L;
        return true;
    }
    const int i = lds32(order + 4u * (kPlanRange + 3)) + k;
    const int N = pf_decode(p, 0u, tiles, i, false, it, nk_all);
    if (N == 0) return false;
    const int off = lds32(order + 4u * uint32_t(i));
    const int kb = max(lds32(order + 4u * (kPlanRange + 1)) - off, 0);
    const int ke = min(lds32(order + 4u * (kPlanRange + 2)) - off, N);
    if (ke <= kb) return false;
    // a piece that starts inside the item is its CTA's first (slot 2c); one
    // that starts the item is the CTA's last, or its only one (slot 2c + 1)
    it.slot = 2 * int(blockIdx.x) + (kb > 0 ? 0 : 1);
    it.kb = kb;
    it.split = kb > 0 || ke < N;
#pragma unroll
    for (int t = 0; t < kTcTiles; ++t) it.nk[t] = max(min(nk_all[t], ke) - kb, 0);
    it.nkt = ke - kb;
    it.tail = ke == N && N * kTcKeys > it.L;
    return true;
}

// This CTA's m-th item: whole items in bands of gridDim.x items, dealt
// forwards in even bands and backwards in odd ones (so that every CTA gets a
// similar share of the ranked work; the item count fits an int, the launcher
// checks); under the key split the CTA's pieces in order.
template <bool kSplit>
__device__ __forceinline__ int pf_item_index(int m) {
    if (kSplit) return m;
    const int G = int(gridDim.x), c = int(blockIdx.x);
    return m * G + ((m & 1) ? G - 1 - c : c);
}

// Key split: the plan, alike in every CTA, in one of two layouts. off[i]
// (shared memory, i = 0 .. items) counts the key tiles of items before i
// (T in all); a piece is an item's tiles within one CTA's range [start, end).
// - Ranges: CTA c takes tiles [c r, min((c + 1) r, T)) of all items end to
//   end, r at least ceil(T / grid), long enough that no item meets more than
//   `parts` ranges (an item of N tiles meets at most ceil((N - 1) / r) + 1)
//   and at least min(kMinPartTiles, the longest item). A range can hold the
//   end of one item and the start of the next.
// - Parts (at most grid / items CTAs per item and 16, p of them): CTA c takes part
//   c % p of item c / p, whose N tiles go to min(p, ceil(N / kMinPartTiles))
//   equal parts; every CTA holds one piece at most.
// Either way an item's pieces sit in consecutive CTAs from c0. The plan takes
// the layout whose longest CTA (key tiles, plus kPieceCost per piece) is the
// shorter: parts, when the items are about equal and divide the SMs well.
// Every thread of the CTA calls it.
constexpr int kPieceCost = 4;   // a piece's fixed cost (Q copy, epilogue, merge) in key tiles
constexpr int kMaxItemParts = 16;  // CTAs per item in the parts layout at most
__device__ __forceinline__ void pf_split_plan(const PrefillParams &p, int tiles, int items, int *off,
                                              bool report) {
    for (int i = int(threadIdx.x); i < items; i += int(blockDim.x)) {
        PfItem it;
        int nk_all[kTcTiles];
        off[i + 1] = pf_decode(p, 0u, tiles, i, report, it, nk_all);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        const int lane = int(threadIdx.x);
        const int G = int(gridDim.x);
        // CTAs per item in the parts layout (0: it does not fit the grid; more
        // than 16 parts cost the merge more than their shorter key loop saves)
        const int pp = min(min(p.key_parts, kMaxItemParts), G / max(items, 1));
        // a lane per run of items: the run's sum, maximum and longest part, then the prefix
        const int per = (items + 31) / 32;
        const int lo = min(lane * per, items), hi = min(lo + per, items);
        int sum = 0, mx = 0, part_mx = 0;
        for (int i = lo; i < hi; ++i) {
            const int n = off[i + 1];
            sum += n;
            mx = max(mx, n);
            if (pp > 0) {
                const int eff = min(pp, max(1, (n + kMinPartTiles - 1) / kMinPartTiles));
                part_mx = max(part_mx, (n + eff - 1) / eff);
            }
        }
        int incl = sum;
        for (int d = 1; d < 32; d <<= 1) {
            const int y = __shfl_up_sync(kAll, incl, d);
            if (lane >= d) incl += y;
        }
        for (int d = 16; d >= 1; d >>= 1) {
            mx = max(mx, __shfl_xor_sync(kAll, mx, d));
            part_mx = max(part_mx, __shfl_xor_sync(kAll, part_mx, d));
        }
        int run = incl - sum;
        for (int i = lo; i < hi; ++i) {
            run += off[i + 1];
            off[i + 1] = run;
        }
        const int T = __shfl_sync(kAll, incl, 31);
        if (lane == 0) {
            off[0] = 0;
            int r = (T + G - 1) / G;
            if (mx > 1) r = max(r, (mx - 2) / (p.key_parts - 1) + 1);
            r = max(r, max(min(kMinPartTiles, mx), 1));
            const int c = int(blockIdx.x);
            long long start, end;
            int first, count;
            // the ranges' longest CTA: a range and two pieces (the end of one
            // item, the start of the next) unless the items are shorter
            const bool parts_layout = pp > 0 && part_mx + kPieceCost <= r + 2 * kPieceCost;
            if (parts_layout) {
                const int i = c / pp, q = c - i * pp;
                const int n = i < items ? off[i + 1] - off[i] : 0;
                const int eff = min(pp, max(1, (n + kMinPartTiles - 1) / kMinPartTiles));
                first = i;
                count = n > 0 && q < eff ? 1 : 0;
                start = count ? off[i] + (long long)n * q / eff : 0;
                end = count ? off[i] + (long long)n * (q + 1) / eff : 0;
            } else {
                start = min((long long)c * r, (long long)T);
                end = min(start + r, (long long)T);
                // the first item holding a tile at or past start, the last one
                // holding a tile before end (off is non-decreasing)
                int lo2 = 0, hi2 = items;
                while (lo2 < hi2) {
                    const int mid = (lo2 + hi2) >> 1;
                    if (off[mid + 1] > start) hi2 = mid;
                    else lo2 = mid + 1;
                }
                first = lo2;
                lo2 = first;
                hi2 = items;
                while (lo2 < hi2) {
                    const int mid = (lo2 + hi2) >> 1;
                    if (off[mid + 1] >= end) hi2 = mid;
                    else lo2 = mid + 1;
                }
                count = start < end ? lo2 - first + 1 : 0;
            }
            off[kPlanRange] = r;
            off[kPlanRange + 1] = int(start);
            off[kPlanRange + 2] = int(end);
            off[kPlanRange + 3] = first;
            off[kPlanRange + 4] = count;
            off[kPlanRange + 5] = parts_layout ? pp : 0;
        }
    }
}

}  // namespace

template <typename T, int D, bool kSplit>
__global__ void __launch_bounds__(kTcThreads, 1)
paged_prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap,
                        const __grid_constant__ CUtensorMap qmap, const PrefillParams p, int tiles) {
    using Ly = TcLayout<D>;
    constexpr bool kBf16 = Elem<T>::kBf16;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *const sm = smem_raw + (base - raw);
    const uint32_t flag = base + Ly::kFlag;   // the abort flag
    auto aborted = [&]() { return lds32(flag) != 0; };
    auto bar = [&](int i) { return base + Ly::kBars + 8u * uint32_t(i); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int B = p.block_size;
    const int g = p.group;
    const int all_items = p.num_seqs * tiles * p.n_kv_heads;

    if (threadIdx.x == 0) {
        for (int k = 0; k < kTcStages; ++k) {
            mbar_init(bar(kKvFull + k), 1);
            mbar_init(bar(kKvEmpty + k), kTcTiles);   // one commit per issuer and key tile
        }
        for (int t = 0; t < kTcTiles; ++t) {
            for (int b = 0; b < 2; ++b) {
                mbar_init(bar(bar_s(t, b)), 1);
                mbar_init(bar(bar_p(t, b)), kTcRows / 32);   // one arrival per softmax warp
                mbar_init(bar(bar_o(t, b)), 1);
            }
            mbar_init(bar(bar_qfull(t)), 1);   // the Q copy's arrival and bytes
            mbar_init(bar(bar_qfree(t)), 1);
        }
        mbar_init(bar(kDone), kTcTiles);
        for (int k = 0; k < kTcStages; ++k) mbar_init(bar(kTailV + k), 1);
        sts32(flag, 0);
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(base + Ly::kTmemSlot, kTcTiles * kTmemTile);
        tmem_relinquish();
    }
    // sequences ranked by decreasing context length (ties by index), when some
    // CTA gets more than one item; the lengths are the caller's, read before
    // any grid dependency
    // (whole items), or the key split's plan: the item order's shared address
    uint32_t order = 0;    // 0: the sequences' own order
    if (!kSplit && p.num_seqs > 1 && p.num_seqs <= kMaxRankedSeqs && all_items > int(gridDim.x)) {
        order = base + Ly::kOrder;
        int *ids = reinterpret_cast<int *>(sm + Ly::kOrder);
        int *lens = ids + kMaxRankedSeqs;
        for (int s = threadIdx.x; s < p.num_seqs; s += blockDim.x) lens[s] = __ldg(p.context_lens + s);
        __syncthreads();
        for (int s = threadIdx.x; s < p.num_seqs; s += blockDim.x) {
            const int Ls = lens[s];
            int rank = 0;
            for (int u = 0; u < p.num_seqs; ++u) {
                const int Lu = lens[u];
                rank += (Lu > Ls || (Lu == Ls && u < s)) ? 1 : 0;
            }
            ids[rank] = s;
        }
    }
    if (kSplit) {
        // (the launcher keeps the split to at most kMaxSplitItems items)
        order = base + Ly::kOrder;
        pf_split_plan(p, tiles, all_items, reinterpret_cast<int *>(sm + Ly::kOrder), blockIdx.x == 0);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(sm + Ly::kTmemSlot);
    // items (key split: this CTA's pieces) to work through
    const int num_items = kSplit ? lds32(order + 4u * (kPlanRange + 4)) : all_items;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // Per key tile, lane 0 waits for a free stage and arms its barrier;
        // then one lane per (box, column block, operand) issues that copy (a
        // single thread issuing all of a tile's copies took about 100 cycles
        // each, most of a key tile's period at D = 128). Stages run on across
        // the CTA's items, so the next item's first tiles load while the
        // current one finishes.
        if (lane == 0) {
            tma_prefetch_descriptor(&kmap);
            tma_prefetch_descriptor(&vmap);
        }
        // the pools as the kernels before this one left them (launched as
        // the programmatic dependent of an append that may still be running)
        grid_dependency_wait();
        if (kSplit && blockIdx.x == 0) {
            // for the merge, per item: the CTA c0 of its first piece (bits 0-15)
            // and its piece count (bits 16-31; fewer than 2: not split); written
            // once the grids before this one are done with the workspace
            const int *off = reinterpret_cast<const int *>(sm + Ly::kOrder);
            const int r = off[kPlanRange], pp = off[kPlanRange + 5];
            for (int i = lane; i < all_items; i += 32) {
                const int o = off[i], n = off[i + 1] - o;
                int c0 = 0, pieces = 0;
                if (n > 0 && pp > 0) {
                    c0 = i * pp;
                    pieces = min(pp, max(1, (n + kMinPartTiles - 1) / kMinPartTiles));
                } else if (n > 0) {
                    c0 = o / r;
                    pieces = (o + n - 1) / r - c0 + 1;
                }
                p.ws_plan[i] = c0 | (pieces << 16);
            }
        }
        const int rows_per_box = B >= 16 ? 16 : 8;
        // this lane's copy: box ci (rows_per_box keys), column block csl, operand cop
        constexpr int kCopies = 2 * Ly::kSlabs;              // per box
        const int ci = lane / kCopies, csl = (lane / 2) % Ly::kSlabs, cop = lane & 1;
        int kt = 0;          // key tiles armed before this item (position in the ring)
        int armed = 0;
        bool ok = true;
        for (int m = 0; ok; ++m) {
            const int k = pf_item_index<kSplit>(m);
            if (k >= num_items) break;
            PfItem it;
            if (!pf_item<kSplit>(p, order, tiles, k, lane == 0, it)) continue;
            const int32_t *table = p.block_tables + size_t(it.s) * p.max_blocks;
            for (int j = 0; j < it.nkt; ++j) {
                const int gk = kt + j;
                const int st = gk % kTcStages;
                const int k0 = (it.kb + j) * kTcKeys;
                const int present = min(kTcKeys, it.L - k0);
                const int boxes = (present + rows_per_box - 1) / rows_per_box;
                const bool last_tail = it.tail && j == it.nkt - 1;
                const bool mine = ci < boxes && ci < kTcKeys / 8;
                // the lane's block id first, while the slot may still be busy
                int pb = mine ? __ldg(table + ((k0 + rows_per_box * ci) >> p.log2_block)) : 0;
                const uint32_t half = uint32_t(boxes * Ly::kSlabs * rows_per_box * 128);
                bool got = true;
                if (lane == 0) {
                    got = !aborted() &&
                          mbar_wait(bar(kKvEmpty + st), uint32_t((gk / kTcStages) & 1) ^ 1u, p.err);
                    if (got && !last_tail) {
                        mbar_arrive_expect_tx(bar(kKvFull + st), 2 * half);
                    } else if (got) {
                        // K completes on the stage's barrier, whose arrival comes from
                        // the zeroing warp once the V rows past the context are zero;
                        // V lands on the stage's tail barrier
                        mbar_expect_tx(bar(kKvFull + st), half);
                        mbar_arrive_expect_tx(bar(kTailV + st), half);
                    }
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
                    const uint32_t done = (cop && last_tail) ? bar(kTailV + st) : bar(kKvFull + st);
                    tma_load_4d(dst, cop ? &vmap : &kmap, 0, z, csl, it.h, done);
                }
                ++armed;
            }
            kt += it.nkt;
        }
        if (!ok && lane == 0) {
            // stop everyone, then wait (bounded) for this CTA's copies still in flight
            // (a tail stage completes only with the zeroing warp's arrival: when that
            // warp stopped too, the wait ends at its time limit, its copies long done)
            sts32(flag, 1);
            const int first = armed > kTcStages ? armed - kTcStages : 0;
            for (int x = first; x < armed; ++x)
                mbar_wait(bar(kKvFull + x % kTcStages), uint32_t((x / kTcStages) & 1), p.err);
        }
        __syncwarp();
    } else if (warp == kZeroWarp) {
        // ------------------------------------------------ Q copies and V tails
        // Q: lane 0 copies each Q tile of an item with one TMA box per
        // 64-column block ([tq = 128/g whole tokens][g heads][64 columns],
        // which lands as the tile's first tq*g rows (token, head) in the
        // swizzled layout the tensor core reads; the rows past them, when g
        // does not divide 128, hold whatever they held: the softmax masks every
        // key of such a row), as soon as every S MMA of the item
        // before has completed: about two key tiles before the softmax warps
        // finish that item, so the copy is off their path.
        // V: the rows past a context (never written for the sequence, or left
        // in the stage by an earlier tile) become zeros once the tile's V
        // copies have landed: the tensor core would turn 0 * NaN into NaN.
        // Then the stage is complete (its K copies may still be landing). The
        // issuers reach that tile's S two key tiles ahead of its P V, which
        // hides the wait. An item's Q copies go first: its S MMAs, which the
        // item's last stage waits for, need them.
        if (lane == 0) tma_prefetch_descriptor(&qmap);
        // key split: the merge that follows on the stream may launch now (it
        // waits for this grid before it reads the states or exits; should this
        // warp's signal not count for the CTA, it launches at the grid's end)
        if (kSplit) grid_launch_dependents();
        const int tq = kTcRows / g;
        int kt = 0;
        int i = 0;
        // per Q tile, the last item that took a phase of its Q full barrier (a
        // copy or a plain arrival): each phase waits for the one before to be
        // consumed, so that phase is the only one that may still be pending
        int qlast[kTcTiles] = {-1, -1};
        uint32_t parity = 0;   // bit st: phase parity of stage st's tail barrier
        bool ok = true;
        for (int m = 0; ok; ++m) {
            const int k = pf_item_index<kSplit>(m);
            if (k >= num_items) break;
            PfItem it;
            if (!pf_item<kSplit>(p, order, tiles, k, false, it)) continue;
            {
                bool got = true;
                if (lane == 0) {
#pragma unroll
                    for (int t = 0; t < kTcTiles; ++t) {
                        if (i > 0) got = got && !aborted() &&
                                         mbar_wait(bar(bar_qfree(t)), uint32_t((i - 1) & 1), p.err);
                        if (!got) break;
                        if (it.nk[t] > 0) {
                            const uint32_t full = bar(bar_qfull(t));
                            mbar_arrive_expect_tx(full, uint32_t(Ly::kSlabs * tq * g * 128));
                            // rows past the item are another sequence's tokens, or zeros past
                            // the last token: the softmax masks every key of such a row
                            const int tok = it.q0 + it.j0 + t * tq;
                            for (int sl = 0; sl < Ly::kSlabs; ++sl)
                                tma_load_4d(base + Ly::kQ + t * Ly::kQTile + sl * Ly::kQSlab, &qmap, 0, sl,
                                            it.h * g, tok, full);
                        } else {
                            // no row of this tile: the issuer still takes the phase
                            mbar_arrive(bar(bar_qfull(t)));
                        }
                        qlast[t] = i;
                    }
                }
                if (!__shfl_sync(kAll, got ? 1 : 0, 0)) {
                    ok = false;
                    break;
                }
            }
            if (it.tail) {
                const int st = (kt + it.nkt - 1) % kTcStages;
                const int present = it.L - (it.kb + it.nkt - 1) * kTcKeys;
                bool got = true;
                if (lane == 0)
                    got = !aborted() && mbar_wait(bar(kTailV + st), (parity >> st) & 1u, p.err);
                if (!__shfl_sync(kAll, got ? 1 : 0, 0)) {
                    ok = false;
                    break;
                }
                parity ^= 1u << st;
                const uint32_t vbase = base + Ly::kKv + st * Ly::kStage + Ly::kHalf;
                for (int x = lane; x < (kTcKeys - present) * Ly::kSlabs * 8; x += 32) {
                    const int r = present + x / (Ly::kSlabs * 8);
                    const int sl = (x / 8) % Ly::kSlabs;
                    sts128(vbase + sl * Ly::kKvSlab + r * 128 + (x & 7) * 16, make_uint4(0u, 0u, 0u, 0u));
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(kKvFull + st));
            }
            kt += it.nkt;
            ++i;
        }
        if (lane == 0) {
            if (!ok) sts32(flag, 1);
            // this CTA's Q copies have landed before it may exit (a bounded
            // wait; the issuers have waited for them unless the CTA stopped)
#pragma unroll
            for (int t = 0; t < kTcTiles; ++t)
                if (qlast[t] >= 0) mbar_wait(bar(bar_qfull(t)), uint32_t(qlast[t] & 1), p.err);
        }
        __syncwarp();
    } else if (warp == 1 || warp == kIssuer1Warp) {
        // ------------------------------------------------------- MMA issuers
        // One warp per Q tile issues that tile's MMAs. A thread that issues
        // tcgen05.mma runs only about two MMAs ahead of the tensor core, so
        // every wait of an issuing warp is idle tensor time; with one issuer
        // per tile, one tile's MMAs go in while the other's issuer waits. The
        // whole warp runs the loop and its waits (so that the descriptors and
        // addresses are warp-uniform values), and lane 0 alone issues each
        // tcgen05.mma and tcgen05.commit (a commit tracks its own thread's MMAs).
        {
            const int t = warp == 1 ? 0 : 1;
            const bool leader = lane == 0;
            constexpr uint32_t kIdS = tc_idesc_f16(kBf16, false, kTcRows, kTcKeys);
            constexpr uint32_t kIdO = tc_idesc_f16(kBf16, true, kTcRows, D);
            // every lane waits; the warp goes on only if all of them saw the phase
            // (a phase already complete passes at once; the abort flag is read only
            // when the lane has to wait)
            auto wait = [&](int i, int phase) {
                bool got = mbar_try_wait(bar(i), uint32_t(phase & 1));
                if (!got) got = !aborted() && mbar_wait(bar(i), uint32_t(phase & 1), p.err);
                return __all_sync(kAll, got);
            };
            auto commit = [&](int i) {
                if (leader) tc_commit(bar(i));
            };
            // The issuing warp shares its SM sub-partition with two softmax warps,
            // so every instruction it spends per MMA slows the MMAs' issue: the
            // shared-memory descriptors are built once (Q's for the whole kernel,
            // a stage's per use) and a K step only offsets a descriptor's start
            // address, a constant once the loop is unrolled.
            const uint32_t qb = base + Ly::kQ + t * Ly::kQTile;
            uint64_t qdesc[D / 16];
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
                qdesc[kk] = tc_desc_sw128(qb + (kk >> 2) * Ly::kQSlab + (kk & 3) * 32, 16, 1024);
            // S of key tile gk of the ring (gj-th key tile of this Q tile) into S buffer gj & 1
            auto issue_s = [&](int gk, int gj) {
                const uint64_t kdesc = tc_desc_sw128(base + Ly::kKv + (gk % kTcStages) * Ly::kStage, 16, 1024);
                const uint32_t d = tmem + uint32_t(t * kTmemTile + (gj & 1) * kTcKeys);
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        // (start addresses stay below 2^18 bytes: the offset never carries
                        // out of the descriptor's 14-bit address field)
                        const uint64_t b = kdesc + uint64_t(((kk >> 2) * Ly::kKvSlab + (kk & 3) * 32) >> 4);
                        tc_mma_f16(d, qdesc[kk], b, kIdS, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(bar(bar_s(t, gj & 1)));
                }
            };
            // O (+)= P V; `first` starts the item's accumulator
            auto issue_pv = [&](int gk, int gj, bool first) {
                const uint64_t vdesc =
                    tc_desc_sw128(base + Ly::kKv + (gk % kTcStages) * Ly::kStage + Ly::kHalf, Ly::kKvSlab, 1024);
                // P: the first 32 columns of S buffer gj & 1 (16 keys per 8 columns)
                const uint32_t pa = tmem + uint32_t(t * kTmemTile + (gj & 1) * kTcKeys);
                const uint32_t d = tmem + uint32_t(t * kTmemTile + 2 * kTcKeys);
                if (leader) {
#pragma unroll
                    for (int kk = 0; kk < kTcKeys / 16; ++kk)
                        tc_mma_f16_tmem_a(d, pa + uint32_t(8 * kk), vdesc + uint64_t((kk * 2048) >> 4), kIdO,
                                          (!first || kk > 0) ? 1u : 0u);
                    tc_commit(bar(bar_o(t, gj & 1)));
                }
            };
            int kt = 0;   // ring position of the item's first key tile
            int jt = 0;   // key tiles of this Q tile before the item (S, P and O barrier phases)
            int i = 0;    // items so far
            bool ok = true;
            for (int m = 0; ok; ++m) {
                const int k = pf_item_index<kSplit>(m);
                if (k >= num_items) break;
                PfItem it;
                if (!pf_item<kSplit>(p, order, tiles, k, false, it)) continue;
                const int nk = it.nk[t];
                // the item's Q rows of this tile are in shared memory
                ok = wait(bar_qfull(t), i);
                if (!ok) break;
                if (nk > 0) {
                    for (int j = 0; ok && j < 2 && j < nk; ++j) {
                        ok = wait(kKvFull + (kt + j) % kTcStages, (kt + j) / kTcStages);
                        if (!ok) break;
                        tc_fence_after_sync();
                        issue_s(kt + j, jt + j);
                    }
                    if (!ok) break;
                    // Q may be overwritten once the item's last S has completed
                    if (nk <= 2) commit(bar_qfree(t));
                }
                for (int j = 0; ok && j < it.nkt; ++j) {
                    const int gk = kt + j;
                    if (j < nk) {
                        // P of key tile j (the first P of an item comes after the softmax
                        // warps have read the previous item's O: its P V may start O
                        // afresh); beside it, without blocking, whether the K/V of key
                        // tile j + 2 has landed, so that the P V and the S go in as one run
                        // (a check between them, with both issuers making it at the same
                        // time, left the tensor core idle for hundreds of cycles per key
                        // tile). Only when the K/V is not there yet (an item's first key
                        // tiles) does the warp wait for it, after the P V
                        ok = wait(bar_p(t, (jt + j) & 1), (jt + j) >> 1);
                        const bool ahead = j + 2 < nk;
                        const int gk2 = gk + 2;
                        const bool kv_in = __all_sync(
                            kAll, ok && ahead &&
                                      mbar_test_wait(bar(kKvFull + gk2 % kTcStages), uint32_t((gk2 / kTcStages) & 1)));
                        if (!ok) break;
                        tc_fence_after_sync();
                        issue_pv(gk, jt + j, j == 0);
                        // the stage of key tile j is free once this P V (the last MMA of
                        // this thread that reads it) completes
                        commit(kKvEmpty + gk % kTcStages);
                        // this tile's S two key tiles ahead (its S buffer is free once the
                        // P V just issued has read P)
                        if (ahead) {
                            if (!kv_in) {
                                ok = wait(kKvFull + gk2 % kTcStages, gk2 / kTcStages);
                                if (!ok) break;
                                tc_fence_after_sync();
                            }
                            issue_s(gk2, jt + j + 2);
                            if (j + 2 == nk - 1) commit(bar_qfree(t));
                        }
                    } else {
                        // a key tile this Q tile skips: its stage may be released only
                        // after it landed (the arrival belongs to this phase of the slot)
                        ok = wait(kKvFull + gk % kTcStages, gk / kTcStages);
                        if (!ok) break;
                        commit(kKvEmpty + gk % kTcStages);
                    }
                }
                if (!ok) break;
                // no MMA of this tile reads Q in this item: Q is free at once
                if (nk == 0 && leader) mbar_arrive(bar(bar_qfree(t)));
                kt += it.nkt;
                jt += nk;
                ++i;
            }
            if (leader) {
                if (!ok) sts32(flag, 1);
                // every MMA of both issuers has completed before tensor memory is freed
                tc_commit(bar(kDone));
                mbar_wait(bar(kDone), 0, p.err);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int t = (warp - 2) >> 2;                 // Q tile of this warp
        const int quarter = warp & 3;                  // tensor-memory lanes this warp may read
        const int r = 32 * quarter + lane;             // row within the Q tile
        const int R = t * kTcRows + r;                 // row slot within the item
        const int tq = kTcRows / g;                    // whole tokens per Q tile
        const uint32_t trow = tmem + (uint32_t(32 * quarter) << 16) + uint32_t(t * kTmemTile);
        const uint32_t otile = trow + uint32_t(2 * kTcKeys);
        bool ok = true;
        // the previous item's results, stored once its O is complete (while this
        // tile's MMAs of the next item already run); its output row waits in
        // shared memory (all ones: a row past the item)
        const uint32_t out_row = base + Ly::kOutRow + 8u * uint32_t(R);
        const uint32_t ref_row = base + Ly::kRefRow + 4u * uint32_t(R);
        int prev_nk = 0, prev_jend = 0;
        float prev_l = 0.f;
        auto epilogue = [&]() -> bool {
            const unsigned long long v_row = (unsigned long long)(unsigned)lds32(out_row) |
                                             ((unsigned long long)(unsigned)lds32(out_row + 4) << 32);
            const bool prev_row = v_row != ~0ull;
            const unsigned long long prev_qrow = prev_row ? v_row & ((1ull << 48) - 1) : 0ull;
            const bool split = kSplit && prev_row && ((v_row >> 62) & 1ull);
            // key split: every row of the item leaves its piece's state in the
            // piece's slot, m = -inf when the piece held none of its keys (its O
            // is then not written)
            const size_t wrow = size_t((v_row >> 48) & 0x3fffull) * size_t(kTcTiles * kTcRows) + size_t(R);
            if (split && prev_row) {
                p.ws_m[wrow] = prev_nk > 0 ? __int_as_float(lds32(ref_row)) : -INFINITY;
                p.ws_l[wrow] = prev_nk > 0 ? prev_l : 0.f;
            }
            if (prev_nk == 0) return true;
            // the last P V's completion covers every earlier MMA of the issuing thread
            const int e = prev_jend - 1;
            const bool got = !aborted() && mbar_wait(bar(bar_o(t, e & 1)), uint32_t((e >> 1) & 1), p.err);
            if (!__all_sync(kAll, got)) return false;
            tc_fence_after_sync();
            // the row normalised into `out`, or (key split) its part's O as it is
            const float inv = prev_l > 0.f ? 1.f / prev_l : 0.f;
            const bool keep = prev_row && (!split || prev_l > 0.f);
            uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<T *>(p.out) + prev_qrow * D);
            float4 *wo = reinterpret_cast<float4 *>(p.ws_o + wrow * D);
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                float v[32];
                tmem_ld32(otile + uint32_t(32 * c), v);
                if (keep && split) {
#pragma unroll
                    for (int e4 = 0; e4 < 8; ++e4)
                        wo[8 * c + e4] = make_float4(v[4 * e4], v[4 * e4 + 1], v[4 * e4 + 2], v[4 * e4 + 3]);
                } else if (keep) {
#pragma unroll
                    for (int e4 = 0; e4 < 4; ++e4) {
                        uint4 w;
                        w.x = Elem<T>::pack2(v[8 * e4 + 0] * inv, v[8 * e4 + 1] * inv);
                        w.y = Elem<T>::pack2(v[8 * e4 + 2] * inv, v[8 * e4 + 3] * inv);
                        w.z = Elem<T>::pack2(v[8 * e4 + 4] * inv, v[8 * e4 + 5] * inv);
                        w.w = Elem<T>::pack2(v[8 * e4 + 6] * inv, v[8 * e4 + 7] * inv);
                        dst[4 * c + e4] = w;
                    }
                }
            }
            return true;
        };
        int jt = 0;   // key tiles of this Q tile before the item
        int i = 0;
        for (int m = 0; ok; ++m) {
            const int k = pf_item_index<kSplit>(m);
            if (k >= num_items) break;
            PfItem it;
            if (!pf_item<kSplit>(p, order, tiles, k, false, it)) continue;
            const int nk = it.nk[t];
            // this thread's row: token tok of the item (t*tq + r/g), head r%g of the
            // group; none past the tile's tq*g rows or the item's tokens
            const int tok = t * tq + r / g;
            const bool row = r < tq * g && tok < it.ntok;
            const int pos = row ? it.pos0 + tok : -1;
            const unsigned long long qrow =
                (unsigned long long)(it.q0 + it.j0 + (row ? tok : 0)) * p.n_q_heads + it.h * g + (row ? r % g : 0);
            // the previous item's output (its tensor-memory loads complete before
            // this warp's next arrival on a P barrier, which lets O be overwritten)
            if (i > 0 && !epilogue()) {
                ok = false;
                break;
            }
            {
                // (a piece of a split item: its slot in bits 48-61, bit 62 set)
                const unsigned long long v =
                    row ? (kSplit ? qrow | ((unsigned long long)it.slot << 48) | (it.split ? 1ull << 62 : 0ull) : qrow)
                        : ~0ull;
                sts32(out_row, int(unsigned(v)));
                sts32(out_row + 4, int(unsigned(v >> 32)));
            }
            float ref = -INFINITY;   // reference maximum (base 2) that P and O are relative to
            float l = 0.f;
            for (int j = 0; j < nk; ++j) {
                const int gj = jt + j;
                const int b = gj & 1;
                // (a phase already complete passes at once; the abort flag is read
                // only when the warp has to wait)
                bool got = mbar_try_wait(bar(bar_s(t, b)), uint32_t((gj >> 1) & 1));
                if (!got) got = !aborted() && mbar_wait(bar(bar_s(t, b)), uint32_t((gj >> 1) & 1), p.err);
                if (!__all_sync(kAll, got)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                float sc[kTcKeys];
                tmem_ld64(trow + uint32_t(b * kTcKeys), sc);
                const int k0 = (it.kb + j) * kTcKeys;   // absolute key index of the tile's first key
                if (k0 + kTcKeys - 1 > pos) {
#pragma unroll
                    for (int x = 0; x < kTcKeys; ++x) sc[x] = k0 + x <= pos ? sc[x] : -INFINITY;
                }
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int x = 0; x < kTcKeys; x += 8) {
                    m4[0] = fmax3(m4[0], sc[x], sc[x + 1]);
                    m4[1] = fmax3(m4[1], sc[x + 2], sc[x + 3]);
                    m4[2] = fmax3(m4[2], sc[x + 4], sc[x + 5]);
                    m4[3] = fmax3(m4[3], sc[x + 6], sc[x + 7]);
                }
                const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3])) * p.scale_log2;
                const bool move = mx > ref + kRescaleLog2;
                const float alpha = move ? fast_exp2(ref - mx) : 1.f;   // 0 while no key was seen
                if (move) ref = mx;
                if (j > 0 && __any_sync(kAll, move)) {
                    // rescale this warp's rows of O (every earlier P V has completed first)
                    got = !aborted() &&
                          mbar_wait(bar(bar_o(t, (gj - 1) & 1)), uint32_t(((gj - 1) >> 1) & 1), p.err);
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
                for (int x = 0; x < kTcKeys; x += 2) {
                    ffma2(sc[x], sc[x + 1], p.scale_log2, nu);
                    sc[x] = fast_exp2(sc[x]);
                    sc[x + 1] = fast_exp2(sc[x + 1]);
                    if (x & 2) fadd2(s4[2], s4[3], sc[x], sc[x + 1]);
                    else fadd2(s4[0], s4[1], sc[x], sc[x + 1]);
                }
                l = l * alpha + ((s4[0] + s4[1]) + (s4[2] + s4[3]));
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
            if (!ok) break;
            prev_nk = nk;
            prev_jend = jt + nk;
            prev_l = l;
            if (kSplit) sts32(ref_row, __float_as_int(ref));
            jt += nk;
            ++i;
        }
        // the last item's output
        if (ok && i > 0 && !epilogue()) ok = false;
        if (!ok) sts32(flag, 1);
    }

    // ---- every role is done: release the tensor memory
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTcTiles * kTmemTile);
    }
}

// Key split: the merge. A warp per row of an item (a CTA per 4 row slots of
// one (sequence, query tile, kv head)): the item's pieces are its ranges'
// CTAs c0 .. c0 + n - 1, the first in slot 2 c0 + 1, the others in slot 2c;
// lane q loads piece q's (m, l), the warp reduces M = max m_q and
// den = sum 2^(m_q - M) l_q (m_q in the kernel's base-2 units), and each lane
// accumulates its columns of out = sum 2^(m_q - M) O_q / den, loading the
// pieces' O kChunk at a time (the first kChunk in the same round trip as the
// states). 8 at a time keeps 8 CTAs on an SM; 16 at a time holds more
// registers and pays only where items have 9 or more pieces: the launcher
// takes it for calls of at most SMs / 9 items, where every item may (a call
// of more items with one long one among them takes 8 at a time, in more round
// trips).
// A piece that held none of the row's keys left m_q = -inf and is skipped
// (its O was not written). An item not split, or of a flagged sequence, is
// left as the kernel left it.
constexpr int kMergeRowsPerCta = 4;
static_assert(kMaxSplitParts <= 32, "a lane per piece");

template <typename T, int D, int kChunk>
__global__ void __launch_bounds__(32 * kMergeRowsPerCta, kChunk > 8 ? 4 : 8)
paged_prefill_merge_kernel(const PrefillParams p, int tiles) {
    constexpr int E = D / 32;
    constexpr int kSlices = kTcTiles * kTcRows / kMergeRowsPerCta;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int grp = blockIdx.x / kSlices;
    const int R = (blockIdx.x - grp * kSlices) * kMergeRowsPerCta + warp;   // row slot of the item
    PfItem it;
    int nk_all[kTcTiles];
    const bool valid = pf_decode(p, 0u, tiles, grp, false, it, nk_all) > 0;
    const int g = p.group, tq = kTcRows / g;
    const int t = R / kTcRows, r = R - t * kTcRows;
    const int tok = t * tq + r / g;
    // the plan and the states (and, for the stream's order, the kernel's end:
    // this grid does not complete before it)
    grid_dependency_wait();
    if (!valid || r >= tq * g || tok >= it.ntok) return;
    const int word = __ldcg(p.ws_plan + grp);
    const int n = word >> 16, c0 = word & 0xffff;
    if (n < 2) return;
    const size_t qrow = size_t(it.q0 + it.j0 + tok) * p.n_q_heads + size_t(it.h) * g + r % g;
    auto slot_row = [&](int q) {
        return size_t(2 * (c0 + q) + (q == 0 ? 1 : 0)) * size_t(kTcTiles * kTcRows) + size_t(R);
    };
    float mp = -INFINITY, lp = 0.f;
    if (lane < n) {
        mp = __ldcg(p.ws_m + slot_row(lane));
        lp = __ldcg(p.ws_l + slot_row(lane));
    }
    float x[kChunk][E];
    auto load = [&](int q0) {
#pragma unroll
        for (int q = 0; q < kChunk; ++q) {
            const bool in = q0 + q < n;
            const float *o = p.ws_o + slot_row(in ? q0 + q : 0) * D + lane * E;
#pragma unroll
            for (int e = 0; e < E; ++e) x[q][e] = in ? __ldcg(o + e) : 0.f;
        }
    };
    load(0);
    float M = mp;
#pragma unroll
    for (int mask = 16; mask >= 1; mask >>= 1) M = fmaxf(M, __shfl_xor_sync(kAll, M, mask));
    const float w = mp > -INFINITY ? exp2f(mp - M) : 0.f;
    float den = w * lp;
#pragma unroll
    for (int mask = 16; mask >= 1; mask >>= 1) den += __shfl_xor_sync(kAll, den, mask);
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    for (int q0 = 0; q0 < n; q0 += kChunk) {
        if (q0 > 0) load(q0);
#pragma unroll
        for (int q = 0; q < kChunk; ++q) {
            const float wq = __shfl_sync(kAll, w, (q0 + q) & 31);
            const bool use = q0 + q < n && wq != 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e) acc[e] = use ? fmaf(wq, x[q][e], acc[e]) : acc[e];
        }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    T *dst = reinterpret_cast<T *>(p.out) + qrow * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; e += 2)
        *reinterpret_cast<uint32_t *>(dst + e) = Elem<T>::pack2(acc[e] * inv, acc[e + 1] * inv);
}

int prefill_tc_smem_bytes(int head_dim) {
    return (head_dim == 64 ? TcLayout<64>::kTotal : TcLayout<128>::kTotal) + 1024;
}

template <typename T, int D, bool kSplit>
static cudaError_t launch_tc_instance(const CUtensorMap &kmap, const CUtensorMap &vmap,
                                      const CUtensorMap &qmap, const PrefillParams &p, int max_query_len, int num_sms,
                                      cudaStream_t stream) {
    auto kernel = paged_prefill_tc_kernel<T, D, kSplit>;
    const int smem = TcLayout<D>::kTotal + 1024;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static std::atomic<unsigned long long> opened[kLaunchCacheDevices];
    e = open_dynamic_smem(opened, dev, kernel, smem);
    if (e != cudaSuccess) return e;
    // persistent: one CTA per SM (its shared memory allows no second), each
    // working through its share of the items
    // items (and a CTA's band index, at most items + grid) must fit an int
    // (the API refuses larger calls)
    const long long tiles_ll = ((long long)max_query_len + p.tile_tokens - 1) / p.tile_tokens;
    const long long per_seq = tiles_ll * p.n_kv_heads;
    if (per_seq > (INT_MAX / 2) / p.num_seqs) return cudaErrorInvalidValue;
    const int tiles = int(tiles_ll);
    const long long items = per_seq * p.num_seqs;
    // (key split: every SM, each CTA a range of the call's key tiles)
    if (kSplit && (items > kMaxSplitItems || p.key_parts < 2 || p.key_parts > kMaxSplitParts))
        return cudaErrorInvalidValue;
    const dim3 grid(unsigned(kSplit ? num_sms : items < num_sms ? items : num_sms));
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
    return cudaLaunchKernelEx(&cfg, kernel, kmap, vmap, qmap, p, tiles);
}

template <typename T, int D>
static cudaError_t launch_merge_instance(const PrefillParams &p, int max_query_len, int num_sms,
                                         cudaStream_t stream) {
    const long long tiles = ((long long)max_query_len + p.tile_tokens - 1) / p.tile_tokens;
    const long long groups = tiles * p.n_kv_heads * p.num_seqs;
    const long long ctas = groups * (kTcTiles * kTcRows / kMergeRowsPerCta);
    if (ctas > INT_MAX) return cudaErrorInvalidValue;
    // the programmatic dependent of the prefill kernel: its launch and its
    // items' set-up overlap the kernel's end
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(ctas));
    cfg.blockDim = dim3(32 * kMergeRowsPerCta);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // (in calls of at most SMs / 9 items every item may have 9 or more pieces)
    if (groups * 9 <= num_sms) return cudaLaunchKernelEx(&cfg, paged_prefill_merge_kernel<T, D, 16>, p, int(tiles));
    return cudaLaunchKernelEx(&cfg, paged_prefill_merge_kernel<T, D, 8>, p, int(tiles));
}

cudaError_t launch_prefill_merge(int dtype, int head_dim, const PrefillParams &p, int max_query_len,
                                 int num_sms, cudaStream_t stream) {
    const bool bf16 = dtype == PAGEDKV_BF16;
    if (head_dim == 64)
        return bf16 ? launch_merge_instance<__nv_bfloat16, 64>(p, max_query_len, num_sms, stream)
                    : launch_merge_instance<__half, 64>(p, max_query_len, num_sms, stream);
    return bf16 ? launch_merge_instance<__nv_bfloat16, 128>(p, max_query_len, num_sms, stream)
                : launch_merge_instance<__half, 128>(p, max_query_len, num_sms, stream);
}

cudaError_t launch_prefill_tc(int dtype, int head_dim, const CUtensorMap &kmap,
                              const CUtensorMap &vmap, const CUtensorMap &qmap,
                              const PrefillParams &p, int max_query_len, int num_sms,
                              cudaStream_t stream) {
    const bool bf16 = dtype == PAGEDKV_BF16;
    // the key split has an instance of its own: the whole-item kernel keeps
    // none of its per-item arithmetic
    if (p.key_parts > 1) {
        if (head_dim == 64)
            return bf16 ? launch_tc_instance<__nv_bfloat16, 64, true>(kmap, vmap, qmap, p, max_query_len, num_sms, stream)
                        : launch_tc_instance<__half, 64, true>(kmap, vmap, qmap, p, max_query_len, num_sms, stream);
        return bf16 ? launch_tc_instance<__nv_bfloat16, 128, true>(kmap, vmap, qmap, p, max_query_len, num_sms, stream)
                    : launch_tc_instance<__half, 128, true>(kmap, vmap, qmap, p, max_query_len, num_sms, stream);
    }
    if (head_dim == 64)
        return bf16 ? launch_tc_instance<__nv_bfloat16, 64, false>(kmap, vmap, qmap, p, max_query_len, num_sms, stream)
                    : launch_tc_instance<__half, 64, false>(kmap, vmap, qmap, p, max_query_len, num_sms, stream);
    return bf16 ? launch_tc_instance<__nv_bfloat16, 128, false>(kmap, vmap, qmap, p, max_query_len, num_sms, stream)
                : launch_tc_instance<__half, 128, false>(kmap, vmap, qmap, p, max_query_len, num_sms, stream);
}

}  // namespace pkv
