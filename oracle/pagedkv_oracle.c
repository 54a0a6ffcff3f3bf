/*
 * pagedkv_oracle.c -- plain, slow, fp64 CPU oracle for attention over a
 * block-paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY. The test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg are the only callers. The CUDA library never
 * links or calls this file and shares no code, header or table with it.
 *
 * What each function follows (page title, then section):
 *
 *   oracle_slot, oracle_slot_mapping
 *     "How a serving engine actually works", section "The one formula":
 *         physical(seq, i) = block_table[seq][floor(i / B)] * B + (i mod B)
 *     and section "The block table, printed small enough to read" (a 10-token
 *     sequence at B = 4 that lives in physical blocks 5, 2, 9, then grows).
 *
 *   oracle_append
 *     "Paged-KV + Continuous Batching From Scratch", section 1 "Paging is
 *     really about not reserving": one K and one V pool per layer, shaped
 *     (num_blocks, block_size, n_kv_heads, head_dim) and indexed by physical
 *     block. Appending a token stores its K/V row at its physical slot; the
 *     same page's closing section says the append is plain indexing.
 *
 *   oracle_copy_blocks
 *     "How a serving engine actually works", section "Copy-on-write, because
 *     you have used fork()": a sequence about to write into a block that others
 *     still reference gets a fresh block; the fresh block must first hold the
 *     shared block's contents. Whole-block copy, K and V, pairs in order.
 *
 *   oracle_swap_blocks
 *     "Paged Attention and the Block Manager", section "Running out of memory
 *     becomes a scheduling decision": a preempted sequence can keep its cache
 *     by having it copied out to host memory and back in later. The copy moves
 *     whole blocks (K and V) from one pool to another pool of the same block
 *     shape; the two pools may hold different numbers of blocks.
 *
 *   oracle_gather
 *     "Paged Attention and the Block Manager", section "The measurement": a
 *     sequence's cache is copied out of its blocks, in logical order, into a
 *     contiguous [length][head_dim] array per kv head. The oracle keeps this
 *     deliberate copy; the CUDA path is the thing that removes it.
 *
 *   oracle_decode_units
 *     "Paged-KV + Continuous Batching From Scratch", section "What's
 *     deliberately still missing": paged attention is the same mathematics as
 *     ordinary attention, only the addressing differs ("How a serving engine
 *     actually works", section "A serving engine is an operating system":
 *     attention never changes). So decode is textbook softmax attention over
 *     the gathered keys and values, for every query head of the kv head's
 *     group (query head qh reads kv head qh / (n_q_heads / n_kv_heads); the
 *     pages are silent on grouping, this is the consecutive-group reading).
 *
 *   oracle_prefill_units
 *     "How a serving engine actually works", section "Prefill and decode are
 *     two different jobs": a long prompt is prefilled in slices, one chunk per
 *     iteration. Reading taken (the pages give the schedule, not the
 *     attention): a chunk's K/V are appended to the cache first, so with
 *     L = tokens cached (the chunk included) and n = the chunk's length, its
 *     query j is the token at position L - n + j and attends, by the same
 *     softmax attention as decode, over the keys at positions 0 .. L - n + j
 *     (the earlier chunks and itself, causally). Decode is the case n = 1.
 *
 *   oracle_decode_partition, oracle_lse_merge
 *     The pages do not split a context. These two state the split-context
 *     form used by the partitioned kernel: over tokens [t0, t1) of one query
 *     head, m = max z, l = sum exp(z - m), o = sum exp(z - m) v; partitions
 *     combine as out = sum_p e^(m_p - M) o_p / sum_p e^(m_p - M) l_p with
 *     M = max_p m_p. This is an identity of the softmax, not an approximation.
 *
 * Element types: 0 = fp32, 1 = fp16 (IEEE binary16), 2 = bf16 (upper half of
 * an IEEE binary32). Stored values are widened exactly to double; the fp16
 * and bf16 decoders below are written from the formats' definitions.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_BF16 = 2 };

/* ------------------------------------------------------------------------ */
/* Exact widening of stored elements to double.                              */
/* ------------------------------------------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double mag;
    if (expo == 0)
        mag = ldexp((double)frac, -24);                 /* zero or subnormal: frac * 2^-24 */
    else if (expo == 31)
        mag = frac ? NAN : INFINITY;
    else
        mag = ldexp((double)(1024 + frac), expo - 25);  /* (1 + frac/1024) * 2^(expo-15) */
    return sign ? -mag : mag;
}

/* bfloat16: the upper 16 bits of a binary32 value. */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t bits = (uint32_t)b << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
}

static double widen(const void *base, int64_t index, int dtype)
{
    if (dtype == ORACLE_F32) {
        float f;
        memcpy(&f, (const char *)base + 4 * index, 4);
        return (double)f;
    }
    uint16_t bits;
    memcpy(&bits, (const char *)base + 2 * index, 2);
    return dtype == ORACLE_F16 ? oracle_f16_to_double(bits) : oracle_bf16_to_double(bits);
}

/* ------------------------------------------------------------------------ */
/* Address translation ("The one formula").                                  */
/* ------------------------------------------------------------------------ */

/* Physical slot of logical position pos of sequence seq. */
int64_t oracle_slot(const int32_t *block_tables, int max_blocks_per_seq,
                    int seq, int64_t pos, int block_size)
{
    int64_t logical_block = pos / block_size;
    int64_t offset = pos % block_size;
    int64_t physical_block = block_tables[(int64_t)seq * max_blocks_per_seq + logical_block];
    return physical_block * block_size + offset;
}

/* slot_mapping[t] for each new token t = (token_seq[t], token_pos[t]).
 * A negative position is padding and maps to -1. Returns 0, or -1 if a
 * position falls outside the block table (nothing is written for it then). */
int oracle_slot_mapping(const int32_t *block_tables, int max_blocks_per_seq,
                        const int32_t *token_seq, const int32_t *token_pos,
                        int64_t num_tokens, int block_size, int64_t *slot_mapping)
{
    int status = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        if (token_pos[t] < 0) {
            slot_mapping[t] = -1;
            continue;
        }
        if (token_pos[t] / block_size >= max_blocks_per_seq) {
            slot_mapping[t] = -1;
            status = -1;
            continue;
        }
        slot_mapping[t] = oracle_slot(block_tables, max_blocks_per_seq,
                                      token_seq[t], token_pos[t], block_size);
    }
    return status;
}

/* ------------------------------------------------------------------------ */
/* Append: store each token's K and V row at its physical slot.              */
/* ------------------------------------------------------------------------ */

/* k_rows, v_rows: [num_tokens][row_bytes] where row_bytes is one token's
 * n_kv_heads * head_dim elements. The pools are [num_slots][row_bytes], i.e.
 * (num_blocks, block_size, n_kv_heads, head_dim) with num_slots =
 * num_blocks * block_size. A negative slot is padding and is skipped.
 * Returns the number of slots that were out of range (those are skipped). */
int64_t oracle_append(const uint8_t *k_rows, const uint8_t *v_rows,
                      const int64_t *slot_mapping, int64_t num_tokens,
                      uint8_t *k_cache, uint8_t *v_cache,
                      int64_t num_slots, int64_t row_bytes)
{
    int64_t bad = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0)
            continue;
        if (slot >= num_slots) {
            ++bad;
            continue;
        }
        memcpy(k_cache + slot * row_bytes, k_rows + t * row_bytes, (size_t)row_bytes);
        memcpy(v_cache + slot * row_bytes, v_rows + t * row_bytes, (size_t)row_bytes);
    }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Copy-on-write: copy whole blocks (K and V) from src to dst.               */
/* ------------------------------------------------------------------------ */

/* pairs: [num_pairs][2] = {src, dst}. block_bytes = block_size * row bytes.
 * Returns the number of pairs skipped because an id was outside the pool. */
int64_t oracle_copy_blocks(uint8_t *k_cache, uint8_t *v_cache, const int32_t *pairs,
                           int64_t num_pairs, int64_t num_blocks, int64_t block_bytes)
{
    int64_t bad = 0;
    for (int64_t i = 0; i < num_pairs; ++i) {
        int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            ++bad;
            continue;
        }
        memcpy(k_cache + dst * block_bytes, k_cache + src * block_bytes, (size_t)block_bytes);
        memcpy(v_cache + dst * block_bytes, v_cache + src * block_bytes, (size_t)block_bytes);
    }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Swap: copy whole blocks (K and V) from one pool into another.             */
/* ------------------------------------------------------------------------ */

/* pairs: [num_pairs][2] = {block in the source pools, block in the destination
 * pools}. Returns the number of pairs skipped because an id was outside its
 * pool. */
int64_t oracle_swap_blocks(const uint8_t *src_k, const uint8_t *src_v, int64_t src_blocks,
                           uint8_t *dst_k, uint8_t *dst_v, int64_t dst_blocks,
                           const int32_t *pairs, int64_t num_pairs, int64_t block_bytes)
{
    int64_t bad = 0;
    for (int64_t i = 0; i < num_pairs; ++i) {
        int64_t from = pairs[2 * i], to = pairs[2 * i + 1];
        if (from < 0 || from >= src_blocks || to < 0 || to >= dst_blocks) {
            ++bad;
            continue;
        }
        memcpy(dst_k + to * block_bytes, src_k + from * block_bytes, (size_t)block_bytes);
        memcpy(dst_v + to * block_bytes, src_v + from * block_bytes, (size_t)block_bytes);
    }
    return bad;
}

/* ------------------------------------------------------------------------ */
/* Gather: copy one sequence's cache for one kv head out of its blocks.      */
/* ------------------------------------------------------------------------ */

/* dst[i][d] = cache[physical(seq, i)][kv_head][d] for i < length. */
void oracle_gather(const void *cache, const int32_t *block_tables, int max_blocks_per_seq,
                   int seq, int length, int kv_head, int n_kv_heads, int head_dim,
                   int block_size, int dtype, double *dst)
{
    for (int i = 0; i < length; ++i) {
        int64_t slot = oracle_slot(block_tables, max_blocks_per_seq, seq, i, block_size);
        int64_t row = (slot * n_kv_heads + kv_head) * (int64_t)head_dim;
        for (int d = 0; d < head_dim; ++d)
            dst[(int64_t)i * head_dim + d] = widen(cache, row + d, dtype);
    }
}

/* ------------------------------------------------------------------------ */
/* Decode attention.                                                         */
/* ------------------------------------------------------------------------ */

/* Textbook softmax attention of one query against `length` contiguous keys
 * and values (all double): z_i = scale * q.K_i, out = softmax(z) V. */
static void attend(const double *q, const double *K, const double *V, int length,
                   int head_dim, double scale, double *z, double *out)
{
    for (int d = 0; d < head_dim; ++d)
        out[d] = 0.0;
    if (length <= 0)
        return;                                  /* empty context: zeros by convention */
    double zmax = -INFINITY;
    for (int i = 0; i < length; ++i) {
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
            dot += q[d] * K[(int64_t)i * head_dim + d];
        z[i] = scale * dot;
        if (z[i] > zmax)
            zmax = z[i];
    }
    double denom = 0.0;
    for (int i = 0; i < length; ++i) {
        z[i] = exp(z[i] - zmax);
        denom += z[i];
    }
    for (int i = 0; i < length; ++i)
        for (int d = 0; d < head_dim; ++d)
            out[d] += z[i] * V[(int64_t)i * head_dim + d];
    for (int d = 0; d < head_dim; ++d)
        out[d] /= denom;
}

/*
 * Decode attention for the listed (seq, kv_head) units; units holds pairs
 * {seq, kv_head}. For each unit the sequence's K and V are gathered for that
 * kv head, then every query head of its group attends over them.
 *   q            [num_seqs][n_q_heads][head_dim]                 (dtype)
 *   k/v_cache    [num_blocks][block_size][n_kv_heads][head_dim]  (dtype)
 *   block_tables [num_seqs][max_blocks_per_seq]
 *   context_lens [num_seqs]  number of tokens each sequence attends over
 *   out          [num_seqs][n_q_heads][head_dim] double; only the rows of the
 *                listed units are written.
 * Returns 0, or -1 on an argument that cannot be honoured.
 */
int oracle_decode_units(const void *q, const void *k_cache, const void *v_cache,
                        const int32_t *block_tables, const int32_t *context_lens,
                        double scale, int num_seqs, int n_q_heads, int n_kv_heads,
                        int head_dim, int block_size, int max_blocks_per_seq, int dtype,
                        const int32_t *units, int64_t num_units, double *out, int threads)
{
    if (n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0)
        return -1;
    int group = n_q_heads / n_kv_heads;
    int status = 0;
    (void)num_seqs;
    (void)threads;
#ifdef _OPENMP
    if (threads <= 0)
        threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads)
#endif
    for (int64_t u = 0; u < num_units; ++u) {
        int seq = units[2 * u];
        int kv_head = units[2 * u + 1];
        int length = context_lens[seq];
        if (length < 0 || length > max_blocks_per_seq * block_size) {
            status = -1;
            continue;
        }
        int n = length > 0 ? length : 1;
        double *K = (double *)malloc(sizeof(double) * (size_t)n * head_dim);
        double *V = (double *)malloc(sizeof(double) * (size_t)n * head_dim);
        double *qd = (double *)malloc(sizeof(double) * (size_t)head_dim);
        double *z = (double *)malloc(sizeof(double) * (size_t)n);
        oracle_gather(k_cache, block_tables, max_blocks_per_seq, seq, length, kv_head,
                      n_kv_heads, head_dim, block_size, dtype, K);
        oracle_gather(v_cache, block_tables, max_blocks_per_seq, seq, length, kv_head,
                      n_kv_heads, head_dim, block_size, dtype, V);
        for (int j = 0; j < group; ++j) {
            int qh = kv_head * group + j;
            int64_t qrow = ((int64_t)seq * n_q_heads + qh) * head_dim;
            for (int d = 0; d < head_dim; ++d)
                qd[d] = widen(q, qrow + d, dtype);
            attend(qd, K, V, length, head_dim, scale, z, out + qrow);
        }
        free(K);
        free(V);
        free(qd);
        free(z);
    }
    return status;
}

/*
 * Chunked-prefill attention for the listed (seq, kv_head) units.
 *   q             [num_tokens][n_q_heads][head_dim] (dtype): the chunks' query
 *                 rows, sequence after sequence
 *   query_start   [num_seqs + 1]: sequence s owns query rows
 *                 query_start[s] .. query_start[s + 1] - 1
 *   context_lens  [num_seqs]: tokens in the cache, the chunk included
 *   out           [num_tokens][n_q_heads][head_dim] double; only the rows of the
 *                 listed units are written.
 * Query row j of sequence s, whose chunk holds n rows, is the token at position
 * context_lens[s] - n + j; it attends over the keys at positions 0 .. that
 * position. Returns 0, or -1 on a length that cannot be honoured.
 */
int oracle_prefill_units(const void *q, const void *k_cache, const void *v_cache,
                         const int32_t *block_tables, const int32_t *query_start,
                         const int32_t *context_lens, double scale, int n_q_heads,
                         int n_kv_heads, int head_dim, int block_size, int max_blocks_per_seq,
                         int dtype, const int32_t *units, int64_t num_units, double *out,
                         int threads)
{
    if (n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0)
        return -1;
    int group = n_q_heads / n_kv_heads;
    int status = 0;
    (void)threads;
#ifdef _OPENMP
    if (threads <= 0)
        threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads)
#endif
    for (int64_t u = 0; u < num_units; ++u) {
        int seq = units[2 * u];
        int kv_head = units[2 * u + 1];
        int length = context_lens[seq];
        int first = query_start[seq];
        int rows = query_start[seq + 1] - first;
        if (length < 0 || length > max_blocks_per_seq * block_size || rows < 0 || rows > length) {
            status = -1;
            continue;
        }
        if (rows == 0)
            continue;
        double *K = (double *)malloc(sizeof(double) * (size_t)length * head_dim);
        double *V = (double *)malloc(sizeof(double) * (size_t)length * head_dim);
        double *qd = (double *)malloc(sizeof(double) * (size_t)head_dim);
        double *z = (double *)malloc(sizeof(double) * (size_t)length);
        oracle_gather(k_cache, block_tables, max_blocks_per_seq, seq, length, kv_head,
                      n_kv_heads, head_dim, block_size, dtype, K);
        oracle_gather(v_cache, block_tables, max_blocks_per_seq, seq, length, kv_head,
                      n_kv_heads, head_dim, block_size, dtype, V);
        for (int r = 0; r < rows; ++r) {
            int position = length - rows + r;
            for (int e = 0; e < group; ++e) {
                int qh = kv_head * group + e;
                int64_t qrow = ((int64_t)(first + r) * n_q_heads + qh) * head_dim;
                for (int d = 0; d < head_dim; ++d)
                    qd[d] = widen(q, qrow + d, dtype);
                attend(qd, K, V, position + 1, head_dim, scale, z, out + qrow);
            }
        }
        free(K);
        free(V);
        free(qd);
        free(z);
    }
    return status;
}

/*
 * Unnormalised attention state of query head qh of sequence seq over the
 * token range [t0, t1): m = max_i z_i, l = sum_i exp(z_i - m),
 * o[d] = sum_i exp(z_i - m) V_i[d], z_i = scale * q.K_i. An empty range gives
 * m = -inf, l = 0, o = 0.
 */
int oracle_decode_partition(const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, double scale, int n_q_heads,
                            int n_kv_heads, int head_dim, int block_size,
                            int max_blocks_per_seq, int dtype, int seq, int qh,
                            int t0, int t1, double *o, double *m, double *l)
{
    if (n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0 || t0 < 0 || t1 < t0 ||
        t1 > max_blocks_per_seq * block_size)
        return -1;
    int group = n_q_heads / n_kv_heads;
    int kv_head = qh / group;
    int length = t1;
    int n = length > 0 ? length : 1;
    double *K = (double *)malloc(sizeof(double) * (size_t)n * head_dim);
    double *V = (double *)malloc(sizeof(double) * (size_t)n * head_dim);
    double *qd = (double *)malloc(sizeof(double) * (size_t)head_dim);
    double *z = (double *)malloc(sizeof(double) * (size_t)n);
    oracle_gather(k_cache, block_tables, max_blocks_per_seq, seq, length, kv_head,
                  n_kv_heads, head_dim, block_size, dtype, K);
    oracle_gather(v_cache, block_tables, max_blocks_per_seq, seq, length, kv_head,
                  n_kv_heads, head_dim, block_size, dtype, V);
    int64_t qrow = ((int64_t)seq * n_q_heads + qh) * head_dim;
    for (int d = 0; d < head_dim; ++d) {
        qd[d] = widen(q, qrow + d, dtype);
        o[d] = 0.0;
    }
    double zmax = -INFINITY;
    for (int i = t0; i < t1; ++i) {
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
            dot += qd[d] * K[(int64_t)i * head_dim + d];
        z[i] = scale * dot;
        if (z[i] > zmax)
            zmax = z[i];
    }
    double sum = 0.0;
    for (int i = t0; i < t1; ++i) {
        double w = exp(z[i] - zmax);
        sum += w;
        for (int d = 0; d < head_dim; ++d)
            o[d] += w * V[(int64_t)i * head_dim + d];
    }
    *m = zmax;
    *l = sum;
    free(K);
    free(V);
    free(qd);
    free(z);
    return 0;
}

/* Combine n partition states (m[p], l[p], o[p][head_dim]) into one
 * normalised output row. All-empty input gives zeros. */
void oracle_lse_merge(int n, const double *m, const double *l, const double *o,
                      int head_dim, double *out)
{
    double M = -INFINITY;
    for (int p = 0; p < n; ++p)
        if (m[p] > M)
            M = m[p];
    for (int d = 0; d < head_dim; ++d)
        out[d] = 0.0;
    if (M == -INFINITY)
        return;
    double denom = 0.0;
    for (int p = 0; p < n; ++p) {
        double w = exp(m[p] - M);
        denom += w * l[p];
        for (int d = 0; d < head_dim; ++d)
            out[d] += w * o[(int64_t)p * head_dim + d];
    }
    for (int d = 0; d < head_dim; ++d)
        out[d] /= denom;
}

/* Number of threads an OpenMP region would use (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
