/*
 * pagedkv_oracle.c -- plain CPU oracle for paged single-token decode attention,
 * slot-mapped KV writes and copy-on-write block copies.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
 * CPU-baseline / reference legs load this file. The product path never calls it,
 * and it shares no code, header, table or helper with the CUDA library.
 *
 * It is deliberately slow and obvious: every score, weight and output element is
 * computed in fp64 from the stored element values, token by token, in logical
 * order, with no blocking, fusion or reordering beyond the definitions below.
 *
 * What is computed, and where the pages define it:
 *
 *  - Block-table addressing.  "Why vLLM Uses PagedAttention", section "Split the KV
 *    cache into 16-token blocks": a sequence's cache is cut into fixed-size blocks and
 *    a per-request block table maps logical block j to a physical block.  "Paged
 *    Attention" (vanos001), section "Paged Attention's Approach": the kernel reads
 *    block_table[request * MAX_BLOCKS + logical_block] and the cache entry
 *    kv_cache[physical_block, in_block, head].  Logical position p therefore lives in
 *    physical block block_table[p / bs] at in-block offset p % bs.
 *
 *  - Attention itself.  "PagedAttention: how vLLM manages the KV cache", section
 *    "PagedAttention changes addressing inside attention": the computation is that of
 *    ordinary attention; only the addressing of the cache changes.  For one decode query
 *    q (one token, one head) over the L cached tokens of its sequence:
 *        s_p   = scale * <q, K_p>                      p = 0 .. L-1
 *        out   = sum_p softmax(s)_p * V_p
 *    evaluated with the maximum subtracted before exponentiation.
 *
 *  - Partitioned form (split context).  The same result written as per-partition
 *    (max, sum of exponentials, unnormalised weighted V) triples merged by
 *    log-sum-exp; exact up to rounding order.
 *
 *  - Slot writes.  "Why vLLM Uses PagedAttention" ("blocks are allocated on demand
 *    and filled left to right as tokens generate") and "PagedAttention: how vLLM
 *    manages the KV cache", section "Walk one request through the allocator": a new
 *    token's key and value go into one slot, slot = physical_block * bs + offset.
 *
 *  - Block copies.  "PagedAttention: how vLLM manages the KV cache", section
 *    "Copy-on-write makes shared prefixes practical": the manager allocates a new
 *    block and copies only that block.
 *
 *  - Chunked prefill.  "Paged Attention: How vLLM Solves the KV Cache Memory Problem",
 *    section "Continuous Batching and Chunked Prefill": a long prompt is processed in
 *    chunks interleaved with decode steps.  A chunk of n query tokens of a sequence whose
 *    cache holds L tokens (the chunk's own keys and values written last) sits at
 *    positions L-n .. L-1; query i of the chunk attends the positions 0 .. L-n+i (causal
 *    attention, as in any prefill).  Decode is the case n = 1.
 *
 * Layout conventions (the readings taken where the pages are silent):
 *  - cache tensors are [num_blocks, block_size, num_kv_heads, head_dim], row-major;
 *    K and V are separate tensors of the same shape;
 *  - q and the output are [num_seqs, num_q_heads, head_dim];
 *  - query head h reads KV head h / (num_q_heads / num_kv_heads);
 *  - exactly context_lens[s] tokens (positions 0 .. L-1) are attended; L = 0 gives 0.
 *
 * Element types: 0 = fp32, 1 = bf16 (raw 16-bit patterns), 2 = fp16 (raw patterns).
 * All are widened exactly to fp64 before any arithmetic.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define PKVO_OK 0
#define PKVO_EINVAL (-1)
#define PKVO_ENOMEM (-2)
#define PKVO_EDATA 1 /* out-of-range ids were found; those units were skipped */

/* ---- exact widening of stored elements to fp64 ---------------------------------- */

static double bf16_bits_to_double(uint16_t bits) {
    /* bf16 is the upper half of an IEEE binary32 pattern. */
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

static double f16_bits_to_double(uint16_t bits) {
    /* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
    int sign = (bits >> 15) & 1;
    int e = (bits >> 10) & 0x1f;
    int m = bits & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m + 1024), e - 25); /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

static double elem(const void* base, size_t idx, int dtype) {
    switch (dtype) {
    case 0: return (double)((const float*)base)[idx];
    case 1: return bf16_bits_to_double(((const uint16_t*)base)[idx]);
    default: return f16_bits_to_double(((const uint16_t*)base)[idx]);
    }
}

static size_t elem_size(int dtype) { return dtype == 0 ? 4u : 2u; }

/* ---- block-table addressing -------------------------------------------------------- */

int64_t pkvo_num_blocks(int64_t num_tokens, int block_size) {
    if (num_tokens <= 0) return 0;
    return (num_tokens + block_size - 1) / block_size;
}

void pkvo_locate(const int32_t* block_table_row, int64_t pos, int block_size,
                 int32_t* physical_block, int32_t* offset) {
    *physical_block = block_table_row[pos / block_size];
    *offset = (int32_t)(pos % block_size);
}

int64_t pkvo_slot(const int32_t* block_table_row, int64_t pos, int block_size) {
    int32_t phys, off;
    pkvo_locate(block_table_row, pos, block_size, &phys, &off);
    return (int64_t)phys * block_size + off;
}

/* Index of element d of the (physical block, offset, kv head) row of a cache tensor. */
static size_t cache_index(int32_t phys, int32_t off, int g, int d, int block_size,
                          int num_kv_heads, int head_dim) {
    size_t row = (size_t)phys * (size_t)block_size + (size_t)off;
    return (row * (size_t)num_kv_heads + (size_t)g) * (size_t)head_dim + (size_t)d;
}

static int check_shapes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                        int block_size, int max_blocks_per_seq, int num_blocks, int dtype) {
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
    if (block_size <= 0 || max_blocks_per_seq < 0 || num_blocks < 0) return 0;
    if (num_q_heads % num_kv_heads != 0) return 0;
    if (dtype < 0 || dtype > 2) return 0;
    return 1;
}

/* Every block a sequence's live tokens touch must be a valid physical id. */
static int check_tables(const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                        int block_size, int max_blocks_per_seq, int num_blocks) {
    for (int s = 0; s < num_seqs; ++s) {
        int64_t L = context_lens[s];
        if (L < 0) return 0;
        int64_t nb = pkvo_num_blocks(L, block_size);
        if (nb > max_blocks_per_seq) return 0;
        for (int64_t j = 0; j < nb; ++j) {
            int32_t b = block_tables[(size_t)s * max_blocks_per_seq + j];
            if (b < 0 || b >= num_blocks) return 0;
        }
    }
    return 1;
}

/* Scores s_p = scale * <q, K_p> for p = 0 .. L-1 of sequence s, query head h. */
static void scores_for(double* sc, const void* q, const void* k_cache, int dtype,
                       const int32_t* bt_row, int64_t L, int s, int h, int num_q_heads,
                       int num_kv_heads, int head_dim, int block_size, double scale) {
    int group = num_q_heads / num_kv_heads;
    int g = h / group;
    size_t qbase = ((size_t)s * num_q_heads + h) * (size_t)head_dim;
    for (int64_t p = 0; p < L; ++p) {
        int32_t phys, off;
        pkvo_locate(bt_row, p, block_size, &phys, &off);
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
            dot += elem(q, qbase + d, dtype) *
                   elem(k_cache, cache_index(phys, off, g, d, block_size, num_kv_heads, head_dim), dtype);
        sc[p] = scale * dot;
    }
}

/* ---- paged decode attention: the definition ----------------------------------------- */

int pkvo_paged_decode(double* out, const void* q, const void* k_cache, const void* v_cache,
                      int dtype, const int32_t* block_tables, const int32_t* context_lens,
                      int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                      int block_size, int max_blocks_per_seq, int num_blocks, double scale,
                      int num_threads) {
    if (!check_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                      max_blocks_per_seq, num_blocks, dtype))
        return PKVO_EINVAL;
    if (!check_tables(block_tables, context_lens, num_seqs, block_size, max_blocks_per_seq,
                      num_blocks))
        return PKVO_EINVAL;
    int group = num_q_heads / num_kv_heads;
    int64_t units = (int64_t)num_seqs * num_q_heads;
    int failed = 0;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
    for (int64_t u = 0; u < units; ++u) {
        int s = (int)(u / num_q_heads);
        int h = (int)(u % num_q_heads);
        int g = h / group;
        double* o = out + (size_t)u * head_dim;
        int64_t L = context_lens[s];
        for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
        if (L == 0) continue;
        const int32_t* bt_row = block_tables + (size_t)s * max_blocks_per_seq;
        double* w = (double*)malloc((size_t)L * sizeof(double));
        if (!w) { failed = 1; continue; }
        scores_for(w, q, k_cache, dtype, bt_row, L, s, h, num_q_heads, num_kv_heads, head_dim,
                   block_size, scale);
        double m = -INFINITY;
        for (int64_t p = 0; p < L; ++p) if (w[p] > m) m = w[p];
        double z = 0.0;
        for (int64_t p = 0; p < L; ++p) { w[p] = exp(w[p] - m); z += w[p]; }
        for (int64_t p = 0; p < L; ++p) {
            int32_t phys, off;
            pkvo_locate(bt_row, p, block_size, &phys, &off);
            for (int d = 0; d < head_dim; ++d)
                o[d] += w[p] * elem(v_cache, cache_index(phys, off, g, d, block_size, num_kv_heads,
                                                         head_dim), dtype);
        }
        for (int d = 0; d < head_dim; ++d) o[d] /= z;
        free(w);
    }
    return failed ? PKVO_ENOMEM : PKVO_OK;
}

/* ---- paged decode attention: split context, merged by log-sum-exp ------------------- */
/*
 * The context is cut into partitions of partition_size tokens.  Partition i yields
 *     m_i = max_{p in i} s_p,  l_i = sum_{p in i} exp(s_p - m_i),
 *     o_i = sum_{p in i} exp(s_p - m_i) V_p,
 * and the partials merge as  M = max_i m_i,
 *     out = sum_i exp(m_i - M) o_i / sum_i exp(m_i - M) l_i,
 * which equals the definition above up to rounding order.
 */
int pkvo_paged_decode_partitioned(double* out, const void* q, const void* k_cache,
                                  const void* v_cache, int dtype, const int32_t* block_tables,
                                  const int32_t* context_lens, int num_seqs, int num_q_heads,
                                  int num_kv_heads, int head_dim, int block_size,
                                  int max_blocks_per_seq, int num_blocks, double scale,
                                  int partition_size, int num_threads) {
    if (!check_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                      max_blocks_per_seq, num_blocks, dtype) || partition_size <= 0)
        return PKVO_EINVAL;
    if (!check_tables(block_tables, context_lens, num_seqs, block_size, max_blocks_per_seq,
                      num_blocks))
        return PKVO_EINVAL;
    int group = num_q_heads / num_kv_heads;
    int64_t units = (int64_t)num_seqs * num_q_heads;
    int failed = 0;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
    for (int64_t u = 0; u < units; ++u) {
        int s = (int)(u / num_q_heads);
        int h = (int)(u % num_q_heads);
        int g = h / group;
        double* o = out + (size_t)u * head_dim;
        int64_t L = context_lens[s];
        for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
        if (L == 0) continue;
        const int32_t* bt_row = block_tables + (size_t)s * max_blocks_per_seq;
        int64_t np = (L + partition_size - 1) / partition_size;
        double* sc = (double*)malloc((size_t)L * sizeof(double));
        double* mi = (double*)malloc((size_t)np * sizeof(double));
        double* li = (double*)malloc((size_t)np * sizeof(double));
        double* oi = (double*)calloc((size_t)np * head_dim, sizeof(double));
        if (!sc || !mi || !li || !oi) {
            failed = 1;
            free(sc); free(mi); free(li); free(oi);
            continue;
        }
        scores_for(sc, q, k_cache, dtype, bt_row, L, s, h, num_q_heads, num_kv_heads, head_dim,
                   block_size, scale);
        for (int64_t i = 0; i < np; ++i) {
            int64_t p0 = i * partition_size;
            int64_t p1 = p0 + partition_size < L ? p0 + partition_size : L;
            double m = -INFINITY;
            for (int64_t p = p0; p < p1; ++p) if (sc[p] > m) m = sc[p];
            double l = 0.0;
            for (int64_t p = p0; p < p1; ++p) {
                double e = exp(sc[p] - m);
                int32_t phys, off;
                pkvo_locate(bt_row, p, block_size, &phys, &off);
                l += e;
                for (int d = 0; d < head_dim; ++d)
                    oi[(size_t)i * head_dim + d] +=
                        e * elem(v_cache, cache_index(phys, off, g, d, block_size, num_kv_heads,
                                                      head_dim), dtype);
            }
            mi[i] = m;
            li[i] = l;
        }
        double M = -INFINITY;
        for (int64_t i = 0; i < np; ++i) if (mi[i] > M) M = mi[i];
        double den = 0.0;
        for (int64_t i = 0; i < np; ++i) {
            double c = exp(mi[i] - M);
            den += c * li[i];
            for (int d = 0; d < head_dim; ++d) o[d] += c * oi[(size_t)i * head_dim + d];
        }
        for (int d = 0; d < head_dim; ++d) o[d] /= den;
        free(sc); free(mi); free(li); free(oi);
    }
    return failed ? PKVO_ENOMEM : PKVO_OK;
}

/* ---- chunked prefill: several query tokens per sequence, causal ------------------ */
/*
 * q and out are [num_q_tokens, num_q_heads, head_dim]; sequence s owns query rows
 * query_start[s] .. query_start[s+1]-1 (query_start[0] = 0, query_start[num_seqs] =
 * num_q_tokens, non-decreasing).  With n = query_start[s+1] - query_start[s] and
 * L = context_lens[s] (n <= L), row query_start[s] + i, head h, is
 *     pos   = L - n + i
 *     s_p   = scale * <q_row,h, K_p>                   p = 0 .. pos
 *     out   = sum_p softmax(s)_p * V_p
 * with K_p, V_p read through sequence s's block table as for decode.
 */
int pkvo_paged_prefill(double* out, const void* q, const void* k_cache, const void* v_cache,
                       int dtype, const int32_t* block_tables, const int32_t* context_lens,
                       const int32_t* query_start, int num_seqs, int num_q_tokens,
                       int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                       int max_blocks_per_seq, int num_blocks, double scale, int num_threads) {
    if (!check_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                      max_blocks_per_seq, num_blocks, dtype) || num_q_tokens < 0)
        return PKVO_EINVAL;
    if (!check_tables(block_tables, context_lens, num_seqs, block_size, max_blocks_per_seq,
                      num_blocks))
        return PKVO_EINVAL;
    if (num_seqs > 0 && (query_start[0] != 0 || query_start[num_seqs] != num_q_tokens))
        return PKVO_EINVAL;
    for (int s = 0; s < num_seqs; ++s) {
        int64_t n = (int64_t)query_start[s + 1] - query_start[s];
        if (n < 0 || n > context_lens[s]) return PKVO_EINVAL;
    }
    int group = num_q_heads / num_kv_heads;
    int64_t units = (int64_t)num_q_tokens * num_q_heads;
    int failed = 0;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
    for (int64_t u = 0; u < units; ++u) {
        int64_t t = u / num_q_heads;
        int h = (int)(u % num_q_heads);
        int g = h / group;
        int s = 0;
        while (query_start[s + 1] <= t) ++s;  /* the sequence that owns query row t */
        int64_t n = (int64_t)query_start[s + 1] - query_start[s];
        int64_t i = t - query_start[s];
        int64_t pos = (int64_t)context_lens[s] - n + i;
        double* o = out + (size_t)u * head_dim;
        for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
        const int32_t* bt_row = block_tables + (size_t)s * max_blocks_per_seq;
        size_t qbase = ((size_t)t * num_q_heads + h) * (size_t)head_dim;
        double* w = (double*)malloc((size_t)(pos + 1) * sizeof(double));
        if (!w) { failed = 1; continue; }
        double m = -INFINITY;
        for (int64_t p = 0; p <= pos; ++p) {
            int32_t phys, off;
            pkvo_locate(bt_row, p, block_size, &phys, &off);
            double dot = 0.0;
            for (int d = 0; d < head_dim; ++d)
                dot += elem(q, qbase + d, dtype) *
                       elem(k_cache, cache_index(phys, off, g, d, block_size, num_kv_heads,
                                                 head_dim), dtype);
            w[p] = scale * dot;
            if (w[p] > m) m = w[p];
        }
        double z = 0.0;
        for (int64_t p = 0; p <= pos; ++p) { w[p] = exp(w[p] - m); z += w[p]; }
        for (int64_t p = 0; p <= pos; ++p) {
            int32_t phys, off;
            pkvo_locate(bt_row, p, block_size, &phys, &off);
            for (int d = 0; d < head_dim; ++d)
                o[d] += w[p] * elem(v_cache, cache_index(phys, off, g, d, block_size, num_kv_heads,
                                                         head_dim), dtype);
        }
        for (int d = 0; d < head_dim; ++d) o[d] /= z;
        free(w);
    }
    return failed ? PKVO_ENOMEM : PKVO_OK;
}

/* ---- slot-mapped write of new tokens ---------------------------------------------- */
/*
 * Token i's key row k[i] (num_kv_heads * head_dim elements, row_bytes bytes) goes to
 * cache row slot_mapping[i], i.e. physical block slot / bs, offset slot % bs; likewise
 * for v.  A negative slot is padding and is skipped.  A slot at or past
 * num_blocks * block_size is out of range: it is skipped and PKVO_EDATA is returned.
 */
int pkvo_kv_cache_write(const void* k, const void* v, void* k_cache, void* v_cache,
                        const int64_t* slot_mapping, int num_tokens, size_t row_bytes,
                        int num_blocks, int block_size) {
    if (num_tokens < 0 || num_blocks < 0 || block_size <= 0) return PKVO_EINVAL;
    int64_t rows = (int64_t)num_blocks * block_size;
    int bad = 0;
    for (int i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if (slot >= rows) { bad = 1; continue; }
        int64_t blk = slot / block_size, off = slot % block_size;
        size_t dst = ((size_t)blk * block_size + (size_t)off) * row_bytes;
        memcpy((char*)k_cache + dst, (const char*)k + (size_t)i * row_bytes, row_bytes);
        memcpy((char*)v_cache + dst, (const char*)v + (size_t)i * row_bytes, row_bytes);
    }
    return bad ? PKVO_EDATA : PKVO_OK;
}

/* ---- copy-on-write block copies ------------------------------------------------------ */
/*
 * For each pair (src, dst): the whole physical block dst becomes a byte copy of block
 * src (block_bytes bytes).  src == dst leaves the block as it is.  A pair naming an id
 * outside [0, num_blocks) is skipped and PKVO_EDATA is returned.
 */
int pkvo_copy_blocks(void* cache, const int64_t* src_dst_pairs, int num_pairs,
                     size_t block_bytes, int num_blocks) {
    if (num_pairs < 0 || num_blocks < 0) return PKVO_EINVAL;
    int bad = 0;
    for (int i = 0; i < num_pairs; ++i) {
        int64_t src = src_dst_pairs[2 * (size_t)i], dst = src_dst_pairs[2 * (size_t)i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) { bad = 1; continue; }
        if (src == dst) continue;
        memcpy((char*)cache + (size_t)dst * block_bytes,
               (const char*)cache + (size_t)src * block_bytes, block_bytes);
    }
    return bad ? PKVO_EDATA : PKVO_OK;
}

/* ---- block copies between two pools (swap out / swap in) ---------------------------- */
/*
 * For each pair (src, dst): block dst of dst_cache becomes a byte copy of block src of
 * src_cache.  "PagedAttention" (papermap), chapter 05 "vLLM -- The Engine": under memory
 * pressure requests are swapped out or recomputed; "PagedAttention: how vLLM manages the
 * KV cache", section "PagedAttention does not solve admission control": the scheduler
 * must queue, preempt, recompute, swap or reject.  A pair naming an id outside its pool
 * is skipped and PKVO_EDATA is returned.
 */
int pkvo_swap_blocks(void* dst_cache, const void* src_cache, const int64_t* src_dst_pairs,
                     int num_pairs, size_t block_bytes, int dst_num_blocks, int src_num_blocks) {
    if (num_pairs < 0 || dst_num_blocks < 0 || src_num_blocks < 0) return PKVO_EINVAL;
    int bad = 0;
    for (int i = 0; i < num_pairs; ++i) {
        int64_t src = src_dst_pairs[2 * (size_t)i], dst = src_dst_pairs[2 * (size_t)i + 1];
        if (src < 0 || src >= src_num_blocks || dst < 0 || dst >= dst_num_blocks) { bad = 1; continue; }
        memcpy((char*)dst_cache + (size_t)dst * block_bytes,
               (const char*)src_cache + (size_t)src * block_bytes, block_bytes);
    }
    return bad ? PKVO_EDATA : PKVO_OK;
}

/* ---- fp8 (E4M3) KV blocks --------------------------------------------------------- */
/*
 * "PagedAttention: how vLLM manages the KV cache", section "Keep the tensor formula beside
 * the allocator model": lower-precision cache formats reduce the bytes per element.  The
 * cache then holds 8-bit E4M3 codes (1 sign, 4 exponent bits with bias 7, 3 fraction
 * bits; no infinities; the all-ones pattern 0x7F / 0xFF is NaN; largest finite 448), and
 * a per-tensor scale: the stored element stands for code_value * scale.
 */

double pkvo_e4m3_to_double(uint8_t c) {
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);  /* subnormal: (m / 8) * 2^(1 - 7) */
    else
        v = ldexp((double)(m + 8), e - 10);  /* (1 + m/8) * 2^(e - 7) */
    return sign ? -v : v;
}

/* Nearest E4M3 code to x (ties to the even code), magnitudes above 448 saturating to
 * +-448; NaN maps to 0x7F.  Found by search over the 127 non-negative finite codes, which
 * are ordered by value. */
uint8_t pkvo_e4m3_from_double(double x) {
    if (x != x) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs(x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    int best = 0;
    for (int c = 1; c <= 0x7E; ++c) {
        double vc = pkvo_e4m3_to_double((uint8_t)c), vb = pkvo_e4m3_to_double((uint8_t)best);
        double dc = fabs(vc - a), db = fabs(vb - a);
        if (dc < db || (dc == db && (c & 1) == 0 && (best & 1) == 1)) best = c;
    }
    return (uint8_t)(sign | best);
}

/* Decode with fp8 caches: K_p = e4m3(k_code) * k_scale, V_p = e4m3(v_code) * v_scale; q in
 * `dtype` (0 f32, 1 bf16, 2 f16).  Otherwise the same definition as pkvo_paged_decode. */
int pkvo_paged_decode_fp8kv(double* out, const void* q, const uint8_t* k_cache,
                            const uint8_t* v_cache, int dtype, const int32_t* block_tables,
                            const int32_t* context_lens, int num_seqs, int num_q_heads,
                            int num_kv_heads, int head_dim, int block_size,
                            int max_blocks_per_seq, int num_blocks, double scale, double k_scale,
                            double v_scale, int num_threads) {
    if (!check_shapes(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                      max_blocks_per_seq, num_blocks, dtype))
        return PKVO_EINVAL;
    if (!check_tables(block_tables, context_lens, num_seqs, block_size, max_blocks_per_seq,
                      num_blocks))
        return PKVO_EINVAL;
    int group = num_q_heads / num_kv_heads;
    int64_t units = (int64_t)num_seqs * num_q_heads;
    int failed = 0;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
#endif
    for (int64_t u = 0; u < units; ++u) {
        int s = (int)(u / num_q_heads);
        int h = (int)(u % num_q_heads);
        int g = h / group;
        double* o = out + (size_t)u * head_dim;
        int64_t L = context_lens[s];
        for (int d = 0; d < head_dim; ++d) o[d] = 0.0;
        if (L == 0) continue;
        const int32_t* bt_row = block_tables + (size_t)s * max_blocks_per_seq;
        size_t qbase = ((size_t)s * num_q_heads + h) * (size_t)head_dim;
        double* w = (double*)malloc((size_t)L * sizeof(double));
        if (!w) { failed = 1; continue; }
        for (int64_t p = 0; p < L; ++p) {
            int32_t phys, off;
            pkvo_locate(bt_row, p, block_size, &phys, &off);
            double dot = 0.0;
            for (int d = 0; d < head_dim; ++d)
                dot += elem(q, qbase + d, dtype) *
                       (pkvo_e4m3_to_double(k_cache[cache_index(phys, off, g, d, block_size,
                                                                num_kv_heads, head_dim)]) *
                        k_scale);
            w[p] = scale * dot;
        }
        double m = -INFINITY;
        for (int64_t p = 0; p < L; ++p) if (w[p] > m) m = w[p];
        double z = 0.0;
        for (int64_t p = 0; p < L; ++p) { w[p] = exp(w[p] - m); z += w[p]; }
        for (int64_t p = 0; p < L; ++p) {
            int32_t phys, off;
            pkvo_locate(bt_row, p, block_size, &phys, &off);
            for (int d = 0; d < head_dim; ++d)
                o[d] += w[p] * (pkvo_e4m3_to_double(v_cache[cache_index(
                                    phys, off, g, d, block_size, num_kv_heads, head_dim)]) *
                                v_scale);
        }
        for (int d = 0; d < head_dim; ++d) o[d] /= z;
        free(w);
    }
    return failed ? PKVO_ENOMEM : PKVO_OK;
}

/* Slot write into fp8 caches: each element x of token i's key row becomes the code of
 * (x / k_scale) -- the division done in fp32, the precision the GPU writes with -- at row
 * slot_mapping[i] (same for values with v_scale).  Slot rules as pkvo_kv_cache_write. */
int pkvo_kv_cache_write_fp8(const void* k, const void* v, uint8_t* k_cache, uint8_t* v_cache,
                            const int64_t* slot_mapping, int num_tokens, int row_elems,
                            int dtype, int num_blocks, int block_size, float k_scale,
                            float v_scale) {
    if (num_tokens < 0 || num_blocks < 0 || block_size <= 0 || row_elems <= 0) return PKVO_EINVAL;
    int64_t rows = (int64_t)num_blocks * block_size;
    int bad = 0;
    for (int i = 0; i < num_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if (slot >= rows) { bad = 1; continue; }
        for (int e = 0; e < row_elems; ++e) {
            size_t src = (size_t)i * row_elems + e, dst = (size_t)slot * row_elems + e;
            float xk = (float)elem(k, src, dtype) / k_scale;
            float xv = (float)elem(v, src, dtype) / v_scale;
            k_cache[dst] = pkvo_e4m3_from_double((double)xk);
            v_cache[dst] = pkvo_e4m3_from_double((double)xv);
        }
    }
    return bad ? PKVO_EDATA : PKVO_OK;
}

int pkvo_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
