/*
 * pagedkv.h -- C ABI of libpagedkv: paged KV-cache decode attention for GB300 (sm_103a).
 *
 * Three operations make up the data-parallel hot path of PagedAttention:
 *
 *   paged_attn_decode  single-token decode attention whose keys and values are gathered
 *                      from fixed-size, non-contiguous physical KV blocks through a
 *                      per-sequence block table (with a split-context variant for long
 *                      contexts, merged by log-sum-exp);
 *   kv_cache_write     writes each new token's key/value rows into the cache slot its
 *                      slot mapping names;
 *   kv_copy_blocks     copies whole physical blocks (copy-on-write of a shared block).
 *
 * Common conventions
 *   - Every pointer argument is caller-owned DEVICE memory of the current CUDA device,
 *     except where stated.  The library keeps no pointer after a call returns and
 *     allocates no device memory.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the legacy
 *     default stream).  Return codes report argument and launch errors only.
 *   - Tensors are dense and row-major (C order).
 *   - Cache layout: k_cache and v_cache are separate tensors of shape
 *         [num_blocks, block_size, num_kv_heads, head_dim]
 *     so token slot `slot` (= physical_block * block_size + offset) is row `slot` of the
 *     cache seen as [num_blocks * block_size, num_kv_heads, head_dim].  This follows the
 *     kernel sketch on the "Paged Attention" page (section "Paged Attention's Approach"),
 *     whose cache is [num_blocks, block_size, hidden] indexed
 *     [physical_block, in_block, head].
 *   - Data errors found on the device (a block id, slot or pair id out of range, a
 *     context length outside the block table) never trap: the offending unit is
 *     skipped or clamped, a bit is set in the library's device error word, and
 *     pkv_device_error() reports it.
 *
 * Element types: PKV_F32, PKV_BF16, PKV_F16.  Accumulation is always fp32.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle; binary-compatible with cudaStream_t / CUstream. */
typedef struct CUstream_st* pkv_stream_t;

typedef enum { PKV_F32 = 0, PKV_BF16 = 1, PKV_F16 = 2 } pkv_dtype;

/* Return codes (host side). */
#define PKV_OK 0
#define PKV_EINVAL (-1)      /* null pointer, bad size, misaligned pointer, Hq % Hkv != 0 */
#define PKV_ENOMEM (-2)      /* workspace smaller than paged_attn_decode_workspace_size() */
#define PKV_ECUDA (-3)       /* the CUDA runtime reported an error while launching */
#define PKV_EUNSUPPORTED (-4)/* head_dim / block_size / dtype combination not implemented */
#define PKV_ESCRATCH (-5)    /* needs more scratch than paged_attn_decode_noalloc has */
#define PKV_ENODEVMEM (-6)   /* no device memory left to load paged_attn_decode_noalloc's array */

/* Device error bits (OR-ed together, reported by pkv_device_error). */
#define PKV_DERR_BLOCK_ID 1u /* a live block-table entry outside [0, num_blocks) */
#define PKV_DERR_SLOT 2u     /* a slot >= num_blocks * block_size */
#define PKV_DERR_PAIR 4u     /* a copy pair naming a block outside [0, num_blocks) */
#define PKV_DERR_CONTEXT 8u  /* context_len < 0 or > max_blocks_per_seq * block_size */
#define PKV_DERR_TIMEOUT 16u /* a pipeline wait gave up after ~1 s (the call's output is void) */

/*
 * paged_attn_decode -- one decode query token per sequence attends to that sequence's
 * cached keys and values, read block by block through its block table.
 *
 * What it computes ("PagedAttention: how vLLM manages the KV cache", section
 * "PagedAttention changes addressing inside attention": the attention computation is
 * unchanged, only the addressing of the cache differs).  For sequence s with
 * L = context_lens[s], query head h and G = num_q_heads / num_kv_heads, the query reads
 * KV head g = h / G (consecutive groups; "Grouped-query attention can reduce the
 * KV-head term", same page, section "Keep the tensor formula beside the allocator
 * model").  Logical position p (0 <= p < L) lives in physical block
 * block_tables[s][p / block_size] at offset p % block_size ("Why vLLM Uses
 * PagedAttention", section "Split the KV cache into 16-token blocks").  Then
 *     out[s][h] = sum_p softmax_p( scale * <q[s][h], K_p> ) * V_p.
 * L = 0 gives a zero output row.  The values of block-table entries past
 * ceil(L / block_size) never matter (the kernel may load an entry of the row early,
 * before it knows L, but never dereferences one past the context), and cache slots past
 * L are never read.
 *
 * The query heads of one KV head are processed together, so every cached byte is read
 * from memory once.  Contexts longer than `partition_size` tokens are split into
 * partitions whose partial results (running max, sum of exponentials, unnormalised
 * output) are merged by log-sum-exp inside the same launch; the result equals the
 * single-pass one up to rounding order.
 *
 * Arguments
 *   out          [num_seqs, num_q_heads, head_dim], element type `dtype` (written).
 *   q            [num_seqs, num_q_heads, head_dim], `dtype`.
 *   k_cache,
 *   v_cache      [num_blocks, block_size, num_kv_heads, head_dim], `dtype`; 16-byte aligned.
 *   block_tables int32 [num_seqs, max_blocks_per_seq]; physical block ids.
 *   context_lens int32 [num_seqs]; tokens attended per sequence (0 allowed).
 *   scale        multiplies q.k before the softmax (typically 1/sqrt(head_dim)).
 *   partition_size  tokens per split-context partition: a positive multiple of
 *                block_size, or 0 for the library's choice -- the largest of 2048, 1024
 *                and 512 tokens that still gives at least 2048 work units (sequences x
 *                KV heads x partitions, every sequence counted at the block table's full
 *                length).  paged_attn_decode_workspace_size makes the same choice.
 *   workspace    device scratch of at least paged_attn_decode_workspace_size() bytes
 *                (may be NULL when that size is 0), 16-byte aligned.  Its contents need
 *                not be initialised: a call writes every workspace byte before it reads
 *                it.  Calls that may run concurrently must not share a workspace.
 * Launches on `stream`: one decode grid when the workspace size is 0; otherwise a
 * one-CTA kernel that orders the work longest first (left out when the batch has more
 * than 65536 sequence x partition items), the decode grid, and a grid that merges the
 * partitions' partial results by log-sum-exp.  The later grids use programmatic stream
 * serialization (they may start while the grid ahead drains and wait for it on the GPU);
 * work enqueued on `stream` afterwards still runs after all of them.
 *   stream       CUDA stream to launch on.
 * Supported: head_dim in {32, 64, 128, 256} (fp32 and fp16/bf16); the tensor-core path
 * serves fp16/bf16 with head_dim 64 or 128, block_size 16, 32 or 64 and at most 16
 * query heads per KV head; other shapes use the CUDA-core path.
 * Returns PKV_OK, PKV_EINVAL, PKV_ENOMEM, PKV_EUNSUPPORTED or PKV_ECUDA.
 */
int paged_attn_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                      int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                      int max_blocks_per_seq, int num_blocks, float scale, pkv_dtype dtype,
                      int partition_size, void* workspace, size_t workspace_bytes,
                      pkv_stream_t stream);

/*
 * Bytes of workspace paged_attn_decode needs for these sizes (0 when no sequence can
 * span more than one partition).  Pure host function; no CUDA call.
 */
size_t paged_attn_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                        int head_dim, int block_size, int max_blocks_per_seq,
                                        int partition_size);

/*
 * The partition size (tokens) paged_attn_decode uses for these sizes and this
 * `partition_size` argument (0 resolves to the library's choice), or PKV_EINVAL.  Pure
 * host function; no CUDA call.
 */
int paged_attn_decode_partition_tokens(int num_seqs, int num_q_heads, int num_kv_heads,
                                       int block_size, int max_blocks_per_seq,
                                       int partition_size);

/*
 * kv_cache_write -- store new tokens' keys and values in their cache slots
 * (the reshape-and-cache step).
 *
 * Blocks fill left to right as tokens are generated ("Why vLLM Uses PagedAttention",
 * section "Split the KV cache into 16-token blocks"; "PagedAttention: how vLLM manages
 * the KV cache", section "Walk one request through the allocator"): the caller's block
 * manager picks each token's slot, slot = physical_block * block_size + offset, and
 * this call copies the token's rows there:
 *     k_cache[slot / block_size][slot % block_size][:][:] = k[i][:][:]   (same for v)
 * A negative slot marks padding and is skipped.  A slot >= num_blocks * block_size is
 * skipped and sets PKV_DERR_SLOT.  Two tokens naming the same slot in one call leave
 * that slot undefined.  The copy is bit-exact.
 *
 *   k, v          [num_tokens, num_kv_heads, head_dim], `dtype`.
 *   k_cache,
 *   v_cache       [num_blocks, block_size, num_kv_heads, head_dim], `dtype` (written).
 *   slot_mapping  int64 [num_tokens].
 * Returns PKV_OK, PKV_EINVAL or PKV_ECUDA.  num_tokens = 0 is a no-op.
 */
int kv_cache_write(const void* k, const void* v, void* k_cache, void* v_cache,
                   const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                   int block_size, int num_blocks, pkv_dtype dtype, pkv_stream_t stream);

/*
 * paged_attn_prefill -- chunked-prefill attention: several query tokens per sequence
 * over the paged cache, causal within the chunk.
 *
 * "Paged Attention: How vLLM Solves the KV Cache Memory Problem", section "Continuous
 * Batching and Chunked Prefill": a long prompt is cut into chunks that are processed
 * between decode steps.  Sequence s contributes the n_s = query_start[s+1] -
 * query_start[s] query rows query_start[s] .. query_start[s+1]-1 of q.  Its cache already
 * holds L_s = context_lens[s] tokens, the chunk's own keys and values last (written with
 * kv_cache_write), so chunk token i sits at position L_s - n_s + i and attends positions
 * 0 .. L_s - n_s + i:
 *     out[t][h] = sum_{p <= L_s - n_s + i} softmax_p( scale * <q[t][h], K_p> ) * V_p,
 * t = query_start[s] + i, K_p and V_p of KV head h / (num_q_heads / num_kv_heads) read
 * through block_tables[s] as in paged_attn_decode.  A chunk of one token is a decode.
 *
 *   out, q       [num_q_tokens, num_q_heads, head_dim], `dtype` (PKV_BF16 or PKV_F16).
 *   k_cache, v_cache, block_tables, context_lens, num_blocks: as in paged_attn_decode.
 *   query_start  int32 [num_seqs + 1], device; query_start[0] = 0, non-decreasing,
 *                query_start[num_seqs] = num_q_tokens.
 *   max_query_len  an upper bound on every n_s (sizes the grid; host value).
 * All pointers are caller-owned device memory; the call is asynchronous on `stream` and
 * allocates nothing.  head_dim 64 or 128, block_size 16, 32 or 64, any finite scale (a
 * negative one is computed exactly as (-q) . k times |scale|).
 * Device-side data errors set PKV_DERR_* bits (see pkv_device_error) and skip the unit:
 * a chunk longer than its context or than max_query_len, a context longer than the table
 * or rows outside [0, num_q_tokens) set PKV_DERR_CONTEXT and leave that sequence's rows
 * unwritten; an out-of-range live block id sets PKV_DERR_BLOCK_ID and reads as zeros.
 * Returns PKV_OK, PKV_EINVAL, PKV_EUNSUPPORTED or PKV_ECUDA.
 */
int paged_attn_prefill(void* out, const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const int32_t* context_lens,
                       const int32_t* query_start, int num_seqs, int num_q_tokens,
                       int max_query_len, int num_q_heads, int num_kv_heads, int head_dim,
                       int block_size, int max_blocks_per_seq, int num_blocks, float scale,
                       pkv_dtype dtype, pkv_stream_t stream);

/*
 * paged_attn_decode_shared_prefix -- paged_attn_decode for sequences that share a
 * physical prefix, reading each shared block once per group instead of once per sequence.
 *
 * "PagedAttention: how vLLM manages the KV cache", section "Copy-on-write makes shared
 * prefixes practical": sequences forked from one prompt map the same physical blocks for
 * their common prefix.  The result is paged_attn_decode's:
 *     out[s][h] = sum_{p < L_s} softmax_p( scale * <q[s][h], K_p> ) * V_p,
 * computed as a cascade: a prefix pass in which all queries of a group meet each prefix
 * block once (tensor cores), a suffix pass (the decode kernel) over each sequence's own
 * tokens, and a log-sum-exp merge of their partial results.
 *
 *   out, q, k_cache, v_cache, block_tables, context_lens, num_seqs, ..., dtype:
 *                as in paged_attn_decode (dtype PKV_BF16 or PKV_F16, head_dim 128,
 *                block_size 16, 32 or 64, any finite scale).
 *   group_start  int32 [num_groups + 1], device: group g is the run of sequences
 *                group_start[g] .. group_start[g+1]-1 (non-decreasing, within
 *                [0, num_seqs]); sequences outside every run have no shared prefix.
 *   prefix_lens  int32 [num_groups], device: the group's shared prefix in tokens, a
 *                multiple of block_size, at most every member's context length.  The
 *                members' block tables must hold the same physical ids for those blocks
 *                (the first member's are read).
 *   max_group_size, max_prefix_tokens  host upper bounds of the group sizes and prefix
 *                lengths (they size the grids and the workspace).
 *   workspace    device scratch of paged_attn_decode_shared_prefix_workspace_size() bytes
 *                (16-byte aligned); it needs no initialisation.
 * A group that breaks these rules sets PKV_DERR_CONTEXT; its members are then attended
 * without the prefix pass (still correctly, if their tables are valid).
 * When to call it instead of paged_attn_decode: the cascade saves the HBM reads of the
 * repeated prefix blocks and costs three more launches and the partials' traffic.  It
 * pays when the groups' distinct prefix bytes (sum over groups of prefix_lens[g] *
 * num_kv_heads * head_dim * 2 element bytes, keys and values) exceed the L2 cache (about
 * 126 MB on GB300): then plain decode reads every member's copy of the prefix from HBM.
 * Measured on one GB300: 64 prompts of 4096 tokens shared by 8 sequences each (1 GB of
 * prefix) ran x1.77 faster than paged_attn_decode; 256 sequences sharing one 992-token
 * prefix (4 MB, held in L2 across the batch) ran x0.92 as fast.
 * Returns PKV_OK, PKV_EINVAL, PKV_ENOMEM, PKV_EUNSUPPORTED or PKV_ECUDA.
 */
size_t paged_attn_decode_shared_prefix_workspace_size(int num_seqs, int num_groups,
                                                      int num_q_heads, int num_kv_heads,
                                                      int block_size, int max_blocks_per_seq,
                                                      int max_group_size, int max_prefix_tokens);
int paged_attn_decode_shared_prefix(void* out, const void* q, const void* k_cache,
                                    const void* v_cache, const int32_t* block_tables,
                                    const int32_t* context_lens, const int32_t* group_start,
                                    const int32_t* prefix_lens, int num_seqs, int num_groups,
                                    int max_group_size, int max_prefix_tokens, int num_q_heads,
                                    int num_kv_heads, int head_dim, int block_size,
                                    int max_blocks_per_seq, int num_blocks, float scale,
                                    pkv_dtype dtype, void* workspace, size_t workspace_bytes,
                                    pkv_stream_t stream);

/*
 * paged_attn_decode_fp8 -- paged_attn_decode over caches of 8-bit E4M3 codes.
 *
 * "PagedAttention: how vLLM manages the KV cache", section "Keep the tensor formula
 * beside the allocator model": lower-precision cache formats reduce the bytes per element
 * (paging itself does not).  k_cache and v_cache hold E4M3 codes (uint8, 1 sign, 4
 * exponent bits with bias 7, 3 fraction bits, largest finite 448), laid out
 * [num_blocks, block_size, num_kv_heads, head_dim] like the 16-bit caches; element e
 * stands for value(e) * k_scale (keys) or value(e) * v_scale (values), per-tensor scales.
 * The result is paged_attn_decode's on those values:
 *     out[s][h] = sum_p softmax_p( scale * <q[s][h], K_p> ) * V_p.
 * q and out are `dtype` (PKV_BF16 or PKV_F16).  Codes convert exactly to fp16, so the
 * products run on the tensor cores in fp16 with fp32 accumulation.  head_dim must be 128
 * and block_size 16, 32 or 64.  Other arguments, the workspace and the return codes are
 * those of paged_attn_decode, except the default partition (partition_size 0): the
 * candidates grow by half to 3072, 1536 and 768 tokens (same 2048-work-unit rule).  At
 * one byte per element a token carries half the bytes, but its conversions cost more
 * instructions, and a 1.5x unit takes about as long as a 16-bit one.  The workspace is
 * sized by paged_attn_decode_fp8_workspace_size.
 */
int paged_attn_decode_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                          int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                          int max_blocks_per_seq, int num_blocks, float scale, float k_scale,
                          float v_scale, pkv_dtype dtype, int partition_size, void* workspace,
                          size_t workspace_bytes, pkv_stream_t stream);

/*
 * Bytes of workspace paged_attn_decode_fp8 needs for these sizes (0 when no sequence can
 * span more than one partition), and the partition size (tokens) it uses for this
 * `partition_size` argument, or PKV_EINVAL.  Pure host functions; no CUDA call.
 */
size_t paged_attn_decode_fp8_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                            int head_dim, int block_size, int max_blocks_per_seq,
                                            int partition_size);
int paged_attn_decode_fp8_partition_tokens(int num_seqs, int num_q_heads, int num_kv_heads,
                                           int block_size, int max_blocks_per_seq,
                                           int partition_size);

/*
 * kv_cache_write_fp8 -- kv_cache_write into E4M3 caches.
 *
 * Element x of token i's key row becomes the E4M3 code nearest to x / k_scale (the
 * division in IEEE fp32; ties to the even code; magnitudes beyond 448 saturate to +-448;
 * NaN stays NaN), stored at row slot_mapping[i] of k_cache; likewise for values with
 * v_scale.  k and v are [num_tokens, num_kv_heads, head_dim] in `dtype` (any of the three
 * types); num_kv_heads * head_dim must be a multiple of 8.  Slot rules and return codes
 * are those of kv_cache_write.  The copies are deterministic: equal inputs give equal
 * codes.
 */
int kv_cache_write_fp8(const void* k, const void* v, void* k_cache, void* v_cache,
                       const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                       int head_dim, int block_size, int num_blocks, pkv_dtype dtype,
                       float k_scale, float v_scale, pkv_stream_t stream);

/*
 * kv_copy_blocks -- copy whole physical blocks of one cache tensor, for copy-on-write.
 *
 * "PagedAttention: how vLLM manages the KV cache", section "Copy-on-write makes shared
 * prefixes practical": when a branch must modify a shared last block, the manager
 * allocates a new block and copies only that block.  For each pair i,
 *     cache[dst_i] = cache[src_i]          (block_bytes bytes, bit-exact)
 * with (src_i, dst_i) = (src_dst_pairs[2i], src_dst_pairs[2i+1]).  src == dst is a no-op.
 * The destinations must be distinct and disjoint from the sources of the same call
 * (otherwise the result is undefined).  A pair naming an id outside [0, num_blocks) is
 * skipped and sets PKV_DERR_PAIR.  Call once for the key cache and once for the value
 * cache.
 *
 *   cache          [num_blocks] blocks of block_bytes bytes each (written).
 *   src_dst_pairs  int64 [num_pairs, 2], device memory.
 *   block_bytes    bytes per block = block_size * num_kv_heads * head_dim * element size.
 * Returns PKV_OK, PKV_EINVAL or PKV_ECUDA.  num_pairs = 0 is a no-op.
 */
int kv_copy_blocks(void* cache, const int64_t* src_dst_pairs, int num_pairs, size_t block_bytes,
                   int num_blocks, pkv_stream_t stream);

/*
 * paged_attn_decode_noalloc -- paged_attn_decode for callers that cannot allocate.
 *
 * The pages have no counterpart to this call; it exists for users of this library.
 * paged_attn_decode needs scratch memory (the `workspace`), which its caller allocates.
 * Some callers cannot: a host program that owns the device's whole memory budget and
 * passes the library nothing but the tensors of each call, or a hot path on which no
 * allocation may happen.  This variant takes the same arguments minus the workspace and
 * uses instead a scratch array compiled into the library: PKV_NOALLOC_SCRATCH_BYTES of
 * device memory that every GPU which loads the library holds until the process exits.
 * It never allocates (no cudaMalloc or cudaFree, no allocating library routine).
 *
 *   - A problem whose scratch (paged_attn_decode_workspace_size) exceeds
 *     PKV_NOALLOC_SCRATCH_BYTES is rejected with PKV_ESCRATCH before any device work;
 *     use paged_attn_decode with a workspace for it, or a larger partition_size.
 *   - The first call on each device looks up the scratch array's device address (once,
 *     with that device current); make that first call before any stream capture.  That
 *     lookup also loads the part of the library holding the array, which is when its
 *     bytes are committed on the device (modules load lazily by default): make the first
 *     call at start-up, while memory is still free.  If the device has no room left for
 *     the array then, the call returns PKV_ENODEVMEM.  The address is cached per device
 *     together with the id of the current context; a call that finds a different context
 *     (the previous one was destroyed, e.g. by cudaDeviceReset) looks it up again, and
 *     that call is again a first call in the sense above.
 *   - All calls on a device share the one array, and it keeps the last call's contents
 *     (no call depends on them: each writes what it reads first).
 *     Calls whose work can overlap on the GPU (different streams without ordering
 *     between them) race on the array and give wrong results; order them.
 * Otherwise it behaves exactly as paged_attn_decode, with the same return codes.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (32u << 20)
int paged_attn_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, const int32_t* context_lens,
                              int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                              int block_size, int max_blocks_per_seq, int num_blocks, float scale,
                              pkv_dtype dtype, int partition_size, pkv_stream_t stream);

/*
 * kv_swap_blocks -- copy whole blocks from one pool to another (swap out / swap in).
 *
 * "PagedAttention" explainer, chapter 05 ("vLLM -- The Engine"): under memory pressure
 * requests are recomputed or swapped out; "PagedAttention: how vLLM manages the KV cache",
 * section "PagedAttention does not solve admission control": the scheduler must queue,
 * preempt, recompute, swap or reject.  For each pair i,
 *     dst_cache[dst_i] = src_cache[src_i]        (block_bytes bytes, bit-exact)
 * with (src_i, dst_i) = (src_dst_pairs[2i], src_dst_pairs[2i+1]).  Unlike kv_copy_blocks
 * the two pools are different tensors: either may be device memory or host memory the
 * device can address (pinned host memory; on Grace-Blackwell the kernel reaches it over
 * NVLink-C2C), so one launch gathers a preempted request's blocks out to a host pool, or
 * back in.  Destination blocks must be distinct.  A pair naming an id outside its pool is
 * skipped and sets PKV_DERR_PAIR.  Call once for the key pools and once for the value
 * pools.
 *
 *   dst_cache      [dst_num_blocks] blocks of block_bytes bytes (written).
 *   src_cache      [src_num_blocks] blocks of block_bytes bytes.
 *   src_dst_pairs  int64 [num_pairs, 2], device-addressable memory.
 * Returns PKV_OK, PKV_EINVAL or PKV_ECUDA.  num_pairs = 0 is a no-op.
 */
int kv_swap_blocks(void* dst_cache, const void* src_cache, const int64_t* src_dst_pairs,
                   int num_pairs, size_t block_bytes, int dst_num_blocks, int src_num_blocks,
                   pkv_stream_t stream);

/*
 * Synchronise `stream`, then return and clear the device error bits (PKV_DERR_*) that
 * kernels of this library set on the current device since the last call.  Returns a
 * negative PKV_ECUDA if the synchronisation itself failed.
 */
int pkv_device_error(pkv_stream_t stream);

/*
 * pkv_selftest_bounded_wait -- exercise the kernels' bounded-wait failure path.
 *
 * Launches one thread that waits on a fresh shared-memory mbarrier through the same
 * bounded wait the decode pipeline uses, for at most `wait_us` microseconds (at most one
 * second).  With arrive = 0 nothing ever completes the barrier, so the wait runs out,
 * the kernel sets PKV_DERR_TIMEOUT and returns normally: the context stays usable and
 * pkv_device_error() reports the bit.  With arrive != 0 the barrier completes at once
 * and no bit is set.  Asynchronous on `stream`.  Returns PKV_OK, PKV_EINVAL or
 * PKV_ECUDA.
 */
int pkv_selftest_bounded_wait(unsigned wait_us, int arrive, pkv_stream_t stream);

/* Static description of a return code or device error bit. */
const char* pkv_strerror(int code);

/* Library version, e.g. 0x000100 for 0.1.0. */
int pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
