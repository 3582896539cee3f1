// internal.h -- host-side interfaces between the C-ABI layer (api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pagedkv.h"

namespace pkv {

constexpr int kDefaultPartitionTokens = 512;
constexpr int kMaxPartitionBlocks = 2048;

struct DecodeArgs {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  int num_seqs, num_q_heads, num_kv_heads, head_dim, block_size;
  int max_blocks_per_seq, num_blocks;
  float scale;
  pkv_dtype dtype;
  int partition_tokens;  // resolved: a positive multiple of block_size
  void* workspace;
  size_t workspace_bytes;
  unsigned* err;  // device error word
  bool kv_fp8;    // caches hold E4M3 codes (then k_scale / v_scale apply)
  float k_scale, v_scale;
  // every context writes (m, l, o) partials to the workspace (layout of workspace_layout
  // with partials = true) instead of `out`; no merge grid runs
  bool partials_out;
};

// Resolved partition size in tokens, or -1 if `partition_size` is not acceptable.
// 0 selects a default from the batch's shape and the cache's bytes per element
// (`kv_elem_bytes`: 2 for 16-bit caches, 1 for E4M3; pure host arithmetic).
int resolve_partition_tokens(int partition_size, int block_size, int num_seqs, int num_q_heads,
                             int num_kv_heads, int max_blocks_per_seq, int kv_elem_bytes = 2);

// Workspace layout shared by the size query and the launcher.
struct WorkspaceLayout {
  size_t o_offset, ml_offset, order_offset, total;
  int max_parts;
};
// partials: lay the partials out even when no context can span two partitions.
WorkspaceLayout workspace_layout(int num_seqs, int num_q_heads, int head_dim, int block_size,
                                 int max_blocks_per_seq, int partition_tokens,
                                 bool partials = false);

// Whether the tensor-core path serves this shape (otherwise the CUDA-core path does).
bool decode_uses_tensor_cores(pkv_dtype dtype, int head_dim, int block_size);
// Whether any decode path serves this shape.
bool decode_supported(pkv_dtype dtype, int head_dim, int block_size);

// Whether the fp8-cache decode serves this q/out type and shape.
bool decode_fp8_supported(pkv_dtype dtype, int head_dim, int block_size);

int launch_decode(const DecodeArgs& a, cudaStream_t stream);

struct PrefillArgs {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start;
  int num_seqs, num_q_tokens, max_query_len, num_q_heads, num_kv_heads, head_dim, block_size;
  int max_blocks_per_seq, num_blocks;
  float scale;
  pkv_dtype dtype;
  unsigned* err;
  // options of the tcgen05 kernel (zero / null for chunked prefill)
  const int32_t* kv_start;    // per sequence, first attended position (a block multiple)
  const int32_t* table_rows;  // per sequence, the block-table row it reads
  bool non_causal;            // every row attends all of [kv_start, context_len)
  float* part_o;              // write (m, l, o) partials instead of `out`
  float* part_ml;
  int ksplit;                 // key ranges per sequence, one partial each (non-causal)
};

// Whether the chunked-prefill kernel's tcgen05 path (the one with the options above)
// serves this shape.
bool prefill_umma_supported(pkv_dtype dtype, int head_dim, int block_size, int group,
                            float scale);

// Whether the chunked-prefill kernel serves this element type and shape.
bool prefill_supported(pkv_dtype dtype, int head_dim, int block_size);

int launch_prefill(const PrefillArgs& a, cudaStream_t stream);

struct SharedPrefixArgs {
  void* out;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* group_start;  // [num_groups + 1]: group g = sequences group_start[g] ..
  const int32_t* prefix_lens;  // [num_groups]: shared prefix tokens (whole blocks)
  int num_seqs, num_groups, max_group_size, max_prefix_tokens;
  int num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq, num_blocks;
  float scale;
  pkv_dtype dtype;
  void* workspace;
  size_t workspace_bytes;
  unsigned* err;
};

size_t shared_prefix_workspace_size(int num_seqs, int num_groups, int num_q_heads,
                                    int num_kv_heads, int block_size, int max_blocks_per_seq,
                                    int max_group_size, int max_prefix_tokens);
int launch_shared_prefix(const SharedPrefixArgs& a, cudaStream_t stream);

int launch_kv_cache_write_fp8(const void* k, const void* v, void* k_cache, void* v_cache,
                              const int64_t* slot_mapping, int num_tokens, int row_elems,
                              pkv_dtype src_dtype, long long num_rows, float k_scale,
                              float v_scale, unsigned* err, cudaStream_t stream);

int launch_kv_cache_write(const void* k, const void* v, void* k_cache, void* v_cache,
                          const int64_t* slot_mapping, int num_tokens, size_t row_bytes,
                          long long num_rows, unsigned* err, cudaStream_t stream);

int launch_kv_copy_blocks(void* cache, const int64_t* pairs, int num_pairs, size_t block_bytes,
                          int num_blocks, unsigned* err, cudaStream_t stream);

int launch_kv_swap_blocks(void* dst, const void* src, const int64_t* pairs, int num_pairs,
                          size_t block_bytes, int dst_blocks, int src_blocks, unsigned* err,
                          cudaStream_t stream);

size_t dtype_size(pkv_dtype dtype);

}  // namespace pkv
