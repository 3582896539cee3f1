// api.cu -- the extern "C" entry points of libpagedkv: argument validation, dispatch to
// the kernel launchers, and the device error word.
#include <cuda_runtime.h>

#include <climits>
#include <mutex>

#include "device_common.cuh"
#include "internal.h"
#include "pagedkv.h"

namespace pkv {
namespace {

// Data errors found by kernels (PKV_DERR_* bits); one word per device.
__device__ unsigned g_error_word;

constexpr int kMaxDevices = 64;

// Device address of this device's error word (host code may not take it directly).
unsigned* error_word() {
  static unsigned* addr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<unsigned*>(p);
  }
  return addr[dev];
}

bool aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

// One thread waits on a fresh mbarrier, through the same bounded wait the pipelines use,
// for at most `limit_ns`; the barrier completes only if `arrive` is set.  A wait that
// runs out sets PKV_DERR_TIMEOUT and the kernel returns normally.
__global__ void bounded_wait_selftest(unsigned long long limit_ns, int arrive, unsigned* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  const uint32_t b = smem_addr(&bar);
  mbar_init(b, 1);
  fence_mbar_init();
  if (arrive) mbar_arrive_expect_tx(b, 0);
  if (!mbar_wait_for(b, 0, limit_ns)) raise_error(err, PKV_DERR_TIMEOUT);
}

bool valid_dtype(pkv_dtype d) { return d == PKV_F32 || d == PKV_BF16 || d == PKV_F16; }

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" {

int paged_attn_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                      int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                      int max_blocks_per_seq, int num_blocks, float scale, pkv_dtype dtype,
                      int partition_size, void* workspace, size_t workspace_bytes,
                      pkv_stream_t stream) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      block_size <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || !valid_dtype(dtype))
    return PKV_EINVAL;
  if (num_q_heads % num_kv_heads != 0) return PKV_EINVAL;
  if (static_cast<long long>(num_blocks) * block_size >= INT_MAX) return PKV_EINVAL;
  if (static_cast<long long>(max_blocks_per_seq) * block_size >= INT_MAX) return PKV_EINVAL;
  const int ptok = resolve_partition_tokens(partition_size, block_size, num_seqs, num_q_heads,
                                           num_kv_heads, max_blocks_per_seq);
  if (ptok < 0) return PKV_EINVAL;
  if (!decode_supported(dtype, head_dim, block_size)) return PKV_EUNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PKV_EINVAL;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 4) || !aligned(out, 4) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4))
    return PKV_EINVAL;
  if (workspace && !aligned(workspace, 16)) return PKV_EINVAL;
  unsigned* err = error_word();
  if (!err) return PKV_ECUDA;
  DecodeArgs a{};
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.scale = scale;
  a.dtype = dtype;
  a.partition_tokens = ptok;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.err = err;
  return launch_decode(a, reinterpret_cast<cudaStream_t>(stream));
}

int paged_attn_decode_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, const int32_t* context_lens, int num_seqs,
                          int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                          int max_blocks_per_seq, int num_blocks, float scale, float k_scale,
                          float v_scale, pkv_dtype dtype, int partition_size, void* workspace,
                          size_t workspace_bytes, pkv_stream_t stream) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      block_size <= 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || !valid_dtype(dtype))
    return PKV_EINVAL;
  if (num_q_heads % num_kv_heads != 0) return PKV_EINVAL;
  if (!(k_scale > 0.f) || !(v_scale > 0.f)) return PKV_EINVAL;
  if (static_cast<long long>(num_blocks) * block_size >= INT_MAX) return PKV_EINVAL;
  if (static_cast<long long>(max_blocks_per_seq) * block_size >= INT_MAX) return PKV_EINVAL;
  const int ptok = resolve_partition_tokens(partition_size, block_size, num_seqs, num_q_heads,
                                            num_kv_heads, max_blocks_per_seq, 1);
  if (ptok < 0) return PKV_EINVAL;
  if (!decode_fp8_supported(dtype, head_dim, block_size)) return PKV_EUNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PKV_EINVAL;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 4) || !aligned(out, 4) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4))
    return PKV_EINVAL;
  if (workspace && !aligned(workspace, 16)) return PKV_EINVAL;
  unsigned* err = error_word();
  if (!err) return PKV_ECUDA;
  DecodeArgs a{};
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.scale = scale;
  a.dtype = dtype;
  a.partition_tokens = ptok;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.err = err;
  a.kv_fp8 = true;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  return launch_decode(a, reinterpret_cast<cudaStream_t>(stream));
}

size_t paged_attn_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                        int head_dim, int block_size, int max_blocks_per_seq,
                                        int partition_size) {
  if (num_seqs <= 0 || num_q_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      max_blocks_per_seq <= 0)
    return 0;
  const int ptok = resolve_partition_tokens(partition_size, block_size, num_seqs, num_q_heads,
                                           num_kv_heads, max_blocks_per_seq);
  if (ptok < 0) return 0;
  return workspace_layout(num_seqs, num_q_heads, head_dim, block_size, max_blocks_per_seq, ptok)
      .total;
}

int paged_attn_decode_partition_tokens(int num_seqs, int num_q_heads, int num_kv_heads,
                                       int block_size, int max_blocks_per_seq,
                                       int partition_size) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || block_size <= 0 ||
      max_blocks_per_seq <= 0)
    return PKV_EINVAL;
  const int ptok = resolve_partition_tokens(partition_size, block_size, num_seqs, num_q_heads,
                                            num_kv_heads, max_blocks_per_seq);
  return ptok < 0 ? PKV_EINVAL : ptok;
}

size_t paged_attn_decode_fp8_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads,
                                            int head_dim, int block_size, int max_blocks_per_seq,
                                            int partition_size) {
  if (num_seqs <= 0 || num_q_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      max_blocks_per_seq <= 0)
    return 0;
  const int ptok = resolve_partition_tokens(partition_size, block_size, num_seqs, num_q_heads,
                                            num_kv_heads, max_blocks_per_seq, 1);
  if (ptok < 0) return 0;
  return workspace_layout(num_seqs, num_q_heads, head_dim, block_size, max_blocks_per_seq, ptok)
      .total;
}

int paged_attn_decode_fp8_partition_tokens(int num_seqs, int num_q_heads, int num_kv_heads,
                                           int block_size, int max_blocks_per_seq,
                                           int partition_size) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || block_size <= 0 ||
      max_blocks_per_seq <= 0)
    return PKV_EINVAL;
  const int ptok = resolve_partition_tokens(partition_size, block_size, num_seqs, num_q_heads,
                                            num_kv_heads, max_blocks_per_seq, 1);
  return ptok < 0 ? PKV_EINVAL : ptok;
}

int paged_attn_prefill(void* out, const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const int32_t* context_lens,
                       const int32_t* query_start, int num_seqs, int num_q_tokens,
                       int max_query_len, int num_q_heads, int num_kv_heads, int head_dim,
                       int block_size, int max_blocks_per_seq, int num_blocks, float scale,
                       pkv_dtype dtype, pkv_stream_t stream) {
  if (num_seqs < 0 || num_q_tokens < 0 || max_query_len < 0 || num_q_heads <= 0 ||
      num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || max_blocks_per_seq <= 0 ||
      num_blocks <= 0 || !valid_dtype(dtype))
    return PKV_EINVAL;
  if (num_q_heads % num_kv_heads != 0) return PKV_EINVAL;
  if (static_cast<long long>(num_blocks) * block_size >= INT_MAX) return PKV_EINVAL;
  if (static_cast<long long>(max_blocks_per_seq) * block_size >= INT_MAX) return PKV_EINVAL;
  if (!prefill_supported(dtype, head_dim, block_size)) return PKV_EUNSUPPORTED;
  if (num_seqs == 0 || num_q_tokens == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start)
    return PKV_EINVAL;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 4) || !aligned(out, 4) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(query_start, 4))
    return PKV_EINVAL;
  unsigned* err = error_word();
  if (!err) return PKV_ECUDA;
  PrefillArgs a{};
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.query_start = query_start;
  a.num_seqs = num_seqs;
  a.num_q_tokens = num_q_tokens;
  a.max_query_len = max_query_len;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.scale = scale;
  a.dtype = dtype;
  a.err = err;
  return launch_prefill(a, reinterpret_cast<cudaStream_t>(stream));
}

size_t paged_attn_decode_shared_prefix_workspace_size(int num_seqs, int num_groups,
                                                      int num_q_heads, int num_kv_heads,
                                                      int block_size, int max_blocks_per_seq,
                                                      int max_group_size, int max_prefix_tokens) {
  if (num_seqs <= 0 || num_groups < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      num_q_heads % num_kv_heads != 0 || block_size <= 0 || max_blocks_per_seq <= 0 ||
      max_group_size < 0 || max_prefix_tokens < 0)
    return 0;
  return shared_prefix_workspace_size(num_seqs, num_groups, num_q_heads, num_kv_heads,
                                      block_size, max_blocks_per_seq, max_group_size,
                                      max_prefix_tokens);
}

int paged_attn_decode_shared_prefix(void* out, const void* q, const void* k_cache,
                                    const void* v_cache, const int32_t* block_tables,
                                    const int32_t* context_lens, const int32_t* group_start,
                                    const int32_t* prefix_lens, int num_seqs, int num_groups,
                                    int max_group_size, int max_prefix_tokens, int num_q_heads,
                                    int num_kv_heads, int head_dim, int block_size,
                                    int max_blocks_per_seq, int num_blocks, float scale,
                                    pkv_dtype dtype, void* workspace, size_t workspace_bytes,
                                    pkv_stream_t stream) {
  if (num_seqs < 0 || num_groups < 0 || max_group_size < 0 || max_prefix_tokens < 0 ||
      num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      max_blocks_per_seq <= 0 || num_blocks <= 0 || !valid_dtype(dtype))
    return PKV_EINVAL;
  if (num_q_heads % num_kv_heads != 0) return PKV_EINVAL;
  if (static_cast<long long>(num_blocks) * block_size >= INT_MAX) return PKV_EINVAL;
  if (static_cast<long long>(max_blocks_per_seq) * block_size >= INT_MAX) return PKV_EINVAL;
  if (!prefill_umma_supported(dtype, head_dim, block_size, num_q_heads / num_kv_heads, scale))
    return PKV_EUNSUPPORTED;
  if (num_seqs == 0) return PKV_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens ||
      (num_groups > 0 && (!group_start || !prefix_lens)))
    return PKV_EINVAL;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 16) || !aligned(out, 4) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(group_start, 4) ||
      !aligned(prefix_lens, 4) || !aligned(workspace, 16))
    return PKV_EINVAL;
  unsigned* err = error_word();
  if (!err) return PKV_ECUDA;
  SharedPrefixArgs a{};
  a.out = out;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.group_start = group_start;
  a.prefix_lens = prefix_lens;
  a.num_seqs = num_seqs;
  a.num_groups = num_groups;
  a.max_group_size = max_group_size;
  a.max_prefix_tokens = max_prefix_tokens;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.block_size = block_size;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.scale = scale;
  a.dtype = dtype;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.err = err;
  return launch_shared_prefix(a, reinterpret_cast<cudaStream_t>(stream));
}

int kv_cache_write(const void* k, const void* v, void* k_cache, void* v_cache,
                   const int64_t* slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
                   int block_size, int num_blocks, pkv_dtype dtype, pkv_stream_t stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      num_blocks <= 0 || !valid_dtype(dtype))
    return PKV_EINVAL;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PKV_EINVAL;
  if (!aligned(slot_mapping, 8)) return PKV_EINVAL;
  unsigned* err = error_word();
  if (!err) return PKV_ECUDA;
  const size_t row_bytes = static_cast<size_t>(num_kv_heads) * head_dim * dtype_size(dtype);
  const long long rows = static_cast<long long>(num_blocks) * block_size;
  return launch_kv_cache_write(k, v, k_cache, v_cache, slot_mapping, num_tokens, row_bytes, rows,
                               err, reinterpret_cast<cudaStream_t>(stream));
}

int kv_cache_write_fp8(const void* k, const void* v, void* k_cache, void* v_cache,
                       const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                       int head_dim, int block_size, int num_blocks, pkv_dtype dtype,
                       float k_scale, float v_scale, pkv_stream_t stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      num_blocks <= 0 || !valid_dtype(dtype))
    return PKV_EINVAL;
  if (!(k_scale > 0.f) || !(v_scale > 0.f)) return PKV_EINVAL;
  const long long row_elems = static_cast<long long>(num_kv_heads) * head_dim;
  if (row_elems % 8 != 0 || row_elems > INT_MAX) return PKV_EINVAL;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PKV_EINVAL;
  if (!aligned(slot_mapping, 8) || !aligned(k_cache, 8) || !aligned(v_cache, 8)) return PKV_EINVAL;
  unsigned* err = error_word();
  if (!err) return PKV_ECUDA;
  return launch_kv_cache_write_fp8(k, v, k_cache, v_cache, slot_mapping, num_tokens,
                                   static_cast<int>(row_elems), dtype,
                                   static_cast<long long>(num_blocks) * block_size, k_scale,
                                   v_scale, err, reinterpret_cast<cudaStream_t>(stream));
}

int kv_copy_blocks(void* cache, const int64_t* src_dst_pairs, int num_pairs, size_t block_bytes,
                   int num_blocks, pkv_stream_t stream) {
  if (num_pairs < 0 || num_blocks <= 0 || block_bytes == 0) return PKV_EINVAL;
  if (num_pairs == 0) return PKV_OK;
  if (!cache || !src_dst_pairs || !aligned(src_dst_pairs, 8)) return PKV_EINVAL;
  unsigned* err = error_word();
  if (!err) return PKV_ECUDA;
  return launch_kv_copy_blocks(cache, src_dst_pairs, num_pairs, block_bytes, num_blocks, err,
                               reinterpret_cast<cudaStream_t>(stream));
}

int kv_swap_blocks(void* dst_cache, const void* src_cache, const int64_t* src_dst_pairs,
                   int num_pairs, size_t block_bytes, int dst_num_blocks, int src_num_blocks,
                   pkv_stream_t stream) {
  if (num_pairs < 0 || dst_num_blocks <= 0 || src_num_blocks <= 0 || block_bytes == 0)
    return PKV_EINVAL;
  if (num_pairs == 0) return PKV_OK;
  if (!dst_cache || !src_cache || !src_dst_pairs || !aligned(src_dst_pairs, 8)) return PKV_EINVAL;
  unsigned* err = error_word();
  if (!err) return PKV_ECUDA;
  return launch_kv_swap_blocks(dst_cache, src_cache, src_dst_pairs, num_pairs, block_bytes,
                               dst_num_blocks, src_num_blocks, err,
                               reinterpret_cast<cudaStream_t>(stream));
}

int pkv_selftest_bounded_wait(unsigned wait_us, int arrive, pkv_stream_t stream) {
  if (wait_us > 1000000u) return PKV_EINVAL;
  unsigned* err = error_word();
  if (!err) return PKV_ECUDA;
  bounded_wait_selftest<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<unsigned long long>(wait_us) * 1000ull, arrive, err);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

int pkv_device_error(pkv_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PKV_ECUDA;
  unsigned bits = 0;
  if (cudaMemcpyFromSymbol(&bits, g_error_word, sizeof bits) != cudaSuccess) return PKV_ECUDA;
  const unsigned zero = 0;
  if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof zero) != cudaSuccess) return PKV_ECUDA;
  return static_cast<int>(bits);
}

const char* pkv_strerror(int code) {
  switch (code) {
    case PKV_OK: return "success";
    case PKV_EINVAL: return "invalid argument";
    case PKV_ENOMEM: return "workspace too small";
    case PKV_ECUDA: return "CUDA runtime error";
    case PKV_EUNSUPPORTED: return "unsupported head_dim / block_size / dtype combination";
    case PKV_ESCRATCH: return "problem needs more scratch than the no-alloc decode provides";
    case PKV_ENODEVMEM: return "no device memory left to load the no-alloc decode's scratch array";
    case static_cast<int>(PKV_DERR_BLOCK_ID): return "device: block id out of range";
    case static_cast<int>(PKV_DERR_SLOT): return "device: slot out of range";
    case static_cast<int>(PKV_DERR_PAIR): return "device: copy pair id out of range";
    case static_cast<int>(PKV_DERR_CONTEXT): return "device: context length outside the block table";
    case static_cast<int>(PKV_DERR_TIMEOUT): return "device: pipeline wait timed out";
    default: return "unknown code";
  }
}

int pkv_version(void) { return 0x000100; }

}  // extern "C"
