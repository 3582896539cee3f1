// noalloc.cu -- paged_attn_decode for callers that cannot allocate device memory.
//
// The decode kernels need scratch memory when a context spans several partitions: the
// partitions' partial results and the work order of the decode grid.
// paged_attn_decode takes that scratch from the caller.  Some callers have no way to
// provide it: a host program that owns the device's whole memory budget and hands the
// library only the tensors of a call, or a hot path on which allocating is not allowed.
// This entry point serves them from a fixed array compiled into the library instead.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "pagedkv.h"

namespace pkv {
namespace {

// Scratch for paged_attn_decode_noalloc.  Every GPU that loads the library holds these
// bytes until the process exits; all calls on one device share them.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Device address of the scratch on the current device.  Host code cannot use the array's
// name as an address (on the host it names a stand-in object), so the address is looked
// up once per device, with that device current, and cached.
void* scratch_address(int* err) {
  static void* addr[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = PKV_ECUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      *err = PKV_ECUDA;
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace
}  // namespace pkv

extern "C" int paged_attn_decode_noalloc(void* out, const void* q, const void* k_cache,
                                         const void* v_cache, const int32_t* block_tables,
                                         const int32_t* context_lens, int num_seqs,
                                         int num_q_heads, int num_kv_heads, int head_dim,
                                         int block_size, int max_blocks_per_seq, int num_blocks,
                                         float scale, pkv_dtype dtype, int partition_size,
                                         pkv_stream_t stream) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      block_size <= 0 || max_blocks_per_seq <= 0)
    return PKV_EINVAL;
  // reject, before touching the device, a problem whose scratch would not fit
  const size_t need = paged_attn_decode_workspace_size(
      num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
      partition_size);
  if (need > static_cast<size_t>(PKV_NOALLOC_SCRATCH_BYTES)) return PKV_ESCRATCH;
  int err = PKV_OK;
  void* scratch = pkv::scratch_address(&err);
  if (!scratch) return err;
  // nothing in the scratch needs clearing: every byte a call reads it wrote first
  return paged_attn_decode(out, q, k_cache, v_cache, block_tables, context_lens, num_seqs,
                           num_q_heads, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
                           num_blocks, scale, dtype, partition_size, scratch,
                           static_cast<size_t>(PKV_NOALLOC_SCRATCH_BYTES), stream);
}
