// noalloc.cu -- paged_attn_decode for callers that cannot allocate device memory.
//
// The decode kernels need scratch memory when a context spans several partitions: the
// partitions' partial results and the work order of the decode grid.
// paged_attn_decode takes that scratch from the caller.  Some callers have no way to
// provide it: a host program that owns the device's whole memory budget and hands the
// library only the tensors of a call, or a hot path on which allocating is not allowed.
// This entry point serves them from a fixed array compiled into the library instead.
#include <cuda.h>
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

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <class Fn>
Fn driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<Fn>(p);
  return nullptr;
}

// Process-unique id of the context current on this thread (0 if none can be read).
// Context ids are never reused, unlike context handles, so a context destroyed and
// created again (cudaDeviceReset) shows up as a new id.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device address of the scratch in the current device's context.  Host code cannot use
// the array's name as an address (on the host it names a stand-in object), so the address
// is looked up with the device current and cached per device, together with the id of
// the context it belongs to; a call that finds another context current (the old one was
// destroyed, e.g. by cudaDeviceReset) looks it up again.  The first lookup in a context
// loads the library's module holding the array and so commits its bytes on the device;
// if the device has no memory left for it, the call returns PKV_ENODEVMEM.
void* scratch_address(int* err) {
  static void* addr[kMaxDevices] = {};
  static unsigned long long ctx_of[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = PKV_ECUDA;
    return nullptr;
  }
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev] || ctx == 0 || ctx != ctx_of[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      if (e != cudaSuccess) cudaGetLastError();  // do not leave the error to the next call
      *err = e == cudaErrorMemoryAllocation ? PKV_ENODEVMEM : PKV_ECUDA;
      addr[dev] = nullptr;
      return nullptr;
    }
    addr[dev] = p;
    ctx_of[dev] = ctx;
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
