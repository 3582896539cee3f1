// cache_ops.cu -- slot-mapped writes of new tokens and whole-block copies (sm_103a).
//
// Both are pure byte movement, bound by HBM bandwidth: each thread moves 16-byte vectors
// (narrower only when a size or pointer is not 16-byte aligned), grid-stride, with the
// grid sized to a multiple of the SM count.
#include <cuda_fp8.h>

#include <algorithm>

#include "device_common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kThreads = 256;

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

// k_cache row `slot` <- k row i (and the same for v); vec_per_row vectors of type V per row.
template <typename V>
__global__ void __launch_bounds__(kThreads)
    kv_write_kernel(const V* __restrict__ k, const V* __restrict__ v, V* __restrict__ kc,
                    V* __restrict__ vc, const int64_t* __restrict__ slots, long long num_tokens,
                    long long vec_per_row, long long num_rows, unsigned* err) {
  const long long total = num_tokens * vec_per_row;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const long long t = i / vec_per_row;
    const long long col = i - t * vec_per_row;
    // the row loads do not depend on the slot: all three are in flight together
    const long long slot = __ldg(&slots[t]);
    const V kv = __ldg(&k[i]);
    const V vv = __ldg(&v[i]);
    if (slot < 0) continue;  // padding
    if (slot >= num_rows) {
      if (col == 0) raise_error(err, PKV_DERR_SLOT);
      continue;
    }
    kc[slot * vec_per_row + col] = kv;
    vc[slot * vec_per_row + col] = vv;
  }
}

constexpr int kCopyUnroll = 4;  // vectors a thread moves per group (the grid gives it 4)

// cache block dst <- cache block src for every pair; blockIdx.y strides over pairs.
template <typename V>
__global__ void __launch_bounds__(kThreads)
    kv_copy_kernel(V* cache, const int64_t* __restrict__ pairs, int num_pairs,
                   long long vec_per_block, long long num_blocks, unsigned* err) {
  for (int pi = blockIdx.y; pi < num_pairs; pi += gridDim.y) {
    const long long src = __ldg(&pairs[2LL * pi]);
    const long long dst = __ldg(&pairs[2LL * pi + 1]);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      if (blockIdx.x == 0 && threadIdx.x == 0) raise_error(err, PKV_DERR_PAIR);
      continue;
    }
    if (src == dst) continue;
    const V* s = cache + src * vec_per_block;
    V* d = cache + dst * vec_per_block;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    // every load of a group before its stores: destinations never overlap sources (the
    // call's contract), so a thread keeps kCopyUnroll reads in flight instead of one
    for (; i + (kCopyUnroll - 1) * stride < vec_per_block; i += kCopyUnroll * stride) {
      V r[kCopyUnroll];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) r[u] = s[i + u * stride];
#pragma unroll
      for (int u = 0; u < kCopyUnroll; ++u) d[i + u * stride] = r[u];
    }
    for (; i < vec_per_block; i += stride) d[i] = s[i];
  }
}

// dst block <- src block of another pool for every pair; either pool may be device
// memory or host memory the device can address (pinned host memory, reached over
// NVLink-C2C on Grace-Blackwell); blockIdx.y strides over pairs.
template <typename V>
__global__ void __launch_bounds__(kThreads)
    kv_swap_kernel(V* __restrict__ dst, const V* __restrict__ src,
                   const int64_t* __restrict__ pairs, int num_pairs, long long vec_per_block,
                   long long dst_blocks, long long src_blocks, unsigned* err) {
  for (int pi = blockIdx.y; pi < num_pairs; pi += gridDim.y) {
    const long long s = __ldg(&pairs[2LL * pi]);
    const long long d = __ldg(&pairs[2LL * pi + 1]);
    if (s < 0 || s >= src_blocks || d < 0 || d >= dst_blocks) {
      if (blockIdx.x == 0 && threadIdx.x == 0) raise_error(err, PKV_DERR_PAIR);
      continue;
    }
    const V* sp = src + s * vec_per_block;
    V* dp = dst + d * vec_per_block;
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
         i < vec_per_block; i += stride)
      dp[i] = sp[i];
  }
}

// k_cache row `slot` <- E4M3 codes of k row i / k_scale (and v with v_scale); one thread
// per 8 elements.  The division is IEEE fp32; the conversion rounds to nearest even and
// saturates at +-448.
template <typename T>
__global__ void __launch_bounds__(kThreads)
    kv_write_fp8_kernel(const T* __restrict__ k, const T* __restrict__ v,
                        uint8_t* __restrict__ kc, uint8_t* __restrict__ vc,
                        const int64_t* __restrict__ slots, long long num_tokens, int row_elems,
                        long long num_rows, float k_scale, float v_scale, unsigned* err) {
  const int groups = row_elems / 8;
  const long long total = num_tokens * groups;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += stride) {
    const long long t = i / groups;
    const int e0 = static_cast<int>(i - t * groups) * 8;
    // the row loads do not depend on the slot: all of them are in flight together
    const long long slot = __ldg(&slots[t]);
    float fk[8], fv[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      fk[e] = to_f32(k[t * row_elems + e0 + e]);
      fv[e] = to_f32(v[t * row_elems + e0 + e]);
    }
    if (slot < 0) continue;
    if (slot >= num_rows) {
      if (e0 == 0) raise_error(err, PKV_DERR_SLOT);
      continue;
    }
    uint8_t ck[8], cv[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float xk = __fdiv_rn(fk[e], k_scale);
      const float xv = __fdiv_rn(fv[e], v_scale);
      ck[e] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(xk, __NV_SATFINITE, __NV_E4M3));
      cv[e] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(xv, __NV_SATFINITE, __NV_E4M3));
    }
    uint2 pk, pv;
    pk.x = ck[0] | (ck[1] << 8) | (ck[2] << 16) | (static_cast<uint32_t>(ck[3]) << 24);
    pk.y = ck[4] | (ck[5] << 8) | (ck[6] << 16) | (static_cast<uint32_t>(ck[7]) << 24);
    pv.x = cv[0] | (cv[1] << 8) | (cv[2] << 16) | (static_cast<uint32_t>(cv[3]) << 24);
    pv.y = cv[4] | (cv[5] << 8) | (cv[6] << 16) | (static_cast<uint32_t>(cv[7]) << 24);
    *reinterpret_cast<uint2*>(kc + slot * row_elems + e0) = pk;
    *reinterpret_cast<uint2*>(vc + slot * row_elems + e0) = pv;
  }
}

// Widest vector (16, 8, 4, 2 or 1 bytes) dividing `bytes` and every pointer's address.
int vector_bytes(size_t bytes, std::initializer_list<const void*> ptrs) {
  for (int w : {16, 8, 4, 2}) {
    bool ok = bytes % w == 0;
    for (const void* p : ptrs) ok = ok && (reinterpret_cast<uintptr_t>(p) % w == 0);
    if (ok) return w;
  }
  return 1;
}

template <typename V>
int write_with(const void* k, const void* v, void* kc, void* vc, const int64_t* slots,
               int num_tokens, size_t row_bytes, long long num_rows, unsigned* err,
               cudaStream_t stream) {
  const long long vpr = static_cast<long long>(row_bytes / sizeof(V));
  const long long total = static_cast<long long>(num_tokens) * vpr;
  const long long want = (total + kThreads - 1) / kThreads;
  const int grid = static_cast<int>(std::max(1LL, std::min(want, 8LL * sm_count())));
  kv_write_kernel<V><<<grid, kThreads, 0, stream>>>(
      static_cast<const V*>(k), static_cast<const V*>(v), static_cast<V*>(kc), static_cast<V*>(vc),
      slots, num_tokens, vpr, num_rows, err);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

template <typename V>
int copy_with(void* cache, const int64_t* pairs, int num_pairs, size_t block_bytes,
              int num_blocks, unsigned* err, cudaStream_t stream) {
  const long long vpb = static_cast<long long>(block_bytes / sizeof(V));
  // enough CTAs per pair that each thread moves about four vectors, capped so that all
  // pairs together fill the GPU a few times over
  const long long per_pair = std::max(1LL, (vpb + 4LL * kThreads - 1) / (4LL * kThreads));
  const int gy = std::min(num_pairs, 65535);
  const int gx = static_cast<int>(std::min(per_pair, 1024LL));
  kv_copy_kernel<V><<<dim3(gx, gy), kThreads, 0, stream>>>(static_cast<V*>(cache), pairs,
                                                           num_pairs, vpb, num_blocks, err);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

template <typename V>
int swap_with(void* dst, const void* src, const int64_t* pairs, int num_pairs, size_t block_bytes,
              int dst_blocks, int src_blocks, unsigned* err, cudaStream_t stream) {
  const long long vpb = static_cast<long long>(block_bytes / sizeof(V));
  const long long per_pair = std::max(1LL, (vpb + 4LL * kThreads - 1) / (4LL * kThreads));
  const int gy = std::min(num_pairs, 65535);
  const int gx = static_cast<int>(std::min(per_pair, 1024LL));
  kv_swap_kernel<V><<<dim3(gx, gy), kThreads, 0, stream>>>(
      static_cast<V*>(dst), static_cast<const V*>(src), pairs, num_pairs, vpb, dst_blocks,
      src_blocks, err);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

}  // namespace

int launch_kv_swap_blocks(void* dst, const void* src, const int64_t* pairs, int num_pairs,
                          size_t block_bytes, int dst_blocks, int src_blocks, unsigned* err,
                          cudaStream_t stream) {
  if (num_pairs == 0) return PKV_OK;
  switch (vector_bytes(block_bytes, {dst, src})) {
    case 16: return swap_with<uint4>(dst, src, pairs, num_pairs, block_bytes, dst_blocks, src_blocks, err, stream);
    case 8: return swap_with<uint2>(dst, src, pairs, num_pairs, block_bytes, dst_blocks, src_blocks, err, stream);
    case 4: return swap_with<uint32_t>(dst, src, pairs, num_pairs, block_bytes, dst_blocks, src_blocks, err, stream);
    case 2: return swap_with<uint16_t>(dst, src, pairs, num_pairs, block_bytes, dst_blocks, src_blocks, err, stream);
    default: return swap_with<uint8_t>(dst, src, pairs, num_pairs, block_bytes, dst_blocks, src_blocks, err, stream);
  }
}

int launch_kv_cache_write(const void* k, const void* v, void* k_cache, void* v_cache,
                          const int64_t* slot_mapping, int num_tokens, size_t row_bytes,
                          long long num_rows, unsigned* err, cudaStream_t stream) {
  if (num_tokens == 0) return PKV_OK;
  switch (vector_bytes(row_bytes, {k, v, k_cache, v_cache})) {
    case 16: return write_with<uint4>(k, v, k_cache, v_cache, slot_mapping, num_tokens, row_bytes, num_rows, err, stream);
    case 8: return write_with<uint2>(k, v, k_cache, v_cache, slot_mapping, num_tokens, row_bytes, num_rows, err, stream);
    case 4: return write_with<uint32_t>(k, v, k_cache, v_cache, slot_mapping, num_tokens, row_bytes, num_rows, err, stream);
    case 2: return write_with<uint16_t>(k, v, k_cache, v_cache, slot_mapping, num_tokens, row_bytes, num_rows, err, stream);
    default: return write_with<uint8_t>(k, v, k_cache, v_cache, slot_mapping, num_tokens, row_bytes, num_rows, err, stream);
  }
}

int launch_kv_cache_write_fp8(const void* k, const void* v, void* k_cache, void* v_cache,
                              const int64_t* slot_mapping, int num_tokens, int row_elems,
                              pkv_dtype src_dtype, long long num_rows, float k_scale,
                              float v_scale, unsigned* err, cudaStream_t stream) {
  if (num_tokens == 0) return PKV_OK;
  const long long total = static_cast<long long>(num_tokens) * (row_elems / 8);
  const int grid = static_cast<int>(
      std::max(1LL, std::min((total + kThreads - 1) / kThreads, 8LL * sm_count())));
  uint8_t* kc = static_cast<uint8_t*>(k_cache);
  uint8_t* vc = static_cast<uint8_t*>(v_cache);
  switch (src_dtype) {
    case PKV_F32:
      kv_write_fp8_kernel<float><<<grid, kThreads, 0, stream>>>(
          static_cast<const float*>(k), static_cast<const float*>(v), kc, vc, slot_mapping,
          num_tokens, row_elems, num_rows, k_scale, v_scale, err);
      break;
    case PKV_BF16:
      kv_write_fp8_kernel<__nv_bfloat16><<<grid, kThreads, 0, stream>>>(
          static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), kc, vc,
          slot_mapping, num_tokens, row_elems, num_rows, k_scale, v_scale, err);
      break;
    default:
      kv_write_fp8_kernel<__half><<<grid, kThreads, 0, stream>>>(
          static_cast<const __half*>(k), static_cast<const __half*>(v), kc, vc, slot_mapping,
          num_tokens, row_elems, num_rows, k_scale, v_scale, err);
  }
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

int launch_kv_copy_blocks(void* cache, const int64_t* pairs, int num_pairs, size_t block_bytes,
                          int num_blocks, unsigned* err, cudaStream_t stream) {
  if (num_pairs == 0) return PKV_OK;
  switch (vector_bytes(block_bytes, {cache})) {
    case 16: return copy_with<uint4>(cache, pairs, num_pairs, block_bytes, num_blocks, err, stream);
    case 8: return copy_with<uint2>(cache, pairs, num_pairs, block_bytes, num_blocks, err, stream);
    case 4: return copy_with<uint32_t>(cache, pairs, num_pairs, block_bytes, num_blocks, err, stream);
    case 2: return copy_with<uint16_t>(cache, pairs, num_pairs, block_bytes, num_blocks, err, stream);
    default: return copy_with<uint8_t>(cache, pairs, num_pairs, block_bytes, num_blocks, err, stream);
  }
}

}  // namespace pkv
