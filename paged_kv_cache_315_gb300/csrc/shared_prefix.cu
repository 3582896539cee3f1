// shared_prefix.cu -- decode attention for sequences that share a physical prefix.
//
// "PagedAttention: how vLLM manages the KV cache", section "Copy-on-write makes shared
// prefixes practical": sequences forked from one prompt map the same physical blocks for
// their common prefix.  Plain decode reads those blocks once per sequence.  Here a group
// of sequences that share their first prefix_lens[g] tokens (whole blocks) is served as a
// cascade:
//   1. prefix pass: every query of the group meets each prefix block once -- a dense,
//      non-causal multi-query attention on the tensor cores (the chunked-prefill tcgen05
//      kernel, key range split across CTAs), giving (m, l, o) partials per query row;
//   2. suffix pass: the decode kernel over each sequence's own tokens [prefix, L) (its
//      block-table row shifted by the prefix blocks), writing its partition partials;
//   3. merge: out = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i over the partials, which
//      equals the single-pass softmax-weighted sum up to rounding order.
#include <algorithm>
#include <climits>

#include "device_common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kPrepThreads = 256;
constexpr int kMergeWarps = 4;
constexpr int kMinSplitKeys = 128;  // keys per prefix split, at least

// Per (sequence, table entry): the suffix pass's block table (sequence s's row shifted by
// its prefix blocks) and, once per sequence, the prefix length and the suffix length.  A
// group whose run is longer than max_group_size, or whose prefix length is negative, not
// whole blocks, above max_prefix_tokens or longer than a member's context, is flagged and
// its members are served without the prefix pass (the suffix pass covers their context).
__global__ void __launch_bounds__(kPrepThreads)
    shared_prefix_prep(const int32_t* __restrict__ group_start,
                       const int32_t* __restrict__ prefix_lens,
                       const int32_t* __restrict__ context_lens,
                       const int32_t* __restrict__ block_tables, int num_seqs, int num_groups,
                       int block_size, int max_blocks_per_seq, int max_group_size,
                       int max_prefix_tokens, int32_t* seq_prefix, int32_t* suffix_lens,
                       int32_t* suffix_tables, unsigned* err) {
  const long long n = static_cast<long long>(num_seqs) * max_blocks_per_seq;
  for (long long e = static_cast<long long>(blockIdx.x) * kPrepThreads + threadIdx.x; e < n;
       e += static_cast<long long>(gridDim.x) * kPrepThreads) {
    const int s = static_cast<int>(e / max_blocks_per_seq);
    const int j = static_cast<int>(e - static_cast<long long>(s) * max_blocks_per_seq);
    // the group whose run holds s: the last g with group_start[g] <= s
    int lo = 0, hi = num_groups;
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (group_start[mid] <= s) lo = mid; else hi = mid;
    }
    const int L = context_lens[s];
    int pl = 0;
    if (num_groups > 0 && group_start[lo] <= s && s < group_start[lo + 1]) {
      pl = prefix_lens[lo];
      if (pl < 0 || pl % block_size != 0 || pl > max_prefix_tokens || pl > L ||
          group_start[lo + 1] - group_start[lo] > max_group_size) {
        if (j == 0) raise_error(err, PKV_DERR_CONTEXT);
        pl = 0;
      }
    }
    const int jb = j + pl / block_size;
    suffix_tables[e] =
        jb < max_blocks_per_seq ? block_tables[static_cast<size_t>(s) * max_blocks_per_seq + jb] : -1;
    if (j == 0) {
      seq_prefix[s] = pl;
      suffix_lens[s] = L - pl;
    }
  }
}

// One warp per (sequence, query head): merge the prefix pass's ksplit partials (when the
// sequence's group has a prefix) with the suffix decode's partition partials.  Lane i loads
// partial i's (m, l), so the weights take one load round trip; the o slices of all
// partials are then loaded together.
template <typename T>
__global__ void __launch_bounds__(kMergeWarps * 32)
    shared_prefix_merge(T* __restrict__ out, const float* __restrict__ pre_o,
                        const float* __restrict__ pre_ml, const float* __restrict__ dec_o,
                        const float* __restrict__ dec_ml, const int32_t* __restrict__ seq_prefix,
                        const int32_t* __restrict__ suffix_lens, int num_seqs, int num_q_heads,
                        int ksplit, int part_tokens, int max_parts) {
  constexpr int D = 128, V = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * kMergeWarps + warp;
  const long long rows = static_cast<long long>(num_seqs) * num_q_heads;
  if (row >= rows) return;
  const int s = static_cast<int>(row / num_q_heads);
  const int npre = seq_prefix[s] > 0 ? ksplit : 0;
  const int sl = max(suffix_lens[s], 0);
  const int nsuf = min((sl + part_tokens - 1) / part_tokens, max_parts);
  const int np = npre + nsuf;
  auto ml_of = [&](int i) -> const float* {
    return i < npre ? pre_ml + (static_cast<size_t>(i) * rows + row) * 2
                    : dec_ml + (static_cast<size_t>(row) * max_parts + (i - npre)) * 2;
  };
  auto o_of = [&](int i) -> const float* {
    return i < npre ? pre_o + (static_cast<size_t>(i) * rows + row) * D
                    : dec_o + (static_cast<size_t>(row) * max_parts + (i - npre)) * D;
  };
  float acc[V] = {0.f, 0.f, 0.f, 0.f};
  float den = 0.f;
  if (np <= 32) {
    float mi = -INFINITY, li = 0.f;
    if (lane < np) {
      const float2 x = __ldcg(reinterpret_cast<const float2*>(ml_of(lane)));
      mi = x.x;
      li = x.y;
    }
    float M = li > 0.f ? mi : -INFINITY;  // empty key ranges do not count
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float wi = li > 0.f ? exp2f(mi - M) : 0.f;
    den = wi * li;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
#pragma unroll 4
    for (int i = 0; i < np; ++i) {
      const float w = __shfl_sync(0xffffffffu, wi, i);
      if (w == 0.f) continue;
      const float4 x = __ldcg(reinterpret_cast<const float4*>(o_of(i) + lane * V));
      acc[0] += w * x.x;
      acc[1] += w * x.y;
      acc[2] += w * x.z;
      acc[3] += w * x.w;
    }
  } else {
    // more than 32 partials (very long suffixes): a plain two-pass merge
    float M = -INFINITY;
    for (int i = 0; i < np; ++i) {
      const float2 x = __ldcg(reinterpret_cast<const float2*>(ml_of(i)));
      if (x.y > 0.f) M = fmaxf(M, x.x);
    }
    for (int i = 0; i < np; ++i) {
      const float2 x = __ldcg(reinterpret_cast<const float2*>(ml_of(i)));
      if (!(x.y > 0.f)) continue;
      const float w = exp2f(x.x - M);
      den += w * x.y;
      const float4 y = __ldcg(reinterpret_cast<const float4*>(o_of(i) + lane * V));
      acc[0] += w * y.x;
      acc[1] += w * y.y;
      acc[2] += w * y.z;
      acc[3] += w * y.w;
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;  // an empty context gives zeros
  T* o = out + row * D + lane * V;
#pragma unroll
  for (int k = 0; k < V; ++k) o[k] = from_f32<T>(acc[k] * inv);
}

struct Plan {
  int ksplit, part_tokens;
  WorkspaceLayout dec;
  size_t pre_o, pre_ml, dec_off, seq_prefix, suffix_lens, suffix_tables, total;
};

Plan plan(int num_seqs, int num_groups, int num_q_heads, int num_kv_heads, int block_size,
          int max_blocks_per_seq, int max_group_size, int max_prefix_tokens) {
  Plan p{};
  const int group = num_q_heads / num_kv_heads;
  const long long m_tiles = (static_cast<long long>(max_group_size) * group + 127) / 128;
  const long long base =
      std::max(1LL, static_cast<long long>(num_groups) * m_tiles * num_kv_heads);
  // enough prefix-pass CTAs for two per SM, but at least kMinSplitKeys keys each
  const long long want = (2 * 152 + base - 1) / base;
  const long long cap = std::max(1, (max_prefix_tokens + kMinSplitKeys - 1) / kMinSplitKeys);
  p.ksplit = static_cast<int>(std::max(1LL, std::min(want, cap)));
  p.part_tokens = resolve_partition_tokens(0, block_size, num_seqs, num_q_heads, num_kv_heads,
                                           max_blocks_per_seq);
  p.dec = workspace_layout(num_seqs, num_q_heads, 128, block_size, max_blocks_per_seq,
                           p.part_tokens, true);
  const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads;
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  p.pre_o = 0;
  p.pre_ml = p.pre_o + up(p.ksplit * rows * 128 * sizeof(float));
  p.dec_off = p.pre_ml + up(p.ksplit * rows * 2 * sizeof(float));
  p.seq_prefix = p.dec_off + up(p.dec.total);
  p.suffix_lens = p.seq_prefix + up(num_seqs * sizeof(int32_t));
  p.suffix_tables = p.suffix_lens + up(num_seqs * sizeof(int32_t));
  p.total = p.suffix_tables +
            up(static_cast<size_t>(num_seqs) * max_blocks_per_seq * sizeof(int32_t));
  return p;
}

}  // namespace

size_t shared_prefix_workspace_size(int num_seqs, int num_groups, int num_q_heads,
                                    int num_kv_heads, int block_size, int max_blocks_per_seq,
                                    int max_group_size, int max_prefix_tokens) {
  return plan(num_seqs, num_groups, num_q_heads, num_kv_heads, block_size, max_blocks_per_seq,
              max_group_size, max_prefix_tokens)
      .total;
}

int launch_shared_prefix(const SharedPrefixArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0) return PKV_OK;
  const Plan pl = plan(a.num_seqs, a.num_groups, a.num_q_heads, a.num_kv_heads, a.block_size,
                       a.max_blocks_per_seq, a.max_group_size, a.max_prefix_tokens);
  if (pl.part_tokens <= 0) return PKV_EINVAL;
  if (!a.workspace || a.workspace_bytes < pl.total) return PKV_ENOMEM;
  char* ws = static_cast<char*>(a.workspace);
  float* pre_o = reinterpret_cast<float*>(ws + pl.pre_o);
  float* pre_ml = reinterpret_cast<float*>(ws + pl.pre_ml);
  char* dec = ws + pl.dec_off;
  int32_t* seq_prefix = reinterpret_cast<int32_t*>(ws + pl.seq_prefix);
  int32_t* suffix_lens = reinterpret_cast<int32_t*>(ws + pl.suffix_lens);
  int32_t* suffix_tables = reinterpret_cast<int32_t*>(ws + pl.suffix_tables);

  const long long elems = static_cast<long long>(a.num_seqs) * a.max_blocks_per_seq;
  const int pgrid = static_cast<int>(std::min<long long>((elems + kPrepThreads - 1) / kPrepThreads,
                                                         4 * 152));
  shared_prefix_prep<<<pgrid, kPrepThreads, 0, stream>>>(
      a.group_start, a.prefix_lens, a.context_lens, a.block_tables, a.num_seqs, a.num_groups,
      a.block_size, a.max_blocks_per_seq, a.max_group_size, a.max_prefix_tokens, seq_prefix,
      suffix_lens, suffix_tables, a.err);
  if (cudaGetLastError() != cudaSuccess) return PKV_ECUDA;

  const bool prefix_pass = a.num_groups > 0 && a.max_group_size > 0 && a.max_prefix_tokens > 0;
  if (prefix_pass) {
    // prefix pass: "sequence" g = group g, its query rows the members' rows, its keys the
    // prefix blocks of the first member's table (tensor cores, key range split in ksplit)
    PrefillArgs pre{};
    pre.q = a.q;
    pre.k_cache = a.k_cache;
    pre.v_cache = a.v_cache;
    pre.block_tables = a.block_tables;
    pre.num_q_tokens = a.num_seqs;  // q is [num_seqs, Hq, D]: one query row per sequence
    pre.num_q_heads = a.num_q_heads;
    pre.num_kv_heads = a.num_kv_heads;
    pre.head_dim = a.head_dim;
    pre.block_size = a.block_size;
    pre.max_blocks_per_seq = a.max_blocks_per_seq;
    pre.num_blocks = a.num_blocks;
    pre.scale = a.scale;
    pre.dtype = a.dtype;
    pre.err = a.err;
    pre.non_causal = true;
    pre.num_seqs = a.num_groups;
    pre.query_start = a.group_start;
    pre.context_lens = a.prefix_lens;
    pre.table_rows = a.group_start;
    pre.max_query_len = a.max_group_size;
    pre.part_o = pre_o;
    pre.part_ml = pre_ml;
    pre.ksplit = pl.ksplit;
    const int rc = launch_prefill(pre, stream);
    if (rc != PKV_OK) return rc;
  }
  // suffix pass: the decode kernel over each sequence's own tokens, partials out
  DecodeArgs d{};
  d.out = a.out;
  d.q = a.q;
  d.k_cache = a.k_cache;
  d.v_cache = a.v_cache;
  d.block_tables = suffix_tables;
  d.context_lens = suffix_lens;
  d.num_seqs = a.num_seqs;
  d.num_q_heads = a.num_q_heads;
  d.num_kv_heads = a.num_kv_heads;
  d.head_dim = a.head_dim;
  d.block_size = a.block_size;
  d.max_blocks_per_seq = a.max_blocks_per_seq;
  d.num_blocks = a.num_blocks;
  d.scale = a.scale;
  d.dtype = a.dtype;
  d.partition_tokens = pl.part_tokens;
  d.workspace = dec;
  d.workspace_bytes = pl.dec.total;
  d.err = a.err;
  d.partials_out = true;
  int rc = launch_decode(d, stream);
  if (rc != PKV_OK) return rc;

  const long long rows = static_cast<long long>(a.num_seqs) * a.num_q_heads;
  const unsigned grid = static_cast<unsigned>((rows + kMergeWarps - 1) / kMergeWarps);
  const float* dec_o = reinterpret_cast<const float*>(dec + pl.dec.o_offset);
  const float* dec_ml = reinterpret_cast<const float*>(dec + pl.dec.ml_offset);
  const int ks = prefix_pass ? pl.ksplit : 0;
  if (a.dtype == PKV_BF16)
    shared_prefix_merge<__nv_bfloat16><<<grid, kMergeWarps * 32, 0, stream>>>(
        static_cast<__nv_bfloat16*>(a.out), pre_o, pre_ml, dec_o, dec_ml, seq_prefix, suffix_lens,
        a.num_seqs, a.num_q_heads, ks, pl.part_tokens, pl.dec.max_parts);
  else
    shared_prefix_merge<__half><<<grid, kMergeWarps * 32, 0, stream>>>(
        static_cast<__half*>(a.out), pre_o, pre_ml, dec_o, dec_ml, seq_prefix, suffix_lens,
        a.num_seqs, a.num_q_heads, ks, pl.part_tokens, pl.dec.max_parts);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

}  // namespace pkv
