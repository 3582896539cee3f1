// decode.cu -- paged single-token decode attention for sm_103a.
//
// Work unit: one CTA per (sequence s, KV head g, query-head chunk c, context partition p).
// The CTA walks the partition's logical blocks j, resolves each through the block table
// to a physical block, and streams that block's K and V tiles ([block_size, head_dim]
// each, one KV head) into shared memory with TMA.  All query heads of KV head g that
// fall in chunk c are scored against every staged tile, so each cached byte leaves HBM
// once per call ("PagedAttention: how vLLM manages the KV cache": attention itself is
// unchanged, the kernel reads keys and values block by block through the request's
// logical-to-physical mapping).
//
// Pipeline: four consumer warps; logical block j goes to warp j % 4 and to ring stage
// j % S (S a multiple of 4, so every stage belongs to one warp).  Thread 0 issues the
// first S tile loads; afterwards the warp that finishes a stage refills it with the
// block S positions further on.  Each stage has one mbarrier (TMA transaction bytes);
// every wait gives up after ~1 s and sets PKV_DERR_TIMEOUT.
//
// Math per warp, per block: an online softmax in base 2 (scores pre-multiplied by
// scale*log2(e)): running max m, running sum l, unnormalised output o, rescaled by
// 2^(m_old - m_new) whenever the max grows.  The four warps' (m, l, o) are merged in
// shared memory at the end.  Contexts longer than one partition leave (m, l, o) per
// partition in the workspace, and a second grid (decode_merge_kernel, one warp per query
// head) merges them by log-sum-exp and writes the output.  Such split launches run three
// grids: a one-CTA prep kernel that orders the work longest first, the decode grid and
// the merge grid, the later two launched so that they start while the one ahead drains.
//
// With partitions of at most 1024 tokens and at most four query heads per KV head, one
// CTA streams two consecutive partitions through its ring (still one partial each), so
// the next partition's tiles are in flight while the previous one is merged.
//
// Tensor-core path (fp16/bf16, head_dim 64/128, block_size 16/32/64): S = Q.K^T and
// O += P.V with mma.sync m16n8k16 (fp32 accumulate); up to 16 query heads form the M
// rows.  Tiles arrive with the 128-byte TMA swizzle so ldmatrix reads are
// bank-conflict free.  CUDA-core path: everything else (fp32, other head sizes).
#include <algorithm>
#include <climits>
#include <mutex>

#include "device_common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kTcHeads = 16;    // query heads per CTA on the tensor-core path
constexpr int kFp8gHeads = 8;   // ... on the fp8 path with heads in the MMA's N dimension
constexpr int kSimtHeads = 8;   // ... on the CUDA-core path
constexpr int kMaxStageSet = 4; // stages per warp, at most
constexpr int kMaxParts = 1024; // partitions per sequence, at most
constexpr float kRescaleSlack = 8.f;  // see online_softmax
constexpr long long kMinUnits = 2048;  // work units the default partition size aims for

struct Params {
  void* out;
  const void* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* ws_o;
  float* ws_ml;
  unsigned* err;
  int num_seqs, num_q_heads, num_kv_heads, group, head_chunk, num_chunks;
  int max_blocks_per_seq, num_blocks, block_size;
  int partition_blocks, max_parts, stages;
  int tile_bytes;   // bytes of one K (or V) tile
  int tile_stride;  // tile_bytes rounded up to 1024: V tile offset inside a stage
  int stage_bytes, box_bytes, box_cols, boxes, ring_bytes;
  int pair;         // physical blocks per staged tile (2 pairs 16-token blocks for fp8)
  int ppc;          // partitions per CTA: streamed back to back, one partial each
  int max_groups;   // CTAs per (sequence, KV head, head chunk) = ceil(max_parts / ppc)
  int merge_off;    // byte offset of the merge buffer from the ring (0: the ring itself)
  const int32_t* order;  // CTA work order over (sequence, partition group) items, or null
  int force_partials;    // every context leaves (m, l, o) partials, none writes `out`
  int fold;              // a CTA folds its ppc partitions into one partial (see finish_part)
  float scale_log2;
  float out_scale;  // multiplies every output (the V scale of fp8 caches, else 1)
};

struct Work {
  int s, g, c, p;
  int np;         // partitions of this sequence
  int blk0;       // first logical block of the partition
  int nblk;       // blocks in the partition
  int tok_valid;  // tokens of the partition that are live
  int h0, hc;     // first query head and number of heads of this CTA
  int nparts;     // partitions this CTA covers, starting at p
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Decode blockIdx into a work unit: (item, KV head, head chunk) from slowest to fastest,
// so the KV heads of one physical block are read by neighbouring CTAs.  An item is a
// (sequence, group of ppc partitions) pair, taken in sequence-major order or, when the
// launch carries one, in the order decode_prep_kernel wrote.  Returns false when the CTA has nothing to do (after writing zeros for an empty
// context).  `spec_id` receives this thread's entry of the partition's block-table row,
// loaded before the context length is known so that the two loads overlap (an entry past
// the context is loaded but never used).
template <typename T>
__device__ bool decode_work(const Params& P, int D, Work& w, int& spec_id) {
  // Launched behind the prep kernel, this grid may start before it ends: wait for it (a
  // no-op otherwise).  Every CTA has started once all pass here, which lets the merge
  // kernel behind this grid be scheduled into the slots the tail leaves free.
  griddep_wait();
  griddep_launch_dependents();
  long long bid = blockIdx.x;
  w.c = static_cast<int>(bid % P.num_chunks);
  bid /= P.num_chunks;
  w.g = static_cast<int>(bid % P.num_kv_heads);
  bid /= P.num_kv_heads;
  const int item = P.order ? P.order[bid] : static_cast<int>(bid);
  w.p = (item % P.max_groups) * P.ppc;
  w.s = item / P.max_groups;
  w.h0 = w.g * P.group + w.c * P.head_chunk;
  w.hc = min(P.head_chunk, P.group - w.c * P.head_chunk);
  const int jb = w.p * P.partition_blocks + static_cast<int>(threadIdx.x);
  spec_id = (static_cast<int>(threadIdx.x) < P.partition_blocks * P.ppc &&
             jb < P.max_blocks_per_seq)
                ? __ldg(&P.block_tables[static_cast<size_t>(w.s) * P.max_blocks_per_seq + jb])
                : -1;
  int L = P.context_lens[w.s];
  const int Lmax = P.max_blocks_per_seq * P.block_size;
  if (L < 0 || L > Lmax) {
    if (threadIdx.x == 0 && w.p == 0 && w.g == 0 && w.c == 0) raise_error(P.err, PKV_DERR_CONTEXT);
    L = L < 0 ? 0 : Lmax;
  }
  const int ptok = P.partition_blocks * P.block_size;
  w.np = (L + ptok - 1) / ptok;
  if (L == 0) {
    if (w.p == 0) {
      T* out = static_cast<T*>(P.out) + (static_cast<size_t>(w.s) * P.num_q_heads + w.h0) * D;
      for (int i = threadIdx.x; i < w.hc * D; i += kThreads) out[i] = from_f32<T>(0.f);
    }
    return false;
  }
  if (w.p >= w.np) return false;
  w.nparts = min(P.ppc, w.np - w.p);
  w.blk0 = w.p * P.partition_blocks;
  w.tok_valid = min(P.ppc * ptok, L - w.p * ptok);
  w.nblk = (w.tok_valid + P.block_size - 1) / P.block_size;
  return true;
}

struct Smem {
  float* merge;  // [kWarps][head_chunk][D] o, then [kWarps][head_chunk][2] (m, l)
  uint8_t* ring;
  uint64_t* bars;
  int* ycoord;
};

__device__ __forceinline__ Smem carve(uint8_t* raw, const Params& P) {
  Smem s;
  const uint32_t a = smem_addr(raw);
  s.ring = raw + ((1024u - (a & 1023u)) & 1023u);
  s.bars = reinterpret_cast<uint64_t*>(s.ring + P.ring_bytes);
  s.ycoord = reinterpret_cast<int*>(s.bars + P.stages);
  s.merge = reinterpret_cast<float*>(s.ring + P.merge_off);
  return s;
}

// Resolve the partition's block ids to TMA row coordinates (invalid ids point past the
// tensor, so their tiles load as zeros), initialise the stage barriers and issue the
// first S tile loads.  Called by every thread of the CTA.
__device__ __forceinline__ void pipeline_start(const Params& P, const Work& w, const Smem& sm,
                                               const CUtensorMap* kmap, const CUtensorMap* vmap,
                                               int x0, int spec_id);

// Load staged tile v: physical blocks v*pair .. v*pair + pair - 1 of the partition (those
// that exist), stacked row-wise so that two 16-row boxes form the layout of one 32-row box.
__device__ __forceinline__ void issue_tile(const Params& P, const Smem& sm, const CUtensorMap* kmap,
                                           const CUtensorMap* vmap, int v, int x0, int nblk) {
  const int st = v % P.stages;
  const uint32_t bar = smem_addr(&sm.bars[st]);
  const uint32_t kdst = smem_addr(sm.ring + st * P.stage_bytes);
  const uint32_t vdst = kdst + P.tile_stride;
  const int j0 = v * P.pair;
  const int cnt = min(P.pair, nblk - j0);
  mbar_arrive_expect_tx(bar, 2u * cnt * P.tile_bytes);
  for (int i = 0; i < cnt; ++i) {
    const int y = sm.ycoord[j0 + i];
    for (int b = 0; b < P.boxes; ++b) {
      const uint32_t off = b * P.pair * P.box_bytes + i * P.box_bytes;
      tma_load_2d(kdst + off, kmap, bar, x0 + b * P.box_cols, y);
      tma_load_2d(vdst + off, vmap, bar, x0 + b * P.box_cols, y);
    }
  }
}

// Stage and barrier phase of a warp's staged tiles.  Tile v sits in stage v % stages and
// completes phase (v / stages) & 1 of that stage's barrier.  A warp visits tiles v,
// v + kWarps, v + 2 kWarps, ... and the stage count is a multiple of kWarps, so both
// advance without a division.
struct StageCursor {
  int st, ph;
  __device__ __forceinline__ StageCursor(int v, int stages)
      : st(v % stages), ph((v / stages) & 1) {}
  __device__ __forceinline__ void next(int stages) {
    st += kWarps;
    if (st >= stages) {
      st -= stages;
      ph ^= 1;
    }
  }
};

// issue_tile for one physical block per stage (pair 1) with BOXES boxes per row segment,
// into stage `st` (the stage of the tile it replaces); `y` is the block's TMA row.
template <int BOXES>
__device__ __forceinline__ void issue_block(const Params& P, const Smem& sm,
                                            const CUtensorMap* kmap, const CUtensorMap* vmap,
                                            int st, int y, int x0) {
  const uint32_t bar = smem_addr(&sm.bars[st]);
  const uint32_t kdst = smem_addr(sm.ring + st * P.stage_bytes);
  const uint32_t vdst = kdst + P.tile_stride;
  mbar_arrive_expect_tx(bar, 2u * P.tile_bytes);
#pragma unroll
  for (int b = 0; b < BOXES; ++b) {
    tma_load_2d(kdst + b * P.box_bytes, kmap, bar, x0 + b * P.box_cols, y);
    tma_load_2d(vdst + b * P.box_bytes, vmap, bar, x0 + b * P.box_cols, y);
  }
}

__device__ __forceinline__ void pipeline_start(const Params& P, const Work& w, const Smem& sm,
                                               const CUtensorMap* kmap, const CUtensorMap* vmap,
                                               int x0, int spec_id) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto row_of = [&](int id) {
    if (id < 0 || id >= P.num_blocks) {
      raise_error(P.err, PKV_DERR_BLOCK_ID);
      id = P.num_blocks;
    }
    return id * P.block_size;
  };
  // the first kThreads ids were loaded by decode_work (one per thread)
  if (tid < w.nblk) sm.ycoord[tid] = row_of(spec_id);
  if (tid == 0) {
    tma_prefetch_desc(kmap);
    tma_prefetch_desc(vmap);
    for (int i = 0; i < P.stages; ++i) mbar_init(smem_addr(&sm.bars[i]), 1);
    fence_mbar_init();
  }
  __syncthreads();
  // Each warp issues the first tiles of its own stages (tile v: stage v, owner warp v % 4);
  // they need at most stages * pair ids, all among the first kThreads.
  static_assert(kWarps * kMaxStageSet * 2 <= kThreads, "first tiles' ids come from decode_work");
  if (lane == 0) {
    const int nv = (w.nblk + P.pair - 1) / P.pair;
    const int first = min(P.stages, nv);
    for (int v = warp; v < first; v += kWarps) issue_tile(P, sm, kmap, vmap, v, x0, w.nblk);
  }
  // ids past the first kThreads: loaded while the first tiles are in flight
  if (w.nblk > kThreads) {
    const int32_t* bt = P.block_tables + static_cast<size_t>(w.s) * P.max_blocks_per_seq + w.blk0;
    for (int j = tid + kThreads; j < w.nblk; j += kThreads) sm.ycoord[j] = row_of(bt[j]);
    __syncthreads();
  }
}

// After a timed-out wait on block j: wait (bounded) for this warp's loads still in flight.
__device__ __forceinline__ void drain_after_timeout(const Params& P, const Work& w, const Smem& sm,
                                                    int j) {
  const int end = min((w.nblk + P.pair - 1) / P.pair, j + P.stages);
  for (int jj = j; jj < end; jj += kWarps)
    mbar_wait_bounded(smem_addr(&sm.bars[jj % P.stages]), (jj / P.stages) & 1);
}

// Merge the four warps' (m, l, o) of each query head; write the output (a context of one
// partition) or this partition's partial (m, l, o), which decode_merge_kernel reduces.
// O_s: [kWarps][HC][D] floats, ml_s: [kWarps][HC][2] (m in log2 units, l).
template <typename T>
__device__ void finish(const Params& P, const Work& w, int D, int HC, const float* O_s,
                       const float* ml_s) {
  const int tid = threadIdx.x;
  const int n = w.hc * D;
  const bool split = w.np > 1 || P.force_partials;
  T* out = static_cast<T*>(P.out);
  for (int i = tid; i < n; i += kThreads) {
    const int r = i / D, d = i - r * D;
    float M = -INFINITY;
#pragma unroll
    for (int wi = 0; wi < kWarps; ++wi) M = fmaxf(M, ml_s[(wi * HC + r) * 2]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int wi = 0; wi < kWarps; ++wi) {
      const float mw = ml_s[(wi * HC + r) * 2];
      const float cw = mw == -INFINITY ? 0.f : exp2f(mw - M);
      num += cw * O_s[(wi * HC + r) * D + d];
      den += cw * ml_s[(wi * HC + r) * 2 + 1];
    }
    const size_t row = static_cast<size_t>(w.s) * P.num_q_heads + w.h0 + r;
    if (!split) {
      out[row * D + d] = from_f32<T>(num / den * P.out_scale);
    } else {
      const size_t idx = row * P.max_parts + w.p;
      P.ws_o[idx * D + d] = num;
      if (d == 0) {
        P.ws_ml[idx * 2] = M;
        P.ws_ml[idx * 2 + 1] = den;
      }
    }
  }
}

// Partition k of the CTA's group (partitions w.p .. w.p + w.nparts - 1).  Unless the launch
// folds (P.fold: ppc > 1 and no per-partition partials wanted; FOLD = false compiles the
// kernel without this path), this is finish().  Folding, the CTA combines its partitions
// into one (m, l, o) by log-sum-exp as it goes, keeping the running value in the group's
// partial slot w.p / ppc (read back by the same threads), and after the last partition
// writes either the output (the group covers the whole context) or that one partial for
// decode_merge_kernel.  Called by every thread.
template <typename T, bool FOLD>
__device__ void finish_part(const Params& P, const Work& w, int k, int D, int HC,
                            const float* O_s, const float* ml_s) {
  if (!FOLD || !P.fold) {
    Work wk = w;
    wk.p = w.p + k;
    finish<T>(P, wk, D, HC, O_s, ml_s);
    return;
  }
  constexpr int kMaxPer = 4;  // elements per thread: head_chunk * D <= 4 * kThreads
  const int tid = threadIdx.x;
  const int n = w.hc * D;
  const int groups = (w.np + P.ppc - 1) / P.ppc;
  const bool last = k == w.nparts - 1;
  const size_t slot = static_cast<size_t>(w.p / P.ppc);
  float Ms[kMaxPer], Ds[kMaxPer], Ns[kMaxPer];
#pragma unroll
  for (int q = 0; q < kMaxPer; ++q) {
    const int i = tid + q * kThreads;
    if (i >= n) break;
    const int r = i / D, d = i - r * D;
    float M = -INFINITY;
#pragma unroll
    for (int wi = 0; wi < kWarps; ++wi) M = fmaxf(M, ml_s[(wi * HC + r) * 2]);
    float num = 0.f, den = 0.f;
#pragma unroll
    for (int wi = 0; wi < kWarps; ++wi) {
      const float mw = ml_s[(wi * HC + r) * 2];
      const float cw = mw == -INFINITY ? 0.f : exp2f(mw - M);
      num += cw * O_s[(wi * HC + r) * D + d];
      den += cw * ml_s[(wi * HC + r) * 2 + 1];
    }
    if (k > 0) {
      // fold in the running value of the partitions before this one
      const size_t idx = (static_cast<size_t>(w.s) * P.num_q_heads + w.h0 + r) * P.max_parts + slot;
      const float Mp = P.ws_ml[idx * 2], Dp = P.ws_ml[idx * 2 + 1], Np = P.ws_o[idx * D + d];
      const float Mn = fmaxf(M, Mp);
      const float a = Mp == -INFINITY ? 0.f : exp2f(Mp - Mn);
      const float b = M == -INFINITY ? 0.f : exp2f(M - Mn);
      num = Np * a + num * b;
      den = Dp * a + den * b;
      M = Mn;
    }
    Ms[q] = M;
    Ds[q] = den;
    Ns[q] = num;
  }
  // every thread has read the running (m, l) of its rows before any thread rewrites them
  if (k > 0) __syncthreads();
  T* out = static_cast<T*>(P.out);
#pragma unroll
  for (int q = 0; q < kMaxPer; ++q) {
    const int i = tid + q * kThreads;
    if (i >= n) break;
    const int r = i / D, d = i - r * D;
    const size_t row = static_cast<size_t>(w.s) * P.num_q_heads + w.h0 + r;
    if (last && groups <= 1) {
      out[row * D + d] = from_f32<T>(Ns[q] / Ds[q] * P.out_scale);
    } else {
      const size_t idx = row * P.max_parts + slot;
      P.ws_o[idx * D + d] = Ns[q];
      if (d == 0) {
        P.ws_ml[idx * 2] = Ms[q];
        P.ws_ml[idx * 2 + 1] = Ds[q];
      }
    }
  }
}

// ------------------------------------------------------------------------------------------
// tensor-core path
// ------------------------------------------------------------------------------------------

// Byte offset of (row r, column d) in a tile stored as 64-column boxes of 128-byte rows
// with the TMA 128-byte swizzle (16-byte chunk index XOR row % 8); d a multiple of 8.
template <int BS>
__device__ __forceinline__ uint32_t swz(int r, int d) {
  return static_cast<uint32_t>((d >> 6) * (BS * 128) + r * 128 + ((((d & 63) >> 3) ^ (r & 7)) << 4));
}

// The same offsets for the ldmatrix pattern of an m16n8k16 A operand, split into a lane
// part and a step part.  Lane `lane` reads row (lane & 7) + 8 * bit `rbit` of the lane and
// 16-byte chunk 2 s + bit `cbit` of K-step s (s = 0..7, 8 columns per chunk); with the
// tile base 1024-byte aligned,
//     base + swz<BS>(16 t + row, 16 s + 8 cbit) = ((base + lane_off) ^ ((s & 3) << 5))
//                                                 + (s >> 2) * BS * 128 + 2048 t,
// since the step only flips chunk bits 1-2 (byte bits 5-6) of a 1024-byte-aligned row group.
__device__ __forceinline__ uint32_t ldsm_lane_off(int lane, int rbit, int cbit) {
  const int row = (lane & 7) + ((lane >> rbit) & 1) * 8;
  return static_cast<uint32_t>(row * 128 + ((((lane >> cbit) & 1) ^ (lane & 7)) << 4));
}
template <int BS>
__device__ __forceinline__ uint32_t ldsm_step(uint32_t base_lane, int s, int t) {
  return (base_lane ^ static_cast<uint32_t>((s & 3) << 5)) +
         static_cast<uint32_t>((s >> 2) * (BS * 128) + 2048 * t);
}

// One block's online-softmax step on the S fragments of an m16n8 tile row pair: scale into
// log2 units, mask tokens past `valid`, update the running max m and sum l (rows lane/4
// and lane/4 + 8), rescale the output accumulators, and return P = 2^(S - m) rounded to
// the operand type as A fragments for P.V.  The row sums use the rounded weights.
template <typename T, int BS, int ND>
__device__ __forceinline__ void online_softmax(float (&sc)[BS / 8][4], float (&o)[ND][4],
                                               float (&m)[2], float (&l)[2],
                                               uint32_t (&pa)[BS / 16][4], int valid,
                                               float scale_log2, int lane) {
  constexpr int NT = BS / 8;
  // scale into log2 units, mask tokens past the context, row maxima over the quad
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int tok = nt * 8 + (lane & 3) * 2 + (c & 1);
      const float v = sc[nt][c] * scale_log2;
      sc[nt][c] = tok < valid ? v : -INFINITY;
    }
    mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
    mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
  }
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
  // The reference max m moves only when a row's new scores exceed it by more than
  // kRescaleSlack (log2 units): the weights 2^(S - m) then stay below 2^kRescaleSlack,
  // and the accumulators are rescaled only on those (rare) blocks.  o and l always share
  // one m, so the final o / l is unchanged.
  const bool up0 = mx0 > m[0] + kRescaleSlack, up1 = mx1 > m[1] + kRescaleSlack;
  const float mn0 = up0 ? mx0 : m[0], mn1 = up1 ? mx1 : m[1];
  // P = 2^(S - m) rounded to the operand type; the row sums use the rounded weights
  float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const uint32_t lo = Mma<T>::pack(fast_exp2(sc[nt][0] - mn0), fast_exp2(sc[nt][1] - mn0));
    const uint32_t hi = Mma<T>::pack(fast_exp2(sc[nt][2] - mn1), fast_exp2(sc[nt][3] - mn1));
    const float2 flo = Mma<T>::unpack(lo), fhi = Mma<T>::unpack(hi);
    rs0 += flo.x + flo.y;
    rs1 += fhi.x + fhi.y;
    pa[nt >> 1][(nt & 1) * 2 + 0] = lo;
    pa[nt >> 1][(nt & 1) * 2 + 1] = hi;
  }
  if (__any_sync(0xffffffffu, up0 || up1)) {
    const float a0 = fast_exp2(m[0] - mn0), a1 = fast_exp2(m[1] - mn1);  // 1 for rows that kept m
    l[0] *= a0;
    l[1] *= a1;
#pragma unroll
    for (int nd = 0; nd < ND; ++nd) {
      o[nd][0] *= a0;
      o[nd][1] *= a0;
      o[nd][2] *= a1;
      o[nd][3] *= a1;
    }
  }
  m[0] = mn0;
  m[1] = mn1;
  l[0] += rs0;
  l[1] += rs1;
}

template <typename T, int D, int BS>
__device__ __forceinline__ void tc_block(uint32_t kb, uint32_t vb, const uint32_t (&qa)[D / 16][4],
                                         float (&o)[D / 8][4], float (&m)[2], float (&l)[2],
                                         int valid, float scale_log2, int lane) {
  constexpr int NT = BS / 8;  // 8-token column tiles of S
  float sc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
  const int mi = lane >> 3;
  // S = Q . K^T : A = Q fragments (16 heads x 16 dims), B = K rows via ldmatrix.
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int r = nt * 8 + (lane & 7);
#pragma unroll
    for (int kk = 0; kk < D / 16; kk += 2) {
      const int d = (kk + (mi >> 1)) * 16 + (mi & 1) * 8;
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kb + swz<BS>(r, d), b0, b1, b2, b3);
      Mma<T>::run(sc[nt], qa[kk], b0, b1);
      Mma<T>::run(sc[nt], qa[kk + 1], b2, b3);
    }
  }
  uint32_t pa[BS / 16][4];
  online_softmax<T, BS, D / 8>(sc, o, m, l, pa, valid, scale_log2, lane);
  // O += P . V : B = V rows via transposing ldmatrix.
#pragma unroll
  for (int kt = 0; kt < BS / 16; ++kt) {
    const int r = kt * 16 + (mi & 1) * 8 + (lane & 7);
#pragma unroll
    for (int nd = 0; nd < D / 8; nd += 2) {
      const int d = (nd + (mi >> 1)) * 8;
      uint32_t b0, b1, b2, b3;
      ldsm_x4_trans(vb + swz<BS>(r, d), b0, b1, b2, b3);
      Mma<T>::run(o[nd], pa[kt], b0, b1);
      Mma<T>::run(o[nd + 1], pa[kt], b2, b3);
    }
  }
}

// Zero V rows [valid, BS) of a swizzled tile: masked tokens get weight 0, but 0 * NaN
// from stale slots would still poison the product.
template <int D, int BS>
__device__ __forceinline__ void zero_tail_rows(uint8_t* vtile, int valid, int lane) {
  constexpr int kBoxes = D / 64;
  const int rows = BS - valid;
  const int n = kBoxes * rows * 8;  // 16-byte chunks
  for (int i = lane; i < n; i += 32) {
    const int b = i / (rows * 8);
    const int rem = i - b * rows * 8;
    const int r = valid + rem / 8;
    const int ch = rem & 7;
    *reinterpret_cast<uint4*>(vtile + b * BS * 128 + r * 128 + ch * 16) = make_uint4(0, 0, 0, 0);
  }
}

template <typename T, int D, int BS>
__global__ void __launch_bounds__(kThreads)
    decode_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                     const __grid_constant__ CUtensorMap vmap, const Params P) {
  extern __shared__ uint8_t smem_raw[];
  Work w;
  int spec_id;
  if (!decode_work<T>(P, D, w, spec_id)) return;
  const Smem sm = carve(smem_raw, P);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int x0 = w.g * D;
  pipeline_start(P, w, sm, &kmap, &vmap, x0, spec_id);

  // Q fragments (A operand, rows = query heads of this CTA, zero past hc)
  uint32_t qa[D / 16][4];
  {
    const T* qs = static_cast<const T*>(P.q) + (static_cast<size_t>(w.s) * P.num_q_heads + w.h0) * D;
    const int r0 = lane >> 2, cq = (lane & 3) * 2;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int c0 = kk * 16 + cq;
      qa[kk][0] = r0 < w.hc ? __ldg(reinterpret_cast<const uint32_t*>(qs + r0 * D + c0)) : 0u;
      qa[kk][1] = r0 + 8 < w.hc ? __ldg(reinterpret_cast<const uint32_t*>(qs + (r0 + 8) * D + c0)) : 0u;
      qa[kk][2] = r0 < w.hc ? __ldg(reinterpret_cast<const uint32_t*>(qs + r0 * D + c0 + 8)) : 0u;
      qa[kk][3] =
          r0 + 8 < w.hc ? __ldg(reinterpret_cast<const uint32_t*>(qs + (r0 + 8) * D + c0 + 8)) : 0u;
    }
  }
  // The CTA covers w.nparts consecutive partitions; the ring streams across them and each
  // partition's state is merged and written on its own.
  bool dead = false;  // a wait of this warp timed out: the call's output is void
  float o[D / 8][4];
  float m[2], l[2];
  for (int k = 0; k < w.nparts; ++k) {
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
    const int je = min(w.nblk, (k + 1) * P.partition_blocks);
    StageCursor cur(k * P.partition_blocks + warp, P.stages);
    for (int j = k * P.partition_blocks + warp; j < je && !dead;
         j += kWarps, cur.next(P.stages)) {
      const int st = cur.st;
      if (!mbar_wait_bounded(smem_addr(&sm.bars[st]), cur.ph)) {
        if (lane == 0) raise_error(P.err, PKV_DERR_TIMEOUT);
        drain_after_timeout(P, w, sm, j);
        dead = true;
        break;
      }
      uint8_t* ktile = sm.ring + st * P.stage_bytes;
      uint8_t* vtile = ktile + P.tile_stride;
      const int valid = min(BS, w.tok_valid - j * BS);
      if (valid < BS) {
        zero_tail_rows<D, BS>(vtile, valid, lane);
        fence_proxy_async_smem();  // generic writes before the stage's next TMA fill
        __syncwarp();
      }
      tc_block<T, D, BS>(smem_addr(ktile), smem_addr(vtile), qa, o, m, l, valid, P.scale_log2, lane);
      __syncwarp();
      if (lane == 0 && j + P.stages < w.nblk)
        issue_block<D / 64>(P, sm, &kmap, &vmap, st, sm.ycoord[j + P.stages], x0);
    }

    __syncthreads();  // every warp is done with partition k (and, with one partition, the ring)
    const int HC = P.head_chunk;
    float* O_s = sm.merge;
    float* ml_s = O_s + kWarps * HC * D;
    {
      const int r0 = lane >> 2;
#pragma unroll
      for (int nd = 0; nd < D / 8; ++nd) {
        const int col = nd * 8 + (lane & 3) * 2;
        if (r0 < w.hc)
          *reinterpret_cast<float2*>(&O_s[(warp * HC + r0) * D + col]) = make_float2(o[nd][0], o[nd][1]);
        if (r0 + 8 < w.hc)
          *reinterpret_cast<float2*>(&O_s[(warp * HC + r0 + 8) * D + col]) =
              make_float2(o[nd][2], o[nd][3]);
      }
      l[0] += __shfl_xor_sync(0xffffffffu, l[0], 1);
      l[0] += __shfl_xor_sync(0xffffffffu, l[0], 2);
      l[1] += __shfl_xor_sync(0xffffffffu, l[1], 1);
      l[1] += __shfl_xor_sync(0xffffffffu, l[1], 2);
      if ((lane & 3) == 0) {
        if (r0 < w.hc) {
          ml_s[(warp * HC + r0) * 2] = m[0];
          ml_s[(warp * HC + r0) * 2 + 1] = l[0];
        }
        if (r0 + 8 < w.hc) {
          ml_s[(warp * HC + r0 + 8) * 2] = m[1];
          ml_s[(warp * HC + r0 + 8) * 2 + 1] = l[1];
        }
      }
    }
    __syncthreads();
    finish_part<T, BS == 16>(P, w, k, D, HC, O_s, ml_s);
    if (k + 1 < w.nparts) __syncthreads();  // the merge buffer is read before it is reused
  }
}

// ------------------------------------------------------------------------------------------
// fp8 (E4M3) caches: tensor cores in fp16
// ------------------------------------------------------------------------------------------
//
// K and V tiles hold E4M3 codes: rows of head_dim = 128 bytes, one TMA box with the
// 128-byte swizzle.  Every E4M3 value is exactly an fp16 value, so Q is converted to fp16
// and both products run as fp16 mma with fp32 accumulation; the K scale is folded into
// the score scale and the V scale multiplies the output.  head_dim is visited in an order
// that is the same for Q and K (a dot product does not depend on the order of its terms):
// lane c = lane % 4 of a quad owns elements [32c, 32c + 32), so a lane's operand bytes of
// one row are 32 contiguous bytes.  For P.V the lanes own V's columns the same way; an 8x8
// block of V (8 tokens x 8 columns) is read row-wise and transposed in registers with
// movmatrix, and column j of output n-tile nd is head_dim element 32(j/2) + 2nd + j%2.

// Byte offset of 16-byte chunk `chunk` of row r in a tile of 128-byte rows stored with the
// TMA 128-byte swizzle.
__device__ __forceinline__ uint32_t swz_chunk(int r, int chunk) {
  return static_cast<uint32_t>(r * 128 + ((chunk ^ (r & 7)) << 4));
}

template <int BS>
__device__ __forceinline__ void fp8_block(uint32_t kb, uint32_t vb, const uint32_t (&qa)[8][4],
                                          float (&o)[16][4], float (&m)[2], float (&l)[2],
                                          int valid, float scale_log2, int lane) {
  constexpr int NT = BS / 8;
  const int c = lane & 3, r8 = lane >> 2;
  float sc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
    const int r = nt * 8 + r8;
    const uint4 w0 = lds128(kb + swz_chunk(r, 2 * c));
    const uint4 w1 = lds128(kb + swz_chunk(r, 2 * c + 1));
    const uint32_t wk[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t b0, b1;
      e4m3x4_to_f16x2x2(wk[kk], b0, b1);
      Mma<__half>::run(sc[nt], qa[kk], b0, b1);
    }
  }
  uint32_t pa[BS / 16][4];
  online_softmax<__half, BS, 16>(sc, o, m, l, pa, valid, scale_log2, lane);
#pragma unroll
  for (int kt = 0; kt < BS / 16; ++kt) {
    const int ra = kt * 16 + r8, rb = ra + 8;
    const uint4 a0 = lds128(vb + swz_chunk(ra, 2 * c)), a1 = lds128(vb + swz_chunk(ra, 2 * c + 1));
    const uint4 b0 = lds128(vb + swz_chunk(rb, 2 * c)), b1 = lds128(vb + swz_chunk(rb, 2 * c + 1));
    const uint32_t va[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const uint32_t vc[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t a_even, a_odd, c_even, c_odd;  // columns of n-tiles 2i and 2i+1
      e4m3x4_to_f16x2x2(va[i], a_even, a_odd);
      e4m3x4_to_f16x2x2(vc[i], c_even, c_odd);
      Mma<__half>::run(o[2 * i], pa[kt], movmatrix_trans(a_even), movmatrix_trans(c_even));
      Mma<__half>::run(o[2 * i + 1], pa[kt], movmatrix_trans(a_odd), movmatrix_trans(c_odd));
    }
  }
}

__device__ __forceinline__ uint32_t to_f16x2(uint32_t w, __half) { return w; }
__device__ __forceinline__ uint32_t to_f16x2(uint32_t w, __nv_bfloat16) {
  const float2 f = Mma<__nv_bfloat16>::unpack(w);
  return Mma<__half>::pack(f.x, f.y);
}

template <typename T, int BS, int PAIR>
__global__ void __launch_bounds__(kThreads)
    decode_fp8_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const Params P) {
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  Work w;
  int spec_id;
  if (!decode_work<T>(P, D, w, spec_id)) return;
  const Smem sm = carve(smem_raw, P);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int x0 = w.g * D;  // bytes of one KV head's row segment
  pipeline_start(P, w, sm, &kmap, &vmap, x0, spec_id);

  // Q fragments in fp16, head_dim visited as described above
  uint32_t qa[8][4];
  {
    const T* qs = static_cast<const T*>(P.q) + (static_cast<size_t>(w.s) * P.num_q_heads + w.h0) * D;
    const int r0 = lane >> 2, c = lane & 3;
    auto ld = [&](int r, int d) {
      return r < w.hc ? to_f16x2(__ldg(reinterpret_cast<const uint32_t*>(qs + r * D + d)), T()) : 0u;
    };
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int d0 = 32 * c + 4 * kk;
      qa[kk][0] = ld(r0, d0);
      qa[kk][1] = ld(r0 + 8, d0);
      qa[kk][2] = ld(r0, d0 + 2);
      qa[kk][3] = ld(r0 + 8, d0 + 2);
    }
  }
  constexpr int TR = BS * PAIR;  // token rows of a staged tile
  const int nv = (w.nblk + PAIR - 1) / PAIR;
  const int vpp = P.partition_blocks / PAIR;  // staged tiles per partition
  bool dead = false;
  float o[16][4];
  float m[2], l[2];
  for (int k = 0; k < w.nparts; ++k) {
#pragma unroll
    for (int nd = 0; nd < 16; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
    const int ve = min(nv, (k + 1) * vpp);
    StageCursor cur(k * vpp + warp, P.stages);
    for (int v = k * vpp + warp; v < ve && !dead; v += kWarps, cur.next(P.stages)) {
      const int st = cur.st;
      if (!mbar_wait_bounded(smem_addr(&sm.bars[st]), cur.ph)) {
        if (lane == 0) raise_error(P.err, PKV_DERR_TIMEOUT);
        drain_after_timeout(P, w, sm, v);
        dead = true;
        break;
      }
      uint8_t* ktile = sm.ring + st * P.stage_bytes;
      uint8_t* vtile = ktile + P.tile_stride;
      const int valid = min(TR, w.tok_valid - v * TR);
      if (valid < TR) {
        zero_tail_rows<64, TR>(vtile, valid, lane);  // 128-byte rows, one box
        fence_proxy_async_smem();
        __syncwarp();
      }
      fp8_block<TR>(smem_addr(ktile), smem_addr(vtile), qa, o, m, l, valid, P.scale_log2, lane);
      __syncwarp();
      if (lane == 0 && v + P.stages < nv) {
        if constexpr (PAIR == 1)
          issue_block<1>(P, sm, &kmap, &vmap, st, sm.ycoord[v + P.stages], x0);
        else
          issue_tile(P, sm, &kmap, &vmap, v + P.stages, x0, w.nblk);
      }
    }

    __syncthreads();
    const int HC = P.head_chunk;
    float* O_s = sm.merge;
    float* ml_s = O_s + kWarps * HC * D;
    {
      const int r0 = lane >> 2, c = lane & 3;
#pragma unroll
      for (int nd = 0; nd < 16; ++nd) {
        const int col = 32 * c + 2 * nd;
        if (r0 < w.hc)
          *reinterpret_cast<float2*>(&O_s[(warp * HC + r0) * D + col]) = make_float2(o[nd][0], o[nd][1]);
        if (r0 + 8 < w.hc)
          *reinterpret_cast<float2*>(&O_s[(warp * HC + r0 + 8) * D + col]) =
              make_float2(o[nd][2], o[nd][3]);
      }
      l[0] += __shfl_xor_sync(0xffffffffu, l[0], 1);
      l[0] += __shfl_xor_sync(0xffffffffu, l[0], 2);
      l[1] += __shfl_xor_sync(0xffffffffu, l[1], 1);
      l[1] += __shfl_xor_sync(0xffffffffu, l[1], 2);
      if ((lane & 3) == 0) {
        if (r0 < w.hc) {
          ml_s[(warp * HC + r0) * 2] = m[0];
          ml_s[(warp * HC + r0) * 2 + 1] = l[0];
        }
        if (r0 + 8 < w.hc) {
          ml_s[(warp * HC + r0 + 8) * 2] = m[1];
          ml_s[(warp * HC + r0 + 8) * 2 + 1] = l[1];
        }
      }
    }
    __syncthreads();
    finish_part<T, false>(P, w, k, D, HC, O_s, ml_s);
    if (k + 1 < w.nparts) __syncthreads();
  }
}

// ------------------------------------------------------------------------------------------
// CUDA-core path
// ------------------------------------------------------------------------------------------

template <typename T, int E>
__global__ void __launch_bounds__(kThreads)
    decode_simt_kernel(const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap, const Params P) {
  constexpr int D = 32 * E;
  constexpr int HC = kSimtHeads;
  extern __shared__ uint8_t smem_raw[];
  Work w;
  int spec_id;
  if (!decode_work<T>(P, D, w, spec_id)) return;
  const Smem sm = carve(smem_raw, P);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int x0 = w.g * D;
  const int BS = P.block_size;
  pipeline_start(P, w, sm, &kmap, &vmap, x0, spec_id);

  float qr[HC][E];
  {
    const T* qs = static_cast<const T*>(P.q) + (static_cast<size_t>(w.s) * P.num_q_heads + w.h0) * D;
#pragma unroll
    for (int h = 0; h < HC; ++h)
#pragma unroll
      for (int e = 0; e < E; ++e) qr[h][e] = h < w.hc ? to_f32(qs[h * D + lane * E + e]) : 0.f;
  }
  float acc[HC][E], m[HC], l[HC];
#pragma unroll
  for (int h = 0; h < HC; ++h) {
    m[h] = -INFINITY;
    l[h] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[h][e] = 0.f;
  }

  for (int j = warp; j < w.nblk; j += kWarps) {
    const int st = j % P.stages;
    if (!mbar_wait_bounded(smem_addr(&sm.bars[st]), (j / P.stages) & 1)) {
      if (lane == 0) raise_error(P.err, PKV_DERR_TIMEOUT);
      drain_after_timeout(P, w, sm, j);
      break;
    }
    const T* kt = reinterpret_cast<const T*>(sm.ring + st * P.stage_bytes);
    const T* vt = reinterpret_cast<const T*>(sm.ring + st * P.stage_bytes + P.tile_stride);
    const int valid = min(BS, w.tok_valid - j * BS);
    for (int t = 0; t < valid; ++t) {
      float kf[E], vf[E];
#pragma unroll
      for (int e = 0; e < E; ++e) {
        kf[e] = to_f32(kt[t * D + lane * E + e]);
        vf[e] = to_f32(vt[t * D + lane * E + e]);
      }
#pragma unroll
      for (int h = 0; h < HC; ++h) {
        if (h < w.hc) {
          float dot = 0.f;
#pragma unroll
          for (int e = 0; e < E; ++e) dot = fmaf(qr[h][e], kf[e], dot);
          const float sl = warp_sum(dot) * P.scale_log2;
          const float mn = fmaxf(m[h], sl);
          const float a = exp2f(m[h] - mn);
          const float pr = exp2f(sl - mn);
          l[h] = l[h] * a + pr;
#pragma unroll
          for (int e = 0; e < E; ++e) acc[h][e] = fmaf(pr, vf[e], acc[h][e] * a);
          m[h] = mn;
        }
      }
    }
    __syncwarp();
    if (lane == 0 && j + P.stages < w.nblk) issue_tile(P, sm, &kmap, &vmap, j + P.stages, x0, w.nblk);
  }

  __syncthreads();
  float* O_s = sm.merge;
  float* ml_s = O_s + kWarps * HC * D;
#pragma unroll
  for (int h = 0; h < HC; ++h) {
    if (h < w.hc) {
#pragma unroll
      for (int e = 0; e < E; ++e) O_s[(warp * HC + h) * D + lane * E + e] = acc[h][e];
      if (lane == 0) {
        ml_s[(warp * HC + h) * 2] = m[h];
        ml_s[(warp * HC + h) * 2 + 1] = l[h];
      }
    }
  }
  __syncthreads();
  finish<T>(P, w, D, HC, O_s, ml_s);
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// The cache seen as a 2-D tensor: x = num_kv_heads * head_dim elements, y = cache rows.
bool make_cache_map(CUtensorMap* map, const void* base, pkv_dtype dt, bool fp8, int Hkv, int D,
                    long long rows, int box_cols, int box_rows, bool swizzle) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  const CUtensorMapDataType t = fp8              ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                : dt == PKV_F32  ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                : dt == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const size_t esize = fp8 ? 1 : dtype_size(dt);
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(Hkv) * D, static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(Hkv) * D * esize};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(map, t, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE,
                         swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

using KernelFn = void (*)(CUtensorMap, CUtensorMap, Params);

template <typename T>
KernelFn tc_kernel_for(int D, int BS) {
  if (D == 64) {
    if (BS == 16) return decode_tc_kernel<T, 64, 16>;
    if (BS == 32) return decode_tc_kernel<T, 64, 32>;
    if (BS == 64) return decode_tc_kernel<T, 64, 64>;
  } else if (D == 128) {
    if (BS == 16) return decode_tc_kernel<T, 128, 16>;
    if (BS == 32) return decode_tc_kernel<T, 128, 32>;
    if (BS == 64) return decode_tc_kernel<T, 128, 64>;
  }
  return nullptr;
}

template <typename T>
KernelFn simt_kernel_for(int D) {
  switch (D) {
    case 32: return decode_simt_kernel<T, 1>;
    case 64: return decode_simt_kernel<T, 2>;
    case 128: return decode_simt_kernel<T, 4>;
    case 256: return decode_simt_kernel<T, 8>;
    default: return nullptr;
  }
}

// ------------------------------------------------------------------------------------------
// 16-bit decode with the query heads in the N dimension (head_dim 128, at most 8 heads)
// ------------------------------------------------------------------------------------------
//
// S^T = K . Q^T (M = 16 tokens per m-tile, N = 8 heads, K = head_dim) and
// O^T += V^T . P^T (M = head_dim in 8 m-tiles, N = 8 heads, K = 16 tokens per step).  K
// enters as the A operand through ldmatrix, V^T through ldmatrix.trans, and P^T through two
// movmatrix transposes per 16 tokens; Q^T's B fragments stay in registers.  Half the
// accumulator and Q registers of the M = heads layout, so more CTAs fit on an SM.
// kl, vl: ldsm_lane_off(lane, 3, 4) and ldsm_lane_off(lane, 4, 3), computed once per CTA.
template <typename T, int BS>
__device__ __forceinline__ void tcg_block(uint32_t kb, uint32_t vb, uint32_t kl, uint32_t vl,
                                          const uint32_t (&qb)[8][2], float (&o)[8][4],
                                          float (&m)[2], float (&l)[2], int valid,
                                          float scale_log2, int lane) {
  constexpr int MT = BS / 16;
  const int r8 = lane >> 2;
  float sc[MT][4];
  // A fragment rows: token mt*16 + (lane & 7) + 8 * ((lane >> 3) & 1), cols +8 for lanes 16-31
  const uint32_t kbl = kb + kl;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    sc[mt][0] = sc[mt][1] = sc[mt][2] = sc[mt][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t a[4];
      ldsm_x4(ldsm_step<BS>(kbl, kk, mt), a[0], a[1], a[2], a[3]);
      Mma<T>::run(sc[mt], a, qb[kk][0], qb[kk][1]);
    }
  }
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int tok = mt * 16 + r8 + (e >> 1) * 8;
      const float v = sc[mt][e] * scale_log2;
      sc[mt][e] = tok < valid ? v : -INFINITY;
    }
    mx0 = fmaxf(mx0, fmaxf(sc[mt][0], sc[mt][2]));
    mx1 = fmaxf(mx1, fmaxf(sc[mt][1], sc[mt][3]));
  }
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
  }
  const bool up0 = mx0 > m[0] + kRescaleSlack, up1 = mx1 > m[1] + kRescaleSlack;
  const float mn0 = up0 ? mx0 : m[0], mn1 = up1 ? mx1 : m[1];
  uint32_t pb[MT][2];
  float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const uint32_t lo = Mma<T>::pack(fast_exp2(sc[mt][0] - mn0), fast_exp2(sc[mt][1] - mn1));
    const uint32_t hi = Mma<T>::pack(fast_exp2(sc[mt][2] - mn0), fast_exp2(sc[mt][3] - mn1));
    const float2 flo = Mma<T>::unpack(lo), fhi = Mma<T>::unpack(hi);
    rs0 += flo.x + fhi.x;
    rs1 += flo.y + fhi.y;
    pb[mt][0] = movmatrix_trans(lo);  // (head r8, tokens 2c, 2c + 1)
    pb[mt][1] = movmatrix_trans(hi);  // (head r8, tokens 8 + 2c, 9 + 2c)
  }
  if (__any_sync(0xffffffffu, up0 || up1)) {
    const float a0 = fast_exp2(m[0] - mn0), a1 = fast_exp2(m[1] - mn1);
    l[0] *= a0;
    l[1] *= a1;
#pragma unroll
    for (int md = 0; md < 8; ++md) {
      o[md][0] *= a0;
      o[md][1] *= a1;
      o[md][2] *= a0;
      o[md][3] *= a1;
    }
  }
  m[0] = mn0;
  m[1] = mn1;
  l[0] += rs0;
  l[1] += rs1;
  // O^T += V^T . P^T: A fragments of V^T (rows d, cols tokens) by transposing loads of V
  // rows kt*16 + (lane & 7) + 8 * ((lane >> 4) & 1), cols +8 for lanes 8-15 and 24-31
  const uint32_t vbl = vb + vl;
#pragma unroll
  for (int kt = 0; kt < MT; ++kt) {
#pragma unroll
    for (int md = 0; md < 8; ++md) {
      uint32_t a[4];
      ldsm_x4_trans(ldsm_step<BS>(vbl, md, kt), a[0], a[1], a[2], a[3]);
      Mma<T>::run(o[md], a, pb[kt][0], pb[kt][1]);
    }
  }
}

template <typename T, int BS>
__global__ void __launch_bounds__(kThreads, 5)
    decode_tcg_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const Params P) {
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  Work w;
  int spec_id;
  if (!decode_work<T>(P, D, w, spec_id)) return;
  const Smem sm = carve(smem_raw, P);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int x0 = w.g * D;
  pipeline_start(P, w, sm, &kmap, &vmap, x0, spec_id);
  const uint32_t kl = ldsm_lane_off(lane, 3, 4), vl = ldsm_lane_off(lane, 4, 3);

  // Q^T B fragments: head r8, head_dim kk*16 + 2c (+1) and kk*16 + 8 + 2c (+1)
  uint32_t qb[8][2];
  {
    const int r8 = lane >> 2, c = lane & 3;
    const T* qs = static_cast<const T*>(P.q) +
                  (static_cast<size_t>(w.s) * P.num_q_heads + w.h0 + r8) * D;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int d0 = kk * 16 + 2 * c;
      qb[kk][0] = r8 < w.hc ? __ldg(reinterpret_cast<const uint32_t*>(qs + d0)) : 0u;
      qb[kk][1] = r8 < w.hc ? __ldg(reinterpret_cast<const uint32_t*>(qs + d0 + 8)) : 0u;
    }
  }
  bool dead = false;
  float o[8][4];
  float m[2], l[2];
  for (int k = 0; k < w.nparts; ++k) {
#pragma unroll
    for (int md = 0; md < 8; ++md) o[md][0] = o[md][1] = o[md][2] = o[md][3] = 0.f;
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
    const int je = min(w.nblk, (k + 1) * P.partition_blocks);
    StageCursor cur(k * P.partition_blocks + warp, P.stages);
    for (int j = k * P.partition_blocks + warp; j < je && !dead;
         j += kWarps, cur.next(P.stages)) {
      const int st = cur.st;
      if (!mbar_wait_bounded(smem_addr(&sm.bars[st]), cur.ph)) {
        if (lane == 0) raise_error(P.err, PKV_DERR_TIMEOUT);
        drain_after_timeout(P, w, sm, j);
        dead = true;
        break;
      }
      uint8_t* ktile = sm.ring + st * P.stage_bytes;
      uint8_t* vtile = ktile + P.tile_stride;
      const int valid = min(BS, w.tok_valid - j * BS);
      if (valid < BS) {
        zero_tail_rows<D, BS>(vtile, valid, lane);
        fence_proxy_async_smem();
        __syncwarp();
      }
      tcg_block<T, BS>(smem_addr(ktile), smem_addr(vtile), kl, vl, qb, o, m, l, valid,
                       P.scale_log2, lane);
      __syncwarp();
      if (lane == 0 && j + P.stages < w.nblk)
        issue_block<2>(P, sm, &kmap, &vmap, st, sm.ycoord[j + P.stages], x0);
    }

    __syncthreads();
    const int HC = P.head_chunk;
    float* O_s = sm.merge;
    float* ml_s = O_s + kWarps * HC * D;
    {
      const int r8 = lane >> 2, c = lane & 3;
      const int h0 = 2 * c, h1 = 2 * c + 1;
#pragma unroll
      for (int md = 0; md < 8; ++md) {
        const int d = md * 16 + r8;
        if (h0 < w.hc) {
          O_s[(warp * HC + h0) * D + d] = o[md][0];
          O_s[(warp * HC + h0) * D + d + 8] = o[md][2];
        }
        if (h1 < w.hc) {
          O_s[(warp * HC + h1) * D + d] = o[md][1];
          O_s[(warp * HC + h1) * D + d + 8] = o[md][3];
        }
      }
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
        l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
      }
      if (r8 == 0) {
        if (h0 < w.hc) {
          ml_s[(warp * HC + h0) * 2] = m[0];
          ml_s[(warp * HC + h0) * 2 + 1] = l[0];
        }
        if (h1 < w.hc) {
          ml_s[(warp * HC + h1) * 2] = m[1];
          ml_s[(warp * HC + h1) * 2 + 1] = l[1];
        }
      }
    }
    __syncthreads();
    finish_part<T, BS == 16>(P, w, k, D, HC, O_s, ml_s);
    if (k + 1 < w.nparts) __syncthreads();
  }
}

template <typename T>
KernelFn tcg_kernel_for(int BS) {
  if (BS == 16) return decode_tcg_kernel<T, 16>;
  if (BS == 32) return decode_tcg_kernel<T, 32>;
  if (BS == 64) return decode_tcg_kernel<T, 64>;
  return nullptr;
}

// ------------------------------------------------------------------------------------------
// fp8 decode with the query heads in the N dimension (at most 8 query heads per KV head)
// ------------------------------------------------------------------------------------------
//
// S^T = K . Q^T (M = 16 tokens per m-tile, N = 8 heads, K = head_dim) and
// O^T += V^T . P^T (M = head_dim in 8 m-tiles, N = 8 heads, K = 16 tokens per step), so no
// MMA row is spent on absent heads and each thread owns whole columns (heads 2c, 2c+1).
//   - K as the A operand: lane (r8, c) holds tokens r8 and r8 + 8 of an m-tile; head_dim is
//     visited in the permuted order of the other fp8 kernel (lane c owns bytes [32c, 32c+32)
//     of a row), shared with Q's B fragments.
//   - The 16 tokens of an m-tile enter the MMAs in a permuted order: MMA row 2c is token 4c,
//     2c + 1 is 4c + 1, 8 + 2c is 4c + 2 and 9 + 2c is 4c + 3 (c = 0..3), so the K rows a
//     lane loads are tokens 2 r8 or 2 r8 - 1, and 2 r8 + 2 or 2 r8 + 1 (r8 even or odd).
//   - V^T as the A operand: a transposing byte load (ldmatrix .b8 .trans) gives lane (r8, c)
//     tokens 4c .. 4c + 3 of dims 16 md + r8 and 16 md + r8 + 8, which in that token order
//     are exactly its A fragment after one e4m3 -> f16 conversion per 16-bit half.
//   - P^T as the B operand: two movmatrix transposes per 16 tokens.
template <int TR>
__device__ __forceinline__ void fp8g_block(uint32_t kb, uint32_t vb, const uint32_t (&qb)[8][2],
                                           float (&o)[8][4], float (&m)[2], float (&l)[2],
                                           int valid, float scale_log2, int lane) {
  constexpr int MT = TR / 16;
  const int c = lane & 3, r8 = lane >> 2;
  // tokens (within an m-tile) of the MMA rows r8 and r8 + 8 (the permuted order above)
  const int tok_a = (r8 & 1) ? 2 * r8 - 1 : 2 * r8, tok_b = (r8 & 1) ? 2 * r8 + 1 : 2 * r8 + 2;
  float sc[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    sc[mt][0] = sc[mt][1] = sc[mt][2] = sc[mt][3] = 0.f;
    const int ra = mt * 16 + tok_a, rb = mt * 16 + tok_b;
    const uint4 a0 = lds128(kb + swz_chunk(ra, 2 * c)), a1 = lds128(kb + swz_chunk(ra, 2 * c + 1));
    const uint4 b0 = lds128(kb + swz_chunk(rb, 2 * c)), b1 = lds128(kb + swz_chunk(rb, 2 * c + 1));
    const uint32_t wa[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const uint32_t wb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t fa[4];
      e4m3x4_to_f16x2x2(wa[kk], fa[0], fa[2]);
      e4m3x4_to_f16x2x2(wb[kk], fa[1], fa[3]);
      Mma<__half>::run(sc[mt], fa, qb[kk][0], qb[kk][1]);
    }
  }
  // online softmax per head (column): tokens past `valid` are masked
  float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int tok = mt * 16 + ((e >> 1) ? tok_b : tok_a);
      const float v = sc[mt][e] * scale_log2;
      sc[mt][e] = tok < valid ? v : -INFINITY;
    }
    mx0 = fmaxf(mx0, fmaxf(sc[mt][0], sc[mt][2]));
    mx1 = fmaxf(mx1, fmaxf(sc[mt][1], sc[mt][3]));
  }
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
  }
  const bool up0 = mx0 > m[0] + kRescaleSlack, up1 = mx1 > m[1] + kRescaleSlack;
  const float mn0 = up0 ? mx0 : m[0], mn1 = up1 ? mx1 : m[1];
  uint32_t pb[MT][2];
  float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    const uint32_t lo = Mma<__half>::pack(fast_exp2(sc[mt][0] - mn0), fast_exp2(sc[mt][1] - mn1));
    const uint32_t hi = Mma<__half>::pack(fast_exp2(sc[mt][2] - mn0), fast_exp2(sc[mt][3] - mn1));
    const float2 flo = Mma<__half>::unpack(lo), fhi = Mma<__half>::unpack(hi);
    rs0 += flo.x + fhi.x;
    rs1 += flo.y + fhi.y;
    pb[mt][0] = movmatrix_trans(lo);  // (head r8, MMA rows 2c, 2c + 1 = tokens 4c, 4c + 1)
    pb[mt][1] = movmatrix_trans(hi);  // (head r8, MMA rows 8 + 2c, 9 + 2c = tokens 4c + 2, 4c + 3)
  }
  if (__any_sync(0xffffffffu, up0 || up1)) {
    const float a0 = fast_exp2(m[0] - mn0), a1 = fast_exp2(m[1] - mn1);  // 1 for heads that kept m
    l[0] *= a0;
    l[1] *= a1;
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      o[mt][0] *= a0;
      o[mt][1] *= a1;
      o[mt][2] *= a0;
      o[mt][3] *= a1;
    }
  }
  m[0] = mn0;
  m[1] = mn1;
  l[0] += rs0;
  l[1] += rs1;
  // O^T += V^T . P^T, m-tile md = dims 16 md .. 16 md + 15
#pragma unroll
  for (int kt = 0; kt < MT; ++kt) {
    const int row = kt * 16 + (lane & 15);
#pragma unroll
    for (int md = 0; md < 8; ++md) {
      uint32_t x0, x1, fa[4];
      ldsm_b8_trans(vb + swz_chunk(row, md), x0, x1);
      e4m3x4_to_f16x2x2(x0, fa[0], fa[2]);  // dim 16 md + r8: tokens 4c, 4c + 1 | 4c + 2, 4c + 3
      e4m3x4_to_f16x2x2(x1, fa[1], fa[3]);  // dim 16 md + r8 + 8
      Mma<__half>::run(o[md], fa, pb[kt][0], pb[kt][1]);
    }
  }
}

template <typename T, int BS, int PAIR>
__global__ void __launch_bounds__(kThreads, 5)
    decode_fp8g_kernel(const __grid_constant__ CUtensorMap kmap,
                       const __grid_constant__ CUtensorMap vmap, const Params P) {
  constexpr int D = 128;
  extern __shared__ uint8_t smem_raw[];
  Work w;
  int spec_id;
  if (!decode_work<T>(P, D, w, spec_id)) return;
  const Smem sm = carve(smem_raw, P);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int x0 = w.g * D;  // bytes of one KV head's row segment
  pipeline_start(P, w, sm, &kmap, &vmap, x0, spec_id);

  // Q^T B fragments in fp16: head r8, head_dim 32c + 4kk + (0, 1) and (2, 3)
  uint32_t qb[8][2];
  {
    const int r8 = lane >> 2, c = lane & 3;
    const T* qs = static_cast<const T*>(P.q) +
                  (static_cast<size_t>(w.s) * P.num_q_heads + w.h0 + r8) * D;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const int d0 = 32 * c + 4 * kk;
      qb[kk][0] = r8 < w.hc ? to_f16x2(__ldg(reinterpret_cast<const uint32_t*>(qs + d0)), T()) : 0u;
      qb[kk][1] =
          r8 < w.hc ? to_f16x2(__ldg(reinterpret_cast<const uint32_t*>(qs + d0 + 2)), T()) : 0u;
    }
  }
  constexpr int TR = BS * PAIR;  // token rows of a staged tile
  const int nv = (w.nblk + PAIR - 1) / PAIR;
  const int vpp = P.partition_blocks / PAIR;  // staged tiles per partition
  bool dead = false;
  float o[8][4];
  float m[2], l[2];
  for (int k = 0; k < w.nparts; ++k) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    m[0] = m[1] = -INFINITY;
    l[0] = l[1] = 0.f;
    const int ve = min(nv, (k + 1) * vpp);
    StageCursor cur(k * vpp + warp, P.stages);
    for (int v = k * vpp + warp; v < ve && !dead; v += kWarps, cur.next(P.stages)) {
      const int st = cur.st;
      if (!mbar_wait_bounded(smem_addr(&sm.bars[st]), cur.ph)) {
        if (lane == 0) raise_error(P.err, PKV_DERR_TIMEOUT);
        drain_after_timeout(P, w, sm, v);
        dead = true;
        break;
      }
      uint8_t* ktile = sm.ring + st * P.stage_bytes;
      uint8_t* vtile = ktile + P.tile_stride;
      const int valid = min(TR, w.tok_valid - v * TR);
      if (valid < TR) {
        zero_tail_rows<64, TR>(vtile, valid, lane);  // 128-byte rows, one box
        fence_proxy_async_smem();
        __syncwarp();
      }
      fp8g_block<TR>(smem_addr(ktile), smem_addr(vtile), qb, o, m, l, valid, P.scale_log2, lane);
      __syncwarp();
      if (lane == 0 && v + P.stages < nv) {
        if constexpr (PAIR == 1)
          issue_block<1>(P, sm, &kmap, &vmap, st, sm.ycoord[v + P.stages], x0);
        else
          issue_tile(P, sm, &kmap, &vmap, v + P.stages, x0, w.nblk);
      }
    }

    __syncthreads();
    const int HC = P.head_chunk;
    float* O_s = sm.merge;
    float* ml_s = O_s + kWarps * HC * D;
    {
      const int r8 = lane >> 2, c = lane & 3;
      const int h0 = 2 * c, h1 = 2 * c + 1;
#pragma unroll
      for (int md = 0; md < 8; ++md) {
        const int d = md * 16 + r8;  // rows r8 and r8 + 8 of m-tile md
        if (h0 < w.hc) {
          O_s[(warp * HC + h0) * D + d] = o[md][0];
          O_s[(warp * HC + h0) * D + d + 8] = o[md][2];
        }
        if (h1 < w.hc) {
          O_s[(warp * HC + h1) * D + d] = o[md][1];
          O_s[(warp * HC + h1) * D + d + 8] = o[md][3];
        }
      }
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l[0] += __shfl_xor_sync(0xffffffffu, l[0], off);
        l[1] += __shfl_xor_sync(0xffffffffu, l[1], off);
      }
      if (r8 == 0) {
        if (h0 < w.hc) {
          ml_s[(warp * HC + h0) * 2] = m[0];
          ml_s[(warp * HC + h0) * 2 + 1] = l[0];
        }
        if (h1 < w.hc) {
          ml_s[(warp * HC + h1) * 2] = m[1];
          ml_s[(warp * HC + h1) * 2 + 1] = l[1];
        }
      }
    }
    __syncthreads();
    finish_part<T, false>(P, w, k, D, HC, O_s, ml_s);
    if (k + 1 < w.nparts) __syncthreads();
  }
}

template <typename T>
KernelFn fp8g_kernel_for(int BS) {
  if (BS == 16) return decode_fp8g_kernel<T, 16, 1>;  // two 16-token stages per warp
  if (BS == 32) return decode_fp8g_kernel<T, 32, 1>;
  if (BS == 64) return decode_fp8g_kernel<T, 64, 1>;
  return nullptr;
}

template <typename T>
KernelFn fp8_kernel_for(int BS) {
  if (BS == 16) return decode_fp8_kernel<T, 16, 2>;  // two 16-token blocks per staged tile
  if (BS == 32) return decode_fp8_kernel<T, 32, 1>;
  if (BS == 64) return decode_fp8_kernel<T, 64, 1>;
  return nullptr;
}

KernelFn kernel_for(pkv_dtype dt, int D, int BS, bool tc) {
  if (tc) {
    if (dt == PKV_BF16) return tc_kernel_for<__nv_bfloat16>(D, BS);
    if (dt == PKV_F16) return tc_kernel_for<__half>(D, BS);
    return nullptr;
  }
  if (dt == PKV_F32) return simt_kernel_for<float>(D);
  if (dt == PKV_BF16) return simt_kernel_for<__nv_bfloat16>(D);
  return simt_kernel_for<__half>(D);
}

// ------------------------------------------------------------------------------------------
// Work order for split launches
// ------------------------------------------------------------------------------------------

constexpr int kPrepThreads = 1024;
constexpr int kMaxOrderItems = 1 << 16;  // (sequence, group) items a prep launch sorts
constexpr int kMaxOrderBins = 2049;      // live-block counts 0 .. 2048 of a group

// Live blocks of item (sequence s, group q): the blocks the CTAs of that item stream.
__device__ __forceinline__ int item_blocks(const int32_t* context_lens, int item, int groups,
                                           int group_tokens, int block_size, int max_len) {
  const int s = item / groups, q = item - s * groups;
  int L = context_lens[s];
  L = L < 0 ? 0 : (L > max_len ? max_len : L);
  const int t = L - q * group_tokens;
  return t <= 0 ? 0 : min(group_tokens / block_size, (t + block_size - 1) / block_size);
}

// One CTA, run before a split decode launch on the same stream: writes `order`, the (sequence, group) items sorted by live blocks, most
// first (a counting sort).  Dispatching the longest units first and letting the short
// ones fill the end of the grid is longest-processing-time list scheduling: with contexts
// of very different lengths it keeps the SMs streaming until the last wave.  Items with
// equal counts keep no particular order; the decode results do not depend on it.
__global__ void __launch_bounds__(kPrepThreads)
    decode_prep_kernel(const int32_t* __restrict__ context_lens, int num_seqs, int groups,
                       int group_tokens, int block_size, int max_len, int32_t* order) {
  griddep_launch_dependents();  // the decode grid may be scheduled; it waits for this one
  __shared__ int bins[kMaxOrderBins];
  __shared__ int warp_tot[kPrepThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gblocks = group_tokens / block_size;
  const int nbins = gblocks + 1;  // bin b holds the items with gblocks - b live blocks
  const int n = num_seqs * groups;
  for (int b = tid; b < nbins; b += kPrepThreads) bins[b] = 0;
  __syncthreads();
  // the counts of this thread's first kCached items stay in registers for the second pass
  constexpr int kCached = 2;
  int cached[kCached];
#pragma unroll
  for (int k = 0; k < kCached; ++k) {
    const int i = tid + k * kPrepThreads;
    cached[k] = i < n ? item_blocks(context_lens, i, groups, group_tokens, block_size, max_len) : 0;
    if (i < n) atomicAdd(&bins[gblocks - cached[k]], 1);
  }
  for (int i = tid + kCached * kPrepThreads; i < n; i += kPrepThreads)
    atomicAdd(&bins[gblocks - item_blocks(context_lens, i, groups, group_tokens, block_size,
                                           max_len)], 1);
  __syncthreads();
  // exclusive prefix sum of the bins: each thread owns a run of `per` bins
  const int per = (nbins + kPrepThreads - 1) / kPrepThreads;
  const int b0 = min(nbins, tid * per), b1 = min(nbins, b0 + per);
  int own = 0;
  for (int b = b0; b < b1; ++b) own += bins[b];
  int incl = own;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int v = warp_tot[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += y;
    }
    warp_tot[lane] = v;
  }
  __syncthreads();
  int base = incl - own + (warp > 0 ? warp_tot[warp - 1] : 0);
  for (int b = b0; b < b1; ++b) {
    const int c = bins[b];
    bins[b] = base;
    base += c;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kCached; ++k) {
    const int i = tid + k * kPrepThreads;
    if (i < n) order[atomicAdd(&bins[gblocks - cached[k]], 1)] = i;
  }
  for (int i = tid + kCached * kPrepThreads; i < n; i += kPrepThreads)
    order[atomicAdd(&bins[gblocks - item_blocks(context_lens, i, groups, group_tokens, block_size,
                                                max_len)], 1)] = i;
}

// ------------------------------------------------------------------------------------------
// Reduction of the partition partials
// ------------------------------------------------------------------------------------------

constexpr int kMergeWarps = 4;

// One warp per (sequence, query head) row whose context spans np > 1 partitions: the
// log-sum-exp reduction of the partition partials (m_p in log2 units, l_p, o_p):
//   M = max_p m_p,  w_p = 2^(m_p - M) / sum_q 2^(m_q - M) l_q,  out = sum_p w_p o_p,
// which equals the single-pass softmax-weighted sum of values up to rounding order.
// Rows of one partition were written by the decode kernel itself.  Launched right after
// the decode kernel, possibly while it still runs: the partials are read only after the
// grid dependency wait, through L2.
template <typename T, int D>
__global__ void __launch_bounds__(kMergeWarps * 32) decode_merge_kernel(const Params P) {
  constexpr int V = D / 32;  // columns per lane
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * kMergeWarps + warp;
  int np = 0;
  if (row < static_cast<long long>(P.num_seqs) * P.num_q_heads) {
    int L = P.context_lens[row / P.num_q_heads];
    const int Lmax = P.max_blocks_per_seq * P.block_size;
    L = L < 0 ? 0 : (L > Lmax ? Lmax : L);
    // one partial per partition, or per group of ppc partitions when the CTAs fold them
    const int gtok = P.partition_blocks * P.block_size * (P.fold ? P.ppc : 1);
    np = (L + gtok - 1) / gtok;
  }
  // every thread waits, even one with nothing to merge, so that this grid never ends
  // before the decode grid it depends on
  griddep_wait();
  if (np <= 1) return;
  const size_t base = static_cast<size_t>(row) * P.max_parts;
  const float2* ml = reinterpret_cast<const float2*>(P.ws_ml) + base;
  const float* o = P.ws_o + base * D + lane * V;
  auto load_cols = [&](int p, float (&x)[V]) {
    const float* src = o + static_cast<size_t>(p) * D;
    if constexpr (V % 4 == 0) {
#pragma unroll
      for (int k = 0; k < V; k += 4) {
        const float4 v = __ldcg(reinterpret_cast<const float4*>(src + k));
        x[k] = v.x;
        x[k + 1] = v.y;
        x[k + 2] = v.z;
        x[k + 3] = v.w;
      }
    } else if constexpr (V == 2) {
      const float2 v = __ldcg(reinterpret_cast<const float2*>(src));
      x[0] = v.x;
      x[1] = v.y;
    } else {
      x[0] = __ldcg(src);
    }
  };
  // The first 32 partials' (m, l), one per lane, and the first kPre partials' columns are
  // loaded together, before any of the arithmetic that waits for them.
  constexpr int kPre = D >= 256 ? 4 : 8;
  const float2 first = lane < np ? __ldcg(&ml[lane]) : make_float2(-INFINITY, 0.f);
  float pre[kPre][V];
#pragma unroll
  for (int i = 0; i < kPre; ++i)
    if (i < np) load_cols(i, pre[i]);
  float M = first.x;
  for (int p = lane + 32; p < np; p += 32) M = fmaxf(M, __ldcg(&ml[p]).x);
  M = warp_max(M);
  float den = lane < np ? exp2f(first.x - M) * first.y : 0.f;
  for (int p = lane + 32; p < np; p += 32) {
    const float2 v = __ldcg(&ml[p]);
    den += exp2f(v.x - M) * v.y;
  }
  den = warp_sum(den);
  const float inv = 1.f / den;
  float acc[V];
#pragma unroll
  for (int k = 0; k < V; ++k) acc[k] = 0.f;
  for (int p0 = 0; p0 < np; p0 += 32) {
    const int p = p0 + lane;
    const float mp = p0 == 0 ? first.x : (p < np ? __ldcg(&ml[p]).x : -INFINITY);
    const float wp = p < np ? exp2f(mp - M) * inv : 0.f;
    const int cnt = min(32, np - p0);
    int i = 0;
    if (p0 == 0) {
#pragma unroll
      for (int j = 0; j < kPre; ++j) {
        const float wi = __shfl_sync(0xffffffffu, wp, j);
        if (j < cnt) {
#pragma unroll
          for (int k = 0; k < V; ++k) acc[k] += wi * pre[j][k];
        }
      }
      i = kPre;
    }
#pragma unroll 8
    for (; i < cnt; ++i) {
      const float wi = __shfl_sync(0xffffffffu, wp, i);
      float x[V];
      load_cols(p0 + i, x);
#pragma unroll
      for (int k = 0; k < V; ++k) acc[k] += wi * x[k];
    }
  }
  T* out = static_cast<T*>(P.out) + static_cast<size_t>(row) * D + lane * V;
#pragma unroll
  for (int k = 0; k < V; ++k) out[k] = from_f32<T>(acc[k] * P.out_scale);
}

using MergeFn = void (*)(const Params);

template <typename T>
MergeFn merge_kernel_for_type(int D) {
  switch (D) {
    case 32: return decode_merge_kernel<T, 32>;
    case 64: return decode_merge_kernel<T, 64>;
    case 128: return decode_merge_kernel<T, 128>;
    case 256: return decode_merge_kernel<T, 256>;
    default: return nullptr;
  }
}

MergeFn merge_kernel_for(pkv_dtype dt, int D) {
  if (dt == PKV_F32) return merge_kernel_for_type<float>(D);
  if (dt == PKV_BF16) return merge_kernel_for_type<__nv_bfloat16>(D);
  if (dt == PKV_F16) return merge_kernel_for_type<__half>(D);
  return nullptr;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct Geometry {
  int stages, tile_bytes, tile_stride, stage_bytes, ring_bytes, merge_off, smem_bytes;
};

Geometry geometry(pkv_dtype dt, int D, int BS, bool tc, int partition_blocks, int max_parts,
                  bool fp8 = false, int pair = 1, int ppc = 1, int head_chunk = 0,
                  bool shallow = false) {
  Geometry g{};
  g.tile_bytes = BS * D * (fp8 ? 1 : static_cast<int>(dtype_size(dt)));
  g.tile_stride = static_cast<int>(align_up(static_cast<size_t>(pair) * g.tile_bytes, 1024));
  g.stage_bytes = 2 * g.tile_stride;
  // (shallow: the heads-in-N kernels run five CTAs per SM on half the stages)
  const int per_warp =
      std::max(1, std::min(kMaxStageSet, (shallow ? 8192 : 16384) / g.stage_bytes));
  g.stages = kWarps * per_warp;
  const int HC = tc ? kTcHeads : kSimtHeads;
  const size_t epi = (static_cast<size_t>(kWarps) * HC * D + kWarps * HC * 2) * sizeof(float);
  if (ppc == 1) {
    // the merge runs once, after the last tile: it reuses the ring
    g.ring_bytes = static_cast<int>(
        align_up(std::max(static_cast<size_t>(g.stages) * g.stage_bytes, epi), 1024));
    g.merge_off = 0;
  } else {
    // a partition is merged while the next one's tiles stream in: a buffer of its own
    const size_t merge =
        (static_cast<size_t>(kWarps) * head_chunk * D + kWarps * head_chunk * 2) * sizeof(float);
    g.merge_off = static_cast<int>(align_up(static_cast<size_t>(g.stages) * g.stage_bytes, 1024));
    g.ring_bytes = static_cast<int>(align_up(g.merge_off + merge, 128));
  }
  g.smem_bytes = 1024 + g.ring_bytes + 8 * g.stages + 4 * partition_blocks * ppc;
  return g;
}

constexpr int kMaxSmem = 227 * 1024;

}  // namespace

size_t dtype_size(pkv_dtype dtype) { return dtype == PKV_F32 ? 4 : 2; }

int resolve_partition_tokens(int partition_size, int block_size, int num_seqs, int num_q_heads,
                             int num_kv_heads, int max_blocks_per_seq, int kv_elem_bytes) {
  if (block_size <= 0) return -1;
  if (partition_size == 0) {
    // The largest of 2048, 1024, 512 tokens that still leaves at least kMinUnits work units
    // (sequence x KV head x 16-head chunk x partition, counting every sequence at the block
    // table's full length); longer partitions amortise each CTA's start-up cost, shorter
    // ones balance uneven contexts across the SMs.  For 1-byte E4M3 elements the candidates
    // grow by half: a token carries half the bytes, but its conversions cost more
    // instructions, and a 1.5x unit takes about as long as a 16-bit one.
    const long long max_ctx = static_cast<long long>(max_blocks_per_seq) * block_size;
    const int group = num_kv_heads > 0 ? std::max(1, num_q_heads / num_kv_heads) : 1;
    const long long heads = static_cast<long long>(std::max(0, num_seqs)) *
                            std::max(1, num_kv_heads) * ((group + kTcHeads - 1) / kTcHeads);
    const int widen2 = kv_elem_bytes == 1 ? 3 : 2;  // twice the widening factor
    int t = 0;
    for (int cand : {2048, 1024, kDefaultPartitionTokens}) {
      t = std::max(block_size, (widen2 * cand / 2 / block_size) * block_size);
      if (heads * ((max_ctx + t - 1) / t) >= kMinUnits) break;
    }
    return t;
  }
  if (partition_size < 0 || partition_size % block_size != 0) return -1;
  if (partition_size / block_size > kMaxPartitionBlocks) return -1;
  return partition_size;
}

WorkspaceLayout workspace_layout(int num_seqs, int num_q_heads, int head_dim, int block_size,
                                 int max_blocks_per_seq, int partition_tokens, bool partials) {
  WorkspaceLayout w{};
  const long long max_ctx = static_cast<long long>(max_blocks_per_seq) * block_size;
  w.max_parts = static_cast<int>(std::max(1LL, (max_ctx + partition_tokens - 1) / partition_tokens));
  if (w.max_parts <= 1 && !partials) return w;
  const size_t units = static_cast<size_t>(num_seqs) * num_q_heads * w.max_parts;
  w.o_offset = 0;
  w.ml_offset = align_up(units * head_dim * sizeof(float), 256);
  w.order_offset = w.ml_offset + align_up(units * 2 * sizeof(float), 256);
  w.total = w.order_offset +
            align_up(static_cast<size_t>(num_seqs) * w.max_parts * sizeof(int32_t), 256);
  return w;
}

bool decode_uses_tensor_cores(pkv_dtype dtype, int head_dim, int block_size) {
  return (dtype == PKV_BF16 || dtype == PKV_F16) && (head_dim == 64 || head_dim == 128) &&
         (block_size == 16 || block_size == 32 || block_size == 64);
}

bool decode_supported(pkv_dtype dtype, int head_dim, int block_size) {
  if (head_dim != 32 && head_dim != 64 && head_dim != 128 && head_dim != 256) return false;
  if (block_size < 1 || block_size > 256) return false;
  const bool tc = decode_uses_tensor_cores(dtype, head_dim, block_size);
  const Geometry g = geometry(dtype, head_dim, block_size, tc, 1, 1);
  return g.smem_bytes <= kMaxSmem;
}

bool decode_fp8_supported(pkv_dtype dtype, int head_dim, int block_size) {
  return (dtype == PKV_BF16 || dtype == PKV_F16) && head_dim == 128 &&
         (block_size == 16 || block_size == 32 || block_size == 64);
}

int launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.num_seqs == 0) return PKV_OK;
  if (a.kv_fp8 && !decode_fp8_supported(a.dtype, a.head_dim, a.block_size))
    return PKV_EUNSUPPORTED;
  const bool tc = a.kv_fp8 || decode_uses_tensor_cores(a.dtype, a.head_dim, a.block_size);
  const int D = a.head_dim, BS = a.block_size;
  const WorkspaceLayout wl = workspace_layout(a.num_seqs, a.num_q_heads, D, BS,
                                              a.max_blocks_per_seq, a.partition_tokens,
                                              a.partials_out);
  if (wl.max_parts > kMaxParts) return PKV_EUNSUPPORTED;
  if (wl.total > 0 && (a.workspace == nullptr || a.workspace_bytes < wl.total)) return PKV_ENOMEM;

  Params P{};
  P.out = a.out;
  P.q = a.q;
  P.block_tables = a.block_tables;
  P.context_lens = a.context_lens;
  P.err = a.err;
  P.num_seqs = a.num_seqs;
  P.num_q_heads = a.num_q_heads;
  P.num_kv_heads = a.num_kv_heads;
  P.group = a.num_q_heads / a.num_kv_heads;
  // fp8 caches with at most 8 query heads per KV head: the kernel with heads in N
  const bool fp8g = a.kv_fp8 && P.group <= kFp8gHeads;
  // 16-bit caches, head_dim 128, 2 to 8 query heads per KV head (GQA): heads in N as well.
  // (With one head per KV head the deeper ring of the M = heads kernel streams faster.)
  const bool tcg = !a.kv_fp8 && tc && D == 128 && P.group >= 2 && P.group <= kFp8gHeads;
  const bool shallow = fp8g || tcg;
  P.head_chunk = std::min(P.group, tc ? kTcHeads : kSimtHeads);
  P.num_chunks = (P.group + P.head_chunk - 1) / P.head_chunk;
  P.max_blocks_per_seq = a.max_blocks_per_seq;
  P.num_blocks = a.num_blocks;
  P.block_size = BS;
  P.partition_blocks = a.partition_tokens / BS;
  P.max_parts = wl.max_parts;
  P.force_partials = a.partials_out ? 1 : 0;
  if (wl.total > 0) {
    char* ws = static_cast<char*>(a.workspace);
    P.ws_o = reinterpret_cast<float*>(ws + wl.o_offset);
    P.ws_ml = reinterpret_cast<float*>(ws + wl.ml_offset);
  }
  // 16-token E4M3 blocks: the M = heads kernel stacks two per staged tile; the heads-in-N
  // kernel stages them singly, which gives each warp two stages of the same bytes in flight
  P.pair = (a.kv_fp8 && BS == 16 && !fp8g) ? 2 : 1;
  // Short partitions on the tensor-core paths: a CTA streams two of them back to back
  // (one partial each) when its merge buffer still lets three CTAs share an SM.
  P.ppc = 1;
  // (a CTA's group of partitions is folded by threads holding at most 4 elements each:
  // head_chunk * D <= 4 * kThreads)
  if (tc && a.partition_tokens < 1024 && P.head_chunk <= 4 && wl.max_parts > 1 &&
      P.partition_blocks % (4 * P.pair) == 0) {
    const Geometry g2 = geometry(a.dtype, D, BS, tc, P.partition_blocks, wl.max_parts, a.kv_fp8,
                                 P.pair, 2, P.head_chunk, shallow);
    if ((shallow ? 5 : 3) * (g2.smem_bytes + 1024) <= 228 * 1024) P.ppc = 2;
  }
  P.max_groups = (wl.max_parts + P.ppc - 1) / P.ppc;
  // the 16-bit kernels of 16-token blocks fold a CTA's partitions into one partial (their
  // instantiation has the code for it); the others, at the edge of their register budgets,
  // leave one per partition
  P.fold = P.ppc > 1 && !a.partials_out && !a.kv_fp8 && BS == 16 ? 1 : 0;
  const Geometry g = geometry(a.dtype, D, BS, tc, P.partition_blocks, wl.max_parts, a.kv_fp8,
                              P.pair, P.ppc, P.head_chunk, shallow);
  P.merge_off = g.merge_off;
  if (g.smem_bytes > kMaxSmem) return PKV_EUNSUPPORTED;
  P.stages = g.stages;
  P.tile_bytes = g.tile_bytes;
  P.tile_stride = g.tile_stride;
  P.stage_bytes = g.stage_bytes;
  P.ring_bytes = g.ring_bytes;
  P.boxes = a.kv_fp8 ? 1 : (tc ? D / 64 : 1);
  P.box_cols = a.kv_fp8 ? D : (tc ? 64 : D);
  P.box_bytes = tc ? BS * 128 : g.tile_bytes;
  const double k_scale = a.kv_fp8 ? static_cast<double>(a.k_scale) : 1.0;
  P.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * k_scale * 1.4426950408889634);
  P.out_scale = a.kv_fp8 ? a.v_scale : 1.f;

  const long long grid = static_cast<long long>(a.num_seqs) * P.max_groups * a.num_kv_heads *
                         P.num_chunks;
  if (grid > INT_MAX) return PKV_EUNSUPPORTED;

  CUtensorMap kmap, vmap;
  const long long rows = static_cast<long long>(a.num_blocks) * BS;
  if (!make_cache_map(&kmap, a.k_cache, a.dtype, a.kv_fp8, a.num_kv_heads, D, rows, P.box_cols,
                      BS, tc) ||
      !make_cache_map(&vmap, a.v_cache, a.dtype, a.kv_fp8, a.num_kv_heads, D, rows, P.box_cols,
                      BS, tc))
    return PKV_ECUDA;

  KernelFn fn = tcg      ? (a.dtype == PKV_BF16 ? tcg_kernel_for<__nv_bfloat16>(BS)
                                                : tcg_kernel_for<__half>(BS))
                : fp8g     ? (a.dtype == PKV_BF16 ? fp8g_kernel_for<__nv_bfloat16>(BS)
                                                : fp8g_kernel_for<__half>(BS))
                : a.kv_fp8 ? (a.dtype == PKV_BF16 ? fp8_kernel_for<__nv_bfloat16>(BS)
                                                : fp8_kernel_for<__half>(BS))
                           : kernel_for(a.dtype, D, BS, tc);
  if (!fn) return PKV_EUNSUPPORTED;
  const bool split = wl.total > 0;
  // with partials_out the caller merges the partials itself
  MergeFn merge = split && !a.partials_out ? merge_kernel_for(a.dtype, D) : nullptr;
  if (split && !a.partials_out && !merge) return PKV_EUNSUPPORTED;
  // Split launches: the prep kernel orders the items longest first (natural order beyond
  // its item limit), then the decode grid, then the merge grid.  The two later grids are
  // launched with programmatic stream serialization: they may be scheduled before the grid
  // ahead of them ends and wait for it on the device (griddepcontrol), which hides their
  // launch latency.
  bool ordered = false;
  if (split) {
    const long long items = static_cast<long long>(a.num_seqs) * P.max_groups;
    const int group_tokens = P.ppc * a.partition_tokens;
    if (items <= kMaxOrderItems && group_tokens / BS < kMaxOrderBins) {
      int32_t* order = reinterpret_cast<int32_t*>(static_cast<char*>(a.workspace) + wl.order_offset);
      decode_prep_kernel<<<1, kPrepThreads, 0, stream>>>(a.context_lens, a.num_seqs, P.max_groups,
                                                         group_tokens, BS,
                                                         a.max_blocks_per_seq * BS, order);
      if (cudaGetLastError() != cudaSuccess) return PKV_ECUDA;
      P.order = order;
      ordered = true;
    }
  }
  if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                           cudaFuncAttributeMaxDynamicSharedMemorySize, g.smem_bytes) != cudaSuccess)
    return PKV_ECUDA;
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = static_cast<size_t>(g.smem_bytes);
  cfg.stream = stream;
  cfg.attrs = ordered ? pdl : nullptr;
  cfg.numAttrs = ordered ? 1 : 0;
  if (cudaLaunchKernelEx(&cfg, fn, kmap, vmap, P) != cudaSuccess) return PKV_ECUDA;
  if (merge) {
    const long long rows = static_cast<long long>(a.num_seqs) * a.num_q_heads;
    cudaLaunchConfig_t mcfg{};
    mcfg.gridDim = dim3(static_cast<unsigned>((rows + kMergeWarps - 1) / kMergeWarps));
    mcfg.blockDim = dim3(kMergeWarps * 32);
    mcfg.dynamicSmemBytes = 0;
    mcfg.stream = stream;
    mcfg.attrs = pdl;
    mcfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&mcfg, merge, P) != cudaSuccess) return PKV_ECUDA;
  }
  return PKV_OK;
}

}  // namespace pkv
