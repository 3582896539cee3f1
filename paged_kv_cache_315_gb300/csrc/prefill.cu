// prefill.cu -- paged chunked-prefill attention for sm_103a.
//
// A chunk of n query tokens of a sequence whose cache holds L tokens (the chunk's own keys
// and values written last) sits at positions L-n .. L-1, and query i of the chunk attends
// positions 0 .. L-n+i ("Paged Attention: How vLLM Solves the KV Cache Memory Problem",
// section "Continuous Batching and Chunked Prefill": long prompts are processed in chunks
// interleaved with decode steps; "Paged Attention" (vanos001), section "Common Mistakes":
// the kernel does what FlashAttention does, but reads keys and values block by block).
//
// Every shape runs on the 5th-generation tensor cores (tcgen05, accumulators in tensor
// memory); the kernel and its pipeline are described above prefill_umma_kernel below.
#include <algorithm>
#include <cmath>
#include <climits>
#include <mutex>
#include <type_traits>

#include "device_common.cuh"
#include "internal.h"
#include "umma.cuh"

namespace pkv {
namespace {

constexpr float kSlack = 8.f;  // rescale threshold, log2 units

struct PrefillParams {
  void* out;
  const void* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start;
  unsigned* err;
  int num_seqs, num_q_tokens, num_q_heads, num_kv_heads, group, max_query_len;
  int max_blocks_per_seq, num_blocks, block_size, m_tiles;
  // |scale| * log2(e): the exponent of a weight is scale_log2 * s' - m for the score
  // s' = <q', k>, where q' is the query with every sign bit XORed with q_sign.  A negative
  // scale flips the query's signs (q' = -q, exact) and keeps scale_log2 >= 0, so the row
  // maximum of scale * s is always scale_log2 times the maximum of the raw scores s'.
  float scale_log2;
  uint32_t q_sign;  // 0x80008000 when the scale is negative (two 16-bit lanes), else 0
  // Options of the tcgen05 kernel, used by the shared-prefix decode (all off for prefill):
  const int32_t* kv_start;    // per sequence, first attended position (a block multiple), or null
  const int32_t* table_rows;  // per sequence, the block-table row to read, or null (row s)
  int causal;                 // 1: row i sees positions < L - n + i + 1; 0: every row sees < L
  float* part_o;              // when set: unnormalised o [num_q_tokens, num_q_heads, 128] fp32
  float* part_ml;             //   and (m in log2 units, l) [num_q_tokens, num_q_heads, 2]
  int ksplit;                 // key ranges per sequence (non-causal only), one partial each
};

// two fp32 lanes in one 64-bit register: packed FMA and add (sm_100 and later)
__device__ __forceinline__ unsigned long long f2_pack(float a, float b) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long r, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
  unsigned long long r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
  unsigned long long r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}


// ------------------------------------------------------------------------------------------
// tcgen05 path: head_dim 64 or 128
// ------------------------------------------------------------------------------------------
//
// One CTA per (sequence, KV head, 128 packed query rows).  Warps 0-3 run the softmax
// (thread r owns row r, which is tensor-memory lane r), warp 4 loads the Q tile and the
// 64-token K tiles, warp 6 the V tiles, and warp 5 issues the MMAs from one thread.
// With a power-of-two number G of query heads per KV head (at most 128) the Q tile is one
// 3-D TMA box per 64 columns (G heads x 128/G tokens); with any other G, and for a negative
// scale, each softmax thread stages its own query row instead (QT), with its signs flipped
// for a negative scale.
// Tensor memory (256 columns): two 64-column score buffers and the 128-column output (at
// head_dim 64: three score buffers and a 64-column output).
//   S_b = Q . K_j^T       (M 128, N 64, K 128; A and B K-major from shared memory)
//   P_j                   (bf16, written over the first 32 columns of S_b)
//   O  += P_j . V_j       (M 128, N 128, K 64; A from tensor memory, V MN-major)
// The MMA thread issues QK(j) before PV(j-1), so the tensor cores score tile j while the
// softmax warps turn tile j-1's scores into weights.  O stays in tensor memory for the
// whole key range; the softmax reference max moves only when a row's scores exceed it by
// more than kSlack, and only then are O's rows rescaled (after the previous PV is done).

constexpr int kUThreads = 224;
constexpr int kURows = 128;       // packed query rows per CTA
constexpr int kUKeys = 64;        // key tokens per tile
constexpr int kUStages = 2;       // K/V ring depth at head_dim 128 (shared memory allows no more)
constexpr int kUTmemCols = 256;
// bytes of a K (or V) tile, of the Q tile, and the dynamic shared memory, for head_dim D
// (D / 64 boxes of 64 columns per row, each box 128-byte rows)
__host__ __device__ constexpr int u_tile(int D) { return kUKeys * D * 2; }
__host__ __device__ constexpr int u_qbytes(int D) { return kURows * D * 2; }
// K/V ring depth: head_dim 64 tiles take half the bytes, so the rings run deeper
__host__ __device__ constexpr int u_stages(int D) { return D == 64 ? 3 : kUStages; }
__host__ __device__ constexpr int u_smem(int D) {
  return 1024 + u_qbytes(D) + u_stages(D) * 2 * u_tile(D) + 512;
}

template <typename T, int D, int BS, bool QT, bool WI>
__global__ void __launch_bounds__(kUThreads, 2)
    prefill_umma_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap,
                        const __grid_constant__ CUtensorMap qmap, const PrefillParams P) {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  constexpr int NBT = kUKeys / BS;
  constexpr int NBX = D / 64;                  // 64-column boxes per row
  constexpr int kUTile = u_tile(D);
  constexpr int kUQBytes = u_qbytes(D);
  constexpr int ST = u_stages(D);
  constexpr bool kBf16 = sizeof(T) == 2 && !std::is_same<T, __half>::value;
  constexpr uint32_t kIdQK = umma_idesc(kURows, kUKeys, kBf16, false);
  constexpr uint32_t kIdPV = umma_idesc(kURows, D, kBf16, true);
  // score buffers: at head_dim 64 the output takes 64 columns, so a third 64-column buffer
  // fits in the CTA's 256 (QK(j) then waits for PV(j - 3) instead of PV(j - 2))
  constexpr int SB = D == 64 ? 3 : 2;
  // barriers, the tensor-memory address and the flags fit the 512 bytes past the ring
  static_assert((2 + 4 * ST + 3 * SB) * 8 + 16 <= 512, "barrier area");
  extern __shared__ uint8_t smem_raw[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  long long bid = blockIdx.x;
  const int g = static_cast<int>(bid % P.num_kv_heads);
  bid /= P.num_kv_heads;
  const int split = static_cast<int>(bid % P.ksplit);
  bid /= P.ksplit;
  const int mt = P.m_tiles - 1 - static_cast<int>(bid % P.m_tiles);
  const int s = static_cast<int>(bid / P.m_tiles);
  const int q0 = P.query_start[s], q1 = P.query_start[s + 1];
  const int n = q1 - q0;
  const int L = P.context_lens[s];
  const int G = P.group;
  const int row0 = mt * kURows;
  const int ks0 = P.kv_start ? P.kv_start[s] : 0;  // first attended position
  if (q0 < 0 || q1 > P.num_q_tokens || n < 0 || n > P.max_query_len ||
      (P.causal && n > L) || L > P.max_blocks_per_seq * P.block_size || ks0 < 0 ||
      ks0 % BS != 0) {
    if (tid == 0) raise_error(P.err, PKV_DERR_CONTEXT);
    return;
  }
  if (row0 >= n * G) return;
  const int rows = min(kURows, n * G - row0);
  // key range of this split: whole 64-key tiles of [ks0, L), `split` of `ksplit`
  const int span = ((max(L - ks0, 0) + kUKeys - 1) / kUKeys + P.ksplit - 1) / P.ksplit * kUKeys;
  const int ks = ks0 + split * span;
  const int ke = min(L, ks + span);  // one past the last key
  float* part_o = P.part_o ? P.part_o + static_cast<size_t>(split) * P.num_q_tokens *
                                            P.num_q_heads * 128
                           : nullptr;
  float* part_ml = P.part_ml ? P.part_ml + static_cast<size_t>(split) * P.num_q_tokens *
                                              P.num_q_heads * 2
                             : nullptr;
  if (ks >= ke) {
    // nothing to attend: the rows' partials are empty (m = -inf, l = 0, o = 0)
    if (part_o && tid < rows) {
      const int R = row0 + tid, i = R / G;
      const size_t row = static_cast<size_t>(q0 + i) * P.num_q_heads + g * G + (R - i * G);
      for (int d = 0; d < 128; ++d) part_o[row * 128 + d] = 0.f;
      part_ml[row * 2] = -INFINITY;
      part_ml[row * 2 + 1] = 0.f;
    }
    return;
  }
  const int kmax = P.causal ? L - n + (row0 + rows - 1) / G : ke - 1;
  const int ntiles = (kmax - ks) / kUKeys + 1;
  const int live_blocks = (L + BS - 1) / BS;
  const int blk0 = ks / BS;  // first block of tile 0

  uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint8_t* sq = base;
  uint8_t* ring = base + kUQBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + ST * 2 * kUTile);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;                   // [ST]
  uint64_t* k_empty = k_full + ST;               // [ST]
  uint64_t* v_full = k_empty + ST;               // [ST]
  uint64_t* v_empty = v_full + ST;               // [ST]
  uint64_t* s_full = v_empty + ST;               // [SB]
  uint64_t* p_full = s_full + SB;                // [SB]
  uint64_t* pv_done = p_full + SB;               // [SB]: the P.V of the tiles using S_b
  uint64_t* drain = pv_done + SB;
  uint32_t* tmem_base = reinterpret_cast<uint32_t*>(drain + 1);
  // [0] abort, [1] K tiles issued, [2] V tiles issued
  volatile int* flags = reinterpret_cast<volatile int*>(tmem_base + 1);

  if (tid == 0) {
    mbar_init(smem_addr(q_full), QT ? 4 : 1);  // QT: one arrival per softmax warp
    for (int i = 0; i < ST; ++i) {
      mbar_init(smem_addr(&k_full[i]), 1);
      mbar_init(smem_addr(&k_empty[i]), 1);
      mbar_init(smem_addr(&v_full[i]), 1);
      mbar_init(smem_addr(&v_empty[i]), 1);
    }
    for (int i = 0; i < SB; ++i) {
      mbar_init(smem_addr(&s_full[i]), 1);
      mbar_init(smem_addr(&p_full[i]), 4);
      mbar_init(smem_addr(&pv_done[i]), 1);
    }
    mbar_init(smem_addr(drain), 1);
    flags[0] = 0;
    flags[1] = 0;
    flags[2] = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_addr(tmem_base), kUTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tm = *tmem_base;
  const uint32_t tm_o = tm + SB * kUKeys;

  auto fail = [&](void) {
    raise_error(P.err, PKV_DERR_TIMEOUT);
    flags[0] = 1;
  };

  if (warp == 4 || warp == 6) {
    // ---- producers: warp 4 loads Q and the K tiles, warp 6 the V tiles ----------------
    // A K slot frees when the QK that read it completes, a V slot when its PV completes,
    // so each ring runs ahead by its own consumer.
    const bool is_k = warp == 4;
    const CUtensorMap* map = is_k ? &kmap : &vmap;
    uint64_t* fullb = is_k ? k_full : v_full;
    uint64_t* emptyb = is_k ? k_empty : v_empty;
    const uint32_t tile_off = is_k ? 0u : static_cast<uint32_t>(kUTile);
    const int trow = P.table_rows ? P.table_rows[s] : s;
    const int32_t* bt = P.block_tables + static_cast<size_t>(trow) * P.max_blocks_per_seq;
    const int x0 = g * D;
    if (lane == 0) {
      tma_prefetch_desc(map);
      if (is_k && !QT) {
        tma_prefetch_desc(&qmap);
        const uint32_t bar = smem_addr(q_full);
        mbar_arrive_expect_tx(bar, kUQBytes);
#pragma unroll
        for (int b = 0; b < NBX; ++b)
          tma_load_3d(smem_addr(sq) + b * (kURows * 128), &qmap, bar, 64 * b, g * G,
                      q0 + row0 / G);
      }
    }
    // TMA row coordinate of lane k's block of tile j (out of range, so reading zeros, past
    // the context); the next tile's is read while this one waits for its slot
    auto row_of = [&](int j) -> int {
      int y = P.num_blocks * BS;
      if (lane < NBT) {
        const int jb = blk0 + j * NBT + lane;
        if (jb < live_blocks) {
          const int id = bt[jb];
          if (id >= 0 && id < P.num_blocks)
            y = id * BS;
          else if (is_k)
            raise_error(P.err, PKV_DERR_BLOCK_ID);
        }
      }
      return y;
    };
    int issued = 0;
    int ynext = ntiles > 0 ? row_of(0) : 0;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % ST;
      const int y = ynext;
      if (j + 1 < ntiles) ynext = row_of(j + 1);
      int ok = 1;
      if (lane == 0 && j >= ST)
        ok = mbar_wait_bounded(smem_addr(&emptyb[st]), ((j / ST) - 1) & 1) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok || __any_sync(0xffffffffu, flags[0] != 0)) {
        if (lane == 0 && !ok) fail();
        break;
      }
      int ys[NBT];
#pragma unroll
      for (int k = 0; k < NBT; ++k) ys[k] = __shfl_sync(0xffffffffu, y, k);
      if (lane == 0) {
        const uint32_t bar = smem_addr(&fullb[st]);
        const uint32_t dst = smem_addr(ring + st * 2 * kUTile) + tile_off;
        mbar_arrive_expect_tx(bar, kUTile);
#pragma unroll
        for (int k = 0; k < NBT; ++k) {
#pragma unroll
          for (int b = 0; b < NBX; ++b)
            tma_load_2d(dst + b * (kUKeys * 128) + k * (BS * 128), map, bar, x0 + b * 64, ys[k]);
        }
      }
      issued = j + 1;
    }
    if (lane == 0) flags[is_k ? 1 : 2] = issued;
  } else if (warp == 5) {
    // ---- MMA issuer -----------------------------------------------------------------------
    // K-step 0 of Q (a K-step adds its byte offset / 16 to the start-address field; every
    // address stays below 256 KB, so no carry leaves it)
    const uint64_t dq = smem_desc_sw128(smem_addr(sq), 16, 1024);
    int ok = 1;
    if (lane == 0) ok = mbar_wait_bounded(smem_addr(q_full), 0) ? 1 : 0;
    ok = __shfl_sync(0xffffffffu, ok, 0);
    if (!ok && lane == 0) fail();
    int issued_mma = 0;
    auto pv = [&](int i) -> bool {  // O += P_i . V_i
      const int st = i % ST, b = i % SB;
      // lane 0 waits for P_i and V_i and reads the abort flag; one broadcast carries all
      // three, and the __syncwarp after it orders the warp's zero-fill of stale V rows after
      // the tile's arrival
      int okv = 1;
      if (lane == 0) {
        okv = mbar_wait_bounded(smem_addr(&p_full[b]), (i / SB) & 1) ? 1 : 0;
        if (okv) okv = mbar_wait_bounded(smem_addr(&v_full[st]), (i / ST) & 1) ? 1 : 0;
        if (!okv) fail();
        if (flags[0] != 0) okv = 0;
      }
      if (!__shfl_sync(0xffffffffu, okv, 0)) return false;
      __syncwarp();
      uint8_t* vt = ring + st * 2 * kUTile + kUTile;
      // value rows past the context (stale slots of the last block) become zeros before
      // they meet zero weights in P.V
      const int vrows = L - ks - i * kUKeys;
      if (vrows < kUKeys) {
        const int nz = (kUKeys - vrows) * 8;  // 16-byte chunks per box
        for (int e = lane; e < NBX * nz; e += 32) {
          const int bx = e / nz, rem = e - bx * nz;
          *reinterpret_cast<uint4*>(vt + bx * (kUKeys * 128) + (vrows + rem / 8) * 128 +
                                    (rem & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      // K-step 0 of V; a K-step adds its byte offset / 16 to the start-address field
      const uint64_t dv = smem_desc_sw128(smem_addr(vt), kUKeys * 128, 1024);
      if constexpr (WI) {
        // the whole (converged) warp runs the issue; lane 0 performs it
        const uint32_t iss = lane == 0;
        tc_fence_after_sync();
#pragma unroll
        for (int kt = 0; kt < kUKeys / 16; ++kt)
          umma_ts_warp(iss, tm_o, tm + b * kUKeys + kt * 8,
                       dv + static_cast<uint64_t>(kt * 128), kIdPV,
                       (i > 0 || kt > 0) ? 1u : 0u);
        umma_commit_warp(iss, smem_addr(&v_empty[st]));
        umma_commit_warp(iss, smem_addr(&pv_done[b]));
      } else if (lane == 0) {
        tc_fence_after_sync();
#pragma unroll
        for (int kt = 0; kt < kUKeys / 16; ++kt)
          umma_ts(tm_o, tm + b * kUKeys + kt * 8,
                  dv + static_cast<uint64_t>(kt * 128), kIdPV,
                  (i > 0 || kt > 0) ? 1u : 0u);
        umma_commit(smem_addr(&v_empty[st]));
        umma_commit(smem_addr(&pv_done[b]));
      }
      return true;
    };
    for (int j = 0; ok && j < ntiles; ++j) {
      const int st = j % ST, b = j % SB;
      // lane 0 waits for K_j and for S_b to be free, and reads the abort flag; one broadcast
      // carries all three.  S_b still holds P_{j-SB}: the P.V that reads it must be complete
      // before QK(j) overwrites it (that P.V is the ((j - SB) / SB)-th completion of
      // pv_done[b]).
      int okk = 1;
      if (lane == 0) {
        okk = mbar_wait_bounded(smem_addr(&k_full[st]), (j / ST) & 1) ? 1 : 0;
        if (okk && j >= SB)
          okk = mbar_wait_bounded(smem_addr(&pv_done[b]), ((j - SB) / SB) & 1) ? 1 : 0;
        if (!okk) fail();
        if (flags[0] != 0) okk = 0;
      }
      if (!__shfl_sync(0xffffffffu, okk, 0)) {
        ok = 0;
        break;
      }
      const uint64_t dk = smem_desc_sw128(smem_addr(ring + st * 2 * kUTile), 16, 1024);
      if constexpr (WI) {
        const uint32_t iss = lane == 0;
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss_warp(iss, tm + b * kUKeys,
                       dq + static_cast<uint64_t>(((kk >> 2) * (kURows * 128) + (kk & 3) * 32) >> 4),
                       dk + static_cast<uint64_t>(((kk >> 2) * (kUKeys * 128) + (kk & 3) * 32) >> 4),
                       kIdQK, kk > 0 ? 1u : 0u);
        umma_commit_warp(iss, smem_addr(&k_empty[st]));
        umma_commit_warp(iss, smem_addr(&s_full[b]));
      } else if (lane == 0) {
        tc_fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(tm + b * kUKeys,
                  dq + static_cast<uint64_t>(((kk >> 2) * (kURows * 128) + (kk & 3) * 32) >> 4),
                  dk + static_cast<uint64_t>(((kk >> 2) * (kUKeys * 128) + (kk & 3) * 32) >> 4),
                  kIdQK, kk > 0 ? 1u : 0u);
        umma_commit(smem_addr(&k_empty[st]));
        umma_commit(smem_addr(&s_full[b]));
      }
      issued_mma = 1;
      if (j > 0 && !pv(j - 1)) {
        ok = 0;
        break;
      }
    }
    if (ok && ntiles > 0) pv(ntiles - 1);
    // every MMA this thread issued is complete before tensor memory is released
    if (lane == 0 && issued_mma) {
      umma_commit(smem_addr(drain));
      if (!mbar_wait_bounded(smem_addr(drain), 0)) fail();
    }
  } else {
    // ---- softmax warps: thread r owns packed row r -------------------------------------
    const int r = tid;
    const int R = row0 + r;
    const bool live = R < n * G;
    const int Rc = live ? R : n * G - 1;
    const int i = Rc / G;
    const int head = g * G + (Rc - i * G);
    const int lim = (P.causal ? L - n + i : ke - 1) - ks;  // last key, relative to ks
    const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
    if constexpr (QT) {
      // the row's query into the Q tile: D / 64 boxes of 128-byte rows, 16-byte chunk c of
      // row r stored at chunk c ^ (r mod 8) (the 128-byte swizzle the MMA's shared-memory
      // descriptor describes)
      const uint4* qrow = reinterpret_cast<const uint4*>(
          static_cast<const T*>(P.q) + (static_cast<size_t>(q0 + i) * P.num_q_heads + head) * D);
      const uint32_t sg = P.q_sign;
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        uint4 v = __ldg(qrow + c);
        v.x ^= sg;
        v.y ^= sg;
        v.z ^= sg;
        v.w ^= sg;
        *reinterpret_cast<uint4*>(sq + (c >> 3) * (kURows * 128) + r * 128 +
                                  (((c & 7) ^ (r & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(q_full));
    }
    float m = -INFINITY, l = 0.f;
    int done = 0;
    for (int j = 0; j < ntiles; ++j) {
      const int b = j % SB;
      // warp-uniform decisions: the tensor-memory accesses below are warp-collective
      if (__any_sync(0xffffffffu, flags[0] != 0)) break;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(&s_full[b]), (j / SB) & 1))) {
        if (lane == 0) fail();
        break;
      }
      tc_fence_after_sync();
      uint32_t sraw[2][32];
      tmem_ld32(tm + lane_off + b * kUKeys, sraw[0]);
      tmem_ld32(tm + lane_off + b * kUKeys + 32, sraw[1]);
      tmem_ld_wait();
      // scores past the row's causal limit are masked (only tiles that cross it); the
      // maximum is taken on the raw scores and the scale folds into one FFMA per score
      const int rl = lim - j * kUKeys;  // last allowed key index within the tile
      float mxr = -INFINITY;
      if (rl >= kUKeys - 1) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int c = 0; c < 32; ++c) mxr = fmaxf(mxr, __uint_as_float(sraw[h][c]));
      } else {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float v = h * 32 + c <= rl ? __uint_as_float(sraw[h][c]) : -INFINITY;
            sraw[h][c] = __float_as_uint(v);
            mxr = fmaxf(mxr, v);
          }
      }
      const float sl2 = P.scale_log2;  // >= 0 (a negative scale flipped the query's signs)
      const float mx = mxr * sl2;
      const bool up = mx > m + kSlack;
      const float mn = up ? mx : m;
      const float nmn = -mn;
      // score pairs through packed fp32 FMA and add (half the instructions of scalar ones;
      // the row sum accumulates even and odd keys separately)
      uint32_t pk[32];
      unsigned long long rs2 = f2_pack(0.f, 0.f);
      const unsigned long long sl2x2 = f2_pack(sl2, sl2), nmnx2 = f2_pack(nmn, nmn);
      auto weights = [&](auto masked) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            float a0, a1;
            const unsigned long long x2 =
                f2_pack(__uint_as_float(sraw[h][2 * c]), __uint_as_float(sraw[h][2 * c + 1]));
            f2_unpack(f2_fma(x2, sl2x2, nmnx2), a0, a1);
            if constexpr (decltype(masked)::value) {
              // keys past the row's limit weigh 0 whatever the scale (with a zero scale
              // their -inf scores would otherwise give 0 * -inf)
              if (h * 32 + 2 * c > rl) a0 = -INFINITY;
              if (h * 32 + 2 * c + 1 > rl) a1 = -INFINITY;
            }
            const float p0 = fast_exp2(a0), p1 = fast_exp2(a1);
            rs2 = f2_add(rs2, f2_pack(p0, p1));
            pk[h * 16 + c] = Mma<T>::pack(p0, p1);
          }
      };
      if (rl >= kUKeys - 1)
        weights(std::false_type{});
      else
        weights(std::true_type{});
      float rs;
      {
        float r0, r1;
        f2_unpack(rs2, r0, r1);
        rs = r0 + r1;
      }
      const float alpha = exp2f(m - mn);  // 0 on the first tile (m = -inf), 1 if m stays
      if (j > 0 && __any_sync(0xffffffffu, up)) {
        // O's rows move to the new reference: the previous P.V must have landed
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(&pv_done[(j - 1) % SB]),
                                                        ((j - 1) / SB) & 1))) {
          if (lane == 0) fail();
          break;
        }
        tc_fence_after_sync();
#pragma unroll
        for (int part = 0; part < D / 32; ++part) {
          uint32_t ov[32];
          tmem_ld32(tm_o + lane_off + part * 32, ov);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
          tmem_st32(tm_o + lane_off + part * 32, ov);
        }
      }
      l = l * alpha + rs;
      m = mn;
      tmem_st32(tm + lane_off + b * kUKeys, pk);
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&p_full[b]));
      done = j + 1;
    }
    // the last P.V: waited on through `drain`, which the MMA thread commits after it (a
    // parity wait on pv_done[b] cannot tell PV(ntiles-1) from PV(ntiles-1-2SB))
    if (done == ntiles && !__any_sync(0xffffffffu, flags[0] != 0)) {
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(drain), 0))) {
        if (lane == 0) fail();
      } else {
        tc_fence_after_sync();
        const size_t orow_i = static_cast<size_t>(q0 + i) * P.num_q_heads + head;
        if (part_o) {
          // the partial (m, l, o) of this key range, for a log-sum-exp merge
          float* po = part_o + orow_i * D;
#pragma unroll
          for (int part = 0; part < D / 32; ++part) {
            uint32_t ov[32];
            tmem_ld32(tm_o + lane_off + part * 32, ov);
            tmem_ld_wait();
            if (live) {
#pragma unroll
              for (int c = 0; c < 32; c += 4)
                *reinterpret_cast<float4*>(po + part * 32 + c) =
                    make_float4(__uint_as_float(ov[c]), __uint_as_float(ov[c + 1]),
                                __uint_as_float(ov[c + 2]), __uint_as_float(ov[c + 3]));
            }
          }
          if (live) {
            part_ml[orow_i * 2] = m;
            part_ml[orow_i * 2 + 1] = l;
          }
        } else {
          const float inv = 1.f / l;
          T* orow = static_cast<T*>(P.out) + orow_i * D;
#pragma unroll
          for (int part = 0; part < D / 32; ++part) {
            uint32_t ov[32];
            tmem_ld32(tm_o + lane_off + part * 32, ov);
            tmem_ld_wait();
            if (live) {
#pragma unroll
              for (int c = 0; c < 32; c += 8) {
                uint4 v;
                v.x = Mma<T>::pack(__uint_as_float(ov[c]) * inv, __uint_as_float(ov[c + 1]) * inv);
                v.y = Mma<T>::pack(__uint_as_float(ov[c + 2]) * inv, __uint_as_float(ov[c + 3]) * inv);
                v.z = Mma<T>::pack(__uint_as_float(ov[c + 4]) * inv, __uint_as_float(ov[c + 5]) * inv);
                v.w = Mma<T>::pack(__uint_as_float(ov[c + 6]) * inv, __uint_as_float(ov[c + 7]) * inv);
                *reinterpret_cast<uint4*>(orow + part * 32 + c) = v;
              }
            }
          }
        }
      }
    }
  }

  // wait (bounded) for tile loads still in flight after an abort, then free tensor memory
  if ((tid == 4 * 32 || tid == 6 * 32) && flags[0]) {
    const bool is_k = tid == 4 * 32;
    if (is_k && !QT) mbar_wait_bounded(smem_addr(q_full), 0);
    uint64_t* fullb = is_k ? k_full : v_full;
    const int issued = flags[is_k ? 1 : 2];
    for (int j = max(0, issued - ST); j < issued; ++j)
      mbar_wait_bounded(smem_addr(&fullb[j % ST]), (j / ST) & 1);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 0) tmem_dealloc(tm, kUTmemCols);
}

using PrefillUmmaFn = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, PrefillParams);

template <typename T, int D, bool QT, bool WI>
PrefillUmmaFn prefill_umma_for(int BS) {
  if (BS == 16) return prefill_umma_kernel<T, D, 16, QT, WI>;
  if (BS == 32) return prefill_umma_kernel<T, D, 32, QT, WI>;
  if (BS == 64) return prefill_umma_kernel<T, D, 64, QT, WI>;
  return nullptr;
}

// q_tma: the Q tile by TMA (else staged by the softmax threads); warp_issue: MMAs issued by
// the converged warp (causal chunks) rather than from a lane-0 branch (the options of the
// shared-prefix passes), the faster form for each on GB300.  head_dim 64 serves plain chunked
// prefill only (the shared-prefix passes use head_dim 128).
template <typename T>
PrefillUmmaFn prefill_umma_for_type(int D, int BS, bool q_tma, bool warp_issue) {
  if (D == 64) {
    if (!warp_issue) return nullptr;
    return q_tma ? prefill_umma_for<T, 64, false, true>(BS)
                 : prefill_umma_for<T, 64, true, true>(BS);
  }
  if (D != 128) return nullptr;
  if (warp_issue)
    return q_tma ? prefill_umma_for<T, 128, false, true>(BS)
                 : prefill_umma_for<T, 128, true, true>(BS);
  return q_tma ? prefill_umma_for<T, 128, false, false>(BS)
               : prefill_umma_for<T, 128, true, false>(BS);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult qr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &qr) == cudaSuccess &&
        qr == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// A cache tensor seen as 2-D (x = Hkv * D elements, y = cache rows), boxes of 64 columns
// by block_size rows with the 128-byte swizzle.
bool make_kv_map(CUtensorMap* map, const void* base, pkv_dtype dt, int Hkv, int D, long long rows,
                 int BS) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  const CUtensorMapDataType t =
      dt == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(Hkv) * D, static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(Hkv) * D * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(BS)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, t, 2, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// q [T, Hq, D] seen as 3-D (x = head_dim, y = query head, z = token): boxes of 64 columns
// x G heads x 128 / G tokens, i.e. 128 packed rows of 128 bytes, 128-byte swizzle.
bool make_q_map(CUtensorMap* map, const void* base, pkv_dtype dt, int T, int Hq, int D, int G) {
  EncodeTiledFn enc = encode_tiled();
  if (!enc) return false;
  const CUtensorMapDataType t =
      dt == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hq),
                              static_cast<cuuint64_t>(T)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(Hq) * D * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(G), static_cast<cuuint32_t>(128 / G)};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, t, 3, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// Whether the tcgen05 kernel's Q tile is one 3-D TMA box per 64 columns: a power-of-two
// number of query heads per KV head (at most 128) and a scale whose sign needs no flip.
bool umma_q_tma(int group, float scale) {
  return group <= 128 && (group & (group - 1)) == 0 && !(scale < 0.f);
}

}  // namespace

bool prefill_supported(pkv_dtype dtype, int head_dim, int block_size) {
  return (dtype == PKV_BF16 || dtype == PKV_F16) && (head_dim == 64 || head_dim == 128) &&
         (block_size == 16 || block_size == 32 || block_size == 64);
}

// The tcgen05 kernel with the shared-prefix options (partials of 128 columns): head_dim 128.
bool prefill_umma_supported(pkv_dtype dtype, int head_dim, int block_size, int group,
                            float scale) {
  return prefill_supported(dtype, head_dim, block_size) && head_dim == 128 && group >= 1 &&
         scale == scale;
}

int launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  if (!prefill_supported(a.dtype, a.head_dim, a.block_size)) return PKV_EUNSUPPORTED;
  if (a.num_seqs == 0 || a.num_q_tokens == 0 || a.max_query_len == 0) return PKV_OK;
  const int D = a.head_dim, BS = a.block_size;
  PrefillParams P{};
  P.out = a.out;
  P.q = a.q;
  P.block_tables = a.block_tables;
  P.context_lens = a.context_lens;
  P.query_start = a.query_start;
  P.err = a.err;
  P.num_seqs = a.num_seqs;
  P.num_q_tokens = a.num_q_tokens;
  P.num_q_heads = a.num_q_heads;
  P.num_kv_heads = a.num_kv_heads;
  P.group = a.num_q_heads / a.num_kv_heads;
  P.max_query_len = a.max_query_len;
  P.max_blocks_per_seq = a.max_blocks_per_seq;
  P.num_blocks = a.num_blocks;
  P.block_size = BS;
  const long long packed = static_cast<long long>(a.max_query_len) * P.group;
  if (packed > INT_MAX / 2) return PKV_EUNSUPPORTED;
  P.m_tiles = static_cast<int>((packed + kURows - 1) / kURows);
  // a negative scale runs as (-q) . k times |scale|: exact, and the softmax keeps taking
  // the row maximum of the raw scores
  P.scale_log2 =
      static_cast<float>(std::fabs(static_cast<double>(a.scale)) * 1.4426950408889634);
  P.q_sign = a.scale < 0.f ? 0x80008000u : 0u;
  P.kv_start = a.kv_start;
  P.table_rows = a.table_rows;
  P.causal = a.non_causal ? 0 : 1;
  P.part_o = a.part_o;
  P.part_ml = a.part_ml;
  P.ksplit = a.ksplit > 0 ? a.ksplit : 1;
  const bool options = a.kv_start || a.table_rows || a.non_causal || a.part_o || P.ksplit > 1;
  if (options && (D != 128 || (P.ksplit > 1 && P.causal) || (!a.part_o && P.ksplit > 1)))
    return PKV_EUNSUPPORTED;
  const long long grid =
      static_cast<long long>(a.num_seqs) * P.m_tiles * a.num_kv_heads * P.ksplit;
  if (grid > INT_MAX) return PKV_EUNSUPPORTED;

  CUtensorMap kmap, vmap;
  const long long rows = static_cast<long long>(a.num_blocks) * BS;
  if (!make_kv_map(&kmap, a.k_cache, a.dtype, a.num_kv_heads, D, rows, BS) ||
      !make_kv_map(&vmap, a.v_cache, a.dtype, a.num_kv_heads, D, rows, BS))
    return PKV_ECUDA;
  // (with the query rows staged by threads the kernel never reads the Q map)
  const bool q_tma = umma_q_tma(P.group, a.scale);
  CUtensorMap qmap{};
  if (q_tma && !make_q_map(&qmap, a.q, a.dtype, a.num_q_tokens, a.num_q_heads, D, P.group))
    return PKV_ECUDA;
  const bool warp_issue = !options;
  PrefillUmmaFn ufn =
      a.dtype == PKV_BF16 ? prefill_umma_for_type<__nv_bfloat16>(D, BS, q_tma, warp_issue)
                          : prefill_umma_for_type<__half>(D, BS, q_tma, warp_issue);
  if (!ufn) return PKV_EUNSUPPORTED;
  const int usmem = u_smem(D);
  if (cudaFuncSetAttribute(reinterpret_cast<const void*>(ufn),
                           cudaFuncAttributeMaxDynamicSharedMemorySize, usmem) != cudaSuccess)
    return PKV_ECUDA;
  ufn<<<static_cast<unsigned>(grid), kUThreads, usmem, stream>>>(kmap, vmap, qmap, P);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

}  // namespace pkv
