// prefill.cu -- paged chunked-prefill attention for sm_103a.
//
// A chunk of n query tokens of a sequence whose cache holds L tokens (the chunk's own keys
// and values written last) sits at positions L-n .. L-1, and query i of the chunk attends
// positions 0 .. L-n+i ("Paged Attention: How vLLM Solves the KV Cache Memory Problem",
// section "Continuous Batching and Chunked Prefill": long prompts are processed in chunks
// interleaved with decode steps; "Paged Attention" (vanos001), section "Common Mistakes":
// the kernel does what FlashAttention does, but reads keys and values block by block).
//
// Work unit: one CTA per (sequence s, KV head g, tile of 64 packed query rows), a packed
// row being (chunk token i, query head of g), token-major, so the G heads that share KV
// head g sit in neighbouring rows and share the causal limit of their token.  Four
// consumer warps own 16 rows each; a fifth warp produces: it resolves the sequence's block
// table and streams 64-token K and V tiles (one TMA box per physical block and 64
// columns, 128-byte swizzle) into a ring of stages.  Each stage has a "full" mbarrier
// (TMA transaction bytes) and an "empty" mbarrier (one arrival per consumer warp); every
// wait gives up after ~1 s, sets PKV_DERR_TIMEOUT and makes the CTA stop.
//
// Math per consumer warp and tile: S = Q.K^T and O += P.V on mma.sync m16n8k16 with fp32
// accumulation, an online softmax in base 2 with per-row causal limits, P rounded to the
// operand type (row sums of the rounded P).  Keys past a row's limit are masked; value
// rows past the context (stale slots of the last block) are zeroed in registers.
#include <algorithm>
#include <climits>
#include <mutex>

#include "device_common.cuh"
#include "internal.h"

namespace pkv {
namespace {

constexpr int kConsumers = 4;                       // consumer warps
constexpr int kPrefillThreads = 32 * (kConsumers + 1);
constexpr int kWarpRows = 16;                       // packed query rows per consumer warp
constexpr int kTileRows = kConsumers * kWarpRows;   // packed query rows per CTA
constexpr int kKeyTile = 64;                        // key tokens per staged tile
constexpr float kSlack = 8.f;                       // rescale threshold, log2 units

struct PrefillParams {
  void* out;
  const void* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start;
  unsigned* err;
  int num_seqs, num_q_tokens, num_q_heads, num_kv_heads, group, max_query_len;
  int max_blocks_per_seq, num_blocks, block_size, m_tiles, stages, stage_bytes;
  float scale_log2;
};

template <int ROWS>
__device__ __forceinline__ uint32_t swz(int r, int d) {
  return static_cast<uint32_t>((d >> 6) * (ROWS * 128) + r * 128 +
                               ((((d & 63) >> 3) ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t keep_lo_hi(uint32_t w, bool lo, bool hi) {
  return w & ((lo ? 0x0000ffffu : 0u) | (hi ? 0xffff0000u : 0u));
}

template <typename T, int D, int BS>
__global__ void __launch_bounds__(kPrefillThreads)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap, const PrefillParams P) {
  constexpr int NBT = kKeyTile / BS;         // physical blocks per staged tile
  constexpr int TILE = kKeyTile * D * 2;     // bytes of the K (or V) tile
  constexpr int NT = kKeyTile / 8;           // 8-key column tiles of S
  extern __shared__ uint8_t smem_raw[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // (KV head fastest, then query tile, last tile first, then sequence)
  long long bid = blockIdx.x;
  const int g = static_cast<int>(bid % P.num_kv_heads);
  bid /= P.num_kv_heads;
  const int mt = P.m_tiles - 1 - static_cast<int>(bid % P.m_tiles);
  const int s = static_cast<int>(bid / P.m_tiles);
  const int q0 = P.query_start[s], q1 = P.query_start[s + 1];
  const int n = q1 - q0;
  const int L = P.context_lens[s];
  const int G = P.group;
  const int row0 = mt * kTileRows;
  if (q0 < 0 || q1 > P.num_q_tokens || n < 0 || n > P.max_query_len || n > L ||
      L > P.max_blocks_per_seq * P.block_size) {
    if (tid == 0) raise_error(P.err, PKV_DERR_CONTEXT);
    return;
  }
  if (row0 >= n * G) return;
  const int rows = min(kTileRows, n * G - row0);
  const int kmax = L - n + (row0 + rows - 1) / G;  // last key position any row sees
  const int ntiles = kmax / kKeyTile + 1;
  const int live_blocks = (L + BS - 1) / BS;

  uint8_t* ring = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + P.stages * P.stage_bytes);
  uint64_t* empty = full + P.stages;
  volatile int* flags = reinterpret_cast<volatile int*>(empty + P.stages);  // [0] abort, [1] issued
  if (tid == 0) {
    for (int i = 0; i < P.stages; ++i) {
      mbar_init(smem_addr(&full[i]), 1);
      mbar_init(smem_addr(&empty[i]), kConsumers);
    }
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumers) {
    // ---- producer warp: block ids -> TMA tile loads ------------------------------------
    const int32_t* bt = P.block_tables + static_cast<size_t>(s) * P.max_blocks_per_seq;
    const int x0 = g * D;
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
    int issued = 0;
    for (int j = 0; j < ntiles; ++j) {
      const int st = j % P.stages;
      int y = P.num_blocks * BS;  // past the tensor: the box reads as zeros
      if (lane < NBT) {
        const int jb = j * NBT + lane;
        if (jb < live_blocks) {
          const int id = bt[jb];
          if (id >= 0 && id < P.num_blocks)
            y = id * BS;
          else
            raise_error(P.err, PKV_DERR_BLOCK_ID);
        }
      }
      int ok = 1;
      if (lane == 0 && j >= P.stages)
        ok = mbar_wait_bounded(smem_addr(&empty[st]), ((j / P.stages) - 1) & 1) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok || flags[0]) {
        if (lane == 0 && !ok) {
          raise_error(P.err, PKV_DERR_TIMEOUT);
          flags[0] = 1;
        }
        break;
      }
      int ys[NBT];
#pragma unroll
      for (int k = 0; k < NBT; ++k) ys[k] = __shfl_sync(0xffffffffu, y, k);
      if (lane == 0) {
        const uint32_t bar = smem_addr(&full[st]);
        const uint32_t kdst = smem_addr(ring + st * P.stage_bytes);
        const uint32_t vdst = kdst + TILE;
        mbar_arrive_expect_tx(bar, 2u * TILE);
#pragma unroll
        for (int k = 0; k < NBT; ++k) {
#pragma unroll
          for (int b = 0; b < D / 64; ++b) {
            const uint32_t off = b * (kKeyTile * 128) + k * (BS * 128);
            tma_load_2d(kdst + off, &kmap, bar, x0 + b * 64, ys[k]);
            tma_load_2d(vdst + off, &vmap, bar, x0 + b * 64, ys[k]);
          }
        }
      }
      issued = j + 1;
    }
    if (lane == 0) flags[1] = issued;
  } else {
    // ---- consumer warps ------------------------------------------------------------------
    const int r8 = lane >> 2, c = lane & 3;
    int lim[2], qrow[2], head[2];
    bool live[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int R = row0 + warp * kWarpRows + r8 + 8 * e;
      live[e] = R < n * G;
      const int Rc = live[e] ? R : n * G - 1;  // dead rows follow the last live one
      const int i = Rc / G;
      head[e] = g * G + (Rc - i * G);
      qrow[e] = q0 + i;
      lim[e] = L - n + i;
    }
    int wlim = max(lim[0], lim[1]);
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) wlim = max(wlim, __shfl_xor_sync(0xffffffffu, wlim, o));

    uint32_t qa[D / 16][4];
    {
      const T* q = static_cast<const T*>(P.q);
      const T* qr0 = q + (static_cast<size_t>(qrow[0]) * P.num_q_heads + head[0]) * D;
      const T* qr1 = q + (static_cast<size_t>(qrow[1]) * P.num_q_heads + head[1]) * D;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const int col = kk * 16 + 2 * c;
        qa[kk][0] = live[0] ? __ldg(reinterpret_cast<const uint32_t*>(qr0 + col)) : 0u;
        qa[kk][1] = live[1] ? __ldg(reinterpret_cast<const uint32_t*>(qr1 + col)) : 0u;
        qa[kk][2] = live[0] ? __ldg(reinterpret_cast<const uint32_t*>(qr0 + col + 8)) : 0u;
        qa[kk][3] = live[1] ? __ldg(reinterpret_cast<const uint32_t*>(qr1 + col + 8)) : 0u;
      }
    }

    float o[D / 8][4];
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.f, 0.f};
    const int mi = lane >> 3;

    for (int j = 0; j < ntiles; ++j) {
      const int st = j % P.stages;
      const int t0 = j * kKeyTile;
      if (t0 <= wlim) {
        if (flags[0]) break;
        if (!mbar_wait_bounded(smem_addr(&full[st]), (j / P.stages) & 1)) {
          if (lane == 0) {
            raise_error(P.err, PKV_DERR_TIMEOUT);
            flags[0] = 1;
          }
          break;
        }
        const uint32_t kb = smem_addr(ring + st * P.stage_bytes);
        const uint32_t vb = kb + TILE;

        // S = Q . K^T
        float sc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
          const int r = nt * 8 + (lane & 7);
#pragma unroll
          for (int kk = 0; kk < D / 16; kk += 2) {
            const int d = (kk + (mi >> 1)) * 16 + (mi & 1) * 8;
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kb + swz<kKeyTile>(r, d), b0, b1, b2, b3);
            Mma<T>::run(sc[nt], qa[kk], b0, b1);
            Mma<T>::run(sc[nt], qa[kk + 1], b2, b3);
          }
        }

        // online softmax with per-row causal limits
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int kp = t0 + nt * 8 + 2 * c + (e & 1);
            const float v = sc[nt][e] * P.scale_log2;
            sc[nt][e] = kp <= lim[e >> 1] ? v : -INFINITY;
          }
          mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
          mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        // the reference max moves only when a row's scores exceed it by more than kSlack
        const bool up0 = mx0 > m[0] + kSlack, up1 = mx1 > m[1] + kSlack;
        const float mn0 = up0 ? mx0 : m[0], mn1 = up1 ? mx1 : m[1];
        uint32_t pa[kKeyTile / 16][4];
        float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          const uint32_t lo = Mma<T>::pack(exp2f(sc[nt][0] - mn0), exp2f(sc[nt][1] - mn0));
          const uint32_t hi = Mma<T>::pack(exp2f(sc[nt][2] - mn1), exp2f(sc[nt][3] - mn1));
          const float2 flo = Mma<T>::unpack(lo), fhi = Mma<T>::unpack(hi);
          rs0 += flo.x + flo.y;
          rs1 += fhi.x + fhi.y;
          pa[nt >> 1][(nt & 1) * 2 + 0] = lo;
          pa[nt >> 1][(nt & 1) * 2 + 1] = hi;
        }
        if (__any_sync(0xffffffffu, up0 || up1)) {
          const float a0 = exp2f(m[0] - mn0), a1 = exp2f(m[1] - mn1);
          l[0] *= a0;
          l[1] *= a1;
#pragma unroll
          for (int nd = 0; nd < D / 8; ++nd) {
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

        // O += P . V (value rows past the context are stale slots: zeroed here)
        const int vlim = L - t0;
#pragma unroll
        for (int kt = 0; kt < kKeyTile / 16; ++kt) {
          const int r = kt * 16 + (mi & 1) * 8 + (lane & 7);
          const int tlo = kt * 16 + 2 * c;  // token of b0/b2's low half; b1/b3 are 8 further
#pragma unroll
          for (int nd = 0; nd < D / 8; nd += 2) {
            const int d = (nd + (mi >> 1)) * 8;
            uint32_t b0, b1, b2, b3;
            ldsm_x4_trans(vb + swz<kKeyTile>(r, d), b0, b1, b2, b3);
            if (vlim < kKeyTile) {
              b0 = keep_lo_hi(b0, tlo < vlim, tlo + 1 < vlim);
              b2 = keep_lo_hi(b2, tlo < vlim, tlo + 1 < vlim);
              b1 = keep_lo_hi(b1, tlo + 8 < vlim, tlo + 9 < vlim);
              b3 = keep_lo_hi(b3, tlo + 8 < vlim, tlo + 9 < vlim);
            }
            Mma<T>::run(o[nd], pa[kt], b0, b1);
            Mma<T>::run(o[nd + 1], pa[kt], b2, b3);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&empty[st]));
    }

    // out = o / l for the live rows
    l[0] += __shfl_xor_sync(0xffffffffu, l[0], 1);
    l[0] += __shfl_xor_sync(0xffffffffu, l[0], 2);
    l[1] += __shfl_xor_sync(0xffffffffu, l[1], 1);
    l[1] += __shfl_xor_sync(0xffffffffu, l[1], 2);
    if (!flags[0]) {
      T* out = static_cast<T*>(P.out);
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        if (!live[e]) continue;
        const float inv = 1.f / l[e];
        T* orow = out + (static_cast<size_t>(qrow[e]) * P.num_q_heads + head[e]) * D;
#pragma unroll
        for (int nd = 0; nd < D / 8; ++nd) {
          *reinterpret_cast<uint32_t*>(orow + nd * 8 + 2 * c) =
              Mma<T>::pack(o[nd][2 * e] * inv, o[nd][2 * e + 1] * inv);
        }
      }
    }
  }

  __syncthreads();
  // after an abort, wait (bounded) for the tile loads still in flight before exiting
  if (tid == kConsumers * 32 && flags[0]) {
    const int issued = flags[1];
    for (int j = max(0, issued - P.stages); j < issued; ++j)
      mbar_wait_bounded(smem_addr(&full[j % P.stages]), (j / P.stages) & 1);
  }
}

using PrefillFn = void (*)(CUtensorMap, CUtensorMap, PrefillParams);

template <typename T>
PrefillFn prefill_kernel_for_type(int D, int BS) {
  if (D == 64) {
    if (BS == 16) return prefill_tc_kernel<T, 64, 16>;
    if (BS == 32) return prefill_tc_kernel<T, 64, 32>;
    if (BS == 64) return prefill_tc_kernel<T, 64, 64>;
  } else if (D == 128) {
    if (BS == 16) return prefill_tc_kernel<T, 128, 16>;
    if (BS == 32) return prefill_tc_kernel<T, 128, 32>;
    if (BS == 64) return prefill_tc_kernel<T, 128, 64>;
  }
  return nullptr;
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

constexpr int kMaxPrefillSmem = 227 * 1024;

}  // namespace

bool prefill_supported(pkv_dtype dtype, int head_dim, int block_size) {
  return (dtype == PKV_BF16 || dtype == PKV_F16) && (head_dim == 64 || head_dim == 128) &&
         (block_size == 16 || block_size == 32 || block_size == 64);
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
  P.m_tiles = static_cast<int>((packed + kTileRows - 1) / kTileRows);
  P.stage_bytes = 2 * kKeyTile * D * 2;
  P.stages = D == 128 ? 3 : 4;
  P.scale_log2 = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
  const long long grid = static_cast<long long>(a.num_seqs) * P.m_tiles * a.num_kv_heads;
  if (grid > INT_MAX) return PKV_EUNSUPPORTED;
  const int smem = 1024 + P.stages * P.stage_bytes + 16 * P.stages + 16;
  if (smem > kMaxPrefillSmem) return PKV_EUNSUPPORTED;

  CUtensorMap kmap, vmap;
  const long long rows = static_cast<long long>(a.num_blocks) * BS;
  if (!make_kv_map(&kmap, a.k_cache, a.dtype, a.num_kv_heads, D, rows, BS) ||
      !make_kv_map(&vmap, a.v_cache, a.dtype, a.num_kv_heads, D, rows, BS))
    return PKV_ECUDA;
  PrefillFn fn = a.dtype == PKV_BF16 ? prefill_kernel_for_type<__nv_bfloat16>(D, BS)
                                     : prefill_kernel_for_type<__half>(D, BS);
  if (!fn) return PKV_EUNSUPPORTED;
  if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return PKV_ECUDA;
  fn<<<static_cast<unsigned>(grid), kPrefillThreads, smem, stream>>>(kmap, vmap, P);
  return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ECUDA;
}

}  // namespace pkv
