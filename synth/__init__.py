"""Seeded synthetic decode workloads for paged KV-cache attention.

This module is the one place both sides of every check take their inputs from:
the fp64 oracle (tests, CPU baseline) and the CUDA library (tests, benchmark).
It holds none of the attention arithmetic.  It only

  * draws random tensors (``numpy`` counter-seeded generators, one independent
    stream per tensor and per chunk, so results do not depend on thread count),
  * rounds fp32 draws to bf16 / fp16 storage, and re-encodes pools as E4M3 codes for
    fp8 caches (torch's float8 conversion),
  * hands out physical blocks with a trivial allocator: the pool's ids are shuffled
    once and each sequence takes the next ``ceil(L / block_size)`` of them in order,
  * records, from that allocation, which cache slots hold live tokens (for
    NaN-poisoning the rest).

Workload recipes mirror the five decode batches the benchmark and the tests use;
see ``CONFIGS``.  Everything is returned as numpy arrays (16-bit element types
as raw ``uint16`` bit patterns); ``to_torch`` moves a workload to a device.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import numpy as np

BASE_SEED = 315

_CHUNK = 1 << 22  # elements per independently seeded draw
_POISON_BITS = {"bf16": 0x7FC0, "f16": 0x7E00}


# ---------------------------------------------------------------------------------------
# element storage
# ---------------------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to bf16 (nearest, ties to even); return the bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    b = b + (np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1)))
    return (b >> np.uint32(16)).astype(np.uint16)


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to IEEE fp16 (numpy's conversion); return the bit patterns."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def storage_dtype(dtype: str):
    return np.float32 if dtype == "f32" else np.uint16


def to_storage(x: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "f32":
        return np.ascontiguousarray(x, dtype=np.float32)
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    if dtype == "f16":
        return f32_to_f16_bits(x)
    raise ValueError(dtype)


def storage_to_f64(x: np.ndarray, dtype: str) -> np.ndarray:
    """Widen stored elements to float64 exactly (for comparisons in tests)."""
    if dtype == "f32":
        return x.astype(np.float64)
    if dtype == "bf16":
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    if dtype == "f16":
        return x.view(np.float16).astype(np.float64)
    raise ValueError(dtype)


def _threads() -> int:
    return max(1, min(16, os.cpu_count() or 1))


def normal_storage(seed, shape, dtype: str, row_scale=None) -> np.ndarray:
    """N(0, 1) draws of ``shape`` in ``dtype`` storage.

    ``seed`` is a ``numpy.random.SeedSequence``; the array is cut into fixed chunks,
    each drawn from its own child sequence, so the result is the same for any
    number of worker threads.  ``row_scale`` (optional, shape ``shape[:-1]``)
    multiplies whole last-axis rows before rounding.
    """
    shape = tuple(int(s) for s in shape)
    n = int(np.prod(shape)) if shape else 1
    out = np.empty(n, dtype=storage_dtype(dtype))
    row = shape[-1] if shape else 1
    chunk = max(row, (_CHUNK // row) * row)
    nchunks = (n + chunk - 1) // chunk
    children = seed.spawn(nchunks) if nchunks else []
    rs = None if row_scale is None else np.ascontiguousarray(row_scale, np.float32).reshape(-1)

    def work(i):
        lo = i * chunk
        hi = min(n, lo + chunk)
        g = np.random.Generator(np.random.PCG64(children[i]))
        x = g.standard_normal(hi - lo, dtype=np.float32)
        if rs is not None:
            x = (x.reshape(-1, row) * rs[lo // row: hi // row, None]).reshape(-1)
        out[lo:hi] = to_storage(x, dtype)

    if nchunks <= 1:
        for i in range(nchunks):
            work(i)
    else:
        with ThreadPoolExecutor(max_workers=_threads()) as ex:
            list(ex.map(work, range(nchunks)))
    return out.reshape(shape)


# ---------------------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------------------

@dataclass
class Workload:
    """One decode batch over a paged KV pool (numpy, host)."""
    name: str
    dtype: str                      # "f32" | "bf16" | "f16"
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    scale: float
    q: np.ndarray                   # [B, Hq, D]
    k_cache: np.ndarray             # [NB, bs, Hkv, D]
    v_cache: np.ndarray             # [NB, bs, Hkv, D]
    block_tables: np.ndarray        # int32 [B, MB]; unused entries hold table_pad
    context_lens: np.ndarray        # int32 [B]
    partition_size: int = 0         # 0: library's choice
    # new tokens written before attention (kv_cache_write)
    k_new: np.ndarray | None = None         # [N, Hkv, D]
    v_new: np.ndarray | None = None
    slot_mapping: np.ndarray | None = None  # int64 [N]
    # copy-on-write pairs applied before the writes (kv_copy_blocks)
    copy_pairs: np.ndarray | None = None    # int64 [P, 2]
    # chunked prefill: query rows of every sequence's chunk (the chunk's keys and values
    # are the last n cached tokens, already in the pool)
    chunk_q: np.ndarray | None = None       # [T, Hq, D]
    query_start: np.ndarray | None = None   # int32 [B + 1]
    info: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    def kv_bytes(self) -> int:
        """Live-token K+V bytes, each sequence's tokens counted once."""
        return int(self.context_lens.astype(np.int64).sum()) * 2 * self.num_kv_heads * \
            self.head_dim * self.elem_bytes


def _blocks_for(L: int, bs: int) -> int:
    return (int(L) + bs - 1) // bs if L > 0 else 0


def allocate(context_lens, block_size: int, perm: np.ndarray, max_blocks_per_seq: int,
             table_pad: int = -1) -> np.ndarray:
    """Give each sequence the next blocks of the shuffled pool ``perm``, in order."""
    B = len(context_lens)
    bt = np.full((B, max_blocks_per_seq), table_pad, dtype=np.int32)
    nxt = 0
    for s, L in enumerate(context_lens):
        nb = _blocks_for(L, block_size)
        if nb > max_blocks_per_seq:
            raise ValueError("context longer than the block table allows")
        bt[s, :nb] = perm[nxt:nxt + nb]
        nxt += nb
    if nxt > len(perm):
        raise ValueError("pool too small")
    return bt


def live_slot_mask(w: Workload) -> np.ndarray:
    """bool [NB, bs]: True where the allocation put a live token."""
    bs = w.block_size
    mask = np.zeros((w.num_blocks, bs), dtype=bool)
    for s in range(w.num_seqs):
        L = int(w.context_lens[s])
        nb = _blocks_for(L, bs)
        for j in range(nb):
            used = bs if j < nb - 1 else L - (nb - 1) * bs
            mask[w.block_tables[s, j], :used] = True
    return mask


def poison_unused(w: Workload) -> None:
    """Fill every cache slot that holds no live token with NaN, in place."""
    dead = ~live_slot_mask(w)
    for c in (w.k_cache, w.v_cache):
        if w.dtype == "f32":
            c[dead] = np.nan
        else:
            c[dead] = _POISON_BITS[w.dtype]


def make_workload(name: str, *, seed: int, dtype: str, context_lens, num_q_heads: int,
                  num_kv_heads: int, head_dim: int, block_size: int, scale: float | None = None,
                  pool_slack: float = 0.10, num_blocks: int | None = None, shuffle: bool = True,
                  max_blocks_per_seq: int | None = None, table_pad: int = -1,
                  partition_size: int = 0, key_outlier_frac: float = 0.0,
                  key_outlier_scale: float = 8.0) -> Workload:
    """A decode batch with the given context lengths over a shuffled physical pool."""
    ss = np.random.SeedSequence(seed)
    s_q, s_k, s_v, s_perm, s_mask = ss.spawn(5)
    lens = np.asarray(context_lens, dtype=np.int32)
    B = len(lens)
    bs = block_size
    need = int(sum(_blocks_for(L, bs) for L in lens))
    NB = num_blocks if num_blocks is not None else max(1, math.ceil((1.0 + pool_slack) * need))
    if NB < need:
        raise ValueError("num_blocks below what the context lengths need")
    MB = max_blocks_per_seq if max_blocks_per_seq is not None else \
        max(1, max(_blocks_for(L, bs) for L in lens) if B else 1)
    perm = np.random.Generator(np.random.PCG64(s_perm)).permutation(NB).astype(np.int32) \
        if shuffle else np.arange(NB, dtype=np.int32)
    bt = allocate(lens, bs, perm, MB, table_pad)
    row_scale = None
    if key_outlier_frac > 0:
        g = np.random.Generator(np.random.PCG64(s_mask))
        hit = g.random((NB, bs, num_kv_heads)) < key_outlier_frac
        row_scale = np.where(hit, np.float32(key_outlier_scale), np.float32(1.0))
    q = normal_storage(s_q, (B, num_q_heads, head_dim), dtype)
    k = normal_storage(s_k, (NB, bs, num_kv_heads, head_dim), dtype, row_scale=row_scale)
    v = normal_storage(s_v, (NB, bs, num_kv_heads, head_dim), dtype)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return Workload(name=name, dtype=dtype, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                    head_dim=head_dim, block_size=bs, scale=float(scale), q=q, k_cache=k,
                    v_cache=v, block_tables=bt, context_lens=lens, partition_size=partition_size,
                    info={"seed": seed, "pool_blocks_needed": need})


def add_new_tokens(w: Workload, seed: int) -> None:
    """One new token per sequence, written before attention at position L - 1.

    The slot is the one the allocation gave position L - 1: the block holding the
    sequence's last token and the offset of that token inside it.  ``context_lens``
    already counts the new token.
    """
    ss = np.random.SeedSequence([seed, 1])
    s_k, s_v = ss.spawn(2)
    B, Hkv, D, bs = w.num_seqs, w.num_kv_heads, w.head_dim, w.block_size
    slots = np.full(B, -1, dtype=np.int64)
    for s in range(B):
        L = int(w.context_lens[s])
        if L == 0:
            continue
        # the allocator's cursor: the last slot it filled in the sequence's last block
        nb = _blocks_for(L, bs)
        last_block = int(w.block_tables[s, nb - 1])
        used_in_last = L - (nb - 1) * bs
        slots[s] = last_block * bs + (used_in_last - 1)
    w.k_new = normal_storage(s_k, (B, Hkv, D), w.dtype)
    w.v_new = normal_storage(s_v, (B, Hkv, D), w.dtype)
    w.slot_mapping = slots


def make_prefill_workload(name: str, *, seed: int, dtype: str, prior_lens, chunk_lens,
                          num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                          **kw) -> Workload:
    """Chunks of ``chunk_lens[s]`` query tokens after ``prior_lens[s]`` cached tokens.

    The pool holds ``prior + chunk`` tokens per sequence (the chunk's own keys and values
    included, as after its slot writes); ``chunk_q`` holds the chunk's query rows, packed
    sequence after sequence, and ``query_start`` their offsets.
    """
    prior = np.asarray(prior_lens, dtype=np.int64)
    chunk = np.asarray(chunk_lens, dtype=np.int64)
    if prior.shape != chunk.shape or (prior < 0).any() or (chunk < 0).any():
        raise ValueError("prior_lens and chunk_lens must be non-negative and of equal length")
    w = make_workload(name, seed=seed, dtype=dtype, context_lens=(prior + chunk).astype(np.int32),
                      num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                      block_size=block_size, **kw)
    qs = np.zeros(len(chunk) + 1, dtype=np.int32)
    qs[1:] = np.cumsum(chunk)
    s_q = np.random.SeedSequence([seed, 11])
    w.chunk_q = normal_storage(s_q, (int(qs[-1]), num_q_heads, head_dim), dtype)
    w.query_start = qs
    return w


# the chunked-prefill batch: 16 sequences of the 70B-like GQA shape, each with a 512-token
# chunk after a prior context uniform in [0, 3584] tokens
PREFILL_RECIPE = ("chunked prefill bf16: 16 sequences, a 512-token chunk each after a prior "
                  "context uniform in [0, 3584] tokens, 64 q heads over 8 KV heads, head_dim 128, "
                  "block_size 16, shuffled pool sized to need + 10%, q/K/V ~ N(0,1)")


def prefill_workload(*, seed: int = BASE_SEED + 6, num_seqs: int = 16, chunk: int = 512,
                     max_prior: int = 3584, head_dim: int = 128) -> Workload:
    """The chunked-prefill batch (seeded); ``head_dim`` 64 gives the same batch with
    64-wide heads."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 7])))
    prior = rng.integers(0, max_prior, size=num_seqs, endpoint=True)
    name = "chunked-prefill-70b-gqa8-c512" + ("" if head_dim == 128 else f"-d{head_dim}")
    return make_prefill_workload(name, seed=seed, dtype="bf16",
                                 prior_lens=prior, chunk_lens=[chunk] * num_seqs, num_q_heads=64,
                                 num_kv_heads=8, head_dim=head_dim, block_size=16,
                                 max_blocks_per_seq=(max_prior + chunk + 15) // 16)


def grouped_prefix_workload(*, seed: int = BASE_SEED + 7, groups: int = 64, members: int = 8,
                            prefix_tokens: int = 4096, suffix_range=(1, 256), num_q_heads: int = 32,
                            num_kv_heads: int = 8, head_dim: int = 128, block_size: int = 16,
                            dtype: str = "bf16") -> Workload:
    """Groups of sequences forked from one prompt each (parallel sampling, beam search).

    Group g's members are consecutive sequences whose first ``prefix_tokens`` (whole
    blocks) map the group's own physical prefix blocks; each member then owns a suffix of
    U[suffix_range] tokens in private blocks.  ``info`` holds ``group_start`` and
    ``prefix_lens`` (the shared-prefix description of the batch).
    """
    if prefix_tokens % block_size:
        raise ValueError("prefix_tokens must be whole blocks")
    ss = np.random.SeedSequence(seed)
    s_q, s_k, s_v, s_perm, s_len = ss.spawn(5)
    bs = block_size
    B = groups * members
    g = np.random.Generator(np.random.PCG64(s_len))
    suffix = g.integers(suffix_range[0], suffix_range[1], size=B, endpoint=True)
    lens = (prefix_tokens + suffix).astype(np.int32)
    pre_blocks = prefix_tokens // bs
    own = [_blocks_for(int(x), bs) for x in suffix]
    need = groups * pre_blocks + int(sum(own))
    NB = math.ceil(1.1 * need)
    perm = np.random.Generator(np.random.PCG64(s_perm)).permutation(NB).astype(np.int32)
    MB = pre_blocks + _blocks_for(suffix_range[1], bs)
    bt = np.full((B, MB), -1, dtype=np.int32)
    nxt = 0
    for gi in range(groups):
        ids = perm[nxt:nxt + pre_blocks]
        nxt += pre_blocks
        for m in range(members):
            s = gi * members + m
            bt[s, :pre_blocks] = ids
            bt[s, pre_blocks:pre_blocks + own[s]] = perm[nxt:nxt + own[s]]
            nxt += own[s]
    q = normal_storage(s_q, (B, num_q_heads, head_dim), dtype)
    k = normal_storage(s_k, (NB, bs, num_kv_heads, head_dim), dtype)
    v = normal_storage(s_v, (NB, bs, num_kv_heads, head_dim), dtype)
    return Workload(name=f"grouped-prefix-{groups}x{members}-p{prefix_tokens}-{dtype}", dtype=dtype,
                    num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                    block_size=bs, scale=1.0 / math.sqrt(head_dim), q=q, k_cache=k, v_cache=v,
                    block_tables=bt, context_lens=lens,
                    info={"seed": seed, "group_start": np.arange(0, B + 1, members, dtype=np.int32),
                          "prefix_lens": np.full(groups, prefix_tokens, dtype=np.int32),
                          "shared_prefix_tokens": prefix_tokens, "pool_blocks_needed": need})


GROUPED_PREFIX_RECIPE = ("grouped shared prefixes bf16: 64 groups x 8 sequences (parallel "
                         "sampling), each group sharing a 4096-token prompt in 256 physical "
                         "blocks, private suffixes uniform in [1,256] tokens, 32 q heads over 8 KV "
                         "heads, head_dim 128, block_size 16, shuffled pool sized to need + 10%")


# ---------------------------------------------------------------------------------------
# the five decode batches
# ---------------------------------------------------------------------------------------

CONFIGS = {
    1: "tiny fp32 check: 4 seqs, context_lens {1,17,33,100}, 4 q heads = 4 KV heads, head_dim 64, "
       "block_size 16, 64-block pool, block tables from a seeded permutation, scale 1/8",
    2: "13B-like MHA decode bf16: batch 64, 40 q heads = 40 KV heads, head_dim 128, block_size 16, "
       "context_lens uniform in [1,2048], shuffled pool sized to need + 10%",
    3: "70B-like GQA decode bf16: batch 128, 64 q heads over 8 KV heads, head_dim 128, block_size 16, "
       "context_lens log-uniform in [128,8192], shuffled pool, plus a slot write of one new token "
       "per sequence",
    4: "shared-prefix copy-on-write bf16: 256 seqs sharing a 1008-token prefix in 32 physical blocks "
       "(block_size 32), unique suffixes uniform in [16,512] tokens, 32 q heads over 8 KV heads, "
       "head_dim 128; the last shared (partial) block is copied to a private block before the "
       "suffix is written",
    5: "long-context split-context bf16: batch 32, every context 32768 tokens, 32 q heads over 8 KV "
       "heads, head_dim 128, block_size 16, shuffled pool, 1% of key rows scaled x8, partitions of "
       "512 tokens",
}


def config_workload(cfg: int, *, with_writes: bool = True) -> Workload:
    """Build decode batch ``cfg`` (1..5) with seed ``315 + cfg``."""
    seed = BASE_SEED + cfg
    lens_rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 7])))
    if cfg == 1:
        w = make_workload("tiny-fp32-mha", seed=seed, dtype="f32", context_lens=[1, 17, 33, 100],
                          num_q_heads=4, num_kv_heads=4, head_dim=64, block_size=16,
                          scale=1.0 / 8.0, num_blocks=64)
        return w
    if cfg == 2:
        lens = lens_rng.integers(1, 2048, size=64, endpoint=True)
        return make_workload("13b-mha-b64-bf16", seed=seed, dtype="bf16", context_lens=lens,
                             num_q_heads=40, num_kv_heads=40, head_dim=128, block_size=16,
                             max_blocks_per_seq=2048 // 16)
    if cfg == 3:
        lens = np.rint(np.exp(lens_rng.uniform(math.log(128), math.log(8192), size=128)))
        lens = np.clip(lens, 128, 8192).astype(np.int32)
        w = make_workload("70b-gqa8-b128-bf16", seed=seed, dtype="bf16", context_lens=lens,
                          num_q_heads=64, num_kv_heads=8, head_dim=128, block_size=16,
                          max_blocks_per_seq=8192 // 16)
        if with_writes:
            add_new_tokens(w, seed)
        return w
    if cfg == 4:
        return shared_prefix_workload(seed=seed, with_writes=with_writes)
    if cfg == 5:
        return make_workload("longctx-32k-gqa4-b32-bf16", seed=seed, dtype="bf16",
                             context_lens=[32768] * 32, num_q_heads=32, num_kv_heads=8,
                             head_dim=128, block_size=16, max_blocks_per_seq=32768 // 16,
                             partition_size=512, key_outlier_frac=0.01)
    raise ValueError(f"unknown config {cfg}")


def shared_prefix_workload(*, seed: int, num_seqs: int = 256, prefix_tokens: int = 1008,
                           suffix_range=(16, 512), num_q_heads: int = 32, num_kv_heads: int = 8,
                           head_dim: int = 128, block_size: int = 32,
                           with_writes: bool = True) -> Workload:
    """Sequences sharing one refcounted prefix, diverging by copy-on-write.

    All sequences' tables start with the same physical prefix blocks.  The prefix
    ends inside its last block, so before a sequence's first suffix token is written
    that shared partial block is copied to a private block (``copy_pairs``), the
    sequence's table points at the copy, and the suffix tokens are written from the
    copy's first free slot onward (``slot_mapping`` over ``k_new`` / ``v_new``).
    Before the copies and writes the private blocks hold unrelated data.
    """
    ss = np.random.SeedSequence(seed)
    s_q, s_k, s_v, s_perm, s_len, s_new_k, s_new_v = ss.spawn(7)
    bs = block_size
    shared = _blocks_for(prefix_tokens, bs)
    prefix_partial = prefix_tokens % bs != 0
    g = np.random.Generator(np.random.PCG64(s_len))
    suffix = g.integers(suffix_range[0], suffix_range[1], size=num_seqs, endpoint=True)
    lens = (prefix_tokens + suffix).astype(np.int32)
    private = [_blocks_for(L, bs) - shared + (1 if prefix_partial else 0) for L in lens]
    need = shared + int(sum(private))
    NB = math.ceil(1.1 * need)
    perm = np.random.Generator(np.random.PCG64(s_perm)).permutation(NB).astype(np.int32)
    MB = _blocks_for(prefix_tokens + suffix_range[1], bs)
    bt = np.full((num_seqs, MB), -1, dtype=np.int32)
    shared_ids = perm[:shared]
    nxt = shared
    pairs = []
    slots = []
    for s, L in enumerate(lens):
        nb = _blocks_for(L, bs)
        bt[s, :shared] = shared_ids
        own = perm[nxt:nxt + private[s]]
        nxt += private[s]
        if prefix_partial:
            bt[s, shared - 1] = own[0]
            pairs.append((int(shared_ids[-1]), int(own[0])))
            bt[s, shared:nb] = own[1:]
        else:
            bt[s, shared:nb] = own
        # the allocator fills the sequence's own blocks left to right, starting at the
        # copy's first free slot
        remaining = int(L) - prefix_tokens
        first_free = prefix_tokens % bs
        for i, blk in enumerate(own):
            for off in range(first_free if i == 0 else 0, bs):
                if remaining == 0:
                    break
                slots.append(int(blk) * bs + off)
                remaining -= 1
    B = num_seqs
    q = normal_storage(s_q, (B, num_q_heads, head_dim), "bf16")
    k = normal_storage(s_k, (NB, bs, num_kv_heads, head_dim), "bf16")
    v = normal_storage(s_v, (NB, bs, num_kv_heads, head_dim), "bf16")
    w = Workload(name="shared-prefix-cow-b256-bf16", dtype="bf16", num_q_heads=num_q_heads,
                 num_kv_heads=num_kv_heads, head_dim=head_dim, block_size=bs,
                 scale=1.0 / math.sqrt(head_dim), q=q, k_cache=k, v_cache=v, block_tables=bt,
                 context_lens=lens,
                 info={"seed": seed, "prefix_tokens": prefix_tokens, "shared_blocks": shared,
                       "shared_ids": shared_ids.copy(), "pool_blocks_needed": need,
                       # tokens in the blocks every sequence still maps after its copy
                       "shared_prefix_tokens": (shared - (1 if prefix_partial else 0)) * bs})
    if with_writes:
        n = len(slots)
        w.slot_mapping = np.asarray(slots, dtype=np.int64)
        w.k_new = normal_storage(s_new_k, (n, num_kv_heads, head_dim), "bf16")
        w.v_new = normal_storage(s_new_v, (n, num_kv_heads, head_dim), "bf16")
        w.copy_pairs = np.asarray(pairs, dtype=np.int64).reshape(-1, 2)
    return w


def storage_to_torch(a: np.ndarray, dtype: str, device):
    """A torch tensor on ``device`` holding the elements stored in ``a``."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype != "f32":
        t = t.view(torch.int16).view({"bf16": torch.bfloat16, "f16": torch.float16}[dtype])
    return t.to(device)


def e4m3_codes(values: np.ndarray, scale: float) -> np.ndarray:
    """E4M3 codes (uint8) of values / scale, by torch's float8_e4m3fn conversion (nearest,
    ties to even) after clamping to the format's +-448."""
    import torch

    x = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float32)) / np.float32(scale)
    x = x.clamp(-448.0, 448.0)
    return x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def fp8_kv(w: Workload, k_scale: float, v_scale: float):
    """The workload's K and V pools re-encoded as E4M3 codes with per-tensor scales."""
    k = storage_to_f64(w.k_cache, w.dtype).astype(np.float32)
    v = storage_to_f64(w.v_cache, w.dtype).astype(np.float32)
    return e4m3_codes(k, k_scale), e4m3_codes(v, v_scale)


def to_torch(w: Workload, device):
    """Device copies of a workload's arrays, as a dict of torch tensors."""
    import torch

    def elems(a):
        return storage_to_torch(a, w.dtype, device)

    out = {
        "q": elems(w.q),
        "k_cache": elems(w.k_cache),
        "v_cache": elems(w.v_cache),
        "block_tables": torch.from_numpy(np.ascontiguousarray(w.block_tables)).to(device),
        "context_lens": torch.from_numpy(np.ascontiguousarray(w.context_lens)).to(device),
    }
    if w.k_new is not None:
        out["k_new"] = elems(w.k_new)
        out["v_new"] = elems(w.v_new)
        out["slot_mapping"] = torch.from_numpy(np.ascontiguousarray(w.slot_mapping)).to(device)
    if w.copy_pairs is not None:
        out["copy_pairs"] = torch.from_numpy(np.ascontiguousarray(w.copy_pairs)).to(device)
    if w.chunk_q is not None:
        out["chunk_q"] = elems(w.chunk_q)
        out["query_start"] = torch.from_numpy(np.ascontiguousarray(w.query_start)).to(device)
    return out


def tensor_to_storage(t) -> np.ndarray:
    """Host numpy storage (uint16 bits for 16-bit floats) of a torch tensor."""
    import torch

    t = t.detach().contiguous().cpu()
    if t.dtype in (torch.bfloat16, torch.float16):
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()
