"""Parity of the CUDA path (through the C ABI) with the fp64 oracle, on the GPU.

Acceptance: slot writes and block copies bit-exact; decode outputs within max abs error
1e-5 for fp32, and within |gpu - oracle| <= 2e-2 + 1e-2 |oracle| for bf16 / fp16.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

ATOL_F32 = 1e-5
ATOL_16, RTOL_16 = 2e-2, 1e-2


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_315_gb300 as m

    m.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    m.pkv_device_error()  # clear bits left by earlier modules
    return m


def assert_close(got: np.ndarray, ref: np.ndarray, dtype: str, what: str = ""):
    got = got.astype(np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    if dtype == "f32":
        assert err.max() <= ATOL_F32, f"{what}: max abs err {err.max():.3e}"
    else:
        bad = err > ATOL_16 + RTOL_16 * np.abs(ref)
        assert not bad.any(), f"{what}: {bad.sum()} elements out of tolerance, max err {err.max():.3e}"


def gpu_decode(pkv, w, t, partition_size=None, block_tables=None, context_lens=None):
    out = torch.empty_like(t["q"])
    pkv.paged_attn_decode(out, t["q"], t["k_cache"], t["v_cache"],
                          t["block_tables"] if block_tables is None else block_tables,
                          t["context_lens"] if context_lens is None else context_lens, w.scale,
                          partition_size=w.partition_size if partition_size is None else partition_size)
    return out


def host_out(out: torch.Tensor) -> np.ndarray:
    return out.float().cpu().numpy()


def oracle_decode(w, k=None, v=None, bt=None, seqs=None):
    k = w.k_cache if k is None else k
    v = w.v_cache if v is None else v
    bt = w.block_tables if bt is None else bt
    q, lens = w.q, w.context_lens
    if seqs is not None:
        q, bt, lens = q[seqs], bt[seqs], lens[seqs]
    return oracle.paged_decode(q, k, v, bt, lens, w.scale, w.dtype)


# ------------------------------------------------------------------------------------------
# slot writes and block copies: bit-exact
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,Hkv,D", [("bf16", 8, 128), ("f32", 4, 64), ("f16", 3, 32),
                                         ("bf16", 1, 40)])
def test_kv_cache_write_bit_exact(pkv, dtype, Hkv, D):
    w = synth.make_workload("w", seed=3, dtype=dtype, context_lens=[50, 100, 7], num_q_heads=Hkv,
                            num_kv_heads=Hkv, head_dim=D, block_size=16, pool_slack=0.5)
    rng = np.random.default_rng(4)
    NB, bs = w.num_blocks, w.block_size
    n = 37
    slots = rng.choice(NB * bs, size=n, replace=False).astype(np.int64)
    slots[[3, 11]] = -1
    k_new = synth.to_storage(rng.standard_normal((n, Hkv, D)), dtype)
    v_new = synth.to_storage(rng.standard_normal((n, Hkv, D)), dtype)
    t = synth.to_torch(w, "cuda")
    pkv.kv_cache_write(synth.storage_to_torch(k_new, dtype, "cuda"),
                       synth.storage_to_torch(v_new, dtype, "cuda"), t["k_cache"], t["v_cache"],
                       torch.from_numpy(slots).cuda())
    assert pkv.pkv_device_error() == 0
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    assert oracle.kv_cache_write(k_new, v_new, kc, vc, slots) == 0
    assert np.array_equal(synth.tensor_to_storage(t["k_cache"]), kc)
    assert np.array_equal(synth.tensor_to_storage(t["v_cache"]), vc)


def test_kv_cache_write_flags_out_of_range_slot(pkv):
    kc = torch.zeros(4, 16, 2, 64, dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    k = torch.ones(2, 2, 64, dtype=torch.bfloat16, device="cuda")
    pkv.kv_cache_write(k, k, kc, vc, torch.tensor([5, 4 * 16], dtype=torch.int64, device="cuda"))
    assert pkv.pkv_device_error() == pkv.PKV_DERR_SLOT
    assert kc.view(64, 2, 64)[5].eq(1).all() and kc.view(64, 2, 64)[6:].eq(0).all()
    assert pkv.pkv_device_error() == 0


@pytest.mark.parametrize("dtype,bs,Hkv,D", [("bf16", 32, 8, 128), ("f32", 16, 2, 64),
                                            ("f16", 8, 1, 24)])
def test_kv_copy_blocks_bit_exact(pkv, dtype, bs, Hkv, D):
    w = synth.make_workload("c", seed=5, dtype=dtype, context_lens=[bs * 20], num_q_heads=Hkv,
                            num_kv_heads=Hkv, head_dim=D, block_size=bs, num_blocks=40)
    pairs = np.array([[0, 30], [3, 31], [7, 7], [12, 39], [1, 25]], np.int64)
    t = synth.to_torch(w, "cuda")
    tp = torch.from_numpy(pairs).cuda()
    pkv.kv_copy_blocks(t["k_cache"], tp)
    pkv.kv_copy_blocks(t["v_cache"], tp)
    assert pkv.pkv_device_error() == 0
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    oracle.copy_blocks(kc, pairs)
    oracle.copy_blocks(vc, pairs)
    assert np.array_equal(synth.tensor_to_storage(t["k_cache"]), kc)
    assert np.array_equal(synth.tensor_to_storage(t["v_cache"]), vc)


def test_kv_copy_blocks_flags_bad_pair(pkv):
    c = torch.arange(4 * 16 * 64, dtype=torch.float32, device="cuda").view(4, 16, 1, 64)
    before = c.clone()
    pkv.kv_copy_blocks(c, torch.tensor([[0, 4], [1, 2]], dtype=torch.int64, device="cuda"))
    assert pkv.pkv_device_error() == pkv.PKV_DERR_PAIR
    assert torch.equal(c[2], before[1]) and torch.equal(c[[0, 1, 3]], before[[0, 1, 3]])


# ------------------------------------------------------------------------------------------
# decode: small shapes, every path, against the oracle on all outputs
# ------------------------------------------------------------------------------------------

SHAPES = [
    # dtype, Hq, Hkv, D, bs, partition
    ("bf16", 4, 4, 128, 16, 0),
    ("bf16", 8, 1, 128, 16, 64),
    ("bf16", 16, 2, 128, 32, 128),
    ("bf16", 64, 8, 128, 16, 256),
    ("bf16", 40, 2, 128, 16, 512),   # 20 heads per KV head: two head chunks
    ("bf16", 6, 3, 64, 64, 128),
    ("f16", 32, 8, 128, 16, 96),
    ("f16", 2, 2, 64, 32, 0),
    ("f32", 4, 4, 64, 16, 0),
    ("f32", 8, 2, 128, 8, 64),
    ("f32", 12, 1, 32, 16, 48),
    ("bf16", 4, 2, 256, 16, 128),    # CUDA-core path for 16-bit types
    ("bf16", 16, 4, 128, 8, 64),     # block_size 8: CUDA-core path
    ("bf16", 32, 8, 128, 64, 256),   # 64-token blocks staged as four 16-token slices
    ("f16", 12, 4, 128, 32, 0),      # 32-token blocks as two slices, 3 heads per KV head
]


@pytest.mark.parametrize("dtype,Hq,Hkv,D,bs,part", SHAPES)
def test_decode_matches_oracle(pkv, dtype, Hq, Hkv, D, bs, part):
    lens = [1, bs - 1, bs, bs + 1, 5 * bs + 3, 333, 1000, 0, 2 * bs]
    w = synth.make_workload("d", seed=7 + Hq + D + bs, dtype=dtype, context_lens=lens,
                            num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=bs,
                            partition_size=part, key_outlier_frac=0.02)
    t = synth.to_torch(w, "cuda")
    out = gpu_decode(pkv, w, t)
    assert pkv.pkv_device_error() == 0
    ref = oracle_decode(w)
    assert_close(host_out(out), ref, dtype, f"{dtype} Hq{Hq} Hkv{Hkv} D{D} bs{bs} P{part}")
    assert (host_out(out)[7] == 0).all()  # empty context


# Partitions of at most 512 tokens with at most 4 query heads per KV head: one CTA streams
# two consecutive partitions.  With 16-token blocks (bf16, f16) it folds them into one
# partial, or writes the output when they cover the whole context; otherwise it writes a
# partial for each.  Lengths end on, before and after partition edges so that CTAs see one
# or two live partitions, groups that cover the whole context, odd partition counts and
# ragged tails.
PAIRED_LENS = [1, 511, 512, 513, 1024, 1025, 1543, 2048, 2660, 0, 3000, 257]


@pytest.mark.parametrize("dtype,Hq,Hkv,bs,part", [("bf16", 4, 4, 16, 512), ("bf16", 16, 8, 32, 512),
                                                   ("f16", 32, 8, 16, 256), ("bf16", 8, 2, 64, 512),
                                                   ("bf16", 12, 4, 16, 384)])
def test_two_partitions_per_cta_match_oracle(pkv, dtype, Hq, Hkv, bs, part):
    w = synth.make_workload("pp", seed=50 + Hq + bs + part, dtype=dtype, context_lens=PAIRED_LENS,
                            num_q_heads=Hq, num_kv_heads=Hkv, head_dim=128, block_size=bs,
                            partition_size=part, key_outlier_frac=0.02)
    t = synth.to_torch(w, "cuda")
    out = gpu_decode(pkv, w, t)
    assert pkv.pkv_device_error() == 0
    assert_close(host_out(out), oracle_decode(w), dtype, f"{dtype} Hq{Hq} Hkv{Hkv} bs{bs} P{part}")
    assert (host_out(out)[9] == 0).all()


@pytest.mark.parametrize("bs,part", [(16, 512), (32, 256), (64, 512)])
def test_fp8_two_partitions_per_cta_match_oracle(pkv, bs, part):
    w = synth.make_workload("pp8", seed=70 + bs + part, dtype="bf16", context_lens=PAIRED_LENS,
                            num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=bs,
                            partition_size=part, key_outlier_frac=0.02)
    ks, vs = 0.0625, 0.03
    k8, v8, t = _fp8_setup(w, ks, vs)
    out = torch.empty_like(t["q"])
    pkv.paged_attn_decode_fp8(out, t["q"], t["k8"], t["v8"], t["block_tables"], t["context_lens"],
                              w.scale, ks, vs, partition_size=part)
    assert pkv.pkv_device_error() == 0
    ref = oracle.paged_decode_fp8kv(w.q, k8, v8, w.block_tables, w.context_lens, w.scale, ks, vs,
                                    "bf16")
    assert_close(host_out(out), ref, "bf16", f"fp8 bs{bs} P{part}")
    assert (host_out(out)[9] == 0).all()


def test_batch_beyond_the_ordering_limit_matches_oracle(pkv):
    # 2100 sequences x 32 partitions of 64 tokens = 67200 items: more than the one-CTA work
    # ordering sorts, so the launch leaves the prep kernel out and keeps natural order
    # (8 query heads per KV head: one partition per CTA)
    rng = np.random.default_rng(5)
    lens = rng.integers(1, 256, size=2100, endpoint=True)
    lens[::97] = 2048
    lens[1::89] = 1000
    w = synth.make_workload("many", seed=5, dtype="bf16", context_lens=lens, num_q_heads=8,
                            num_kv_heads=1, head_dim=64, block_size=16, max_blocks_per_seq=128,
                            partition_size=64)
    t = synth.to_torch(w, "cuda")
    out = gpu_decode(pkv, w, t)
    assert pkv.pkv_device_error() == 0
    seqs = np.r_[0:40, 970:1000, 2060:2100]
    assert_close(host_out(out)[seqs], oracle_decode(w, seqs=seqs), "bf16", "67200 items")


def test_config1_tiny_fp32(pkv):
    w = synth.config_workload(1)
    t = synth.to_torch(w, "cuda")
    out = gpu_decode(pkv, w, t)
    assert pkv.pkv_device_error() == 0
    assert_close(host_out(out), oracle_decode(w), "f32", "config 1")


# ------------------------------------------------------------------------------------------
# decode: invariants
# ------------------------------------------------------------------------------------------

def test_physical_block_permutation_gives_identical_bits(pkv):
    w = synth.make_workload("p", seed=9, dtype="bf16", context_lens=[17, 500, 1234, 64],
                            num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                            pool_slack=0.4, partition_size=256)
    t = synth.to_torch(w, "cuda")
    base = gpu_decode(pkv, w, t)
    perm = torch.from_numpy(np.random.default_rng(1).permutation(w.num_blocks)).cuda()
    k2 = torch.empty_like(t["k_cache"])
    v2 = torch.empty_like(t["v_cache"])
    k2[perm] = t["k_cache"]
    v2[perm] = t["v_cache"]
    bt = t["block_tables"]
    bt2 = torch.where(bt >= 0, perm[bt.clamp(min=0).long()].int(), bt)
    out = torch.empty_like(base)
    pkv.paged_attn_decode(out, t["q"], k2, v2, bt2, t["context_lens"], w.scale, partition_size=256)
    assert torch.equal(out, base)


@pytest.mark.parametrize("dtype,D,bs", [("bf16", 128, 16), ("bf16", 64, 32), ("f32", 64, 16),
                                        ("bf16", 128, 32), ("bf16", 128, 64)])
def test_poisoned_dead_slots_and_table_tail_are_never_read(pkv, dtype, D, bs):
    w = synth.make_workload("n", seed=10, dtype=dtype, context_lens=[1, bs - 3, bs + 1, 301],
                            num_q_heads=8, num_kv_heads=2, head_dim=D, block_size=bs,
                            pool_slack=0.5, partition_size=4 * bs, table_pad=2 ** 30)
    t = synth.to_torch(w, "cuda")
    clean = gpu_decode(pkv, w, t)
    synth.poison_unused(w)
    t2 = synth.to_torch(w, "cuda")
    out = gpu_decode(pkv, w, t2)
    assert pkv.pkv_device_error() == 0
    assert torch.isfinite(out.float()).all()
    assert torch.equal(out, clean)


def test_split_context_matches_single_pass(pkv):
    w = synth.make_workload("s", seed=11, dtype="bf16", context_lens=[4000, 2500, 8000, 77],
                            num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                            key_outlier_frac=0.01)
    t = synth.to_torch(w, "cuda")
    ref = oracle_decode(w)
    outs = {}
    for part in (128, 512, 2048, 8192):
        outs[part] = host_out(gpu_decode(pkv, w, t, partition_size=part))
        assert_close(outs[part], ref, "bf16", f"partition {part}")
    # one partition covers every context: no workspace traffic at all
    assert np.abs(outs[8192] - outs[128]).max() < 2e-2


def test_repeated_calls_reuse_the_workspace(pkv):
    w = synth.make_workload("r", seed=12, dtype="bf16", context_lens=[3000, 10, 1500],
                            num_q_heads=16, num_kv_heads=4, head_dim=128, block_size=16,
                            partition_size=256)
    t = synth.to_torch(w, "cuda")
    first = gpu_decode(pkv, w, t)
    for _ in range(3):
        assert torch.equal(gpu_decode(pkv, w, t), first)


def test_one_workspace_serves_changing_shapes(pkv):
    """A serving loop's batch changes every step; one uninitialised workspace buffer
    (filled with garbage between calls) must serve all of them."""
    ws = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    for i, (B, Hq, Hkv, lens) in enumerate([(3, 8, 2, [900, 40, 2000]), (5, 16, 4, [3000] * 5),
                                            (2, 8, 2, [700, 1300])]):
        ws.random_(0, 256)
        w = synth.make_workload("ws", seed=40 + i, dtype="bf16", context_lens=lens,
                                num_q_heads=Hq, num_kv_heads=Hkv, head_dim=128, block_size=16,
                                partition_size=256)
        t = synth.to_torch(w, "cuda")
        out = torch.empty_like(t["q"])
        pkv.paged_attn_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                              t["context_lens"], w.scale, partition_size=256, workspace=ws)
        assert_close(host_out(out), oracle_decode(w), "bf16", f"shape {i}")


@pytest.mark.parametrize("dtype,Hq,Hkv,D,bs,part", [
    ("bf16", 8, 8, 128, 16, 256),    # M = heads kernel, two partitions per CTA folded
    ("bf16", 32, 8, 128, 32, 256),   # heads in N, two partitions per CTA, one partial each
    ("f16", 64, 4, 64, 16, 512),     # 16-head chunks, head_dim 64
    ("f32", 8, 2, 256, 16, 256),     # CUDA-core path
])
def test_split_contexts_from_a_dirty_workspace(pkv, dtype, Hq, Hkv, D, bs, part):
    """Split contexts on every kernel family, with garbage in the workspace (work order and
    partials) before each call: two calls give the oracle's result and identical bits (the
    order in which CTAs finish does not change the merge)."""
    lens = [1, 255, 256, 257, 511, 512, 513, 1400, 2048, 0, 3100, 777]
    w = synth.make_workload("tm", seed=80 + D + bs, dtype=dtype, context_lens=lens,
                            num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=bs,
                            partition_size=part, key_outlier_frac=0.01)
    t = synth.to_torch(w, "cuda")
    need = pkv.paged_attn_decode_workspace_size(len(lens), Hq, Hkv, D, bs,
                                                w.block_tables.shape[1], part)
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        ws.random_(0, 256)
        out = torch.full_like(t["q"], float("nan"))
        pkv.paged_attn_decode(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                              t["context_lens"], w.scale, partition_size=part, workspace=ws)
        assert pkv.pkv_device_error() == 0
        outs.append(out)
    assert_close(host_out(outs[0]), oracle_decode(w), dtype, f"{dtype} Hq{Hq} D{D} bs{bs}")
    assert torch.equal(outs[0], outs[1])


def test_single_token_context_returns_v0_exactly(pkv):
    w = synth.make_workload("one", seed=13, dtype="bf16", context_lens=[1, 1, 1], num_q_heads=8,
                            num_kv_heads=2, head_dim=128, block_size=16)
    t = synth.to_torch(w, "cuda")
    out = gpu_decode(pkv, w, t)
    bt = t["block_tables"][:, 0].long()
    v0 = t["v_cache"][bt, 0]                         # [B, Hkv, D]
    assert torch.equal(out, v0.repeat_interleave(4, dim=1))


def test_uniform_keys_give_mean_of_values(pkv):
    w = synth.make_workload("u", seed=14, dtype="bf16", context_lens=[5, 100, 700], num_q_heads=8,
                            num_kv_heads=8, head_dim=128, block_size=16, shuffle=False,
                            partition_size=256)
    w.k_cache[...] = synth.to_storage(np.full(1, 0.5, np.float32), "bf16")[0]
    t = synth.to_torch(w, "cuda")
    out = host_out(gpu_decode(pkv, w, t))
    V = synth.storage_to_f64(w.v_cache, "bf16").reshape(-1, 8, 128)
    for s in range(3):
        start = int(w.block_tables[s, 0]) * 16
        mean = V[start:start + int(w.context_lens[s])].mean(axis=0)
        assert_close(out[s], mean, "bf16", f"uniform keys seq {s}")


def test_gqa_matches_replicated_mha(pkv):
    w = synth.make_workload("g", seed=15, dtype="bf16", context_lens=[33, 900, 2000],
                            num_q_heads=16, num_kv_heads=2, head_dim=128, block_size=16,
                            partition_size=512)
    t = synth.to_torch(w, "cuda")
    gqa = host_out(gpu_decode(pkv, w, t))
    k_rep = t["k_cache"].repeat_interleave(8, dim=2).contiguous()
    v_rep = t["v_cache"].repeat_interleave(8, dim=2).contiguous()
    mha = torch.empty_like(t["q"])
    pkv.paged_attn_decode(mha, t["q"], k_rep, v_rep, t["block_tables"], t["context_lens"], w.scale,
                          partition_size=512)
    assert np.abs(host_out(mha) - gqa).max() < 1e-2


# ------------------------------------------------------------------------------------------
# decode: device-side data errors are reported, not trapped
# ------------------------------------------------------------------------------------------

def test_bad_block_id_and_context_are_reported(pkv):
    w = synth.make_workload("e", seed=16, dtype="bf16", context_lens=[40, 40], num_q_heads=4,
                            num_kv_heads=4, head_dim=128, block_size=16)
    t = synth.to_torch(w, "cuda")
    bt = t["block_tables"].clone()
    bt[0, 1] = w.num_blocks + 5
    out = gpu_decode(pkv, w, t, block_tables=bt)
    assert pkv.pkv_device_error() & pkv.PKV_DERR_BLOCK_ID
    assert torch.isfinite(out.float()).all()
    lens = t["context_lens"].clone()
    lens[1] = w.max_blocks_per_seq * 16 + 1
    gpu_decode(pkv, w, t, context_lens=lens)
    assert pkv.pkv_device_error() & pkv.PKV_DERR_CONTEXT
    assert pkv.pkv_device_error() == 0


# ------------------------------------------------------------------------------------------
# the five decode batches at full size (outputs sampled where the oracle would be slow)
# ------------------------------------------------------------------------------------------

def _sample(w, n, seed):
    rng = np.random.default_rng(seed)
    if n >= w.num_seqs:
        return np.arange(w.num_seqs)
    # always include the longest and the shortest context
    pick = set(rng.choice(w.num_seqs, size=n - 2, replace=False).tolist())
    pick |= {int(np.argmax(w.context_lens)), int(np.argmin(w.context_lens))}
    return np.array(sorted(pick))


def test_config2_mha_13b_full(pkv):
    w = synth.config_workload(2)
    t = synth.to_torch(w, "cuda")
    out = gpu_decode(pkv, w, t)
    assert pkv.pkv_device_error() == 0
    assert_close(host_out(out), oracle_decode(w), "bf16", "config 2")


def test_config3_gqa_70b_with_slot_write(pkv):
    w = synth.config_workload(3)
    t = synth.to_torch(w, "cuda")
    pkv.kv_cache_write(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["slot_mapping"])
    out = gpu_decode(pkv, w, t)
    assert pkv.pkv_device_error() == 0
    k, v = w.k_cache.copy(), w.v_cache.copy()
    assert oracle.kv_cache_write(w.k_new, w.v_new, k, v, w.slot_mapping) == 0
    rows = w.slot_mapping
    kc = synth.tensor_to_storage(t["k_cache"]).reshape(-1, w.num_kv_heads, w.head_dim)
    assert np.array_equal(kc[rows], k.reshape(-1, w.num_kv_heads, w.head_dim)[rows])
    seqs = _sample(w, 24, 3)
    assert_close(host_out(out)[seqs], oracle_decode(w, k, v, seqs=seqs), "bf16", "config 3")


def test_config4_shared_prefix_copy_on_write(pkv):
    w = synth.config_workload(4)
    t = synth.to_torch(w, "cuda")
    shared_last = int(w.info["shared_ids"][-1])
    shared_before = t["k_cache"][shared_last].clone()
    pkv.kv_copy_blocks(t["k_cache"], t["copy_pairs"])
    pkv.kv_copy_blocks(t["v_cache"], t["copy_pairs"])
    pkv.kv_cache_write(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["slot_mapping"])
    out = gpu_decode(pkv, w, t)
    assert pkv.pkv_device_error() == 0
    k, v = w.k_cache.copy(), w.v_cache.copy()
    oracle.copy_blocks(k, w.copy_pairs)
    oracle.copy_blocks(v, w.copy_pairs)
    assert oracle.kv_cache_write(w.k_new, w.v_new, k, v, w.slot_mapping) == 0
    assert np.array_equal(synth.tensor_to_storage(t["k_cache"]), k)
    assert np.array_equal(synth.tensor_to_storage(t["v_cache"]), v)
    assert torch.equal(t["k_cache"][shared_last], shared_before)  # the shared block is untouched
    seqs = _sample(w, 24, 4)
    assert_close(host_out(out)[seqs], oracle_decode(w, k, v, seqs=seqs), "bf16", "config 4")


def test_config5_long_context_split(pkv):
    w = synth.config_workload(5)
    t = synth.to_torch(w, "cuda")
    out = gpu_decode(pkv, w, t)
    assert pkv.pkv_device_error() == 0
    seqs = _sample(w, 3, 5)
    assert_close(host_out(out)[seqs], oracle_decode(w, seqs=seqs), "bf16", "config 5")


# ------------------------------------------------------------------------------------------
# failure detection: a wait that runs out is reported, and the context stays usable
# ------------------------------------------------------------------------------------------

def test_bounded_wait_runs_out_and_reports(pkv):
    import time

    torch.cuda.synchronize()
    t0 = time.perf_counter()
    pkv.pkv_selftest_bounded_wait(20000, arrive=False)       # nothing ever arrives
    assert pkv.pkv_device_error() == pkv.PKV_DERR_TIMEOUT
    waited = time.perf_counter() - t0
    assert 0.015 < waited < 1.0
    pkv.pkv_selftest_bounded_wait(20000, arrive=True)        # completes at once
    assert pkv.pkv_device_error() == 0
    # the context is still usable: a decode right after gives the oracle's answer
    w = synth.make_workload("after", seed=77, dtype="bf16", context_lens=[40, 700],
                            num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16)
    t = synth.to_torch(w, "cuda")
    assert_close(host_out(gpu_decode(pkv, w, t)), oracle_decode(w), "bf16", "after timeout")


# ------------------------------------------------------------------------------------------
# swap out / swap in between the device pool and a pinned host pool
# ------------------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,bs,Hkv,D", [("bf16", 16, 8, 128), ("f32", 32, 2, 64),
                                            ("f16", 16, 1, 24)])
def test_swap_out_to_host_and_back_in_bit_exact(pkv, dtype, bs, Hkv, D):
    w = synth.make_workload("sw", seed=21, dtype=dtype, context_lens=[bs * 30, bs * 7 + 3],
                            num_q_heads=Hkv, num_kv_heads=Hkv, head_dim=D, block_size=bs,
                            pool_slack=1.0)
    t = synth.to_torch(w, "cuda")
    nb = -(-int(w.context_lens[1]) // bs)
    blocks = w.block_tables[1, :nb].astype(np.int64)
    host_shape = (12,) + tuple(t["k_cache"].shape[1:])
    hk = torch.zeros(host_shape, dtype=t["k_cache"].dtype).pin_memory()
    hv = torch.zeros_like(hk).pin_memory()
    out_pairs = np.stack([blocks, np.arange(nb) + 3], axis=1)
    tp = torch.from_numpy(out_pairs).cuda()
    pkv.kv_swap_blocks(hk, t["k_cache"], tp)                   # device -> host
    pkv.kv_swap_blocks(hv, t["v_cache"], tp)
    assert pkv.pkv_device_error() == 0
    hk_ref = np.zeros((12,) + w.k_cache.shape[1:], w.k_cache.dtype)
    hv_ref = np.zeros_like(hk_ref)
    oracle.swap_blocks(hk_ref, w.k_cache, out_pairs)
    oracle.swap_blocks(hv_ref, w.v_cache, out_pairs)
    assert np.array_equal(synth.tensor_to_storage(hk), hk_ref)
    assert np.array_equal(synth.tensor_to_storage(hv), hv_ref)
    # swap back in to fresh device blocks, pairs given in pinned host memory
    used = set(w.block_tables[w.block_tables >= 0].tolist())
    free = np.array([b for b in range(w.num_blocks) if b not in used][:nb], np.int64)
    in_pairs = np.stack([np.arange(nb) + 3, free], axis=1)
    tin = torch.from_numpy(in_pairs).pin_memory()
    pkv.kv_swap_blocks(t["k_cache"], hk, tin)                   # host -> device
    pkv.kv_swap_blocks(t["v_cache"], hv, tin)
    assert pkv.pkv_device_error() == 0
    k_ref, v_ref = w.k_cache.copy(), w.v_cache.copy()
    oracle.swap_blocks(k_ref, hk_ref, in_pairs)
    oracle.swap_blocks(v_ref, hv_ref, in_pairs)
    assert np.array_equal(synth.tensor_to_storage(t["k_cache"]), k_ref)
    assert np.array_equal(synth.tensor_to_storage(t["v_cache"]), v_ref)


def test_swap_flags_ids_outside_either_pool(pkv):
    dev = torch.arange(4 * 16 * 64, dtype=torch.float32, device="cuda").view(4, 16, 1, 64)
    host = torch.zeros(2, 16, 1, 64).pin_memory()
    pkv.kv_swap_blocks(host, dev, torch.tensor([[3, 1], [0, 2], [9, 0]], device="cuda"))
    assert pkv.pkv_device_error() == pkv.PKV_DERR_PAIR
    assert torch.equal(host[1], dev[3].cpu()) and host[0].eq(0).all()


# ------------------------------------------------------------------------------------------
# fp8 (E4M3) caches
# ------------------------------------------------------------------------------------------

def _fp8_setup(w, ks, vs):
    k8, v8 = synth.fp8_kv(w, ks, vs)
    t = synth.to_torch(w, "cuda")
    t["k8"] = torch.from_numpy(k8).cuda()
    t["v8"] = torch.from_numpy(v8).cuda()
    return k8, v8, t


@pytest.mark.parametrize("dtype,Hq,Hkv,bs,part", [("bf16", 8, 8, 16, 0), ("bf16", 64, 8, 16, 256),
                                                   ("f16", 32, 8, 32, 512), ("bf16", 12, 2, 64, 128),
                                                   ("bf16", 40, 2, 16, 512)])
def test_fp8_decode_matches_oracle(pkv, dtype, Hq, Hkv, bs, part):
    lens = [1, bs - 1, bs, bs + 1, 5 * bs + 3, 333, 1000, 0, 2 * bs]
    w = synth.make_workload("f8", seed=31 + Hq + bs, dtype=dtype, context_lens=lens,
                            num_q_heads=Hq, num_kv_heads=Hkv, head_dim=128, block_size=bs,
                            partition_size=part, key_outlier_frac=0.02)
    ks, vs = 0.0625, 0.03
    k8, v8, t = _fp8_setup(w, ks, vs)
    out = torch.empty_like(t["q"])
    pkv.paged_attn_decode_fp8(out, t["q"], t["k8"], t["v8"], t["block_tables"], t["context_lens"],
                              w.scale, ks, vs, partition_size=part)
    assert pkv.pkv_device_error() == 0
    ref = oracle.paged_decode_fp8kv(w.q, k8, v8, w.block_tables, w.context_lens, w.scale, ks, vs,
                                    dtype)
    assert_close(host_out(out), ref, dtype, f"fp8 {dtype} Hq{Hq} Hkv{Hkv} bs{bs} P{part}")
    assert (host_out(out)[7] == 0).all()


def test_fp8_poisoned_dead_slots_are_never_read(pkv):
    w = synth.make_workload("f8n", seed=33, dtype="bf16", context_lens=[1, 13, 17, 301],
                            num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                            pool_slack=0.5, partition_size=64, table_pad=2 ** 30)
    k8, v8, t = _fp8_setup(w, 0.05, 0.05)
    out = torch.empty_like(t["q"])
    pkv.paged_attn_decode_fp8(out, t["q"], t["k8"], t["v8"], t["block_tables"], t["context_lens"],
                              w.scale, 0.05, 0.05, partition_size=64)
    dead = torch.from_numpy(~synth.live_slot_mask(w)).cuda()
    t["k8"][dead] = 0x7F     # E4M3 NaN
    t["v8"][dead] = 0x7F
    out2 = torch.empty_like(out)
    pkv.paged_attn_decode_fp8(out2, t["q"], t["k8"], t["v8"], t["block_tables"], t["context_lens"],
                              w.scale, 0.05, 0.05, partition_size=64)
    assert pkv.pkv_device_error() == 0
    assert torch.isfinite(out2.float()).all() and torch.equal(out, out2)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_fp8_slot_write_bit_exact(pkv, dtype):
    NB, bs, Hkv, D = 20, 16, 8, 128
    rng = np.random.default_rng(6)
    n = 29
    slots = rng.choice(NB * bs, size=n, replace=False).astype(np.int64)
    slots[[2, 9]] = -1
    k_new = synth.to_storage(rng.standard_normal((n, Hkv, D)) * 4, dtype)
    v_new = synth.to_storage(rng.standard_normal((n, Hkv, D)) * 4, dtype)
    k_new[0, 0, :4] = synth.to_storage(np.array([6e4, -6e4, 0.0, -0.0]), dtype)  # saturation
    kc = np.full((NB, bs, Hkv, D), 0x11, np.uint8)
    vc = kc.copy()
    tk, tv = torch.from_numpy(kc).cuda(), torch.from_numpy(vc).cuda()
    ks, vs = 0.0371, 0.0529
    pkv.kv_cache_write_fp8(synth.storage_to_torch(k_new, dtype, "cuda"),
                           synth.storage_to_torch(v_new, dtype, "cuda"), tk, tv,
                           torch.from_numpy(slots).cuda(), ks, vs)
    assert pkv.pkv_device_error() == 0
    assert oracle.kv_cache_write_fp8(k_new, v_new, kc, vc, slots, ks, vs, dtype) == 0
    assert np.array_equal(tk.cpu().numpy(), kc)
    assert np.array_equal(tv.cpu().numpy(), vc)


def test_fp8_config3_gqa_full_size(pkv):
    """The 70B-like GQA batch with fp8 caches: slot write of the new tokens, then decode."""
    w = synth.config_workload(3)
    ks, vs = 0.0625, 0.0625
    k8, v8, t = _fp8_setup(w, ks, vs)
    pkv.kv_cache_write_fp8(t["k_new"], t["v_new"], t["k8"], t["v8"], t["slot_mapping"], ks, vs)
    out = torch.empty_like(t["q"])
    pkv.paged_attn_decode_fp8(out, t["q"], t["k8"], t["v8"], t["block_tables"], t["context_lens"],
                              w.scale, ks, vs)
    assert pkv.pkv_device_error() == 0
    assert oracle.kv_cache_write_fp8(w.k_new, w.v_new, k8, v8, w.slot_mapping, ks, vs, "bf16") == 0
    assert np.array_equal(t["k8"].cpu().numpy(), k8)
    seqs = _sample(w, 16, 8)
    ref = oracle.paged_decode_fp8kv(w.q[seqs], k8, v8, w.block_tables[seqs], w.context_lens[seqs],
                                    w.scale, ks, vs, "bf16")
    assert_close(host_out(out)[seqs], ref, "bf16", "fp8 config 3")


@pytest.mark.parametrize("cfg", [2, 4, 5])
def test_fp8_full_size_benchmark_batches(pkv, cfg):
    """E4M3 caches on the decode batches bench.py times with --kv-dtype fp8, with its
    scales, cache state, per-step writes and partition size: sampled sequences (always
    the longest and the shortest) against the oracle, and the caches byte for byte."""
    import bench

    w = bench.bench_workload(cfg)
    ks, vs = bench.fp8_scales(cfg)
    k8, v8, t = _fp8_setup(w, ks, vs)
    if cfg == 4:
        # the batch's state: copy-on-write copies, then every suffix token
        sk = synth.storage_to_torch(w.info["setup_k"], "bf16", "cuda")
        sv = synth.storage_to_torch(w.info["setup_v"], "bf16", "cuda")
        ss = torch.from_numpy(w.info["setup_slots"]).cuda()
        pkv.kv_copy_blocks(t["k8"], t["copy_pairs"])
        pkv.kv_copy_blocks(t["v8"], t["copy_pairs"])
        pkv.kv_cache_write_fp8(sk, sv, t["k8"], t["v8"], ss, ks, vs)
        oracle.copy_blocks(k8, w.copy_pairs)
        oracle.copy_blocks(v8, w.copy_pairs)
        assert oracle.kv_cache_write_fp8(w.info["setup_k"], w.info["setup_v"], k8, v8,
                                         w.info["setup_slots"], ks, vs, "bf16") == 0
        # one step: the copies again, then each sequence's next token
        pkv.kv_copy_blocks(t["k8"], t["copy_pairs"])
        pkv.kv_copy_blocks(t["v8"], t["copy_pairs"])
        oracle.copy_blocks(k8, w.copy_pairs)
        oracle.copy_blocks(v8, w.copy_pairs)
    pkv.kv_cache_write_fp8(t["k_new"], t["v_new"], t["k8"], t["v8"], t["slot_mapping"], ks, vs)
    assert oracle.kv_cache_write_fp8(w.k_new, w.v_new, k8, v8, w.slot_mapping, ks, vs,
                                     "bf16") == 0
    # the partition size bench.py launches E4M3 decode with
    part = pkv.paged_attn_decode_fp8_partition_tokens(w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                                      w.block_size, w.max_blocks_per_seq,
                                                      w.partition_size)
    out = torch.empty_like(t["q"])
    pkv.paged_attn_decode_fp8(out, t["q"], t["k8"], t["v8"], t["block_tables"], t["context_lens"],
                              w.scale, ks, vs, partition_size=part)
    assert pkv.pkv_device_error() == 0
    assert np.array_equal(t["k8"].cpu().numpy(), k8)
    assert np.array_equal(t["v8"].cpu().numpy(), v8)
    seqs = _sample(w, 3 if cfg == 5 else 16, 20 + cfg)
    ref = oracle.paged_decode_fp8kv(w.q[seqs], k8, v8, w.block_tables[seqs], w.context_lens[seqs],
                                    w.scale, ks, vs, "bf16")
    assert_close(host_out(out)[seqs], ref, "bf16", f"fp8 config {cfg}")
