"""Shared-prefix (cascade) decode on the GPU against the fp64 decode oracle.

The call computes paged_attn_decode's result; the oracle is the decode definition on the
same tables.  Acceptance: |gpu - oracle| <= 2e-2 + 1e-2 |oracle| (bf16 / fp16).
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

ATOL_16, RTOL_16 = 2e-2, 1e-2


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_315_gb300 as m

    m.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    m.pkv_device_error()
    return m


def assert_close(got, ref, what=""):
    got = got.astype(np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bad = err > ATOL_16 + RTOL_16 * np.abs(ref)
    assert not bad.any(), f"{what}: {bad.sum()} elements out of tolerance, max err {err.max():.3e}"


def cascade(pkv, w, t, group_start, prefix_lens, max_group=None, max_prefix=None):
    gs = torch.tensor(group_start, dtype=torch.int32, device="cuda")
    pl = torch.tensor(prefix_lens, dtype=torch.int32, device="cuda")
    out = torch.full_like(t["q"], float("nan"))
    sizes = np.diff(np.asarray(group_start)) if len(group_start) > 1 else np.array([0])
    pkv.paged_attn_decode_shared_prefix(
        out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"], t["context_lens"], gs, pl,
        int(sizes.max()) if max_group is None else max_group,
        int(max(prefix_lens, default=0)) if max_prefix is None else max_prefix, w.scale)
    return out.float().cpu().numpy()


def share_prefix(w, group_start, prefix_lens):
    """Point every member's first prefix blocks at the first member's physical blocks."""
    bs = w.block_size
    for g in range(len(prefix_lens)):
        a, b = group_start[g], group_start[g + 1]
        nb = prefix_lens[g] // bs
        for s in range(a + 1, b):
            w.block_tables[s, :nb] = w.block_tables[a, :nb]


@pytest.mark.parametrize("Hq,Hkv,bs,dtype", [(8, 2, 16, "bf16"), (16, 2, 32, "f16"),
                                             (4, 4, 64, "bf16"), (12, 4, 16, "bf16"),
                                             (10, 2, 32, "f16")])
def test_groups_of_mixed_sizes_match_oracle(pkv, Hq, Hkv, bs, dtype):
    lens = [200, 70, 64, 900, 33, 40, 1, 300, 64, 0, 17, 500]
    group_start = [0, 4, 5, 9]       # runs [0,4), [4,5), [5,9); 9..11 outside every group
    prefix_lens = [64, 32, 0]        # sequence 2 is all prefix (L == prefix)
    if bs == 64:
        prefix_lens = [64, 0, 0]
    w = synth.make_workload("sp", seed=60 + Hq + bs, dtype=dtype, context_lens=lens,
                            num_q_heads=Hq, num_kv_heads=Hkv, head_dim=128, block_size=bs,
                            key_outlier_frac=0.02)
    share_prefix(w, group_start, prefix_lens)
    t = synth.to_torch(w, "cuda")
    out = cascade(pkv, w, t, group_start, prefix_lens)
    assert pkv.pkv_device_error() == 0
    ref = oracle.paged_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                              w.dtype)
    assert_close(out, ref, f"Hq{Hq} Hkv{Hkv} bs{bs}")
    assert (out[9] == 0).all()  # empty context


@pytest.mark.parametrize("mult", [-1.0, 0.0])
def test_cascade_with_a_non_positive_scale_matches_oracle(pkv, mult):
    # the prefix pass runs (-q) . k times |scale| for a negative scale; the suffix pass and
    # the merge take the scale as it is
    w = synth.make_workload("spn", seed=41, dtype="bf16", context_lens=[200, 77, 129, 64, 300],
                            num_q_heads=16, num_kv_heads=4, head_dim=128, block_size=16)
    share_prefix(w, [0, 3, 5], [64, 48])
    w.scale = mult * w.scale
    t = synth.to_torch(w, "cuda")
    out = cascade(pkv, w, t, [0, 3, 5], [64, 48])
    assert pkv.pkv_device_error() == 0
    ref = oracle.paged_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                              w.dtype)
    assert_close(out, ref, f"cascade, scale {w.scale}")


def test_one_group_with_a_long_prefix_splits_its_keys(pkv):
    # 24 sequences share a 2048-token prefix: the prefix pass splits the keys across CTAs
    lens = 2048 + np.arange(24) * 37 % 300
    w = synth.make_workload("spl", seed=66, dtype="bf16", context_lens=lens, num_q_heads=32,
                            num_kv_heads=8, head_dim=128, block_size=16)
    share_prefix(w, [0, 24], [2048])
    t = synth.to_torch(w, "cuda")
    out = cascade(pkv, w, t, [0, 24], [2048])
    assert pkv.pkv_device_error() == 0
    ref = oracle.paged_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                              w.dtype)
    assert_close(out, ref, "2048-token prefix")


def test_bad_prefix_is_reported_and_served_without_it(pkv):
    lens = [100, 90, 80]
    w = synth.make_workload("spb", seed=67, dtype="bf16", context_lens=lens, num_q_heads=8,
                            num_kv_heads=2, head_dim=128, block_size=16)
    share_prefix(w, [0, 3], [48])
    t = synth.to_torch(w, "cuda")
    ref = oracle.paged_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                              w.dtype)
    out = cascade(pkv, w, t, [0, 3], [40], max_prefix=48)  # 40 is not a whole number of blocks
    assert pkv.pkv_device_error() == pkv.PKV_DERR_CONTEXT
    assert_close(out, ref, "prefix not in whole blocks")
    out = cascade(pkv, w, t, [0, 3], [48], max_group=2)    # a group above max_group_size
    assert pkv.pkv_device_error() & pkv.PKV_DERR_CONTEXT
    assert_close(out, ref, "group above max_group_size")
    out = cascade(pkv, w, t, [0, 3], [48])
    assert pkv.pkv_device_error() == 0
    assert_close(out, ref, "after errors")


def test_config4_shared_prefix_cascade(pkv):
    """The shared-prefix batch at full size, after its copies and writes, in the launch
    bench.py times: sampled sequences against the oracle."""
    w = synth.config_workload(4)
    t = synth.to_torch(w, "cuda")
    pkv.kv_copy_blocks(t["k_cache"], t["copy_pairs"])
    pkv.kv_copy_blocks(t["v_cache"], t["copy_pairs"])
    pkv.kv_cache_write(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["slot_mapping"])
    P = int(w.info["shared_prefix_tokens"])
    out = cascade(pkv, w, t, [0, w.num_seqs], [P])
    assert pkv.pkv_device_error() == 0
    assert np.isfinite(out).all()
    k, v = w.k_cache.copy(), w.v_cache.copy()
    oracle.copy_blocks(k, w.copy_pairs)
    oracle.copy_blocks(v, w.copy_pairs)
    assert oracle.kv_cache_write(w.k_new, w.v_new, k, v, w.slot_mapping) == 0
    rng = np.random.default_rng(4)
    seqs = np.unique(np.r_[0, w.num_seqs - 1, rng.choice(w.num_seqs, 22, replace=False)])
    ref = oracle.paged_decode(w.q[seqs], k, v, w.block_tables[seqs], w.context_lens[seqs],
                              w.scale, w.dtype)
    assert_close(out[seqs], ref, "config 4 cascade")


def test_grouped_prompts_match_oracle(pkv):
    # parallel sampling: 6 prompts x 5 samples, each prompt 512 tokens in shared blocks
    w = synth.grouped_prefix_workload(groups=6, members=5, prefix_tokens=512,
                                      suffix_range=(1, 100), num_q_heads=16, num_kv_heads=4)
    t = synth.to_torch(w, "cuda")
    out = cascade(pkv, w, t, w.info["group_start"].tolist(), w.info["prefix_lens"].tolist())
    assert pkv.pkv_device_error() == 0
    ref = oracle.paged_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                              w.dtype)
    assert_close(out, ref, "grouped prompts")


def test_grouped_prompts_full_size_in_the_benchmarked_launch(pkv):
    """The grouped-prompt batch bench.py times with --grouped-prefix --shared-prefix (64
    prompts of 4096 tokens x 8 samples), after the step's slot write, in that launch:
    sampled sequences (the longest, the shortest and one whole group) against the oracle."""
    w = synth.grouped_prefix_workload()
    synth.add_new_tokens(w, seed=synth.BASE_SEED + 107)
    t = synth.to_torch(w, "cuda")
    pkv.kv_cache_write(t["k_new"], t["v_new"], t["k_cache"], t["v_cache"], t["slot_mapping"])
    gs, pls = w.info["group_start"], w.info["prefix_lens"]
    out = cascade(pkv, w, t, gs.tolist(), pls.tolist())
    assert pkv.pkv_device_error() == 0
    assert np.isfinite(out).all()
    k, v = w.k_cache.copy(), w.v_cache.copy()
    assert oracle.kv_cache_write(w.k_new, w.v_new, k, v, w.slot_mapping) == 0
    rng = np.random.default_rng(7)
    g = int(rng.integers(0, len(pls)))
    seqs = np.unique(np.r_[np.argmax(w.context_lens), np.argmin(w.context_lens),
                           np.arange(gs[g], gs[g + 1]),
                           rng.choice(w.num_seqs, 16, replace=False)])
    ref = oracle.paged_decode(w.q[seqs], k, v, w.block_tables[seqs], w.context_lens[seqs],
                              w.scale, w.dtype)
    assert_close(out[seqs], ref, "grouped prompts, full size")
