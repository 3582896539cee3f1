"""Host-side checks of the seeded workload generators (no GPU)."""
import math

import numpy as np
import pytest

import synth


def test_same_seed_same_arrays_any_thread_count(monkeypatch):
    a = synth.make_workload("a", seed=4, dtype="bf16", context_lens=[300, 5000], num_q_heads=8,
                            num_kv_heads=2, head_dim=128, block_size=16)
    monkeypatch.setattr(synth, "_threads", lambda: 1)
    b = synth.make_workload("b", seed=4, dtype="bf16", context_lens=[300, 5000], num_q_heads=8,
                            num_kv_heads=2, head_dim=128, block_size=16)
    for x, y in ((a.q, b.q), (a.k_cache, b.k_cache), (a.v_cache, b.v_cache),
                 (a.block_tables, b.block_tables)):
        np.testing.assert_array_equal(x, y)


def test_bf16_rounding_is_nearest_even():
    import torch

    x = np.random.default_rng(0).standard_normal(10000).astype(np.float32) * 37
    x[:4] = [1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 0.0]
    bits = synth.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bits, ref)


def test_allocation_gives_each_block_to_one_sequence():
    w = synth.make_workload("t", seed=2, dtype="f32", context_lens=[1, 16, 17, 100, 0],
                            num_q_heads=2, num_kv_heads=2, head_dim=8, block_size=16)
    used = [b for s in range(w.num_seqs)
            for b in w.block_tables[s, :math.ceil(w.context_lens[s] / 16)]]
    assert len(used) == len(set(used)) == 1 + 1 + 2 + 7
    assert w.num_blocks == math.ceil(1.1 * len(used))
    assert (w.block_tables[0, 1:] == -1).all()
    assert synth.live_slot_mask(w).sum() == 1 + 16 + 17 + 100


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_config_shapes(cfg):
    w = synth.config_workload(cfg)
    B, Hq, D = w.q.shape
    NB, bs, Hkv, D2 = w.k_cache.shape
    assert D == D2 and Hq % Hkv == 0
    nb = -(-w.context_lens.astype(np.int64) // bs)
    assert (nb <= w.max_blocks_per_seq).all()
    if cfg == 1:
        assert list(w.context_lens) == [1, 17, 33, 100] and NB == 64 and w.dtype == "f32"
    if cfg == 2:
        assert (B, Hq, Hkv, D, bs) == (64, 40, 40, 128, 16)
        assert w.context_lens.min() >= 1 and w.context_lens.max() <= 2048
    if cfg == 3:
        assert (B, Hq, Hkv, bs) == (128, 64, 8, 16)
        assert w.context_lens.min() >= 128 and w.context_lens.max() <= 8192
        assert w.slot_mapping.shape == (128,)
    if cfg == 4:
        assert (B, Hq, Hkv, bs) == (256, 32, 8, 32)
        shared = w.info["shared_ids"]
        assert len(shared) == 32
        # every sequence shares the 31 full prefix blocks; the partial one was copied
        assert (w.block_tables[:, :31] == shared[:31]).all()
        assert (w.copy_pairs[:, 0] == shared[31]).all()
        assert len(set(w.copy_pairs[:, 1])) == 256
        assert (w.block_tables[:, 31] == w.copy_pairs[:, 1]).all()
        assert w.slot_mapping.shape[0] == int((w.context_lens - 1008).sum())


def test_prefill_workload_packs_chunks_after_prior_context():
    w = synth.make_prefill_workload("t", seed=3, dtype="bf16", prior_lens=[0, 20, 5],
                                    chunk_lens=[4, 1, 30], num_q_heads=4, num_kv_heads=2,
                                    head_dim=32, block_size=16)
    assert w.query_start.tolist() == [0, 4, 5, 35]
    assert w.context_lens.tolist() == [4, 21, 35]
    assert w.chunk_q.shape == (35, 4, 32)
    # the cache holds every token of prior + chunk: blocks for all of them are allocated
    for s, L in enumerate(w.context_lens):
        nb = -(-int(L) // 16)
        assert (w.block_tables[s, :nb] >= 0).all()


def test_prefill_batch_is_seeded_and_shaped():
    a = synth.prefill_workload()
    b = synth.prefill_workload()
    assert np.array_equal(a.context_lens, b.context_lens)
    assert np.array_equal(a.chunk_q, b.chunk_q)
    assert a.num_seqs == 16 and a.chunk_q.shape == (16 * 512, 64, 128)
    prior = a.context_lens - 512
    assert prior.min() >= 0 and prior.max() <= 3584
