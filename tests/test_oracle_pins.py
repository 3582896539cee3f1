"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Each test checks the oracle against something the pages or mathematics fix:
the pages' worked block-table examples, a library attention routine on the same
logical sequence, closed forms, invariants the method must keep, or an
arbitrary-precision brute force on tiny inputs.  The comment on each test names
the mistakes in the oracle it would catch.
"""
import math

import numpy as np
import pytest
import torch

import synth

GOLDEN = __file__.replace("test_oracle_pins.py", "golden/block_table_walks.txt")


# ----------------------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------------------

def _wl(dtype="bf16", lens=(1, 5, 16, 17, 40), Hq=4, Hkv=2, D=64, bs=16, shuffle=True,
        seed=11, scale=None, **kw):
    return synth.make_workload("pin", seed=seed, dtype=dtype, context_lens=list(lens),
                               num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=bs,
                               shuffle=shuffle, scale=scale, **kw)


def _run(oracle_mod, w, **kw):
    return oracle_mod.paged_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                   w.scale, w.dtype, **kw)


def _f64(w, a):
    return synth.storage_to_f64(a, w.dtype)


def _dense_rows(w, s):
    """K, V rows [L, Hkv, D] of sequence s for an unshuffled pool.

    With ``shuffle=False`` the allocator hands each sequence consecutive physical
    blocks, so its tokens are one contiguous run of pool rows; no block-table
    arithmetic is needed to read them.
    """
    NB, bs, Hkv, D = w.k_cache.shape
    start = int(w.block_tables[s, 0]) * bs
    L = int(w.context_lens[s])
    k = _f64(w, w.k_cache).reshape(NB * bs, Hkv, D)[start:start + L]
    v = _f64(w, w.v_cache).reshape(NB * bs, Hkv, D)[start:start + L]
    return k, v


def _torch_bits_to_f64(bits, dtype):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view({"bf16": torch.bfloat16, "f16": torch.float16}[dtype]).double().numpy()


# ----------------------------------------------------------------------------------------
# block-table addressing: the pages' worked examples
# ----------------------------------------------------------------------------------------

def _golden_cases():
    cases, cur = [], None
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, rest = line.partition(" ")
        if key == "case":
            cur = {"name": rest, "checks": []}
            cases.append(cur)
        elif key == "source":
            cur["source"] = rest
        elif key == "block_size":
            cur["bs"] = int(rest)
        elif key == "table":
            cur["table"] = [int(x) for x in rest.split()]
        else:
            cur["checks"].append((key, [int(x) for x in rest.split()]))
    return cases


@pytest.mark.parametrize("case", _golden_cases(), ids=lambda c: c["name"])
def test_golden_block_table_walks(oracle_mod, case):
    """Catches: wrong block index (p % bs vs p / bs), off-by-one in block counts."""
    assert case.get("source")
    bs = case["bs"]
    table = np.asarray(case.get("table", [0]), np.int32)
    for key, vals in case["checks"]:
        if key == "locate":
            pos, phys, off = vals
            assert oracle_mod.locate(table, pos, bs) == (phys, off), (case["name"], vals)
            assert oracle_mod.slot(table, pos, bs) == phys * bs + off
        elif key == "blocks":
            n, nb = vals
            assert oracle_mod.num_blocks(n, bs) == nb, (case["name"], vals)
        elif key == "waste":
            n, waste = vals
            assert oracle_mod.num_blocks(n, bs) * bs - n == waste, (case["name"], vals)
        elif key == "maxwaste":
            (mw,) = vals
            worst = max(oracle_mod.num_blocks(n, bs) * bs - n for n in range(1, 10 * bs))
            assert worst == mw
        else:
            raise AssertionError(f"unknown directive {key}")


# ----------------------------------------------------------------------------------------
# element widening
# ----------------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_single_token_returns_its_value_exactly(oracle_mod, dtype):
    """L = 1: softmax weight is exactly 1, so out = v_0 widened exactly.

    The expected value comes from torch's own bf16/fp16 widening.  Catches: a wrong
    bit-pattern decode, a dropped normalisation, reading the wrong slot or head.
    """
    w = _wl(dtype=dtype, lens=(1, 1, 1), Hq=4, Hkv=2, D=64)
    out = _run(oracle_mod, w)
    G = w.num_q_heads // w.num_kv_heads
    for s in range(w.num_seqs):
        phys = int(w.block_tables[s, 0])
        for h in range(w.num_q_heads):
            row = w.v_cache[phys, 0, h // G]
            want = row.astype(np.float64) if dtype == "f32" else _torch_bits_to_f64(row, dtype)
            np.testing.assert_array_equal(out[s, h], want)


# ----------------------------------------------------------------------------------------
# agreement with a library attention routine on the unpaged sequence
# ----------------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype,Hq,Hkv,D,bs", [
    ("f32", 4, 4, 64, 16), ("bf16", 8, 2, 128, 16), ("f16", 4, 1, 64, 8),
    ("bf16", 16, 2, 128, 32), ("bf16", 6, 3, 32, 16)])
def test_matches_sdpa_on_unpaged_sequence(oracle_mod, dtype, Hq, Hkv, D, bs):
    """Paged attention equals ordinary attention on the same logical sequence.

    Reference: torch.nn.functional.scaled_dot_product_attention in float64 on the
    sequence's contiguous K/V rows (pool unshuffled), GQA by repeating each KV head.
    Catches: dropped or wrong scale, sign errors, transposed operands, wrong head
    mapping, attending L-1 or L+1 tokens.
    """
    lens = (1, bs - 1, bs, bs + 1, 3 * bs + 5, 97)
    w = _wl(dtype=dtype, lens=lens, Hq=Hq, Hkv=Hkv, D=D, bs=bs, shuffle=False, scale=0.37)
    out = _run(oracle_mod, w)
    G = Hq // Hkv
    q = _f64(w, w.q)
    for s in range(w.num_seqs):
        k, v = _dense_rows(w, s)
        kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(G, dim=0)  # [Hq, L, D]
        vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(G, dim=0)
        qt = torch.from_numpy(q[s])[:, None, :]                                  # [Hq, 1, D]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=w.scale)
        np.testing.assert_allclose(out[s], ref[:, 0, :].numpy(), rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------------------------------
# invariants
# ----------------------------------------------------------------------------------------

def test_physical_block_permutation_invariance(oracle_mod):
    """Moving blocks in the pool and renaming them in the tables changes nothing.

    The pages: the gather kernel's correctness is independent of layout.  The
    oracle's arithmetic order depends only on logical positions, so the result is
    bit-identical.  Catches: reading blocks by logical instead of physical id.
    """
    w = _wl(dtype="bf16", lens=(3, 16, 33, 70), Hq=4, Hkv=2, D=64, bs=16, pool_slack=0.5)
    base = _run(oracle_mod, w)
    rng = np.random.default_rng(5)
    perm = rng.permutation(w.num_blocks)
    k2 = np.empty_like(w.k_cache)
    v2 = np.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    bt2 = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    out = oracle_mod.paged_decode(w.q, k2, v2, bt2, w.context_lens, w.scale, w.dtype)
    np.testing.assert_array_equal(out, base)


def test_gqa_equals_mha_with_replicated_kv_heads(oracle_mod):
    """Query head h of a GQA batch reads KV head h // G.

    Replicating each KV head G times (consecutively) and running MHA must give the
    same result.  Catches: h % Hkv head mapping, wrong group size.
    """
    w = _wl(dtype="bf16", lens=(5, 31, 64), Hq=8, Hkv=2, D=64)
    G = 4
    out = _run(oracle_mod, w)
    k_rep = np.repeat(w.k_cache, G, axis=2)
    v_rep = np.repeat(w.v_cache, G, axis=2)
    ref = oracle_mod.paged_decode(w.q, k_rep, v_rep, w.block_tables, w.context_lens, w.scale,
                                  w.dtype)
    np.testing.assert_array_equal(out, ref)


@pytest.mark.parametrize("partition", [16, 32, 48, 512, 1 << 20])
def test_split_context_lse_merge_equals_definition(oracle_mod, partition):
    """Partition partials merged by log-sum-exp give the same attention.

    Catches in the partitioned form: a missing exp(m_i - M) rescale, normalising
    per partition, dropping the last ragged partition.
    """
    w = _wl(dtype="bf16", lens=(1, 17, 100, 700, 1500), Hq=4, Hkv=1, D=64, bs=16,
            key_outlier_frac=0.05)
    ref = _run(oracle_mod, w)
    out = oracle_mod.paged_decode_partitioned(w.q, w.k_cache, w.v_cache, w.block_tables,
                                              w.context_lens, w.scale, w.dtype, partition)
    np.testing.assert_allclose(out, ref, rtol=1e-11, atol=1e-13)


# ----------------------------------------------------------------------------------------
# closed forms
# ----------------------------------------------------------------------------------------

def test_uniform_keys_give_mean_of_values(oracle_mod):
    """All keys equal => all scores equal => out = mean of the L values.

    Catches: a missing normalisation, summing over the wrong token range.
    """
    w = _wl(dtype="f32", lens=(1, 7, 16, 45), Hq=2, Hkv=2, D=32, bs=8, shuffle=False)
    w.k_cache[...] = np.float32(0.75)
    out = _run(oracle_mod, w)
    for s in range(w.num_seqs):
        _, v = _dense_rows(w, s)
        np.testing.assert_allclose(out[s], v.mean(axis=0), rtol=1e-13, atol=1e-14)


def test_zero_scale_gives_mean_of_values(oracle_mod):
    w = _wl(dtype="bf16", lens=(2, 19, 64), Hq=4, Hkv=4, D=64, bs=16, shuffle=False, scale=0.0)
    out = _run(oracle_mod, w)
    for s in range(w.num_seqs):
        _, v = _dense_rows(w, s)
        np.testing.assert_allclose(out[s], v.mean(axis=0), rtol=1e-13, atol=1e-14)


def test_two_tokens_follow_the_logistic_closed_form(oracle_mod):
    """For two tokens, out = v0 + sigmoid(s1 - s0) (v1 - v0), s_i = scale <q, k_i>.

    Catches: a sign error in the exponent, scale applied after softmax.
    """
    w = _wl(dtype="f32", lens=(2, 2, 2), Hq=2, Hkv=1, D=16, bs=4, shuffle=False, scale=0.9)
    out = _run(oracle_mod, w)
    q = _f64(w, w.q)
    for s in range(w.num_seqs):
        k, v = _dense_rows(w, s)
        for h in range(2):
            s0 = w.scale * float(q[s, h] @ k[0, 0])
            s1 = w.scale * float(q[s, h] @ k[1, 0])
            sig = 1.0 / (1.0 + math.exp(-(s1 - s0)))
            want = v[0, 0] + sig * (v[1, 0] - v[0, 0])
            np.testing.assert_allclose(out[s, h], want, rtol=1e-12, atol=1e-13)


def test_dominant_key_selects_its_value_without_overflow(oracle_mod):
    """A key aligned with q and scaled far above the rest takes all the weight.

    Scores reach ~1e4, so exp without the max subtraction overflows.  Catches: a
    missing max subtraction (inf/nan) and selecting the wrong token.
    """
    w = _wl(dtype="f32", lens=(9, 40), Hq=1, Hkv=1, D=16, bs=8, shuffle=False, scale=1.0)
    NB, bs = w.k_cache.shape[:2]
    kf = w.k_cache.reshape(NB * bs, 1, 16)
    for s, hot in ((0, 4), (1, 33)):
        start = int(w.block_tables[s, 0]) * bs
        kf[start + hot, 0] = 400.0 * w.q[s, 0] / np.linalg.norm(w.q[s, 0])
    out = _run(oracle_mod, w)
    assert np.isfinite(out).all()
    for s, hot in ((0, 4), (1, 33)):
        _, v = _dense_rows(w, s)
        np.testing.assert_allclose(out[s, 0], v[hot, 0], rtol=1e-12, atol=1e-12)


def test_empty_context_gives_zeros(oracle_mod):
    w = _wl(dtype="bf16", lens=(0, 5, 0), Hq=2, Hkv=1, D=32, bs=16)
    out = _run(oracle_mod, w)
    assert (out[0] == 0).all() and (out[2] == 0).all()
    assert np.abs(out[1]).sum() > 0


def test_arbitrary_precision_brute_force(oracle_mod):
    """Tiny cases against a 50-digit evaluation of the attention sum (mpmath)."""
    import mpmath

    mpmath.mp.dps = 50
    w = _wl(dtype="bf16", lens=(1, 3, 5), Hq=2, Hkv=1, D=4, bs=2, scale=0.8, seed=3)
    out = _run(oracle_mod, w)
    q = _f64(w, w.q)
    K = _f64(w, w.k_cache)
    V = _f64(w, w.v_cache)
    for s in range(w.num_seqs):
        L = int(w.context_lens[s])
        rows = [(int(w.block_tables[s, p // 2]), p % 2) for p in range(L)]
        for h in range(2):
            sc = [mpmath.mpf(w.scale) * mpmath.fsum(mpmath.mpf(q[s, h, d]) * mpmath.mpf(K[b, o, 0, d])
                                                    for d in range(4)) for b, o in rows]
            e = [mpmath.exp(x) for x in sc]
            z = mpmath.fsum(e)
            for d in range(4):
                want = mpmath.fsum(ei * mpmath.mpf(V[b, o, 0, d]) for ei, (b, o) in zip(e, rows)) / z
                assert abs(out[s, h, d] - float(want)) <= 1e-14 * max(1.0, abs(float(want)))


def test_out_of_range_block_id_is_rejected(oracle_mod):
    w = _wl(dtype="bf16", lens=(5, 20), Hq=2, Hkv=1, D=32, bs=16)
    w.block_tables[1, 1] = w.num_blocks
    with pytest.raises(ValueError):
        _run(oracle_mod, w)


def test_unused_table_entries_and_dead_slots_are_never_read(oracle_mod):
    """Entries past ceil(L / bs) hold -1 and every dead slot holds NaN: no effect."""
    w = _wl(dtype="bf16", lens=(1, 15, 16, 17, 50), Hq=4, Hkv=2, D=64, bs=16, pool_slack=0.3)
    ref = _run(oracle_mod, w)
    synth.poison_unused(w)
    out = _run(oracle_mod, w)
    assert np.isfinite(out).all()
    np.testing.assert_array_equal(out, ref)


# ----------------------------------------------------------------------------------------
# slot writes
# ----------------------------------------------------------------------------------------

def test_slot_write_lands_in_the_row_the_slot_names(oracle_mod):
    """Slot s is row s of the cache viewed as [NB * bs] token rows.

    Catches: swapped block/offset, writing k into v, off-by-one rows.
    """
    w = _wl(dtype="bf16", lens=(40, 40), Hq=2, Hkv=2, D=32, bs=8)
    NB, bs, Hkv, D = w.k_cache.shape
    rng = np.random.default_rng(1)
    slots = rng.choice(NB * bs, size=13, replace=False).astype(np.int64)
    k_new = rng.integers(0, 1 << 16, size=(13, Hkv, D), dtype=np.uint16)
    v_new = rng.integers(0, 1 << 16, size=(13, Hkv, D), dtype=np.uint16)
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    assert oracle_mod.kv_cache_write(k_new, v_new, kc, vc, slots) == 0
    rows_k = kc.reshape(NB * bs, Hkv, D)
    rows_v = vc.reshape(NB * bs, Hkv, D)
    np.testing.assert_array_equal(rows_k[slots], k_new)
    np.testing.assert_array_equal(rows_v[slots], v_new)
    untouched = np.setdiff1d(np.arange(NB * bs), slots)
    np.testing.assert_array_equal(rows_k[untouched], w.k_cache.reshape(NB * bs, Hkv, D)[untouched])
    np.testing.assert_array_equal(rows_v[untouched], w.v_cache.reshape(NB * bs, Hkv, D)[untouched])


def test_slot_write_skips_padding_and_flags_out_of_range(oracle_mod):
    w = _wl(dtype="f32", lens=(10,), Hq=1, Hkv=1, D=8, bs=4)
    NB, bs = w.k_cache.shape[:2]
    k_new = np.ones((3, 1, 8), np.float32)
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    assert oracle_mod.kv_cache_write(k_new, k_new, kc, vc, np.array([-1, NB * bs, -5])) == 1
    np.testing.assert_array_equal(kc, w.k_cache)
    np.testing.assert_array_equal(vc, w.v_cache)


def test_thirty_token_walk_then_decode(oracle_mod):
    """The 30 -> 34 token walk: decoded tokens go to offsets 14, 15 of block 2, then
    offsets 0, 1 of a third block; attention over the 34 tokens is then ordinary
    attention over the sequence in logical order."""
    bs, Hkv, D = 16, 1, 8
    table = np.array([[11, 4, 23]], np.int32)
    rng = np.random.default_rng(2)
    kc = rng.standard_normal((32, bs, Hkv, D)).astype(np.float32)
    vc = rng.standard_normal((32, bs, Hkv, D)).astype(np.float32)
    k_new = rng.standard_normal((4, Hkv, D)).astype(np.float32)
    v_new = rng.standard_normal((4, Hkv, D)).astype(np.float32)
    slots = np.array([oracle_mod.slot(table[0], p, bs) for p in (30, 31, 32, 33)], np.int64)
    assert list(slots) == [4 * bs + 14, 4 * bs + 15, 23 * bs + 0, 23 * bs + 1]
    assert oracle_mod.kv_cache_write(k_new, v_new, kc, vc, slots) == 0
    q = rng.standard_normal((1, 1, D)).astype(np.float32)
    out = oracle_mod.paged_decode(q, kc, vc, table, np.array([34], np.int32), 0.5, "f32")
    K = np.concatenate([kc[11], kc[4], kc[23][:2]])[:, 0].astype(np.float64)
    V = np.concatenate([vc[11], vc[4], vc[23][:2]])[:, 0].astype(np.float64)
    np.testing.assert_array_equal(K[30:], k_new[:, 0])
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q.astype(np.float64))[:, :, None, :][0],
        torch.from_numpy(K)[None], torch.from_numpy(V)[None], scale=0.5)
    np.testing.assert_allclose(out[0], ref[:, 0].numpy(), rtol=1e-12, atol=1e-13)


# ----------------------------------------------------------------------------------------
# block copies (copy-on-write)
# ----------------------------------------------------------------------------------------

def test_copy_blocks_copies_whole_blocks_only(oracle_mod):
    w = _wl(dtype="bf16", lens=(64,), Hq=2, Hkv=2, D=32, bs=16, num_blocks=12)
    pairs = np.array([[3, 7], [5, 5], [0, 11]], np.int64)
    c = w.k_cache.copy()
    assert oracle_mod.copy_blocks(c, pairs) == 0
    np.testing.assert_array_equal(c[7], w.k_cache[3])
    np.testing.assert_array_equal(c[11], w.k_cache[0])
    others = [b for b in range(12) if b not in (7, 11)]
    np.testing.assert_array_equal(c[others], w.k_cache[others])


def test_copy_blocks_flags_out_of_range(oracle_mod):
    w = _wl(dtype="bf16", lens=(16,), Hq=1, Hkv=1, D=16, bs=16, num_blocks=4)
    c = w.k_cache.copy()
    assert oracle_mod.copy_blocks(c, np.array([[0, 4], [-1, 2]], np.int64)) == 1
    np.testing.assert_array_equal(c, w.k_cache)


def test_copy_on_write_leaves_other_sharers_unchanged(oracle_mod):
    """Two sequences share a prefix whose last block is partial.  Sequence 1 copies
    that block to a private one and writes its next token there; sequence 0's output
    and the shared block are unchanged, and sequence 1 then sees the prefix plus its
    own token."""
    bs, Hkv, D = 16, 2, 32
    w = _wl(dtype="bf16", lens=(20, 20), Hq=4, Hkv=Hkv, D=D, bs=bs, num_blocks=8, shuffle=False)
    shared = w.block_tables[0, :2].copy()
    w.block_tables[1, :2] = shared
    before = _run(oracle_mod, w)
    np.testing.assert_array_equal(before[0, :, :], before[0, :, :])
    private = 6
    kc, vc = w.k_cache.copy(), w.v_cache.copy()
    assert oracle_mod.copy_blocks(kc, np.array([[shared[1], private]])) == 0
    assert oracle_mod.copy_blocks(vc, np.array([[shared[1], private]])) == 0
    bt = w.block_tables.copy()
    bt[1, 1] = private
    rng = np.random.default_rng(9)
    k_new = synth.to_storage(rng.standard_normal((1, Hkv, D)), "bf16")
    v_new = synth.to_storage(rng.standard_normal((1, Hkv, D)), "bf16")
    slot = oracle_mod.slot(bt[1], 20, bs)
    assert slot == private * bs + 4
    assert oracle_mod.kv_cache_write(k_new, v_new, kc, vc, np.array([slot])) == 0
    lens = np.array([20, 21], np.int32)
    after = oracle_mod.paged_decode(w.q, kc, vc, bt, lens, w.scale, "bf16")
    np.testing.assert_array_equal(after[0], before[0])
    np.testing.assert_array_equal(kc[shared[1]], w.k_cache[shared[1]])
    np.testing.assert_array_equal(vc[shared[1]], w.v_cache[shared[1]])
    # sequence 1 over the unshared layout equals the same tokens laid out contiguously
    K = np.concatenate([kc[shared[0]], kc[private][:5]]).astype(np.uint16)
    V = np.concatenate([vc[shared[0]], vc[private][:5]]).astype(np.uint16)
    kc2 = np.zeros((2, bs, Hkv, D), np.uint16)
    vc2 = np.zeros((2, bs, Hkv, D), np.uint16)
    kc2.reshape(2 * bs, Hkv, D)[:21] = K
    vc2.reshape(2 * bs, Hkv, D)[:21] = V
    ref = oracle_mod.paged_decode(w.q[1:2], kc2, vc2, np.array([[0, 1]], np.int32),
                                  np.array([21], np.int32), w.scale, "bf16")
    np.testing.assert_allclose(after[1], ref[0], rtol=1e-13, atol=1e-14)


# ----------------------------------------------------------------------------------------
# block copies between pools (swap out / swap in)
# ----------------------------------------------------------------------------------------

def test_swap_out_and_back_in_restores_the_sequence(oracle_mod):
    """Swapping a sequence's blocks to a host pool and back into other device blocks
    (with its table renamed) leaves its attention output bit-identical; the pools' other
    blocks are untouched.  Catches: swapped src/dst, copying from the wrong pool."""
    w = _wl(dtype="bf16", lens=(40, 70), Hq=4, Hkv=2, D=64, bs=16, pool_slack=1.5)
    before = _run(oracle_mod, w)
    nb = -(-70 // 16)
    blocks = w.block_tables[1, :nb].astype(np.int64)
    host_k = np.zeros((8,) + w.k_cache.shape[1:], np.uint16)
    host_v = np.zeros_like(host_k)
    out_pairs = np.stack([blocks, np.arange(nb) + 2], axis=1)       # device -> host slots 2..
    assert oracle_mod.swap_blocks(host_k, w.k_cache, out_pairs) == 0
    assert oracle_mod.swap_blocks(host_v, w.v_cache, out_pairs) == 0
    np.testing.assert_array_equal(host_k[2:2 + nb], w.k_cache[blocks])
    assert (host_k[:2] == 0).all() and (host_k[2 + nb:] == 0).all()
    used = set(w.block_tables[w.block_tables >= 0].tolist())
    free = np.array([b for b in range(w.num_blocks) if b not in used][:nb], np.int64)
    k2, v2 = w.k_cache.copy(), w.v_cache.copy()
    k2[blocks] = 0                                                  # the old blocks are reused
    v2[blocks] = 0
    in_pairs = np.stack([np.arange(nb) + 2, free], axis=1)          # host -> new device blocks
    assert oracle_mod.swap_blocks(k2, host_k, in_pairs) == 0
    assert oracle_mod.swap_blocks(v2, host_v, in_pairs) == 0
    bt = w.block_tables.copy()
    bt[1, :nb] = free
    after = oracle_mod.paged_decode(w.q, k2, v2, bt, w.context_lens, w.scale, "bf16")
    np.testing.assert_array_equal(after, before)


def test_swap_flags_ids_outside_either_pool(oracle_mod):
    a = np.arange(4 * 8, dtype=np.float32).reshape(4, 2, 1, 4)
    b = np.zeros((2, 2, 1, 4), np.float32)
    assert oracle_mod.swap_blocks(b, a, np.array([[3, 1], [0, 2], [4, 0]])) == 1
    np.testing.assert_array_equal(b[1], a[3])
    assert (b[0] == 0).all()


# ----------------------------------------------------------------------------------------
# fp8 (E4M3) KV blocks
# ----------------------------------------------------------------------------------------

def test_e4m3_values_match_torch(oracle_mod):
    """All 256 codes decode to torch's float8_e4m3fn values (NaN where torch has NaN)."""
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    np.testing.assert_array_equal(oracle_mod.e4m3_to_double(codes), ref)


def test_e4m3_rounding_matches_torch(oracle_mod):
    """Encoding rounds to nearest, ties to even, and saturates at 448 like torch's
    conversion of clamped values.  Catches: truncation, ties away from zero, overflow."""
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = oracle_mod.e4m3_to_double(codes)
    np.testing.assert_array_equal(oracle_mod.e4m3_from_double(vals), codes)   # round trip
    finite = np.sort(np.unique(vals))
    mids = (finite[1:] + finite[:-1]) / 2                                       # exact ties
    rng = np.random.default_rng(8)
    x = np.concatenate([mids, rng.standard_normal(4000) * 40, rng.standard_normal(500) * 1e-2,
                        [500.0, -1e4, 447.9, 449.0]]).astype(np.float32)
    ref = torch.from_numpy(np.clip(x, -448, 448)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(oracle_mod.e4m3_from_double(x.astype(np.float64)), ref)


def test_fp8_decode_equals_decode_of_dequantised_cache(oracle_mod):
    """With power-of-two scales the dequantised cache is exact in fp32, so the fp8 decode
    must equal the plain decode of that cache, and SDPA on it.  Catches: a scale applied
    to the wrong tensor, or twice."""
    w = _wl(dtype="bf16", lens=(1, 16, 37, 200), Hq=8, Hkv=2, D=64, bs=16, shuffle=False)
    ks, vs = 2.0 ** -4, 2.0 ** -3
    k8, v8 = synth.fp8_kv(w, ks, vs)
    out = oracle_mod.paged_decode_fp8kv(w.q, k8, v8, w.block_tables, w.context_lens, w.scale,
                                        ks, vs, "bf16")
    kf = (oracle_mod.e4m3_to_double(k8) * ks).astype(np.float32)
    vf = (oracle_mod.e4m3_to_double(v8) * vs).astype(np.float32)
    qf = synth.storage_to_f64(w.q, "bf16").astype(np.float32)
    ref = oracle_mod.paged_decode(qf, kf, vf, w.block_tables, w.context_lens, w.scale, "f32")
    np.testing.assert_array_equal(out, ref)
    NB, bs = kf.shape[:2]
    for s in range(w.num_seqs):
        start, L = int(w.block_tables[s, 0]) * bs, int(w.context_lens[s])
        K = torch.from_numpy(kf.reshape(NB * bs, 2, 64)[start:start + L].astype(np.float64))
        V = torch.from_numpy(vf.reshape(NB * bs, 2, 64)[start:start + L].astype(np.float64))
        qt = torch.from_numpy(qf[s].astype(np.float64))[:, None, :]
        sd = torch.nn.functional.scaled_dot_product_attention(
            qt, K.permute(1, 0, 2).repeat_interleave(4, 0), V.permute(1, 0, 2).repeat_interleave(4, 0),
            scale=w.scale)
        np.testing.assert_allclose(out[s], sd[:, 0].numpy(), rtol=1e-12, atol=1e-13)


def test_fp8_slot_write_quantises_like_torch(oracle_mod):
    """A new token's rows become the codes torch gives x / scale (fp32 division), in the
    slot's row.  Catches: multiplying by the scale, rounding before the division."""
    NB, bs, Hkv, D = 6, 16, 2, 32
    rng = np.random.default_rng(3)
    k_new = synth.to_storage(rng.standard_normal((5, Hkv, D)) * 3, "bf16")
    v_new = synth.to_storage(rng.standard_normal((5, Hkv, D)) * 3, "bf16")
    kc = np.zeros((NB, bs, Hkv, D), np.uint8)
    vc = np.zeros_like(kc)
    slots = np.array([0, 17, -1, 95, 40], np.int64)
    ks, vs = 0.0371, 0.05
    assert oracle_mod.kv_cache_write_fp8(k_new, v_new, kc, vc, slots, ks, vs, "bf16") == 0
    rows_k = kc.reshape(NB * bs, Hkv, D)
    rows_v = vc.reshape(NB * bs, Hkv, D)
    kx = synth.storage_to_f64(k_new, "bf16").astype(np.float32)
    vx = synth.storage_to_f64(v_new, "bf16").astype(np.float32)
    for i, sl in enumerate(slots):
        if sl < 0:
            continue
        np.testing.assert_array_equal(rows_k[sl], synth.e4m3_codes(kx[i], ks))
        np.testing.assert_array_equal(rows_v[sl], synth.e4m3_codes(vx[i], vs))
    assert (rows_k[[1, 2, 3]] == 0).all()


# ----------------------------------------------------------------------------------------
# chunked prefill ("Paged Attention: How vLLM Solves the KV Cache Memory Problem",
# section "Continuous Batching and Chunked Prefill")
# ----------------------------------------------------------------------------------------

def _pf(dtype="bf16", prior=(0, 3, 16, 40), chunk=(5, 1, 17, 9), Hq=4, Hkv=2, D=64, bs=16,
        shuffle=True, seed=21, scale=None, **kw):
    return synth.make_prefill_workload("pin-pf", seed=seed, dtype=dtype, prior_lens=list(prior),
                                       chunk_lens=list(chunk), num_q_heads=Hq, num_kv_heads=Hkv,
                                       head_dim=D, block_size=bs, shuffle=shuffle, scale=scale,
                                       **kw)


def _run_pf(oracle_mod, w, **kw):
    return oracle_mod.paged_prefill(w.chunk_q, w.k_cache, w.v_cache, w.block_tables,
                                    w.context_lens, w.query_start, w.scale, w.dtype, **kw)


@pytest.mark.parametrize("dtype,Hq,Hkv,D,bs", [
    ("f32", 4, 4, 64, 16), ("bf16", 8, 2, 128, 16), ("f16", 6, 3, 32, 32)])
def test_prefill_matches_causal_sdpa_on_unpaged_sequence(oracle_mod, dtype, Hq, Hkv, D, bs):
    """A chunk's rows equal causal attention over the prior context plus the chunk.

    Reference: torch scaled_dot_product_attention in float64 on the sequence's
    contiguous K/V rows (pool unshuffled) with an explicit mask: query i of an n-token
    chunk may see key j iff j <= L - n + i.  Catches: an off-by-one in the causal limit,
    queries placed at the start instead of the end of the context, a mask applied to
    the prior context, wrong query rows per sequence, wrong head mapping.
    """
    w = _pf(dtype=dtype, prior=(0, 7, bs, 2 * bs + 3), chunk=(bs + 2, 1, 5, 2 * bs),
            Hq=Hq, Hkv=Hkv, D=D, bs=bs, shuffle=False, scale=0.29)
    out = _run_pf(oracle_mod, w)
    G = Hq // Hkv
    q = _f64(w, w.chunk_q)
    for s in range(w.num_seqs):
        k, v = _dense_rows(w, s)
        L = int(w.context_lens[s])
        a, b = int(w.query_start[s]), int(w.query_start[s + 1])
        n = b - a
        kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(G, dim=0)  # [Hq, L, D]
        vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(G, dim=0)
        qt = torch.from_numpy(q[a:b]).permute(1, 0, 2)                          # [Hq, n, D]
        mask = torch.arange(L)[None, :] <= (L - n + torch.arange(n))[:, None]   # [n, L]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                               scale=w.scale)
        np.testing.assert_allclose(out[a:b], ref.permute(1, 0, 2).numpy(), rtol=1e-12,
                                   atol=1e-13)


def test_prefill_with_a_negative_scale_matches_sdpa(oracle_mod):
    """A negative scale (the GPU tests use one to reach the mma.sync prefill kernel): the
    rows still equal causal SDPA with that scale, here with 3 query heads per KV head.
    Catches: a scale sign dropped or taken as its magnitude, a GQA map that assumes a
    power-of-two group."""
    w = _pf(dtype="bf16", prior=(0, 9, 40), chunk=(5, 16, 3), Hq=9, Hkv=3, D=64, bs=16,
            shuffle=False, scale=-0.21)
    out = _run_pf(oracle_mod, w)
    G = w.num_q_heads // w.num_kv_heads
    q = _f64(w, w.chunk_q)
    for s in range(w.num_seqs):
        k, v = _dense_rows(w, s)
        L = int(w.context_lens[s])
        a, b = int(w.query_start[s]), int(w.query_start[s + 1])
        n = b - a
        kt = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(G, dim=0)
        vt = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(G, dim=0)
        qt = torch.from_numpy(q[a:b]).permute(1, 0, 2)
        mask = torch.arange(L)[None, :] <= (L - n + torch.arange(n))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask,
                                                               scale=w.scale)
        np.testing.assert_allclose(out[a:b], ref.permute(1, 0, 2).numpy(), rtol=1e-12,
                                   atol=1e-13)


def test_prefill_row_equals_decode_of_truncated_context(oracle_mod):
    """Row i of a chunk is a decode query over the first L - n + i + 1 tokens.

    Reference: the decode oracle (its own pins above) run once per chunk row with the
    context cut at the row's position, on the shuffled pool.  Catches: causal limit
    errors, block-table walks that differ between the two paths, and results that
    depend on tokens after the query.
    """
    w = _pf(prior=(0, 9, 33), chunk=(4, 12, 3), Hq=4, Hkv=2, D=64, bs=16, pool_slack=0.3)
    out = _run_pf(oracle_mod, w)
    for s in range(w.num_seqs):
        L = int(w.context_lens[s])
        a, b = int(w.query_start[s]), int(w.query_start[s + 1])
        n = b - a
        for i in range(n):
            ref = oracle_mod.paged_decode(w.chunk_q[a + i][None], w.k_cache, w.v_cache,
                                          w.block_tables[s:s + 1],
                                          np.array([L - n + i + 1], np.int32), w.scale, w.dtype)
            np.testing.assert_array_equal(out[a + i], ref[0])


def test_prefill_of_one_token_chunks_is_decode(oracle_mod):
    """With one query token per sequence the prefill oracle is the decode oracle.

    Catches: treating the chunk as the first rather than the last n tokens, and any
    special-casing of n = 1.
    """
    w = _pf(prior=(0, 15, 16, 63), chunk=(1, 1, 1, 1), Hq=8, Hkv=2, D=64, bs=16)
    out = _run_pf(oracle_mod, w)
    ref = oracle_mod.paged_decode(w.chunk_q, w.k_cache, w.v_cache, w.block_tables,
                                  w.context_lens, w.scale, w.dtype)
    np.testing.assert_array_equal(out, ref)


def test_prefill_first_chunk_token_of_an_empty_context_returns_its_value(oracle_mod):
    """The first token of a prompt's first chunk sees only itself: its output is V_0.

    Catches: attending a token past the query, normalisation errors.
    """
    w = _pf(dtype="f32", prior=(0, 0), chunk=(3, 1), Hq=2, Hkv=1, D=32, bs=16)
    out = _run_pf(oracle_mod, w)
    for s in range(w.num_seqs):
        a = int(w.query_start[s])
        phys = int(w.block_tables[s, 0])
        v0 = w.v_cache[phys, 0, 0].astype(np.float64)
        for h in range(2):
            np.testing.assert_array_equal(out[a, h], v0)


def test_prefill_rejects_a_chunk_longer_than_its_context(oracle_mod):
    w = _pf(prior=(0, 4), chunk=(3, 2), Hq=2, Hkv=1, D=32, bs=16)
    qs = w.query_start.copy()
    cl = w.context_lens.copy()
    cl[1] = 1  # the second chunk has 2 rows but the context only 1 token
    with pytest.raises(ValueError):
        oracle_mod.paged_prefill(w.chunk_q, w.k_cache, w.v_cache, w.block_tables, cl, qs,
                                 w.scale, w.dtype)
