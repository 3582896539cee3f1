"""Chunked-prefill attention on the GPU (through the C ABI) against the fp64 oracle.

Acceptance: every output within |gpu - oracle| <= 2e-2 + 1e-2 |oracle| (bf16 / fp16).
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


def gpu_prefill(pkv, w, t, max_query_len=None, context_lens=None, block_tables=None):
    out = torch.full_like(t["chunk_q"], float("nan"))
    n = np.diff(w.query_start)
    pkv.paged_attn_prefill(out, t["chunk_q"], t["k_cache"], t["v_cache"],
                           t["block_tables"] if block_tables is None else block_tables,
                           t["context_lens"] if context_lens is None else context_lens,
                           t["query_start"],
                           int(n.max()) if max_query_len is None else max_query_len, w.scale)
    return out


def oracle_prefill(w):
    return oracle.paged_prefill(w.chunk_q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                w.query_start, w.scale, w.dtype)


# prior contexts and chunk lengths cross tile (64 keys), block and 64-row edges
PRIOR = [0, 3, 16, 100, 700, 0, 63]
CHUNK = [1, 17, 64, 5, 130, 70, 65]

SHAPES = [
    # dtype, Hq, Hkv, D, bs     (tcgen05 for head_dim 64 and 128)
    ("bf16", 4, 4, 128, 16),
    ("bf16", 8, 1, 128, 16),
    ("bf16", 64, 8, 128, 16),
    ("f16", 16, 2, 128, 32),
    ("bf16", 16, 4, 128, 64),
    ("bf16", 32, 2, 128, 16),
    ("bf16", 12, 4, 128, 16),    # 3 heads per KV head: a 128-row tile ends inside a token
    ("bf16", 40, 2, 128, 32),    # 20 heads per KV head
    ("f16", 30, 5, 128, 16),     # 6 heads per KV head
    ("bf16", 160, 1, 128, 64),   # 160 heads per KV head: one token spans two tiles
    ("bf16", 12, 4, 64, 64),
    ("bf16", 6, 3, 64, 16),
    ("f16", 2, 2, 64, 32),
]


@pytest.mark.parametrize("dtype,Hq,Hkv,D,bs", SHAPES)
def test_prefill_matches_oracle(pkv, dtype, Hq, Hkv, D, bs):
    w = synth.make_prefill_workload("pf", seed=40 + Hq + D + bs, dtype=dtype, prior_lens=PRIOR,
                                    chunk_lens=CHUNK, num_q_heads=Hq, num_kv_heads=Hkv,
                                    head_dim=D, block_size=bs, key_outlier_frac=0.02)
    t = synth.to_torch(w, "cuda")
    out = gpu_prefill(pkv, w, t)
    assert pkv.pkv_device_error() == 0
    assert_close(out.float().cpu().numpy(), oracle_prefill(w),
                 f"{dtype} Hq{Hq} Hkv{Hkv} D{D} bs{bs}")


@pytest.mark.parametrize("D,mult,Hq,Hkv", [(64, -1.0, 8, 2), (128, -1.0, 8, 2),
                                            (128, -2.5, 12, 4), (128, 0.0, 8, 2),
                                            (64, 0.0, 6, 3), (128, 0.0, 12, 4)])
def test_prefill_non_positive_scale_matches_oracle(pkv, D, mult, Hq, Hkv):
    # a negative scale runs as (-q) . k times |scale| (query rows staged with flipped
    # signs); a zero scale weighs every attended key 1, and keys past a row's causal limit
    # must still weigh 0
    w = synth.make_prefill_workload("pfn", seed=16 + D + Hq, dtype="bf16",
                                    prior_lens=[0, 40, 130], chunk_lens=[17, 64, 9],
                                    num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=16)
    w.scale = mult * w.scale
    t = synth.to_torch(w, "cuda")
    out = gpu_prefill(pkv, w, t)
    assert pkv.pkv_device_error() == 0
    assert_close(out.float().cpu().numpy(), oracle_prefill(w), f"scale {w.scale} D{D} Hq{Hq}")


def test_prefill_of_one_token_chunks_matches_decode_oracle(pkv):
    w = synth.make_prefill_workload("pf1", seed=9, dtype="bf16", prior_lens=[0, 15, 16, 500, 31],
                                    chunk_lens=[1] * 5, num_q_heads=16, num_kv_heads=4,
                                    head_dim=128, block_size=16)
    t = synth.to_torch(w, "cuda")
    out = gpu_prefill(pkv, w, t)
    assert pkv.pkv_device_error() == 0
    ref = oracle.paged_decode(w.chunk_q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                              w.scale, w.dtype)
    assert_close(out.float().cpu().numpy(), ref, "one-token chunks")


def test_prefill_never_reads_dead_slots_or_table_tail(pkv):
    w = synth.make_prefill_workload("pfp", seed=12, dtype="bf16", prior_lens=[5, 40, 0],
                                    chunk_lens=[20, 9, 33], num_q_heads=8, num_kv_heads=2,
                                    head_dim=128, block_size=32, pool_slack=0.5,
                                    table_pad=2 ** 30)
    synth.poison_unused(w)
    t = synth.to_torch(w, "cuda")
    out = gpu_prefill(pkv, w, t)
    assert pkv.pkv_device_error() == 0
    assert_close(out.float().cpu().numpy(), oracle_prefill(w), "poisoned")


def test_prefill_rows_of_other_sequences_are_left_alone(pkv):
    # a larger max_query_len than any chunk only adds empty CTAs
    w = synth.make_prefill_workload("pfm", seed=13, dtype="bf16", prior_lens=[7, 0],
                                    chunk_lens=[3, 40], num_q_heads=4, num_kv_heads=1,
                                    head_dim=64, block_size=16)
    t = synth.to_torch(w, "cuda")
    out = gpu_prefill(pkv, w, t, max_query_len=300)
    assert pkv.pkv_device_error() == 0
    assert_close(out.float().cpu().numpy(), oracle_prefill(w), "max_query_len 300")


def test_prefill_reports_bad_chunks_and_block_ids(pkv):
    w = synth.make_prefill_workload("pfe", seed=14, dtype="bf16", prior_lens=[4, 30],
                                    chunk_lens=[6, 10], num_q_heads=4, num_kv_heads=2,
                                    head_dim=128, block_size=16)
    t = synth.to_torch(w, "cuda")
    ref = oracle_prefill(w)
    # a chunk longer than max_query_len: that sequence's rows are not written
    out = gpu_prefill(pkv, w, t, max_query_len=8)
    assert pkv.pkv_device_error() == pkv.PKV_DERR_CONTEXT
    o = out.float().cpu().numpy()
    assert np.isnan(o[6:16]).all()
    assert_close(o[:6], ref[:6], "the valid sequence")
    # a context shorter than its chunk
    cl = t["context_lens"].clone()
    cl[0] = 3
    gpu_prefill(pkv, w, t, context_lens=cl)
    assert pkv.pkv_device_error() == pkv.PKV_DERR_CONTEXT
    # an out-of-range live block id reads as zeros and is reported
    bt = t["block_tables"].clone()
    bt[1, 1] = w.num_blocks + 5
    gpu_prefill(pkv, w, t, block_tables=bt)
    assert pkv.pkv_device_error() == pkv.PKV_DERR_BLOCK_ID
    # the context is still usable
    out = gpu_prefill(pkv, w, t)
    assert pkv.pkv_device_error() == 0
    assert_close(out.float().cpu().numpy(), ref, "after errors")


@pytest.mark.parametrize("head_dim", [128, 64])
def test_prefill_batch_full_size_sampled_rows(pkv, head_dim):
    """The chunked-prefill batch at full size (bench.py --op prefill [--head-dim 64]), in
    the launch bench.py times.

    Sampled rows are checked one by one: row i of a chunk is a decode query over the
    first L - n + i + 1 tokens (a pinned property of the oracle).
    """
    w = synth.prefill_workload(head_dim=head_dim)
    t = synth.to_torch(w, "cuda")
    out = gpu_prefill(pkv, w, t).float().cpu().numpy()
    assert pkv.pkv_device_error() == 0
    assert np.isfinite(out).all()
    rng = np.random.default_rng(3)
    for s in range(w.num_seqs):
        a, b = int(w.query_start[s]), int(w.query_start[s + 1])
        n, L = b - a, int(w.context_lens[s])
        rows = sorted({0, n - 1, *rng.integers(0, n, size=2).tolist()})
        for i in rows:
            ref = oracle.paged_decode(w.chunk_q[a + i][None], w.k_cache, w.v_cache,
                                      w.block_tables[s:s + 1],
                                      np.array([L - n + i + 1], np.int32), w.scale, w.dtype)
            assert_close(out[a + i], ref[0], f"seq {s} row {i}")
