"""The decode entry point for callers that cannot allocate device memory.

paged_attn_decode_noalloc serves callers with no way to hand the library scratch memory
(a host program that owns the device's whole memory budget, or a hot path on which
nothing may be allocated) from a fixed scratch array built into the library.  These
tests call it through the C ABI and compare it with the fp64 oracle and with
paged_attn_decode, which takes its scratch from the caller, and check that its calls
allocate no device memory.  The file is named to be collected last.
"""
import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-2, 1e-2

# two batches whose contexts span several partitions (so the scratch holds partials):
# (seed, context lengths, query heads, KV heads, partition size)
BATCHES = [(71, [3000, 17, 900, 4096, 1], 32, 8, 256),
           (72, [1500, 2600, 64], 16, 2, 512)]


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_cache_315_gb300 as m

    m.build()
    oracle.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    m.pkv_device_error()
    return m


def _batch(seed, lens, Hq, Hkv, part):
    w = synth.make_workload("noalloc", seed=seed, dtype="bf16", context_lens=lens,
                            num_q_heads=Hq, num_kv_heads=Hkv, head_dim=128, block_size=16,
                            partition_size=part, key_outlier_frac=0.01)
    return w, synth.to_torch(w, "cuda")


def _within(got, want):
    return np.isfinite(got).all() and (np.abs(got - want) <= ATOL + RTOL * np.abs(want)).all()


def test_noalloc_matches_oracle_and_the_workspace_entry_point_on_two_calls_in_a_row(pkv):
    # two different batches back to back: the second call finds the first call's data
    # still in the shared scratch and must not be affected by it
    for seed, lens, Hq, Hkv, part in BATCHES:
        w, t = _batch(seed, lens, Hq, Hkv, part)
        ref = torch.empty_like(t["q"])
        pkv.paged_attn_decode(ref, t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                              t["context_lens"], w.scale, partition_size=part)
        out = torch.full_like(t["q"], float("nan"))
        pkv.paged_attn_decode_noalloc(out, t["q"], t["k_cache"], t["v_cache"], t["block_tables"],
                                      t["context_lens"], w.scale, partition_size=part)
        assert pkv.pkv_device_error() == 0
        got = out.float().cpu().numpy().astype(np.float64)
        want = oracle.paged_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                   w.scale, w.dtype)
        assert _within(got, want), f"batch {seed}: no-alloc decode differs from the oracle"
        assert _within(got, ref.float().cpu().numpy().astype(np.float64)), \
            f"batch {seed}: no-alloc decode differs from paged_attn_decode"


def test_noalloc_calls_allocate_no_device_memory(pkv):
    # after one call of each shape (which loads the kernels they run), further calls of
    # both shapes leave the device's free memory and the caching allocator untouched
    runs = []
    for seed, lens, Hq, Hkv, part in BATCHES:
        w, t = _batch(seed, lens, Hq, Hkv, part)
        runs.append((w, t, part, torch.empty_like(t["q"])))

    def call_all():
        for w, t, part, out in runs:
            pkv.paged_attn_decode_noalloc(out, t["q"], t["k_cache"], t["v_cache"],
                                          t["block_tables"], t["context_lens"], w.scale,
                                          partition_size=part)

    call_all()
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    stats0 = torch.cuda.memory_stats()
    for _ in range(5):
        call_all()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    stats1 = torch.cuda.memory_stats()
    assert pkv.pkv_device_error() == 0
    assert free1 == free0
    for key in ("allocation.all.allocated", "segment.all.allocated", "reserved_bytes.all.current"):
        assert stats1.get(key, 0) == stats0.get(key, 0), key
    # and the results are still right
    for w, t, part, out in runs:
        want = oracle.paged_decode(w.q, w.k_cache, w.v_cache, w.block_tables, w.context_lens,
                                   w.scale, w.dtype)
        assert _within(out.float().cpu().numpy().astype(np.float64), want)


def test_noalloc_rejects_a_problem_larger_than_its_scratch(pkv):
    # 4096 sequences x 64 query heads x 16 partitions of partials do not fit in 32 MiB;
    # the call is refused before any device work, so the dummy tensors are never read
    B, Hq, Hkv, D, bs, MB = 4096, 64, 8, 128, 16, 512
    need = pkv.paged_attn_decode_workspace_size(B, Hq, Hkv, D, bs, MB, 512)
    assert need > 32 << 20
    lib = pkv.load()
    dummy = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    p = dummy.data_ptr()
    rc = lib.paged_attn_decode_noalloc(p, p, p, p, p, p, B, Hq, Hkv, D, bs, MB, 64, 0.1,
                                       pkv.PKV_BF16, 512, None)
    assert rc == pkv.PKV_ESCRATCH
    assert "scratch" in pkv.pkv_strerror(rc)
