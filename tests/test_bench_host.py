"""Host-side pieces of bench.py that need no GPU: the byte counts of the cache operations
reported beside the decode, and the name of the decode kernel each batch runs."""
import numpy as np

import bench
import synth


def test_cache_op_bytes_are_reads_plus_writes():
    w = bench.bench_workload(4)            # copy-on-write pairs + one slot write per suffix token
    t = synth.to_torch(w, "cpu")
    ops = bench.cache_ops(t, w, False, True, copy_ms=0.01, write_ms=0.002)
    pairs, n = w.copy_pairs.shape[0], w.k_new.shape[0]
    block = w.block_size * w.num_kv_heads * w.head_dim * 2          # bf16 block, one tensor
    # each pair reads and writes one block of K and one of V, and its 16-byte id pair is read
    # by both calls
    assert ops["kv_copy_blocks"]["bytes"] == 2 * pairs * (2 * block + 16)
    row = w.num_kv_heads * w.head_dim
    assert ops["kv_cache_write"]["bytes"] == 2 * n * row * (2 + 2) + 8 * n
    assert np.isclose(ops["kv_cache_write"]["GB/s"], ops["kv_cache_write"]["bytes"] / 2e-6 / 1e9,
                      rtol=1e-3)
    # E4M3 cache: one byte per cached element, bf16 inputs
    ops8 = bench.cache_ops(t, w, True, True, copy_ms=0.01, write_ms=0.002)
    assert ops8["kv_copy_blocks"]["bytes"] == 2 * pairs * (2 * block // 2 + 16)
    assert ops8["kv_cache_write_fp8"]["bytes"] == 2 * n * row * (2 + 1) + 8 * n


def test_batches_without_copies_report_only_the_slot_write():
    w = bench.bench_workload(3)
    t = synth.to_torch(w, "cpu")
    assert "copy_pairs" not in t
    ops = bench.cache_ops(t, w, False, False, copy_ms=0.0, write_ms=0.001)
    assert list(ops) == ["kv_cache_write"]
    assert ops["kv_cache_write"]["tokens"] == w.num_seqs


def test_decode_kernel_names_follow_the_launcher():
    # 13B-like MHA: one query head per KV head; 70B-like GQA: 8 per KV head
    assert bench.decode_kernel_name(bench.bench_workload(2), False) == "decode_tc_kernel"
    assert bench.decode_kernel_name(bench.bench_workload(3), False) == "decode_tcg_kernel"
    assert bench.decode_kernel_name(bench.bench_workload(3), True) == "decode_fp8g_kernel"
    # the fp32 correctness batch runs on CUDA cores
    assert bench.decode_kernel_name(bench.bench_workload(1), False) == "decode_simt_kernel"
