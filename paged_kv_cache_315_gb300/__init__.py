"""GB300-native paged KV-cache decode attention.

A thin Python front end to ``libpagedkv.so`` (hand-written CUDA for sm_103a):

* ``paged_attn_decode``  -- single-token decode attention through per-sequence block
  tables, GQA heads batched per KV head, split-context partitions merged by
  log-sum-exp in the same launch;
* ``kv_cache_write``     -- slot-mapped write of new tokens' keys and values;
* ``kv_copy_blocks``     -- whole-block copies for copy-on-write;
* ``kv_swap_blocks``     -- whole-block copies between pools (device / pinned host).

The C ABI is declared in ``include/pagedkv.h``.  PyTorch is used only for device
memory and streams.
"""
from ._binding import (  # noqa: F401
    PKV_BF16,
    PKV_DERR_BLOCK_ID,
    PKV_DERR_CONTEXT,
    PKV_DERR_PAIR,
    PKV_DERR_SLOT,
    PKV_DERR_TIMEOUT,
    PKV_ENODEVMEM,
    PKV_ESCRATCH,
    PKV_F16,
    PKV_F32,
    PagedKVError,
    kv_cache_write,
    kv_cache_write_fp8,
    kv_copy_blocks,
    kv_swap_blocks,
    load,
    paged_attn_decode,
    paged_attn_decode_fp8,
    paged_attn_decode_fp8_partition_tokens,
    paged_attn_decode_fp8_workspace_size,
    paged_attn_decode_noalloc,
    paged_attn_decode_partition_tokens,
    paged_attn_prefill,
    paged_attn_decode_shared_prefix,
    paged_attn_decode_shared_prefix_workspace_size,
    paged_attn_decode_workspace_size,
    pkv_device_error,
    pkv_selftest_bounded_wait,
    pkv_strerror,
    pkv_version,
    workspace_for,
)
from .build import LIB_PATH, build  # noqa: F401
