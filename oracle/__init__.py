"""CPU oracle for paged decode and chunked-prefill attention, slot writes and block copies.

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference legs may import this package. The product
path (the CUDA library and its Python binding) never imports it, and the two
share no code.
"""
from .oracle import (  # noqa: F401
    DTYPE_CODES,
    build,
    copy_blocks,
    e4m3_from_double,
    e4m3_to_double,
    kv_cache_write,
    kv_cache_write_fp8,
    locate,
    max_threads,
    num_blocks,
    paged_decode,
    paged_decode_fp8kv,
    paged_decode_partitioned,
    paged_prefill,
    slot,
    swap_blocks,
)
