"""ctypes front end of the fp64 C oracle in ``pagedkv_oracle.c``.

TEST INFRASTRUCTURE: only the tests, the smoke check and the benchmark's
CPU-baseline / reference legs use it; the product path never does.

Every function here only marshals numpy arrays into the C routines; all the
arithmetic is in the C file, which documents what each routine computes and
which passage of the PagedAttention pages it follows.

Element types are named ``"f32"``, ``"bf16"`` and ``"f16"``. For the 16-bit
types the arrays hold the raw bit patterns (``numpy.uint16``); ``f32`` arrays are
``numpy.float32``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pagedkv_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD_DIR, "liboracle.so")

DTYPE_CODES = {"f32": 0, "bf16": 1, "f16": 2}
_NP_STORAGE = {"f32": np.float32, "bf16": np.uint16, "f16": np.uint16}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, dbl, sz = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_size_t
        lib.pkvo_paged_decode.argtypes = [P, P, P, P, i32, P, P, i32, i32, i32, i32, i32, i32,
                                          i32, dbl, i32]
        lib.pkvo_paged_decode.restype = i32
        lib.pkvo_paged_decode_partitioned.argtypes = [P, P, P, P, i32, P, P, i32, i32, i32, i32,
                                                      i32, i32, i32, dbl, i32, i32]
        lib.pkvo_paged_decode_partitioned.restype = i32
        lib.pkvo_paged_prefill.argtypes = [P, P, P, P, i32, P, P, P, i32, i32, i32, i32, i32,
                                           i32, i32, i32, dbl, i32]
        lib.pkvo_paged_prefill.restype = i32
        lib.pkvo_kv_cache_write.argtypes = [P, P, P, P, P, i32, sz, i32, i32]
        lib.pkvo_kv_cache_write.restype = i32
        lib.pkvo_copy_blocks.argtypes = [P, P, i32, sz, i32]
        lib.pkvo_copy_blocks.restype = i32
        lib.pkvo_swap_blocks.argtypes = [P, P, P, i32, sz, i32, i32]
        lib.pkvo_swap_blocks.restype = i32
        lib.pkvo_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.pkvo_e4m3_to_double.restype = dbl
        lib.pkvo_e4m3_from_double.argtypes = [dbl]
        lib.pkvo_e4m3_from_double.restype = ctypes.c_uint8
        lib.pkvo_paged_decode_fp8kv.argtypes = [P, P, P, P, i32, P, P, i32, i32, i32, i32, i32,
                                                i32, i32, dbl, dbl, dbl, i32]
        lib.pkvo_paged_decode_fp8kv.restype = i32
        lib.pkvo_kv_cache_write_fp8.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32,
                                                ctypes.c_float, ctypes.c_float]
        lib.pkvo_kv_cache_write_fp8.restype = i32
        lib.pkvo_num_blocks.argtypes = [i64, i32]
        lib.pkvo_num_blocks.restype = i64
        lib.pkvo_slot.argtypes = [P, i64, i32]
        lib.pkvo_slot.restype = i64
        lib.pkvo_locate.argtypes = [P, i64, i32, P, P]
        lib.pkvo_locate.restype = None
        lib.pkvo_max_threads.argtypes = []
        lib.pkvo_max_threads.restype = i32
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _check_storage(name: str, a: np.ndarray, dtype: str) -> np.ndarray:
    want = _NP_STORAGE[dtype]
    if a.dtype != want:
        raise TypeError(f"{name}: expected {np.dtype(want).name} storage for {dtype}, got {a.dtype}")
    return np.ascontiguousarray(a)


def max_threads() -> int:
    """Threads the oracle's OpenMP loops use by default."""
    return int(_load().pkvo_max_threads())


def _decode_args(q, k_cache, v_cache, block_tables, context_lens, dtype):
    if dtype not in DTYPE_CODES:
        raise ValueError(f"unknown dtype {dtype!r}")
    q = _check_storage("q", q, dtype)
    k_cache = _check_storage("k_cache", k_cache, dtype)
    v_cache = _check_storage("v_cache", v_cache, dtype)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    if q.ndim != 3 or k_cache.ndim != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("q must be [B, Hq, D]; caches [NB, bs, Hkv, D] of equal shape")
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    if D2 != D or bt.ndim != 2 or bt.shape[0] != B or cl.shape != (B,):
        raise ValueError("shape mismatch between q, caches, block_tables and context_lens")
    return q, k_cache, v_cache, bt, cl, (B, Hq, Hkv, D, bs, bt.shape[1], NB)


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale, dtype,
                 num_threads: int = 0) -> np.ndarray:
    """fp64 paged decode attention by its definition; returns ``[B, Hq, D]`` float64."""
    q, k_cache, v_cache, bt, cl, (B, Hq, Hkv, D, bs, MB, NB) = _decode_args(
        q, k_cache, v_cache, block_tables, context_lens, dtype)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    rc = _load().pkvo_paged_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                   DTYPE_CODES[dtype], _ptr(bt), _ptr(cl), B, Hq, Hkv, D, bs,
                                   MB, NB, float(scale), int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle paged_decode rejected its inputs (code {rc})")
    return out


def paged_decode_partitioned(q, k_cache, v_cache, block_tables, context_lens, scale, dtype,
                             partition_size: int, num_threads: int = 0) -> np.ndarray:
    """fp64 split-context form: per-partition partials merged by log-sum-exp."""
    q, k_cache, v_cache, bt, cl, (B, Hq, Hkv, D, bs, MB, NB) = _decode_args(
        q, k_cache, v_cache, block_tables, context_lens, dtype)
    out = np.zeros((B, Hq, D), dtype=np.float64)
    rc = _load().pkvo_paged_decode_partitioned(
        _ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), DTYPE_CODES[dtype], _ptr(bt), _ptr(cl),
        B, Hq, Hkv, D, bs, MB, NB, float(scale), int(partition_size), int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle paged_decode_partitioned rejected its inputs (code {rc})")
    return out


def paged_prefill(q, k_cache, v_cache, block_tables, context_lens, query_start, scale, dtype,
                  num_threads: int = 0) -> np.ndarray:
    """fp64 chunked-prefill attention by its definition; returns ``[T, Hq, D]`` float64.

    ``q`` is ``[T, Hq, D]``; sequence s owns query rows ``query_start[s] ..
    query_start[s+1]-1``, the last ``n`` positions of its ``context_lens[s]`` cached
    tokens, and each row attends causally (positions ``0 .. L-n+i``).
    """
    q = _check_storage("q", q, dtype)
    k_cache = _check_storage("k_cache", k_cache, dtype)
    v_cache = _check_storage("v_cache", v_cache, dtype)
    T, Hq, D = q.shape
    NB, bs, Hkv, Dk = k_cache.shape
    if Dk != D or v_cache.shape != k_cache.shape:
        raise ValueError("q, k_cache and v_cache disagree on head_dim or shape")
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    qs = _c(query_start, np.int32)
    B = cl.shape[0]
    if bt.ndim != 2 or bt.shape[0] != B or qs.shape != (B + 1,):
        raise ValueError("block_tables / query_start do not match context_lens")
    out = np.zeros((T, Hq, D), dtype=np.float64)
    rc = _load().pkvo_paged_prefill(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                    DTYPE_CODES[dtype], _ptr(bt), _ptr(cl), _ptr(qs), B, T, Hq,
                                    Hkv, D, bs, bt.shape[1], NB, float(scale), int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle paged_prefill rejected its inputs (code {rc})")
    return out


def kv_cache_write(k, v, k_cache, v_cache, slot_mapping) -> int:
    """Scatter token rows ``k[i]``, ``v[i]`` into cache row ``slot_mapping[i]`` in place.

    ``k``/``v`` are ``[N, Hkv, D]``; caches ``[NB, bs, Hkv, D]`` (same storage dtype).
    Returns 0, or 1 when an out-of-range slot was skipped.
    """
    if not (k_cache.flags.c_contiguous and v_cache.flags.c_contiguous):
        raise ValueError("caches must be C-contiguous (written in place)")
    k = np.ascontiguousarray(k)
    v = np.ascontiguousarray(v)
    sm = _c(slot_mapping, np.int64)
    NB, bs = k_cache.shape[0], k_cache.shape[1]
    row_bytes = k_cache[0, 0].nbytes
    if k.dtype != k_cache.dtype or v.dtype != v_cache.dtype or k[0].nbytes != row_bytes:
        raise ValueError("token rows must match the cache's row type and size")
    rc = _load().pkvo_kv_cache_write(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(sm),
                                     int(sm.shape[0]), row_bytes, NB, bs)
    if rc < 0:
        raise ValueError(f"oracle kv_cache_write rejected its inputs (code {rc})")
    return int(rc)


def copy_blocks(cache, src_dst_pairs) -> int:
    """Copy whole physical blocks ``cache[src] -> cache[dst]`` in place, pair by pair.

    Returns 0, or 1 when a pair with an out-of-range id was skipped.
    """
    if not cache.flags.c_contiguous:
        raise ValueError("cache must be C-contiguous (written in place)")
    pairs = _c(src_dst_pairs, np.int64).reshape(-1, 2)
    NB = cache.shape[0]
    block_bytes = cache[0].nbytes
    rc = _load().pkvo_copy_blocks(_ptr(cache), _ptr(pairs), int(pairs.shape[0]), block_bytes, NB)
    if rc < 0:
        raise ValueError(f"oracle copy_blocks rejected its inputs (code {rc})")
    return int(rc)


def swap_blocks(dst_cache, src_cache, src_dst_pairs) -> int:
    """Copy whole blocks ``src_cache[src] -> dst_cache[dst]`` (two pools) in place.

    Returns 0, or 1 when a pair with an out-of-range id was skipped.
    """
    if not dst_cache.flags.c_contiguous:
        raise ValueError("dst_cache must be C-contiguous (written in place)")
    src_cache = np.ascontiguousarray(src_cache)
    if dst_cache[0].nbytes != src_cache[0].nbytes or dst_cache.dtype != src_cache.dtype:
        raise ValueError("pools must have the same block size and element type")
    pairs = _c(src_dst_pairs, np.int64).reshape(-1, 2)
    rc = _load().pkvo_swap_blocks(_ptr(dst_cache), _ptr(src_cache), _ptr(pairs), int(pairs.shape[0]),
                                  dst_cache[0].nbytes, dst_cache.shape[0], src_cache.shape[0])
    if rc < 0:
        raise ValueError(f"oracle swap_blocks rejected its inputs (code {rc})")
    return int(rc)


def e4m3_to_double(codes) -> np.ndarray:
    """Values of E4M3 codes (uint8), exactly, as float64."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.vectorize(lambda x: lib.pkvo_e4m3_to_double(int(x)), otypes=[np.float64])(c)


def e4m3_from_double(x) -> np.ndarray:
    """Nearest E4M3 codes (ties to even, saturating at +-448) of float64 values."""
    lib = _load()
    a = np.asarray(x, dtype=np.float64)
    return np.vectorize(lambda v: lib.pkvo_e4m3_from_double(float(v)), otypes=[np.uint8])(a)


def paged_decode_fp8kv(q, k_cache, v_cache, block_tables, context_lens, scale, k_scale, v_scale,
                       q_dtype, num_threads: int = 0) -> np.ndarray:
    """fp64 decode over E4M3 caches (uint8 codes); q in ``q_dtype`` storage."""
    q = _check_storage("q", q, q_dtype)
    k_cache = np.ascontiguousarray(k_cache, dtype=np.uint8)
    v_cache = np.ascontiguousarray(v_cache, dtype=np.uint8)
    bt = _c(block_tables, np.int32)
    cl = _c(context_lens, np.int32)
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    if D2 != D or k_cache.shape != v_cache.shape or bt.shape[0] != B or cl.shape != (B,):
        raise ValueError("shape mismatch")
    out = np.zeros((B, Hq, D), dtype=np.float64)
    rc = _load().pkvo_paged_decode_fp8kv(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                         DTYPE_CODES[q_dtype], _ptr(bt), _ptr(cl), B, Hq, Hkv, D,
                                         bs, bt.shape[1], NB, float(scale), float(k_scale),
                                         float(v_scale), int(num_threads))
    if rc != 0:
        raise ValueError(f"oracle paged_decode_fp8kv rejected its inputs (code {rc})")
    return out


def kv_cache_write_fp8(k, v, k_cache, v_cache, slot_mapping, k_scale, v_scale, dtype) -> int:
    """Quantise token rows k[i], v[i] ([N, Hkv, D] in ``dtype`` storage) into the E4M3
    caches (uint8 [NB, bs, Hkv, D], written in place) at row slot_mapping[i]."""
    if not (k_cache.flags.c_contiguous and v_cache.flags.c_contiguous):
        raise ValueError("caches must be C-contiguous (written in place)")
    k = _check_storage("k", k, dtype)
    v = _check_storage("v", v, dtype)
    sm = _c(slot_mapping, np.int64)
    NB, bs = k_cache.shape[0], k_cache.shape[1]
    row = int(np.prod(k_cache.shape[2:]))
    if k[0].size != row:
        raise ValueError("token rows must match the cache rows")
    rc = _load().pkvo_kv_cache_write_fp8(_ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(sm),
                                         int(sm.shape[0]), row, DTYPE_CODES[dtype], NB, bs,
                                         float(k_scale), float(v_scale))
    if rc < 0:
        raise ValueError(f"oracle kv_cache_write_fp8 rejected its inputs (code {rc})")
    return int(rc)


def num_blocks(num_tokens: int, block_size: int) -> int:
    """Blocks a sequence of ``num_tokens`` tokens occupies."""
    return int(_load().pkvo_num_blocks(int(num_tokens), int(block_size)))


def locate(block_table_row, pos: int, block_size: int) -> tuple[int, int]:
    """(physical block, in-block offset) of logical position ``pos``."""
    row = _c(block_table_row, np.int32)
    phys = np.zeros(1, np.int32)
    off = np.zeros(1, np.int32)
    _load().pkvo_locate(_ptr(row), int(pos), int(block_size), _ptr(phys), _ptr(off))
    return int(phys[0]), int(off[0])


def slot(block_table_row, pos: int, block_size: int) -> int:
    """Cache slot (physical block * block_size + offset) of logical position ``pos``."""
    row = _c(block_table_row, np.int32)
    return int(_load().pkvo_slot(_ptr(row), int(pos), int(block_size)))
