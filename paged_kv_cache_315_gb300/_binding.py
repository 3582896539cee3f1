"""ctypes binding of libpagedkv (argument marshalling only).

Every function passes device pointers of torch tensors, their sizes and the current
CUDA stream to the C entry point of the same name; all the work happens in the
library's CUDA kernels.  There is no fallback: if the library is not built, or a
tensor is not on a CUDA device, the call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB_PATH

PKV_F32, PKV_BF16, PKV_F16 = 0, 1, 2
_DTYPES = {torch.float32: PKV_F32, torch.bfloat16: PKV_BF16, torch.float16: PKV_F16}

PKV_DERR_BLOCK_ID = 1
PKV_DERR_SLOT = 2
PKV_DERR_PAIR = 4
PKV_DERR_CONTEXT = 8
PKV_DERR_TIMEOUT = 16
PKV_ESCRATCH = -5
PKV_ENODEVMEM = -6

_lock = threading.Lock()
_lib = None
_workspaces: dict = {}


class PagedKVError(RuntimeError):
    """A libpagedkv entry point returned an error code."""

    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed: {pkv_strerror(code)} (code {code})")
        self.code = code


def load() -> ctypes.CDLL:
    """Load libpagedkv.so from the package's build folder (raises if absent)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libpagedkv.so is not built ({LIB_PATH}); run "
                "`python -m paged_kv_cache_315_gb300.build` first")
        lib = ctypes.CDLL(LIB_PATH)
        P, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
        lib.paged_attn_decode.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32,
                                          f32, i32, i32, P, sz, P]
        lib.paged_attn_decode.restype = i32
        lib.paged_attn_decode_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
        lib.paged_attn_decode_workspace_size.restype = sz
        lib.paged_attn_decode_partition_tokens.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.paged_attn_decode_partition_tokens.restype = i32
        lib.paged_attn_decode_fp8_workspace_size.argtypes = [i32, i32, i32, i32, i32, i32, i32]
        lib.paged_attn_decode_fp8_workspace_size.restype = sz
        lib.paged_attn_decode_fp8_partition_tokens.argtypes = [i32, i32, i32, i32, i32, i32]
        lib.paged_attn_decode_fp8_partition_tokens.restype = i32
        lib.paged_attn_decode_noalloc.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32,
                                                  i32, i32, f32, i32, i32, P]
        lib.paged_attn_decode_noalloc.restype = i32
        lib.paged_attn_prefill.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                           i32, i32, i32, f32, i32, P]
        lib.paged_attn_prefill.restype = i32
        lib.paged_attn_decode_shared_prefix_workspace_size.argtypes = [i32, i32, i32, i32, i32,
                                                                       i32, i32, i32]
        lib.paged_attn_decode_shared_prefix_workspace_size.restype = sz
        lib.paged_attn_decode_shared_prefix.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32,
                                                        i32, i32, i32, i32, i32, i32, i32, f32,
                                                        i32, P, sz, P]
        lib.paged_attn_decode_shared_prefix.restype = i32
        lib.kv_cache_write.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, P]
        lib.kv_cache_write.restype = i32
        lib.kv_copy_blocks.argtypes = [P, P, i32, sz, i32, P]
        lib.kv_copy_blocks.restype = i32
        lib.paged_attn_decode_fp8.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                              i32, f32, f32, f32, i32, i32, P, sz, P]
        lib.paged_attn_decode_fp8.restype = i32
        lib.kv_cache_write_fp8.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, f32, f32,
                                           P]
        lib.kv_cache_write_fp8.restype = i32
        lib.kv_swap_blocks.argtypes = [P, P, P, i32, sz, i32, i32, P]
        lib.kv_swap_blocks.restype = i32
        lib.pkv_selftest_bounded_wait.argtypes = [ctypes.c_uint, i32, P]
        lib.pkv_selftest_bounded_wait.restype = i32
        lib.pkv_device_error.argtypes = [P]
        lib.pkv_device_error.restype = i32
        lib.pkv_strerror.argtypes = [i32]
        lib.pkv_strerror.restype = ctypes.c_char_p
        lib.pkv_version.argtypes = []
        lib.pkv_version.restype = i32
        _lib = lib
        return lib


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _cuda(name: str, t: torch.Tensor) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _dtype(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported element type {t.dtype}")
    return _DTYPES[t.dtype]


def _check(fn: str, rc: int) -> None:
    if rc != 0:
        raise PagedKVError(fn, rc)


def pkv_strerror(code: int) -> str:
    return load().pkv_strerror(int(code)).decode()


def pkv_version() -> int:
    return int(load().pkv_version())


def pkv_device_error(stream=None) -> int:
    """Synchronise the stream; return and clear the device error bits (PKV_DERR_*)."""
    rc = load().pkv_device_error(_stream(stream))
    if rc < 0:
        raise PagedKVError("pkv_device_error", rc)
    return rc


def pkv_selftest_bounded_wait(wait_us: int, arrive: bool = False, stream=None) -> None:
    """Run the bounded-wait self-test kernel (see include/pagedkv.h)."""
    _check("pkv_selftest_bounded_wait",
           load().pkv_selftest_bounded_wait(int(wait_us), int(bool(arrive)), _stream(stream)))


def paged_attn_decode_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                     head_dim: int, block_size: int, max_blocks_per_seq: int,
                                     partition_size: int = 0) -> int:
    return int(load().paged_attn_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads,
                                                       head_dim, block_size, max_blocks_per_seq,
                                                       partition_size))


def paged_attn_decode_partition_tokens(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                       block_size: int, max_blocks_per_seq: int,
                                       partition_size: int = 0) -> int:
    rc = int(load().paged_attn_decode_partition_tokens(num_seqs, num_q_heads, num_kv_heads,
                                                        block_size, max_blocks_per_seq,
                                                        partition_size))
    if rc < 0:
        raise PagedKVError("paged_attn_decode_partition_tokens", rc)
    return rc


def paged_attn_decode_fp8_workspace_size(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                         head_dim: int, block_size: int,
                                         max_blocks_per_seq: int,
                                         partition_size: int = 0) -> int:
    return int(load().paged_attn_decode_fp8_workspace_size(num_seqs, num_q_heads, num_kv_heads,
                                                           head_dim, block_size,
                                                           max_blocks_per_seq, partition_size))


def paged_attn_decode_fp8_partition_tokens(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                           block_size: int, max_blocks_per_seq: int,
                                           partition_size: int = 0) -> int:
    rc = int(load().paged_attn_decode_fp8_partition_tokens(num_seqs, num_q_heads, num_kv_heads,
                                                            block_size, max_blocks_per_seq,
                                                            partition_size))
    if rc < 0:
        raise PagedKVError("paged_attn_decode_fp8_partition_tokens", rc)
    return rc


def _reuse(key, nbytes: int, alloc):
    """The cached buffer under ``key`` if it holds ``nbytes``, else a new one from
    ``alloc(nbytes)``, which replaces it in the cache."""
    buf = _workspaces.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = alloc(nbytes)
        _workspaces[key] = buf
    return buf


def workspace_for(device, nbytes: int, stream=None) -> torch.Tensor | None:
    """A byte buffer of at least ``nbytes`` on ``device``, reused across calls.

    One buffer is kept per (device, stream): calls on one stream run in order, and every
    call writes each workspace byte it reads, so they can share a buffer whatever their
    shapes.  Calls on different streams may overlap on the GPU and get different
    buffers.  ``stream`` is a torch.cuda.Stream, a raw handle, or None for the current
    stream.  A caller that passes the same explicit ``workspace`` to calls on different
    streams must order those calls itself.
    """
    if nbytes == 0:
        return None
    dev = torch.device(device)
    return _reuse((dev, _stream(stream)), nbytes,
                  lambda n: torch.empty(n, dtype=torch.uint8, device=dev))


def paged_attn_decode(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                      v_cache: torch.Tensor, block_tables: torch.Tensor,
                      context_lens: torch.Tensor, scale: float, partition_size: int = 0,
                      workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Decode attention over the paged cache; writes and returns ``out`` [B, Hq, D].

    ``q``/``out`` [B, Hq, D]; ``k_cache``/``v_cache`` [NB, bs, Hkv, D];
    ``block_tables`` int32 [B, MB]; ``context_lens`` int32 [B].
    """
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    if D2 != D or tuple(v_cache.shape) != tuple(k_cache.shape) or tuple(out.shape) != (B, Hq, D):
        raise ValueError("shape mismatch between q, out and the caches")
    if not (q.dtype == out.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("q, out and the caches must share one element type")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or tuple(context_lens.shape) != (B,):
        raise ValueError("block_tables must be [B, MB] and context_lens [B]")
    MB = block_tables.shape[1]
    need = paged_attn_decode_workspace_size(B, Hq, Hkv, D, bs, MB, partition_size)
    if workspace is None:
        workspace = workspace_for(q.device, need, stream)
    ws_ptr = _cuda("workspace", workspace) if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = load().paged_attn_decode(
        _cuda("out", out), _cuda("q", q), _cuda("k_cache", k_cache), _cuda("v_cache", v_cache),
        _cuda("block_tables", block_tables), _cuda("context_lens", context_lens), B, Hq, Hkv, D,
        bs, MB, NB, float(scale), _dtype(q), int(partition_size), ws_ptr, ws_bytes,
        _stream(stream))
    _check("paged_attn_decode", rc)
    return out


def paged_attn_prefill(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                       v_cache: torch.Tensor, block_tables: torch.Tensor,
                       context_lens: torch.Tensor, query_start: torch.Tensor,
                       max_query_len: int, scale: float, stream=None) -> torch.Tensor:
    """Chunked-prefill attention over the paged cache; writes and returns ``out``.

    ``q``/``out`` [T, Hq, D]: sequence s owns rows ``query_start[s] .. query_start[s+1]-1``
    (int32 [B + 1] on the device), the last tokens of its ``context_lens[s]`` cached
    tokens, each attending causally.  ``max_query_len`` bounds every chunk length.
    """
    T, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    B = context_lens.shape[0]
    if D2 != D or tuple(v_cache.shape) != tuple(k_cache.shape) or tuple(out.shape) != (T, Hq, D):
        raise ValueError("shape mismatch between q, out and the caches")
    if not (q.dtype == out.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("q, out and the caches must share one element type")
    if (block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32
            or query_start.dtype != torch.int32):
        raise TypeError("block_tables, context_lens and query_start must be int32")
    if (block_tables.dim() != 2 or block_tables.shape[0] != B
            or tuple(query_start.shape) != (B + 1,)):
        raise ValueError("block_tables must be [B, MB] and query_start [B + 1]")
    rc = load().paged_attn_prefill(
        _cuda("out", out), _cuda("q", q), _cuda("k_cache", k_cache), _cuda("v_cache", v_cache),
        _cuda("block_tables", block_tables), _cuda("context_lens", context_lens),
        _cuda("query_start", query_start), B, T, int(max_query_len), Hq, Hkv, D, bs,
        block_tables.shape[1], NB, float(scale), _dtype(q), _stream(stream))
    _check("paged_attn_prefill", rc)
    return out


def paged_attn_decode_shared_prefix_workspace_size(num_seqs: int, num_groups: int,
                                                   num_q_heads: int, num_kv_heads: int,
                                                   block_size: int, max_blocks_per_seq: int,
                                                   max_group_size: int,
                                                   max_prefix_tokens: int) -> int:
    return int(load().paged_attn_decode_shared_prefix_workspace_size(
        num_seqs, num_groups, num_q_heads, num_kv_heads, block_size, max_blocks_per_seq,
        max_group_size, max_prefix_tokens))


def paged_attn_decode_shared_prefix(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                                    v_cache: torch.Tensor, block_tables: torch.Tensor,
                                    context_lens: torch.Tensor, group_start: torch.Tensor,
                                    prefix_lens: torch.Tensor, max_group_size: int,
                                    max_prefix_tokens: int, scale: float,
                                    workspace: torch.Tensor | None = None,
                                    stream=None) -> torch.Tensor:
    """Decode attention for groups of sequences sharing a physical prefix (a cascade).

    Group g is the run of sequences ``group_start[g] .. group_start[g+1]-1`` (int32
    [G + 1]); its first ``prefix_lens[g]`` tokens (int32 [G], whole blocks) are shared.
    Same result as ``paged_attn_decode``.
    """
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    G = prefix_lens.shape[0]
    if D2 != D or tuple(v_cache.shape) != tuple(k_cache.shape) or tuple(out.shape) != (B, Hq, D):
        raise ValueError("shape mismatch between q, out and the caches")
    if not (q.dtype == out.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("q, out and the caches must share one element type")
    for name, t in (("block_tables", block_tables), ("context_lens", context_lens),
                    ("group_start", group_start), ("prefix_lens", prefix_lens)):
        if t.dtype != torch.int32:
            raise TypeError(f"{name} must be int32")
    if tuple(group_start.shape) != (G + 1,):
        raise ValueError("group_start must be [num_groups + 1]")
    need = paged_attn_decode_shared_prefix_workspace_size(B, G, Hq, Hkv, bs, block_tables.shape[1],
                                                          max_group_size, max_prefix_tokens)
    if workspace is None:
        workspace = workspace_for(q.device, need, stream)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = load().paged_attn_decode_shared_prefix(
        _cuda("out", out), _cuda("q", q), _cuda("k_cache", k_cache), _cuda("v_cache", v_cache),
        _cuda("block_tables", block_tables), _cuda("context_lens", context_lens),
        _cuda("group_start", group_start), _cuda("prefix_lens", prefix_lens), B, G,
        int(max_group_size), int(max_prefix_tokens), Hq, Hkv, D, bs, block_tables.shape[1], NB,
        float(scale), _dtype(q), _cuda("workspace", workspace) if workspace is not None else None,
        ws_bytes, _stream(stream))
    _check("paged_attn_decode_shared_prefix", rc)
    return out


def paged_attn_decode_noalloc(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                              v_cache: torch.Tensor, block_tables: torch.Tensor,
                              context_lens: torch.Tensor, scale: float, partition_size: int = 0,
                              stream=None) -> torch.Tensor:
    """``paged_attn_decode`` without a workspace: for callers that may not allocate.

    The library's built-in scratch (``PKV_NOALLOC_SCRATCH_BYTES`` per device) stands in
    for the workspace; calls that overlap on the GPU race on it.  Raises
    ``PagedKVError`` (code -5) when the problem needs more scratch than that.
    """
    B, Hq, D = q.shape
    NB, bs, Hkv, _ = k_cache.shape
    if tuple(v_cache.shape) != tuple(k_cache.shape) or tuple(out.shape) != (B, Hq, D):
        raise ValueError("shape mismatch between q, out and the caches")
    if not (q.dtype == out.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("q, out and the caches must share one element type")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    rc = load().paged_attn_decode_noalloc(
        _cuda("out", out), _cuda("q", q), _cuda("k_cache", k_cache), _cuda("v_cache", v_cache),
        _cuda("block_tables", block_tables), _cuda("context_lens", context_lens), B, Hq, Hkv, D,
        bs, block_tables.shape[1], NB, float(scale), _dtype(q), int(partition_size),
        _stream(stream))
    _check("paged_attn_decode_noalloc", rc)
    return out


def kv_cache_write(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor,
                   v_cache: torch.Tensor, slot_mapping: torch.Tensor, stream=None) -> None:
    """Write token rows ``k[i]``/``v[i]`` [N, Hkv, D] into cache slot ``slot_mapping[i]``."""
    NB, bs, Hkv, D = k_cache.shape
    N = k.shape[0]
    if tuple(k.shape) != (N, Hkv, D) or tuple(v.shape) != (N, Hkv, D):
        raise ValueError("k and v must be [N, Hkv, D] matching the cache")
    if tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("k_cache and v_cache must have the same shape")
    if not (k.dtype == v.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("tokens and caches must share one element type")
    if slot_mapping.dtype != torch.int64 or tuple(slot_mapping.shape) != (N,):
        raise TypeError("slot_mapping must be int64 [N]")
    if N == 0:
        return
    rc = load().kv_cache_write(_cuda("k", k), _cuda("v", v), _cuda("k_cache", k_cache),
                               _cuda("v_cache", v_cache), _cuda("slot_mapping", slot_mapping), N,
                               Hkv, D, bs, NB, _dtype(k), _stream(stream))
    _check("kv_cache_write", rc)


def kv_copy_blocks(cache: torch.Tensor, src_dst_pairs: torch.Tensor, stream=None) -> None:
    """Copy whole blocks ``cache[src] -> cache[dst]`` for each row of ``src_dst_pairs`` [P, 2]."""
    if src_dst_pairs.dtype != torch.int64 or src_dst_pairs.dim() != 2 or \
            src_dst_pairs.shape[1] != 2:
        raise TypeError("src_dst_pairs must be int64 [P, 2]")
    P = src_dst_pairs.shape[0]
    if P == 0:
        return
    NB = cache.shape[0]
    block_bytes = cache[0].numel() * cache.element_size()
    rc = load().kv_copy_blocks(_cuda("cache", cache), _cuda("src_dst_pairs", src_dst_pairs), P,
                               block_bytes, NB, _stream(stream))
    _check("kv_copy_blocks", rc)


def _addressable(name: str, t: torch.Tensor) -> int:
    """Pointer of a contiguous tensor the GPU can address: CUDA or pinned host memory."""
    if not isinstance(t, torch.Tensor) or not (t.is_cuda or t.is_pinned()):
        raise TypeError(f"{name} must be a CUDA tensor or pinned host memory")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def kv_swap_blocks(dst_cache: torch.Tensor, src_cache: torch.Tensor, src_dst_pairs: torch.Tensor,
                   stream=None) -> None:
    """Copy whole blocks ``src_cache[src] -> dst_cache[dst]`` between two pools.

    Either pool may live on the GPU or in pinned host memory (swap out / swap in).
    """
    if src_dst_pairs.dtype != torch.int64 or src_dst_pairs.dim() != 2 or \
            src_dst_pairs.shape[1] != 2:
        raise TypeError("src_dst_pairs must be int64 [P, 2]")
    if dst_cache[0].numel() * dst_cache.element_size() != \
            src_cache[0].numel() * src_cache.element_size():
        raise ValueError("the two pools must have the same block size")
    P = src_dst_pairs.shape[0]
    if P == 0:
        return
    block_bytes = dst_cache[0].numel() * dst_cache.element_size()
    rc = load().kv_swap_blocks(_addressable("dst_cache", dst_cache),
                               _addressable("src_cache", src_cache),
                               _addressable("src_dst_pairs", src_dst_pairs), P, block_bytes,
                               dst_cache.shape[0], src_cache.shape[0], _stream(stream))
    _check("kv_swap_blocks", rc)


def _fp8_cache(name: str, t: torch.Tensor) -> int:
    if t.dtype != torch.uint8:
        raise TypeError(f"{name} must hold E4M3 codes as torch.uint8")
    return _cuda(name, t)


def paged_attn_decode_fp8(out: torch.Tensor, q: torch.Tensor, k_cache: torch.Tensor,
                          v_cache: torch.Tensor, block_tables: torch.Tensor,
                          context_lens: torch.Tensor, scale: float, k_scale: float,
                          v_scale: float, partition_size: int = 0,
                          workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Decode over E4M3 caches (uint8 codes [NB, bs, Hkv, D]); q / out bf16 or fp16."""
    B, Hq, D = q.shape
    NB, bs, Hkv, D2 = k_cache.shape
    if D2 != D or tuple(v_cache.shape) != tuple(k_cache.shape) or tuple(out.shape) != (B, Hq, D):
        raise ValueError("shape mismatch between q, out and the caches")
    if q.dtype != out.dtype:
        raise TypeError("q and out must share one element type")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise TypeError("block_tables and context_lens must be int32")
    MB = block_tables.shape[1]
    need = paged_attn_decode_fp8_workspace_size(B, Hq, Hkv, D, bs, MB, partition_size)
    if workspace is None:
        workspace = workspace_for(q.device, need, stream)
    ws_ptr = _cuda("workspace", workspace) if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = load().paged_attn_decode_fp8(
        _cuda("out", out), _cuda("q", q), _fp8_cache("k_cache", k_cache),
        _fp8_cache("v_cache", v_cache), _cuda("block_tables", block_tables),
        _cuda("context_lens", context_lens), B, Hq, Hkv, D, bs, MB, NB, float(scale),
        float(k_scale), float(v_scale), _dtype(q), int(partition_size), ws_ptr, ws_bytes,
        _stream(stream))
    _check("paged_attn_decode_fp8", rc)
    return out


def kv_cache_write_fp8(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor,
                       v_cache: torch.Tensor, slot_mapping: torch.Tensor, k_scale: float,
                       v_scale: float, stream=None) -> None:
    """Quantise token rows k[i] / v[i] [N, Hkv, D] into E4M3 cache slot slot_mapping[i]."""
    NB, bs, Hkv, D = k_cache.shape
    N = k.shape[0]
    if tuple(k.shape) != (N, Hkv, D) or tuple(v.shape) != (N, Hkv, D):
        raise ValueError("k and v must be [N, Hkv, D] matching the cache")
    if k.dtype != v.dtype:
        raise TypeError("k and v must share one element type")
    if slot_mapping.dtype != torch.int64 or tuple(slot_mapping.shape) != (N,):
        raise TypeError("slot_mapping must be int64 [N]")
    if N == 0:
        return
    rc = load().kv_cache_write_fp8(_cuda("k", k), _cuda("v", v), _fp8_cache("k_cache", k_cache),
                                   _fp8_cache("v_cache", v_cache),
                                   _cuda("slot_mapping", slot_mapping), N, Hkv, D, bs, NB,
                                   _dtype(k), float(k_scale), float(v_scale), _stream(stream))
    _check("kv_cache_write_fp8", rc)
