"""The C ABI without a GPU: the library builds, loads, exports every symbol the header
declares, and its pure-host entry points and argument checks behave as documented."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


def _declared_functions():
    names = []
    for fn in sorted(os.listdir(HEADER_DIR)):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(HEADER_DIR, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        text = re.sub(r"#[^\n]*", "", text)
        for m in re.finditer(r"^[A-Za-z_][\w \t\*]*?\b([A-Za-z_]\w*)\s*\(", text, flags=re.M):
            name = m.group(1)
            if name not in ("if", "while", "for", "return", "sizeof"):
                names.append(name)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from paged_kv_cache_315_gb300 import build

    path = build()
    import torch  # noqa: F401  (loads the CUDA runtime the library links against)

    return ctypes.CDLL(path)


def test_header_declares_the_three_operations():
    names = _declared_functions()
    for n in ("paged_attn_decode", "kv_cache_write", "kv_copy_blocks",
              "paged_attn_decode_workspace_size", "pkv_device_error", "pkv_strerror"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def test_host_only_entry_points(lib):
    import paged_kv_cache_315_gb300 as pkv

    assert pkv.pkv_version() == 0x000100
    assert pkv.pkv_strerror(-1) == "invalid argument"
    # contexts that fit one partition need no workspace
    assert pkv.paged_attn_decode_workspace_size(4, 4, 4, 64, 16, 7, 0) == 0
    # 64 partitions of 512 tokens: o partials, (m, l) pairs and per-unit counters
    n = pkv.paged_attn_decode_workspace_size(32, 32, 8, 128, 16, 2048, 512)
    units = 32 * 32 * 64
    assert n >= units * 128 * 4 + units * 2 * 4 + 32 * 32 * 4
    assert n < units * 130 * 4 + 64 * 1024
    # partition sizes must be multiples of the block size
    assert pkv.paged_attn_decode_workspace_size(32, 32, 8, 128, 16, 2048, 100) == 0


def test_argument_checks_return_before_any_cuda_call(lib):
    """Invalid shapes are rejected on the host (these calls never touch a device)."""
    null = ctypes.c_void_p(0)
    f = lib.paged_attn_decode
    f.restype = ctypes.c_int
    args = lambda hq, hkv, d, bs, dt, part: (  # noqa: E731
        null, null, null, null, null, null, ctypes.c_int(2), ctypes.c_int(hq), ctypes.c_int(hkv),
        ctypes.c_int(d), ctypes.c_int(bs), ctypes.c_int(8), ctypes.c_int(16), ctypes.c_float(0.1),
        ctypes.c_int(dt), ctypes.c_int(part), null, ctypes.c_size_t(0), null)
    assert f(*args(6, 4, 128, 16, 1, 0)) == -1      # Hq % Hkv != 0
    assert f(*args(8, 4, 128, 16, 7, 0)) == -1      # bad dtype
    assert f(*args(8, 4, 128, 16, 1, 24)) == -1     # partition not a multiple of block_size
    assert f(*args(8, 4, 96, 16, 1, 0)) == -4       # head_dim not served
    assert f(*args(8, 4, 128, 16, 1, 0)) == -1      # null pointers
    w = lib.kv_cache_write
    w.restype = ctypes.c_int
    assert w(null, null, null, null, null, ctypes.c_int(-1), 4, 128, 16, 16, 1, null) == -1
    assert w(null, null, null, null, null, ctypes.c_int(0), 4, 128, 16, 16, 1, null) == 0
    c = lib.kv_copy_blocks
    c.restype = ctypes.c_int
    assert c(null, null, ctypes.c_int(0), ctypes.c_size_t(64), 4, null) == 0
    assert c(null, null, ctypes.c_int(3), ctypes.c_size_t(64), 4, null) == -1
    p = lib.paged_attn_prefill
    p.restype = ctypes.c_int
    pargs = lambda hq, hkv, d, bs, dt, ntok: (  # noqa: E731
        null, null, null, null, null, null, null, ctypes.c_int(2), ctypes.c_int(ntok),
        ctypes.c_int(8), ctypes.c_int(hq), ctypes.c_int(hkv), ctypes.c_int(d), ctypes.c_int(bs),
        ctypes.c_int(8), ctypes.c_int(16), ctypes.c_float(0.1), ctypes.c_int(dt), null)
    assert p(*pargs(6, 4, 128, 16, 1, 4)) == -1     # Hq % Hkv != 0
    assert p(*pargs(8, 4, 128, 16, 0, 4)) == -4     # fp32 not served
    assert p(*pargs(8, 4, 96, 16, 1, 4)) == -4      # head_dim not served
    assert p(*pargs(8, 4, 128, 8, 1, 4)) == -4      # block_size not served
    assert p(*pargs(8, 4, 128, 16, 1, 0)) == 0      # no query rows: nothing to do
    assert p(*pargs(8, 4, 128, 16, 1, 4)) == -1     # null pointers
    sp = lib.paged_attn_decode_shared_prefix
    sp.restype = ctypes.c_int
    spargs = lambda hq, hkv, d, bs, dt, scale: (  # noqa: E731
        null, null, null, null, null, null, null, null, ctypes.c_int(4), ctypes.c_int(1),
        ctypes.c_int(4), ctypes.c_int(64), ctypes.c_int(hq), ctypes.c_int(hkv), ctypes.c_int(d),
        ctypes.c_int(bs), ctypes.c_int(8), ctypes.c_int(16), ctypes.c_float(scale),
        ctypes.c_int(dt), null, ctypes.c_size_t(0), null)
    assert sp(*spargs(8, 2, 64, 16, 1, 0.1)) == -4     # head_dim 64 not served
    assert sp(*spargs(12, 4, 128, 16, 1, 0.1)) == -1   # 3 heads per KV head: served (null ptrs)
    assert sp(*spargs(8, 2, 128, 16, 1, -0.1)) == -1   # negative scale: served (null ptrs)
    assert sp(*spargs(8, 2, 128, 16, 1, float("nan"))) == -4   # NaN scale not served
    assert sp(*spargs(8, 2, 128, 16, 1, 0.1)) == -1    # null pointers
    ws = lib.paged_attn_decode_shared_prefix_workspace_size
    ws.restype = ctypes.c_size_t
    assert ws(256, 1, 32, 8, 32, 48, 256, 992) >= 2 * 256 * 32 * 130 * 4


def test_default_partition_size_follows_available_parallelism(lib):
    import paged_kv_cache_315_gb300 as pkv

    f = pkv.paged_attn_decode_partition_tokens
    # 64 seqs x 40 KV heads already give 2560 units at 2048 tokens
    assert f(64, 40, 40, 16, 128, 0) == 2048
    # 128 seqs x 8 KV heads x 4 partitions of 2048 (8192-token tables)
    assert f(128, 64, 8, 16, 512, 0) == 2048
    # a small batch splits finer
    assert f(4, 32, 8, 16, 2048, 0) == 512
    assert f(128, 64, 8, 16, 128, 0) == 1024  # 1024 (seq, head) pairs x 2 partitions
    # an explicit size is kept; block size 48 rounds the default down to a multiple
    assert f(32, 32, 8, 16, 2048, 512) == 512
    assert f(64, 40, 40, 48, 64, 0) % 48 == 0
    with pytest.raises(pkv.PagedKVError):
        f(32, 32, 8, 16, 2048, 100)
    # the workspace query makes the same choice
    assert pkv.paged_attn_decode_workspace_size(4, 32, 8, 128, 16, 2048, 0) == \
        pkv.paged_attn_decode_workspace_size(4, 32, 8, 128, 16, 2048, 512)


def test_fp8_default_partition_is_one_and_a_half_of_the_16_bit_one(lib):
    """At one byte per element the default candidates grow by half (3072, 1536, 768
    tokens) under the same 2048-work-unit rule; explicit sizes are kept."""
    import paged_kv_cache_315_gb300 as pkv

    f8, f16 = pkv.paged_attn_decode_fp8_partition_tokens, pkv.paged_attn_decode_partition_tokens
    # 128 seqs x 8 KV heads x 3 partitions of 3072 (8192-token tables) = 3072 units
    assert f16(128, 64, 8, 16, 512, 0) == 2048
    assert f8(128, 64, 8, 16, 512, 0) == 3072
    # 1024 (seq, head) pairs over 2048-token tables: 3072 gives one partition each (1024
    # units), 1536 gives two
    assert f8(128, 64, 8, 16, 128, 0) == 1536
    # 32 (seq, head) pairs over 32768-token tables: no candidate reaches 2048 units, so
    # the smallest, 768, is taken
    assert f8(4, 32, 8, 16, 2048, 0) == 768
    # block sizes that do not divide 1.5 x 2048 evenly round each candidate down
    assert f8(64, 40, 40, 48, 64, 0) == 3072 - 3072 % 48
    assert f8(32, 32, 8, 16, 2048, 512) == 512
    assert f8(64, 40, 40, 48, 64, 0) % 48 == 0
    with pytest.raises(pkv.PagedKVError):
        f8(32, 32, 8, 16, 2048, 100)
    # the workspace follows the fp8 choice
    ws8, ws16 = pkv.paged_attn_decode_fp8_workspace_size, pkv.paged_attn_decode_workspace_size
    assert ws8(128, 64, 8, 128, 16, 512, 0) == ws16(128, 64, 8, 128, 16, 512, 3072)
    assert ws8(128, 64, 8, 128, 16, 512, 0) < ws16(128, 64, 8, 128, 16, 512, 0)
    assert ws8(4, 32, 8, 128, 16, 2048, 512) == ws16(4, 32, 8, 128, 16, 2048, 512)


def test_binding_argument_lists_match_the_header():
    """Every function the binding declares takes as many arguments as the header says."""
    import paged_kv_cache_315_gb300._binding as bnd

    lib = bnd.load()
    text = "".join(open(os.path.join(HEADER_DIR, f)).read()
                   for f in sorted(os.listdir(HEADER_DIR)) if f.endswith(".h"))
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    for name in _declared_functions():
        m = re.search(r"\b" + name + r"\s*\(([^)]*)\)\s*;", text)
        assert m, name
        params = [p for p in m.group(1).split(",") if p.strip() and p.strip() != "void"]
        fn = getattr(lib, name)
        if fn.argtypes is None:
            continue
        assert len(fn.argtypes) == len(params), (name, len(fn.argtypes), len(params))


def test_workspace_cache_keeps_one_buffer_per_device_and_stream(monkeypatch):
    # calls on one stream share a buffer; a call on another stream gets its own, so two
    # decodes issued on different streams never write the same workspace
    import torch

    from paged_kv_cache_315_gb300 import _binding as b

    monkeypatch.setattr(b, "_workspaces", {})
    made = []

    def alloc(n):
        made.append(n)
        return torch.empty(n, dtype=torch.uint8)

    dev = torch.device("cuda", 0)
    a1 = b._reuse((dev, 111), 64, alloc)
    a2 = b._reuse((dev, 111), 32, alloc)          # smaller request on the same stream
    c1 = b._reuse((dev, 222), 64, alloc)          # another stream
    d1 = b._reuse((torch.device("cuda", 1), 111), 64, alloc)  # another device
    assert a1 is a2
    assert c1 is not a1 and d1 is not a1 and d1 is not c1
    a3 = b._reuse((dev, 111), 128, alloc)         # grows in place of the old one
    assert a3 is not a1 and a3.numel() == 128
    assert b._reuse((dev, 111), 100, alloc) is a3
    assert made == [64, 64, 64, 128]
    assert set(b._workspaces) == {(dev, 111), (dev, 222), (torch.device("cuda", 1), 111)}
