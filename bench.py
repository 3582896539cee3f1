#!/usr/bin/env python
"""Benchmark of the paged decode hot path on one or more GPUs.

One step = one decode pass over a synthetic batch: the copy-on-write block copies (where
the batch has shared blocks), the slot write of every sequence's new token, and paged
decode attention (split partitions merged by log-sum-exp in the same launch).  The KV
pool is device-resident state, as in a serving engine; each step's per-step inputs are
the query, block tables, context lengths and the new tokens.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C]
    python bench.py --impl reference ...      # the fp64 CPU oracle on the host cores

By default one process times the decode batches 2 (13B-like MHA), 3 (70B-like GQA with
slot writes), 4 (shared prefix with copy-on-write) and 5 (32k long context) back to back;
the line's value is batch 5's and the others are under ``per_config``.  ``--config C``
times batch C alone.

Prints one JSON line (rank 0).  Multi-GPU runs (torchrun) are independent replicas: each
rank runs the full batch and the value is the sum of all ranks' bytes over the slowest
rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "paged decode attention KV-read GB/s (% of HBM peak) and queries/s per batch"
PREFILL_METRIC = "paged chunked-prefill attention TFLOP/s (causal chunks over the paged cache)"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

# DRAM bytes (read + write) per launch of the decode kernel, from one ncu capture per
# workload and partition size, valid only for the kernel source whose hash is recorded
# beside it (profiles/ holds the captures).
MEASURED_TRAFFIC: dict = {
    # ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum, one decode launch each (the
    # timed step of `bench.py --steps 1 --warmup 3`)
    "13b-mha-b64-bf16@2048": {"bytes": 1408783360 + 626944, "decode_cu_sha": "03c89ed11f9bee50"},
    "70b-gqa8-b128-bf16@2048": {"bytes": 963344896 + 2590208, "decode_cu_sha": "03c89ed11f9bee50"},
    "shared-prefix-cow-b256-bf16@2048": {"bytes": 328271616 + 1593856, "decode_cu_sha": "03c89ed11f9bee50"},
    "longctx-32k-gqa4-b32-bf16@512": {"bytes": 4300867584 + 32169728, "decode_cu_sha": "03c89ed11f9bee50"},
    "13b-mha-b64-bf16@3072+fp8": {"bytes": 704773376 + 552448, "decode_cu_sha": "03c89ed11f9bee50"},
    "70b-gqa8-b128-bf16@3072+fp8": {"bytes": 482749440 + 1077760, "decode_cu_sha": "03c89ed11f9bee50"},
    "shared-prefix-cow-b256-bf16@3072+fp8": {"bytes": 164968448 + 1629440, "decode_cu_sha": "03c89ed11f9bee50"},
    "longctx-32k-gqa4-b32-bf16@512+fp8": {"bytes": 2148399616 + 31738368, "decode_cu_sha": "03c89ed11f9bee50"},
    "grouped-prefix-64x8-p4096-bf16@2048": {"bytes": 1984763136 + 20503552, "decode_cu_sha": "03c89ed11f9bee50"},
}


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--config", type=int, default=0, choices=[0, 1, 2, 3, 4, 5],
                   help="decode batch; 0 (default): batches 2, 3, 4 and 5 back to back in one "
                        "process, the 32k long-context batch (5) as the headline and the "
                        "others under per_config")
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--partition", type=int, default=-1,
                   help="partition size in tokens (-1: the batch's own, 0: library default)")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="CPU time budget of the oracle baseline sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--flush-l2", action="store_true",
                   help="also time the decode calls with a 2 x L2 scratch write before each "
                        "(reported under l2_flushed)")
    p.add_argument("--kv-dtype", choices=["same", "fp8"], default="same",
                   help="cache element type: the batch's own (default) or fp8 E4M3 codes")
    p.add_argument("--head-dim", type=int, default=128, choices=[64, 128],
                   help="head_dim of the chunked-prefill batch (--op prefill)")
    p.add_argument("--op", choices=["decode", "swap", "prefill"], default="decode",
                   help="decode (default): the decode step; swap: block swaps device <-> host; "
                        "prefill: chunked-prefill attention")
    p.add_argument("--swap-blocks", type=int, default=4096,
                   help="blocks per swap direction for --op swap")
    p.add_argument("--shared-prefix", action="store_true",
                   help="decode the shared-prefix batches (--config 4, --grouped-prefix) as a "
                        "cascade over their shared prefixes (paged_attn_decode_shared_prefix)")
    p.add_argument("--grouped-prefix", action="store_true",
                   help="decode batch: 64 groups x 8 sequences sharing 4096-token prompts "
                        "(parallel sampling) instead of --config")
    return p.parse_args(argv)


# ------------------------------------------------------------------------------------------
# workload
# ------------------------------------------------------------------------------------------

def bench_workload(cfg: int) -> synth.Workload:
    """The decode batch of config ``cfg`` with the per-step writes of a decode step."""
    w = synth.config_workload(cfg)
    if cfg == 4:
        # the copy-on-write state is built once; each step re-copies the shared partial
        # block and writes every sequence's next token into its private copy
        w.info["setup_slots"] = w.slot_mapping
        w.info["setup_k"], w.info["setup_v"] = w.k_new, w.v_new
        suffix = (w.context_lens - w.info["prefix_tokens"]).astype(np.int64)
        starts = np.concatenate([[0], np.cumsum(suffix)[:-1]])  # first suffix token per seq
        w.slot_mapping = w.info["setup_slots"][starts]
        w.k_new = w.info["setup_k"][starts]
        w.v_new = w.info["setup_v"][starts]
    elif w.k_new is None:
        synth.add_new_tokens(w, seed=synth.BASE_SEED + 100 + cfg)
    return w


def fp8_scales(cfg: int) -> tuple[float, float]:
    """Per-tensor scales for E4M3 caches: N(0,1) data (x8 key outliers in batch 5)."""
    return (0.125, 0.0625) if cfg == 5 else (0.0625, 0.0625)


def kv_bytes(w: synth.Workload, fp8: bool) -> int:
    return w.kv_bytes() // w.elem_bytes if fp8 else w.kv_bytes()


def algorithmic_bytes(w: synth.Workload, fp8: bool = False) -> dict:
    """Bytes the decode launch must move at minimum, and its parts."""
    e = w.elem_bytes
    kv = kv_bytes(w, fp8)
    q = w.q.size * e
    out = q
    nblocks = int(sum((int(L) + w.block_size - 1) // w.block_size for L in w.context_lens))
    tables = nblocks * 4
    lens = w.num_seqs * 4
    return {"kv": kv, "q": q, "out": out, "block_tables": tables, "context_lens": lens,
            "total": kv + q + out + tables + lens}


def describe(w: synth.Workload, cfg: int, part: int) -> dict:
    pool = 2 * w.k_cache.nbytes
    recipe = synth.GROUPED_PREFIX_RECIPE if "group_start" in w.info else synth.CONFIGS[cfg]
    d = {"workload": w.name, "recipe": recipe, "batch": w.num_seqs,
         "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
         "block_size": w.block_size,
         "context_tokens": int(w.context_lens.sum()),
         "context_min_mean_max": [int(w.context_lens.min()), float(w.context_lens.mean()),
                                  int(w.context_lens.max())],
         "pool_bytes": pool,
         "l2": f"not flushed: every step reads {w.kv_bytes() / 1e9:.2f} GB of KV, "
               f"{w.kv_bytes() / L2_BYTES:.0f}x the {L2_BYTES >> 20} MiB L2"}
    if "group_start" in w.info:
        d["l2"] = ("not flushed: 64 prompts of 16 MB (1 GB, 8x the L2) are each read by their "
                   "8 sequences in every step; value counts logical bytes")
        d["unique_kv_bytes"] = unique_kv_bytes(w)
    elif cfg == 4:
        d["l2"] = ("not flushed: the 32 shared prefix blocks (4 MB) are read by all 256 "
                   "sequences in every step and stay in L2; value counts logical bytes")
        d["unique_kv_bytes"] = unique_kv_bytes(w)
    return d


def unique_kv_bytes(w: synth.Workload) -> int:
    """KV bytes of distinct (physical block, slot) rows the batch attends to."""
    rows = set()
    bs = w.block_size
    for s in range(w.num_seqs):
        L = int(w.context_lens[s])
        for j in range((L + bs - 1) // bs):
            rows.add((int(w.block_tables[s, j]), min(bs, L - j * bs)))
    per_row = 2 * w.num_kv_heads * w.head_dim * w.elem_bytes
    used = {}
    for b, n in rows:
        used[b] = max(used.get(b, 0), n)
    return sum(used.values()) * per_row


# ------------------------------------------------------------------------------------------
# measurement helpers
# ------------------------------------------------------------------------------------------

def hbm_peak() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) == 9 and parts[1].replace(".", "").isdigit():
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "samples": len(rows), "reasons": reasons}


# DRAM bytes of one shared-prefix cascade call (every kernel of the call: prep, prefix pass,
# suffix ordering and decode, merge), valid only for the recorded sources
CASCADE_TRAFFIC: dict = {
    "grouped-prefix-64x8-p4096-bf16@2048": {"bytes": 1392939264, "sources_sha": "6b6ab9135d74ca0c"},
    "shared-prefix-cow-b256-bf16@2048": {"bytes": 353472768, "sources_sha": "6b6ab9135d74ca0c"},
}
CASCADE_SOURCES = ("prefill.cu", "decode.cu", "shared_prefix.cu")


def cascade_traffic_for(w_name: str, part: int) -> float | None:
    import hashlib

    entry = CASCADE_TRAFFIC.get(f"{w_name}@{part}")
    if not entry:
        return None
    h = hashlib.sha256()
    for f in CASCADE_SOURCES:
        h.update(open(os.path.join(ROOT, "paged_kv_cache_315_gb300", "csrc", f), "rb").read())
    return float(entry["bytes"]) if entry["sources_sha"] == h.hexdigest()[:16] else None


def traffic_for(w_name: str, part: int, fp8: bool = False) -> float | None:
    entry = MEASURED_TRAFFIC.get(f"{w_name}@{part}" + ("+fp8" if fp8 else ""))
    if not entry:
        return None
    import hashlib

    src = os.path.join(ROOT, "paged_kv_cache_315_gb300", "csrc", "decode.cu")
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return float(entry["bytes"]) if entry.get("decode_cu_sha") == digest else None


def decode_kernel_name(w: synth.Workload, fp8: bool) -> str:
    """The decode kernel the library launches for this batch (the launcher's choice)."""
    G = w.num_q_heads // w.num_kv_heads
    if fp8:
        return "decode_fp8g_kernel" if G <= 8 else "decode_fp8_kernel"
    if w.dtype not in ("bf16", "f16") or w.head_dim not in (64, 128) or \
            w.block_size not in (16, 32, 64):
        return "decode_simt_kernel"
    return "decode_tcg_kernel" if w.head_dim == 128 and 2 <= G <= 8 else "decode_tc_kernel"


def cache_ops(t: dict, w: synth.Workload, fp8: bool, has_pairs: bool, copy_ms: float,
              write_ms: float) -> dict:
    """Per-step time and bytes moved (read + write) of the copy-on-write copies and the slot
    write that precede the decode in every step."""
    cache_elem = 1 if fp8 else t["k_cache"].element_size()
    row = w.num_kv_heads * w.head_dim
    out = {}
    if has_pairs:
        pairs = int(t["copy_pairs"].shape[0])
        nbytes = 2 * pairs * (2 * w.block_size * row * cache_elem + 16)  # K and V calls
        out["kv_copy_blocks"] = {"calls": 2, "pairs": pairs, "ms": round(copy_ms, 5),
                                 "bytes": nbytes, "GB/s": round(nbytes / (copy_ms / 1e3) / 1e9, 1)}
    n = int(t["k_new"].shape[0])
    nbytes = 2 * n * row * (t["k_new"].element_size() + cache_elem) + 8 * n
    out["kv_cache_write" + ("_fp8" if fp8 else "")] = {
        "tokens": n, "ms": round(write_ms, 5), "bytes": nbytes,
        "GB/s": round(nbytes / (write_ms / 1e3) / 1e9, 1)}
    return out


def pipelined_e2e(t: dict, names: list, out, step, dev, steps: int, warmup: int, barrier):
    """End-to-end timing through the public calls with host buffers, two steps in flight.

    Every step's inputs (``names`` of ``t``) are copied from one pinned host buffer with one
    cudaMemcpyAsync on a copy-in stream, the step runs on the current stream into one of two
    device outputs, and that output is copied to pinned host memory on a copy-out stream.
    The copy-in of step i+1 and the copy-out of step i-1 overlap step i (device inputs and
    outputs alternate between two buffers), and the host waits for step i-1's output to reach
    the host before it enqueues step i+1, as a serving loop that consumes each step's result
    would.  ``step(inputs, dst=output)`` enqueues one step.  Returns the seconds for ``steps``
    steps (through the last output on the host) and the bytes copied in and out per step."""
    import torch

    offsets, off = {}, 0
    for n in names:
        offsets[n] = off
        off += -(-t[n].numel() * t[n].element_size() // 256) * 256
    host_buf = torch.empty(off, dtype=torch.uint8).pin_memory()
    dev_bufs = [torch.empty(off, dtype=torch.uint8, device=dev) for _ in range(2)]

    def view(buf, n):
        nb = t[n].numel() * t[n].element_size()
        return buf[offsets[n]:offsets[n] + nb].view(t[n].dtype).view(t[n].shape)

    for n in names:
        view(host_buf, n).copy_(t[n].cpu())
    dev_ins = [{n: view(b, n) for n in names} for b in dev_bufs]
    outs = [out, torch.empty_like(out)]
    out_h = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
    h2d = sum(t[n].numel() * t[n].element_size() for n in names)
    d2h = out_h[0].numel() * out_h[0].element_size()
    cs = torch.cuda.current_stream()
    xs = torch.cuda.Stream(device=dev)                 # copies in
    ys = torch.cuda.Stream(device=dev)                 # copies out
    ev_in = [torch.cuda.Event() for _ in range(2)]    # inputs of the step in buffer b copied
    ev_free = [torch.cuda.Event() for _ in range(2)]  # the step using buffers b is done
    ev_out = [torch.cuda.Event() for _ in range(2)]   # its output is on the host

    def one(i):
        b = i & 1
        with torch.cuda.stream(xs):
            if i >= 2:
                xs.wait_event(ev_free[b])
            dev_bufs[b].copy_(host_buf, non_blocking=True)
            ev_in[b].record(xs)
        cs.wait_event(ev_in[b])
        if i >= 2:
            cs.wait_event(ev_out[b])                   # output b copied out before reuse
        step(dev_ins[b], dst=outs[b])
        ev_free[b].record(cs)
        with torch.cuda.stream(ys):
            ys.wait_event(ev_free[b])
            out_h[b].copy_(outs[b], non_blocking=True)
            ev_out[b].record(ys)
        if i >= 1:
            ev_out[(i - 1) & 1].synchronize()

    for i in range(max(3, warmup)):
        one(i)
    torch.cuda.synchronize()
    barrier()
    s0 = time.perf_counter()
    for i in range(steps):
        one(i)
    torch.cuda.synchronize()
    barrier()
    return time.perf_counter() - s0, h2d, d2h


def max_over_ranks(values, world: int) -> list:
    """Element-wise max of ``values`` over all ranks (the values themselves for one rank)."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist

    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" \
        else torch.device("cpu")
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def replica_gbs(bytes_per_step: int, steps: int, world: int, seconds: float) -> float:
    """Whole-job GB/s of ``world`` replicas that each moved ``bytes_per_step`` per step."""
    return bytes_per_step * steps * world / seconds / 1e9


# ------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------

DECODE_CONFIGS = (2, 3, 4, 5)   # the batches one default run times, the last one the headline
NOMINAL_HBM_GBS = 7900.0        # GB300 HBM3e, nominal (published figure, not measured here)


def decode_session(args, cfg: int, dev, pkv):
    """Device state and step functions of one decode batch (``cfg``, or the grouped-prompt
    batch with ``--grouped-prefix``)."""
    import torch

    if args.grouped_prefix:
        w = synth.grouped_prefix_workload()
        synth.add_new_tokens(w, seed=synth.BASE_SEED + 107)
    else:
        w = bench_workload(cfg)
    t = synth.to_torch(w, dev)
    fp8 = args.kv_dtype == "fp8"
    ks, vs = fp8_scales(cfg)
    if fp8:
        k8, v8 = synth.fp8_kv(w, ks, vs)
        t["k_cache"] = torch.from_numpy(k8).to(dev)
        t["v_cache"] = torch.from_numpy(v8).to(dev)
        del k8, v8
    if cfg == 4 and not args.grouped_prefix:
        # state: copy-on-write copies, then every suffix token
        pkv.kv_copy_blocks(t["k_cache"], t["copy_pairs"])
        pkv.kv_copy_blocks(t["v_cache"], t["copy_pairs"])
        sk = synth.storage_to_torch(w.info["setup_k"], "bf16", dev)
        sv = synth.storage_to_torch(w.info["setup_v"], "bf16", dev)
        ss = torch.from_numpy(w.info["setup_slots"]).to(dev)
        if fp8:
            pkv.kv_cache_write_fp8(sk, sv, t["k_cache"], t["v_cache"], ss, ks, vs)
        else:
            pkv.kv_cache_write(sk, sv, t["k_cache"], t["v_cache"], ss)
        del sk, sv, ss
    out = torch.empty_like(t["q"])
    B = w.num_seqs
    part = w.partition_size if args.partition < 0 else args.partition
    ptok_fn = (pkv.paged_attn_decode_fp8_partition_tokens if fp8
               else pkv.paged_attn_decode_partition_tokens)
    ws_fn = (pkv.paged_attn_decode_fp8_workspace_size if fp8
             else pkv.paged_attn_decode_workspace_size)
    part = ptok_fn(B, w.num_q_heads, w.num_kv_heads, w.block_size, w.max_blocks_per_seq, part)
    ws_bytes = ws_fn(B, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                     w.max_blocks_per_seq, part)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None
    has_pairs = "copy_pairs" in t

    cascade = bool(args.shared_prefix)
    sp = {}
    if cascade:
        if "shared_prefix_tokens" not in w.info or fp8:
            raise SystemExit("--shared-prefix applies to the shared-prefix batches (--config 4, "
                             "--grouped-prefix) with the bf16 cache")
        gs = w.info.get("group_start", np.array([0, B], np.int32))
        pls = w.info.get("prefix_lens", np.array([w.info["shared_prefix_tokens"]], np.int32))
        t["group_start"] = torch.from_numpy(np.ascontiguousarray(gs, np.int32)).to(dev)
        t["prefix_lens"] = torch.from_numpy(np.ascontiguousarray(pls, np.int32)).to(dev)
        sp["max_group"] = int(np.diff(gs).max())
        sp["max_prefix"] = int(pls.max())
        nb = pkv.paged_attn_decode_shared_prefix_workspace_size(
            B, len(pls), w.num_q_heads, w.num_kv_heads, w.block_size, w.max_blocks_per_seq,
            sp["max_group"], sp["max_prefix"])
        sp["ws"] = torch.empty(nb, dtype=torch.uint8, device=dev) if nb else None

    def cache_step(inp, ev=None):
        # ev (the separate cache-op timing pass only): start, after the copies, after the write
        if ev is not None:
            ev[0].record()
        if has_pairs:
            pkv.kv_copy_blocks(t["k_cache"], inp["copy_pairs"])
            pkv.kv_copy_blocks(t["v_cache"], inp["copy_pairs"])
        if ev is not None:
            ev[1].record()
        if fp8:
            pkv.kv_cache_write_fp8(inp["k_new"], inp["v_new"], t["k_cache"], t["v_cache"],
                                   inp["slot_mapping"], ks, vs)
        else:
            pkv.kv_cache_write(inp["k_new"], inp["v_new"], t["k_cache"], t["v_cache"],
                               inp["slot_mapping"])
        if ev is not None:
            ev[2].record()

    def step(inp, ev=None, dst=None):
        # ev: events around the decode call, inside the timed steps; dst: the output tensor
        # (the end-to-end pass alternates two)
        o = out if dst is None else dst
        cache_step(inp)
        if ev is not None:
            ev[0].record()
        if cascade:
            pkv.paged_attn_decode_shared_prefix(
                o, inp["q"], t["k_cache"], t["v_cache"], inp["block_tables"],
                inp["context_lens"], t["group_start"], t["prefix_lens"], sp["max_group"],
                sp["max_prefix"], w.scale, workspace=sp["ws"])
        elif fp8:
            pkv.paged_attn_decode_fp8(o, inp["q"], t["k_cache"], t["v_cache"],
                                      inp["block_tables"], inp["context_lens"], w.scale, ks, vs,
                                      partition_size=part, workspace=ws)
        else:
            pkv.paged_attn_decode(o, inp["q"], t["k_cache"], t["v_cache"], inp["block_tables"],
                                  inp["context_lens"], w.scale, partition_size=part, workspace=ws)
        if ev is not None:
            ev[1].record()

    # copies (K and V), the slot write, the decode kernel and, when the batch splits contexts
    # (workspace in use), the one-CTA prep kernel before it and the merge kernel after it
    # (the batches here stay far below the prep kernel's 65536-item limit)
    split = ws is not None
    launches = (2 if has_pairs else 0) + 1 + 1 + (2 if split else 0)
    if cascade:  # prep, prefix pass, suffix ordering + decode, merge
        launches = (2 if has_pairs else 0) + 1 + 5
    names = ["q", "block_tables", "context_lens", "k_new", "v_new", "slot_mapping"]
    if has_pairs:
        names.append("copy_pairs")
    return dict(w=w, t=t, cfg=cfg, fp8=fp8, cascade=cascade, part=part, split=split, out=out,
                step=step, cache_step=cache_step, has_pairs=has_pairs,
                launches_per_step=launches, e2e_names=names)


def time_decode(args, S, dev, world, barrier, pkv) -> dict:
    """Warm-up, then K timed steps (whole-step events and per-call decode events), the cache
    operations in a pass of their own, and the end-to-end pass.  Times are max over ranks."""
    import torch

    step, t = S["step"], S["t"]
    assert pkv.pkv_device_error() == 0
    for _ in range(max(3, args.warmup)):
        step(t)
    torch.cuda.synchronize()
    if pkv.pkv_device_error() != 0:
        raise RuntimeError("device error bits set during warm-up")
    evs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(2))
           for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    barrier()
    t0.record()
    for i in range(args.steps):
        step(t, evs[i])
    t1.record()
    barrier()
    clk = clocks.stop()
    elapsed_ms = t0.elapsed_time(t1)
    per_call = [e[0].elapsed_time(e[1]) for e in evs]
    if pkv.pkv_device_error() != 0:
        raise RuntimeError("device error bits set during the timed steps")
    # the cache operations alone, in a pass of their own (events inside the timed steps
    # would lengthen them).  A busy-wait kernel holds the GPU while the host enqueues the
    # whole pass, so the events time the kernels, not the host's launch rate.
    cevs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(3))
            for _ in range(args.steps)]
    torch.cuda._sleep(int(2e6 + 1e5 * args.steps))
    for i in range(args.steps):
        S["cache_step"](t, cevs[i])
    torch.cuda.synchronize()
    copy_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in cevs)
    write_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in cevs)

    flushed = None
    if args.flush_l2:
        # decode calls with the L2 overwritten before each: a 2 x L2 scratch write on the
        # same stream between the steps, outside the decode call's events
        scratch = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
        fevs = [tuple(torch.cuda.Event(enable_timing=True) for _ in range(2))
                for _ in range(args.steps)]
        for i in range(args.steps):
            scratch.fill_(i & 0xFF)
            step(t, fevs[i])
        torch.cuda.synchronize()
        flushed = statistics.median(a.elapsed_time(b) for a, b in fevs)
        del scratch

    vals = [elapsed_ms, statistics.mean(per_call), statistics.median(per_call), copy_ms,
            write_ms, flushed if flushed is not None else 0.0]
    vals = max_over_ranks(vals, world)
    r = dict(elapsed_ms=vals[0], decode_ms=vals[1], decode_ms_median=vals[2], copy_ms=vals[3],
             write_ms=vals[4], decode_ms_l2_flushed=vals[5] if flushed is not None else None,
             clocks=clk)
    r["e2e"] = None
    if not args.no_e2e:
        e2e_s, h2d, d2h = pipelined_e2e(t, S["e2e_names"], S["out"], step, dev, args.steps,
                                        args.warmup, barrier)
        (e2e_s,) = max_over_ranks([e2e_s], world)
        r["e2e"] = (e2e_s, h2d, d2h)
    return r


def decode_record(args, S, r, world: int) -> dict:
    """The JSON fields of one timed decode batch."""
    w, fp8, cascade, part = S["w"], S["fp8"], S["cascade"], S["part"]
    peak, peak_kind = hbm_peak()
    ab = algorithmic_bytes(w, fp8)
    step_kv = kv_bytes(w, fp8)
    ms = r["elapsed_ms"] / args.steps
    value = replica_gbs(step_kv, args.steps, world, r["elapsed_ms"] / 1e3)
    achieved = ab["total"] / (r["decode_ms"] / 1e3) / 1e9
    traffic = (cascade_traffic_for(w.name, part) if cascade else traffic_for(w.name, part, fp8))
    if cascade:
        kernel = ("paged_attn_decode_shared_prefix (prep, prefix and suffix passes of "
                  "prefill_umma_kernel, merge)")
    else:
        kernel = (("paged_attn_decode_fp8 (" if fp8 else "paged_attn_decode (")
                  + decode_kernel_name(w, fp8) + (" + prep + merge grids)" if S["split"] else ")"))
    roof = {"kernel": kernel, "bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
            "unit": "GB/s", "frac": round(achieved / peak, 4),
            "peak_source": f"{peak_kind} hbm_gbs (copy bandwidth)",
            "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
            "nominal_peak": NOMINAL_HBM_GBS,
            "nominal_source": "GB300 HBM3e nominal 7.9 TB/s (published)",
            "achieved_median": round(ab["total"] / (r["decode_ms_median"] / 1e3) / 1e9, 2),
            "frac_median": round(ab["total"] / (r["decode_ms_median"] / 1e3) / 1e9 / peak, 4),
            "algorithmic_bytes_per_launch": ab, "traffic": traffic}
    rec = {
        "value": round(value, 2), "unit": "GB/s", "ms_per_step": round(ms, 5),
        "hbm_frac": round(value / peak, 4),
        "queries_per_s": round(w.num_seqs * world / (ms / 1e3), 1),
        "query_heads_per_s": round(w.num_seqs * w.num_q_heads * world / (ms / 1e3), 1),
        "decode_ms": round(r["decode_ms"], 5), "decode_ms_median": round(r["decode_ms_median"], 5),
        "partition_tokens": part, "kv_dtype": "e4m3" if fp8 else w.dtype,
        "cache_ops": cache_ops(S["t"], w, fp8, S["has_pairs"], r["copy_ms"], r["write_ms"]),
        "roofline": roof, "gpu_launches": S["launches_per_step"] * args.steps,
        "clocks": r["clocks"],
    }
    if "unique_kv_bytes" in describe(w, S["cfg"], part):
        # logical bytes (what the metric names) count the shared prefix once per sequence;
        # the fractions below count what HBM must deliver at least (unique rows) and what
        # it delivered (ncu DRAM bytes of one call, when recorded for this source)
        ub = unique_kv_bytes(w) // (w.elem_bytes if fp8 else 1)
        uniq = ub + ab["total"] - ab["kv"]
        roof["bytes_basis"] = "logical (each sequence's context counted in full)"
        roof["unique_bytes_per_launch"] = uniq
        roof["frac_unique_bytes"] = round(uniq / (r["decode_ms"] / 1e3) / 1e9 / peak, 4)
        roof["frac_dram_bytes"] = (round(traffic / (r["decode_ms"] / 1e3) / 1e9 / peak, 4)
                                   if traffic else None)
    if r["decode_ms_l2_flushed"] is not None:
        rec["l2_flushed"] = {
            "decode_ms_median": round(r["decode_ms_l2_flushed"], 5),
            "frac": round(ab["total"] / (r["decode_ms_l2_flushed"] / 1e3) / 1e9 / peak, 4),
            "how": "2 x L2 scratch written on the stream before every decode call"}
    if r["e2e"] is not None:
        e2e_s, h2d, d2h = r["e2e"]
        rec["e2e"] = {"value": round(replica_gbs(step_kv, args.steps, world, e2e_s), 2),
                      "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
                      "d2h_bytes_per_step": int(d2h),
                      "ms_per_step": round(e2e_s * 1e3 / args.steps, 4),
                      "path": "per-step inputs packed in one pinned host buffer -> one "
                              "cudaMemcpyAsync on a copy stream (overlapping the previous "
                              "step) -> C-ABI calls -> output to pinned host, each step's "
                              "output waited for one step later"}
    else:
        rec["e2e"] = None
    return rec


def run_ours(args) -> None:
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import paged_kv_cache_315_gb300 as pkv

    pkv.load()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    if args.grouped_prefix:
        cfgs = [0]
    else:
        cfgs = list(DECODE_CONFIGS) if args.config == 0 else [args.config]
    recs, sessions = {}, {}
    for cfg in cfgs:
        S = decode_session(args, cfg, dev, pkv)
        r = time_decode(args, S, dev, world, barrier, pkv)
        rec = decode_record(args, S, r, world)
        rec["config"] = dict(describe(S["w"], cfg, S["part"]),
                             **({"decode": "shared-prefix cascade"} if S["cascade"] else {}))
        recs[cfg] = rec
        sessions[cfg] = S["w"]
        del S
        torch.cuda.empty_cache()

    head_cfg = cfgs[-1]
    head = recs[head_cfg]
    w = sessions[head_cfg]
    fp8 = args.kv_dtype == "fp8"
    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_seconds, fp8_scales(head_cfg) if fp8 else None)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    line = {
        "metric": METRIC,
        "value": head["value"],
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": head["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype if not fp8 else f"{w.dtype} (E4M3 KV cache)",
        "data": "synthetic (seeded N(0,1) q/K/V, shuffled block pool)",
        "config": head["config"],
    }
    for k in ("hbm_frac", "queries_per_s", "query_heads_per_s", "decode_ms", "decode_ms_median",
              "cache_ops", "partition_tokens", "kv_dtype", "roofline"):
        line[k] = head[k]
    if "l2_flushed" in head:
        line["l2_flushed"] = head["l2_flushed"]
    line["cpu_baseline"] = cpu
    line["e2e"] = head["e2e"]
    line["gpu_launches"] = head["gpu_launches"]
    line["clocks"] = head["clocks"]
    if len(cfgs) > 1:
        line["per_config"] = {}
        for cfg in cfgs[:-1]:
            rec = dict(recs[cfg])
            rec["workload"] = rec["config"]["workload"]
            line["per_config"][f"config{cfg}"] = rec
        line["per_config_note"] = (
            "the other decode batches, timed in the same process before the headline batch "
            "with the same steps and warm-up; each entry's gpu_launches counts its own timed "
            "steps")
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


# ------------------------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and reference arm)
# ------------------------------------------------------------------------------------------

def _oracle_seq(w, s, fp8=None, threads: int = 0):
    import oracle

    if fp8 is not None:
        k8, v8, ks, vs = fp8
        return oracle.paged_decode_fp8kv(w.q[s:s + 1], k8, v8, w.block_tables[s:s + 1],
                                         w.context_lens[s:s + 1], w.scale, ks, vs, w.dtype,
                                         num_threads=threads)
    return oracle.paged_decode(w.q[s:s + 1], w.k_cache, w.v_cache, w.block_tables[s:s + 1],
                               w.context_lens[s:s + 1], w.scale, w.dtype, num_threads=threads)


def seq_kv_bytes(w, s) -> int:
    return int(w.context_lens[s]) * 2 * w.num_kv_heads * w.head_dim * w.elem_bytes


def host_cpu() -> dict:
    """The host's CPU model and core counts."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if model is None:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith(("model name", "cpu part")):
                    model = line.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    try:
        usable = len(os.sched_getaffinity(0))
    except Exception:
        usable = os.cpu_count()
    return {"model": model, "os_cpu_count": os.cpu_count(), "usable_cores": usable}


def _oracle_rate(w, seconds: float, fp8, threads: int) -> tuple[float, int, float]:
    """GB/s of the oracle over sequences of the batch (cycling) until ``seconds`` pass."""
    done_bytes, done_seqs = 0, 0
    s0 = time.perf_counter()
    while True:
        s = done_seqs % w.num_seqs
        _oracle_seq(w, s, fp8, threads)
        done_bytes += seq_kv_bytes(w, s) // (w.elem_bytes if fp8 else 1)
        done_seqs += 1
        el = time.perf_counter() - s0
        if el >= seconds or done_seqs >= 4 * w.num_seqs:
            break
    return done_bytes / el / 1e9, done_seqs, el


def cpu_baseline(w, seconds: float, fp8_scale_pair=None) -> dict:
    """The fp64 oracle, as it stands, over sequences of the batch: once on one thread and
    once with OpenMP over every usable core, ``seconds`` each."""
    import oracle

    oracle.build()
    fp8 = None
    if fp8_scale_pair is not None:
        fp8 = (*synth.fp8_kv(w, *fp8_scale_pair), *fp8_scale_pair)
    cpu = host_cpu()
    cores = cpu["usable_cores"]
    v1, n1, e1 = _oracle_rate(w, seconds / 2, fp8, 1)
    vn, nn, en = _oracle_rate(w, seconds, fp8, cores)
    return {"value": round(vn, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{nn} sequences of the batch (all query heads each) in {en:.1f} s on "
                      f"{cores} threads; fp64 C oracle, OpenMP over (sequence, query head)",
            "single_thread": {"value": round(v1, 4), "unit": "GB/s", "cores": 1,
                              "sample": f"{n1} sequences in {e1:.1f} s on one thread"},
            "cpu": cpu}


def run_reference(args) -> None:
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle

    oracle.build()
    cfg = args.config or DECODE_CONFIGS[-1]
    w = bench_workload(cfg)
    part = w.partition_size if args.partition < 0 else args.partition
    cpu = host_cpu()
    cores = cpu["usable_cores"]
    order = list(range(w.num_seqs))
    for i in range(args.warmup):
        _oracle_seq(w, order[i % len(order)], None, cores)
    done_bytes = 0
    s0 = time.perf_counter()
    for i in range(args.steps):
        s = order[i % len(order)]
        _oracle_seq(w, s, None, cores)
        done_bytes += seq_kv_bytes(w, s)
    el = time.perf_counter() - s0
    value = done_bytes / el / 1e9
    ms = el * 1e3 / args.steps
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) q/K/V, shuffled block pool)",
        "config": describe(w, cfg, part),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": "one sequence of the batch (all its query heads) per step, "
                                   "cycling through the batch; fp64 C oracle, OpenMP",
                         "cpu": cpu},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_swap(args) -> None:
    """Swap out / swap in of scattered blocks between the device pool and pinned host memory.

    The 70B-like GQA pool (16-token bf16 blocks, 8 KV heads: 32 KB per block per tensor);
    `--swap-blocks` random blocks go out to a pinned host pool and back in, K and V each.
    The reference ceiling is a contiguous cudaMemcpyAsync of the same bytes, each way.
    """
    import torch

    import paged_kv_cache_315_gb300 as pkv

    torch.cuda.set_device(0)
    pkv.load()
    w = synth.config_workload(3, with_writes=False)
    t = synth.to_torch(w, "cuda")
    n = min(args.swap_blocks, w.num_blocks)
    rng = np.random.default_rng(synth.BASE_SEED + 50)
    blocks = rng.choice(w.num_blocks, size=n, replace=False).astype(np.int64)
    host_k = torch.empty((n,) + tuple(t["k_cache"].shape[1:]), dtype=t["k_cache"].dtype).pin_memory()
    host_v = torch.empty_like(host_k).pin_memory()
    out_pairs = torch.from_numpy(np.stack([blocks, np.arange(n)], axis=1)).cuda()
    in_pairs = torch.from_numpy(np.stack([np.arange(n), blocks], axis=1)).cuda()
    block_bytes = t["k_cache"][0].numel() * t["k_cache"].element_size()
    moved = 2 * n * block_bytes  # K and V, one direction

    def swap_out():
        pkv.kv_swap_blocks(host_k, t["k_cache"], out_pairs)
        pkv.kv_swap_blocks(host_v, t["v_cache"], out_pairs)

    def swap_in():
        pkv.kv_swap_blocks(t["k_cache"], host_k, in_pairs)
        pkv.kv_swap_blocks(t["v_cache"], host_v, in_pairs)

    dev_buf = torch.empty(moved, dtype=torch.uint8, device="cuda")
    host_buf = torch.empty(moved, dtype=torch.uint8).pin_memory()

    def timed(fn):
        for _ in range(max(3, args.warmup)):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(args.steps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / 1e3 / args.steps

    t_out, t_in = timed(swap_out), timed(swap_in)
    if pkv.pkv_device_error() != 0:
        raise RuntimeError("device error bits set during the swaps")
    t_d2h = timed(lambda: host_buf.copy_(dev_buf, non_blocking=True))
    t_h2d = timed(lambda: dev_buf.copy_(host_buf, non_blocking=True))
    out_gbs, in_gbs = moved / t_out / 1e9, moved / t_in / 1e9
    d2h_gbs, h2d_gbs = moved / t_d2h / 1e9, moved / t_h2d / 1e9
    line = {
        "metric": "paged KV block swap GB/s (device pool <-> pinned host pool, K+V)",
        "value": round(2 * moved / (t_out + t_in) / 1e9, 2), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "dtype": "bf16",
        "data": "synthetic", "config": {"workload": w.name, "blocks_per_direction": n,
                                        "block_bytes_per_tensor": block_bytes},
        "swap_out_gbs": round(out_gbs, 2), "swap_in_gbs": round(in_gbs, 2),
        "roofline": {"bound": "host link", "unit": "GB/s",
                     "peak": {"d2h": round(d2h_gbs, 2), "h2d": round(h2d_gbs, 2)},
                     "peak_source": "contiguous cudaMemcpyAsync of the same bytes, same run",
                     "frac": {"out": round(out_gbs / d2h_gbs, 4), "in": round(in_gbs / h2d_gbs, 4)}},
        "gpu_launches": 4 * args.steps,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------
# chunked prefill
# ------------------------------------------------------------------------------------------

# DRAM bytes (read + write) per launch of the chunked-prefill kernel on the chunked-prefill
# batches (head_dim 128 and 64), from one ncu capture each, valid only for the kernel source
# whose hash is recorded.
PREFILL_TRAFFIC = {
    "chunked-prefill-70b-gqa8-c512": {"bytes": 278723328 + 103297792,
                                      "prefill_cu_sha": "9170c7eb63908a79"},
    "chunked-prefill-70b-gqa8-c512-d64": {"bytes": 139379968 + 36869120,
                                          "prefill_cu_sha": "9170c7eb63908a79"},
}


def prefill_traffic(w_name: str) -> float | None:
    """Recorded DRAM bytes of a benchmark prefill batch for the recorded prefill.cu, else
    None."""
    import hashlib

    entry = PREFILL_TRAFFIC.get(w_name)
    if not entry:
        return None
    src = os.path.join(ROOT, "paged_kv_cache_315_gb300", "csrc", "prefill.cu")
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    return float(entry["bytes"]) if entry["prefill_cu_sha"] == digest else None


def prefill_flops(w: synth.Workload, seqs=None) -> int:
    """Attention flops of the chunks: 4 * head_dim per (query row, head, attended key)."""
    n = np.diff(w.query_start).astype(np.int64)
    L = w.context_lens.astype(np.int64)
    total = 0
    for s in (range(w.num_seqs) if seqs is None else seqs):
        ns, Ls = int(n[s]), int(L[s])
        keys = (Ls - ns) * ns + ns * (ns + 1) // 2  # row i attends L - n + i + 1 keys
        total += 4 * w.head_dim * w.num_q_heads * keys
    return total


def tensor_peak() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def _oracle_prefill_seq(w, s, threads: int = 0):
    """The oracle on sequence s alone (all its chunk rows)."""
    import oracle

    a, b = int(w.query_start[s]), int(w.query_start[s + 1])
    return oracle.paged_prefill(w.chunk_q[a:b], w.k_cache, w.v_cache, w.block_tables[s:s + 1],
                                w.context_lens[s:s + 1], np.array([0, b - a], np.int32), w.scale,
                                w.dtype, num_threads=threads)


def _oracle_prefill_head_rows(w, s, r: int, threads: int) -> int:
    """The oracle on the first ``r`` chunk rows of sequence s; returns their flops.

    Rows 0..r-1 of a chunk of n tokens over L cached tokens attend positions 0..L-n+i,
    which is the chunk of r tokens over L-n+r cached tokens: the same arithmetic."""
    import oracle

    a, b = int(w.query_start[s]), int(w.query_start[s + 1])
    r = min(r, b - a)
    Lr = int(w.context_lens[s]) - (b - a) + r
    oracle.paged_prefill(w.chunk_q[a:a + r], w.k_cache, w.v_cache, w.block_tables[s:s + 1],
                         np.array([Lr], np.int32), np.array([0, r], np.int32), w.scale, w.dtype,
                         num_threads=threads)
    keys = (Lr - r) * r + r * (r + 1) // 2
    return 4 * w.head_dim * w.num_q_heads * keys


def _oracle_prefill_rate(w, seconds: float, threads: int, max_seqs: int, rows: int = 0):
    """TFLOP/s of the prefill oracle over whole sequences (or their first ``rows`` chunk
    rows) until ``seconds`` pass."""
    done, nseq = 0, 0
    s0 = time.perf_counter()
    while True:
        s = nseq % w.num_seqs
        if rows:
            done += _oracle_prefill_head_rows(w, s, rows, threads)
        else:
            _oracle_prefill_seq(w, s, threads)
            done += prefill_flops(w, [s])
        nseq += 1
        el = time.perf_counter() - s0
        if el >= seconds or nseq >= max_seqs:
            break
    return done / el / 1e12, nseq, el


def prefill_config(w) -> dict:
    n = np.diff(w.query_start)
    prior = w.context_lens - n
    recipe = synth.PREFILL_RECIPE
    if w.head_dim != 128:
        recipe = recipe.replace("head_dim 128", f"head_dim {w.head_dim}")
    return {"workload": w.name, "recipe": recipe, "sequences": w.num_seqs,
            "chunk_tokens": int(n.max()), "prior_min_mean_max": [int(prior.min()),
                                                                 float(prior.mean()),
                                                                 int(prior.max())],
            "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
            "block_size": w.block_size, "flops_per_step": prefill_flops(w),
            "l2": "not flushed: every step reads 134 MB of queries and ~150 MB of KV and writes "
                  "134 MB, together above the 129 MiB L2"}


def run_prefill(args) -> None:
    import torch

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    w = synth.prefill_workload(head_dim=args.head_dim)
    if args.impl == "reference":
        if rank != 0:
            return
        import oracle

        oracle.build()
        cpu = host_cpu()
        cores = cpu["usable_cores"]
        for i in range(args.warmup):
            _oracle_prefill_seq(w, i % w.num_seqs, cores)
        flops = 0
        s0 = time.perf_counter()
        for i in range(args.steps):
            _oracle_prefill_seq(w, i % w.num_seqs, cores)
            flops += prefill_flops(w, [i % w.num_seqs])
        el = time.perf_counter() - s0
        value = flops / el / 1e12
        line = {"impl": "reference", "metric": PREFILL_METRIC, "value": round(value, 6),
                "unit": "TFLOP/s", "n_gpus": args.gpus, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(el * 1e3 / args.steps, 3),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic (seeded N(0,1) q/K/V, shuffled block pool)",
                "config": prefill_config(w),
                "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s",
                                 "cores": cores, "kind": "oracle",
                                 "sample": "one sequence's whole chunk per step, cycling through "
                                           "the batch; fp64 C oracle, OpenMP", "cpu": cpu},
                "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch.distributed as dist

    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group(backend="nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import paged_kv_cache_315_gb300 as pkv

    pkv.load()
    t = synth.to_torch(w, dev)
    out = torch.empty_like(t["chunk_q"])
    maxq = int(np.diff(w.query_start).max())
    flops = prefill_flops(w)

    def step(inp, ev=None, dst=None):
        if ev is not None:
            ev[0].record()
        pkv.paged_attn_prefill(out if dst is None else dst, inp["chunk_q"], t["k_cache"],
                               t["v_cache"],
                               inp["block_tables"], inp["context_lens"], inp["query_start"], maxq,
                               w.scale)
        if ev is not None:
            ev[1].record()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(max(3, args.warmup)):
        step(t)
    torch.cuda.synchronize()
    if pkv.pkv_device_error() != 0:
        raise RuntimeError("device error bits set during warm-up")
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    barrier()
    t0.record()
    for i in range(args.steps):
        step(t, evs[i])
    t1.record()
    barrier()
    clk = clocks.stop()
    elapsed_ms = t0.elapsed_time(t1)
    kernel_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    if pkv.pkv_device_error() != 0:
        raise RuntimeError("device error bits set during the timed steps")
    elapsed_ms, kernel_ms = max_over_ranks([elapsed_ms, kernel_ms], world)

    e2e = None
    if not args.no_e2e:
        names = ["chunk_q", "block_tables", "context_lens", "query_start"]
        e2e_s, h2d, d2h = pipelined_e2e(t, names, out, step, dev, args.steps, args.warmup,
                                        barrier)
        (e2e_s,) = max_over_ranks([e2e_s], world)
        e2e = {"value": round(flops * world * args.steps / e2e_s / 1e12, 3), "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": round(e2e_s * 1e3 / args.steps, 4),
               "path": "chunk queries and tables packed in one pinned host buffer -> one "
                       "cudaMemcpyAsync on a copy stream (overlapping the previous step) -> C-ABI "
                       "call -> output to pinned host, each step's output waited for one step "
                       "later"}

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle

        oracle.build()
        hc = host_cpu()
        cores = hc["usable_cores"]
        v1, n1, e1 = _oracle_prefill_rate(w, args.cpu_seconds / 2, 1, w.num_seqs, rows=16)
        vn, nn, en = _oracle_prefill_rate(w, args.cpu_seconds, cores, w.num_seqs)
        cpu = {"value": round(vn, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
               "sample": f"{nn} sequences' whole chunks in {en:.1f} s on {cores} threads; fp64 "
                         f"C oracle, OpenMP over (query row, head)",
               "single_thread": {"value": round(v1, 6), "unit": "TFLOP/s", "cores": 1,
                                 "sample": f"the first 16 chunk rows of {n1} sequences in "
                                           f"{e1:.1f} s on one thread"},
               "cpu": hc}
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return
    peak, peak_kind = tensor_peak()
    value = flops * world * args.steps / (elapsed_ms / 1e3) / 1e12
    achieved = flops / (kernel_ms / 1e3) / 1e12
    line = {
        "metric": PREFILL_METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(elapsed_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q/K/V, shuffled block pool)",
        "config": prefill_config(w), "kernel_ms": round(kernel_ms, 5),
        "roofline": {"kernel": "paged_attn_prefill (prefill_umma_kernel)", "bound": "tensor",
                     "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(achieved / peak, 4), "peak_source": f"{peak_kind} bf16_tflops",
                     "algorithmic_flops_per_launch": flops, "traffic": prefill_traffic(w.name),
                     "traffic_unit": "DRAM bytes per launch"},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": args.steps, "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main(argv=None):
    args = parse_args(argv)
    if args.op == "swap":
        run_swap(args)
        return
    if args.op == "prefill":
        run_prefill(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
