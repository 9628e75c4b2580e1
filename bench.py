#!/usr/bin/env python
"""Benchmark of one paged decode step on GB300.

A step is the whole hot path over one batch: copy_blocks (copy-on-write
pairs, if the workload has any), reshape_and_cache of the step's new K/V
rows, and paged decode attention over every sequence's context - all through
the C ABI of libpagedattn.so.  The default workload is the LLaMA-13B-shaped
layer: 256 sequences, 40 heads x 128 dims, block_size 16, long-tailed
context lengths (lognormal, median 300, clipped to [1, 2048]), bf16.

Metric: KV-read HBM GB/s (and us/step).  One JSON line is printed by rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

``--impl reference`` times the CPU oracle (fp64 C, all host cores) on a
bounded sample of the same workload.  Under torchrun (N > 1) every rank runs
its own replica batch (weak scaling, no collective on the data path);
``value`` is the KV bytes of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

WORKLOAD_TEXT = {
    "13b": "LLaMA-13B-shaped decode step, one layer: 256 seqs, 40 heads (MHA), head_dim 128, block_size 16, "
           "context lognormal(median 300, sigma 1) clipped to [1,2048], bf16, reshape_and_cache of each "
           "sequence's new token via a random slot_mapping",
    "13b_fp8": "LLaMA-13B-shaped decode step, one layer, FP8 (e4m3) KV cache with per-tensor scales: 256 seqs, "
               "40 heads, head_dim 128, block_size 16, context lognormal(median 300, sigma 1) clipped to [1,2048], "
               "bf16 queries, quantising reshape_and_cache of each sequence's new token",
    "7b": "LLaMA-7B-shaped decode step, one layer: 64 seqs, 32 heads (MHA), head_dim 128, block_size 16, "
          "context uniform [32,2048], f16",
    "gqa": "GQA long-context decode: 16 seqs, 32 q / 8 kv heads, head_dim 128, block_size 16, context "
           "uniform [16384,32768], 512-token partitions, bf16",
    "gqa32": "GQA long-context decode: 16 seqs, 32 q / 8 kv heads, head_dim 128, block_size 32, context "
             "uniform [16384,32768], 512-token partitions, bf16",
    "prefix": "prefix-sharing decode: 64 prompts x 4 samples sharing a 1000-token prompt, private 0-256 "
              "token suffix, copy-on-write of the shared partial block, 32 heads, head_dim 128, f16",
    "tiny": "tiny paged decode: 4 seqs, context {1,17,35,100}, 4 heads, head_dim 64, block_size 16, f16",
    "prefill": "LLaMA-13B-shaped chunked prefill, one layer: 16 seqs, a 512-token chunk each over a cached "
               "prefix of U{0..2048} tokens, causal, 40 heads (MHA), head_dim 128, block_size 16, bf16, "
               "reshape_and_cache of the chunk's K/V",
    "prefill_gqa": "GQA chunked prefill, one layer: 8 seqs, a 1024-token chunk each over a cached prefix of "
                   "U{0..8192} tokens, causal, 32 q / 8 kv heads, head_dim 128, block_size 16, bf16",
    "prefill_prefix": "prefill after a prefix-cache hit: 64 prompts x 4 samples share a cached 1000-token prompt; "
                      "each sample's private 1-257-token tail is prefilled causally over it (copy-on-write of "
                      "the shared partial block first), 32 heads, head_dim 128, f16",
}
PREFILL_WORKLOADS = {"prefill": "prefill", "prefill_gqa": "prefill_gqa", "prefill_prefix": "prefix"}

MEASURED_PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0


# --------------------------------------------------------------- configs

def decode_config(b, name: str, world: int) -> dict:
    """The decode workload's config, identical in both arms' lines
    (partition_size as requested: 0 = the library's automatic choice)."""
    kvb = kv_bytes(b)
    return {
        "workload": WORKLOAD_TEXT.get(name, name),
        "name": name,
        "num_seqs": b.num_seqs, "num_heads": b.num_heads, "num_kv_heads": b.num_kv_heads,
        "head_dim": b.head_dim, "block_size": b.block_size, "num_blocks": b.num_blocks,
        "dtype": b.dtype, "cache_dtype": b.cache_dtype,
        "tokens": int(b.context_lens.sum()), "max_context_len": b.max_context_len,
        "partition_size": int(b.partition_size), "kv_bytes_per_step": kvb,
        "kv_bytes_unique_per_step": kv_bytes_unique(b),
        "l2": "no flush: each step reads %.2f GB of K/V, far larger than the 126 MB L2" % (kvb / 1e9),
        "parallelism": f"replicas x{world} (independent batches per GPU)",
    }


def prefill_config(b, name: str, world: int) -> dict:
    """The prefill workload's config, identical in both arms' lines."""
    kvb = kv_bytes(b)
    return {
        "workload": WORKLOAD_TEXT[name], "name": name,
        "num_seqs": b.num_seqs, "num_heads": b.num_heads, "num_kv_heads": b.num_kv_heads,
        "head_dim": b.head_dim, "block_size": b.block_size, "num_blocks": b.num_blocks,
        "query_tokens": b.num_tokens, "context_tokens": int(b.context_lens.sum()),
        "flops_per_step": prefill_flops(b), "kv_bytes_read_once": kvb,
        "l2": "no flush: K/V %.2f GB plus queries %.2f GB per step, above the 126 MB L2"
              % (kvb / 1e9, b.q.nbytes / 1e9),
        "parallelism": f"replicas x{world} (independent batches per GPU)",
    }


def cpu_model() -> str:
    """The host CPU's model name (lscpu), for the CPU-baseline record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


# --------------------------------------------------------------- accounting

def kv_bytes(b) -> int:
    """Bytes of K and V a decode step reads: sum_s ctx_s * Hkv * D * 2 (K,V) * element bytes."""
    return int(b.context_lens.astype("int64").sum()) * b.num_kv_heads * b.head_dim * 2 * b.elem_bytes


def kv_bytes_unique(b) -> int:
    """Bytes of K and V in the distinct cache slots a decode step reads: a
    slot that several sequences read through shared blocks counts once (the
    decode kernel loads a shared stage once for all of them)."""
    import numpy as np
    ctx = b.context_lens.astype(np.int64)
    parts = []
    for s in range(b.num_seqs):
        pos = np.arange(int(ctx[s]), dtype=np.int64)
        parts.append(b.block_tables[s, pos // b.block_size].astype(np.int64) * b.block_size + pos % b.block_size)
    slots = np.unique(np.concatenate(parts)) if parts else np.zeros(0, np.int64)
    return int(slots.size) * b.num_kv_heads * b.head_dim * 2 * b.elem_bytes


def decode_bytes(b, partition: int) -> int:
    """Algorithmic bytes of one pa_decode launch: the K/V rows of the distinct
    slots read, queries, outputs, block-table entries, context lengths and the
    split-K partial states (written once, read once by the merge)."""
    import numpy as np
    ctx = b.context_lens.astype(np.int64)
    G = b.num_heads // b.num_kv_heads
    q = b.num_seqs * b.num_heads * b.head_dim * 2
    out = b.num_seqs * b.num_heads * b.head_dim * 2
    tables = int(np.ceil(ctx / b.block_size).sum()) * 4 * b.num_kv_heads
    nparts = np.where(ctx > 0, -(-ctx // partition), 1)
    split = int(nparts[nparts > 1].sum()) * b.num_kv_heads * G * (b.head_dim + 2) * 4 * 2
    return kv_bytes_unique(b) + q + out + tables + b.num_seqs * 4 + split


def step_bytes(b, partition: int) -> int:
    rows = len(b.slot_mapping) * b.num_kv_heads * b.head_dim * 2 * (2 + b.elem_bytes)  # K,V read + write
    copies = len(b.block_mapping) * b.block_size * b.num_kv_heads * b.head_dim * 2 * 2 * b.elem_bytes
    return decode_bytes(b, partition) + rows + copies


def prefill_row_positions(b):
    """Position of every query row of a prefill batch (row i of sequence s:
    ctx_s - q_len_s + i)."""
    import numpy as np
    cu = b.cu_seqlens_q.astype(np.int64)
    ql = np.diff(cu)
    seq = np.repeat(np.arange(b.num_seqs), ql)
    return b.context_lens[seq].astype(np.int64) - ql[seq] + (np.arange(int(cu[-1])) - cu[seq])


def prefill_flops(b, rows=None) -> int:
    """Algorithmic FLOPs of causal prefill attention: every (query row, head)
    attends pos + 1 keys, 2 D FLOPs for QK^T and 2 D for PV each."""
    pos = prefill_row_positions(b)
    if rows is not None:
        pos = pos[rows]
    return int((pos + 1).sum()) * 4 * b.head_dim * b.num_heads


def tensor_peak():
    """Measured dense bf16 tensor throughput (burst), TFLOP/s."""
    try:
        with open(MEASURED_PEAKS) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def hbm_peak():
    try:
        with open(MEASURED_PEAKS) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# ------------------------------------------------------------ distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(backend: str):
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def aggregate(ms_per_step: float, units: float, world: int):
    """Slowest rank's time and the units all ranks processed."""
    if world <= 1:
        return ms_per_step, units
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([ms_per_step], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ clocks

CLOCK_QUERY = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


class ClockSampler:
    """nvidia-smi sampling (every 200 ms) around the timed region."""

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={CLOCK_QUERY}", "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(", ") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        if self.uuid:
            mine = [r for r in rows if len(r) > 1 and r[1].strip() == self.uuid]
            rows = mine or rows
        sm, mx, reasons = [], [], set()
        for r in rows:
            try:
                sm.append(float(r[2]))
                mx.append(float(r[3]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(REASONS, r[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------- GPU arm

def device_tensors(b, device):
    import numpy as np
    import torch
    tdt = torch.float16 if b.dtype == "f16" else torch.bfloat16

    def h(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(tdt)

    host = dict(q=h(b.q), key=h(b.key), value=h(b.value),
                slot_mapping=torch.from_numpy(b.slot_mapping), block_tables=torch.from_numpy(b.block_tables),
                context_lens=torch.from_numpy(b.context_lens),
                block_mapping=torch.from_numpy(np.ascontiguousarray(b.block_mapping)))
    dev = {k: v.to(device) for k, v in host.items()}
    if b.cache_dtype == "fp8":
        dev["k_cache"] = torch.from_numpy(b.k_cache).to(device)
        dev["v_cache"] = torch.from_numpy(b.v_cache).to(device)
    else:
        dev["k_cache"] = h(b.k_cache).to(device)
        dev["v_cache"] = h(b.v_cache).to(device)
    return host, dev


def decode_kernel_name(b):
    """The decode kernel pa_decode / pa_decode_append run for this batch: the
    CTA-cooperative one for 16-bit or e4m3 caches whose KV heads come in groups
    of 8 (head_dim 128, block size a multiple of 16; PA_DECODE_COOP=0 turns it
    off), else the per-warp one."""
    coop = (os.environ.get("PA_DECODE_COOP", "1")[:1] != "0" and b.head_dim == 128
            and b.num_kv_heads % 8 == 0 and b.block_size % 16 == 0)
    return "paged_decode_coop_kernel" if coop else "paged_decode_kernel"


def step_percentiles(marks):
    """p10 / p50 / p90 of the per-step times (us) between consecutive events."""
    ts = sorted(a.elapsed_time(z) * 1e3 for a, z in zip(marks[:-1], marks[1:]))
    if not ts:
        return None
    q = lambda f: round(ts[min(len(ts) - 1, int(f * (len(ts) - 1) + 0.5))], 2)
    return {"p10": q(0.1), "p50": q(0.5), "p90": q(0.9)}


def stage_inputs(tensors, device):
    """One pinned host buffer holding every tensor of ``tensors`` (256-byte
    aligned) and its device twin, with device views shaped like the inputs:
    a step's inputs then cross to the GPU in one copy, as a serving engine
    stages them."""
    import torch
    offs, n = {}, 0
    for k, v in tensors.items():
        offs[k] = n
        n += (v.numel() * v.element_size() + 255) // 256 * 256
    flat_h = torch.empty(max(n, 256), dtype=torch.uint8).pin_memory()
    flat_d = torch.empty(max(n, 256), dtype=torch.uint8, device=device)
    views = {}
    for k, v in tensors.items():
        nb = v.numel() * v.element_size()
        flat_h[offs[k]:offs[k] + nb].copy_(v.contiguous().view(-1).view(torch.uint8))
        views[k] = flat_d[offs[k]:offs[k] + nb].view(v.dtype).view(v.shape)
    return flat_h, flat_d, views


def time_e2e_direct(launch, flat_h, flat_d, out, out_h, stream, K, warmup, world):
    """The end-to-end step with the library's entry points called through the
    Python binding every step (no graph): one pinned-input copy, the calls,
    the output back to pinned host memory, a stream sync.  Host milliseconds
    per step."""
    def one():
        flat_d.copy_(flat_h, non_blocking=True)
        launch()
        out_h.copy_(out, non_blocking=True)
        stream.synchronize()

    for _ in range(max(3, warmup)):
        one()
    barrier(world)
    w0 = time.perf_counter()
    for _ in range(K):
        one()
    ms = (time.perf_counter() - w0) * 1e3 / K
    barrier(world)
    return ms


def time_e2e_pipelined(graphs, flats, outs, outs_h, stream, K, warmup, world):
    """The end-to-end step as a serving loop overlaps it: two sets of device
    inputs and outputs, each step's pinned inputs copied in on one copy
    stream while the previous step computes, and its result copied back to
    pinned host memory on another while the next one does.  Every step still
    moves its own inputs and result across the host link.  Host
    milliseconds per step over K steps (one synchronisation at the end)."""
    import torch
    h2d_s, d2h_s = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()
    copied = [ev(), ev()]
    computed = [ev(), ev()]
    returned = [ev(), ev()]
    started = [False, False]

    def step(k):
        i = k & 1
        with torch.cuda.stream(h2d_s):
            if started[i]:
                h2d_s.wait_event(computed[i])      # step k - 2 is done reading these inputs
            flats[i][1].copy_(flats[i][0], non_blocking=True)
            copied[i].record(h2d_s)
        stream.wait_event(copied[i])
        if started[i]:
            stream.wait_event(returned[i])         # step k - 2's result has left this output
        graphs[i].replay()
        computed[i].record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(computed[i])
            outs_h[i].copy_(outs[i], non_blocking=True)
            returned[i].record(d2h_s)
        started[i] = True

    for k in range(max(3, warmup)):
        step(k)
    torch.cuda.synchronize()
    barrier(world)
    w0 = time.perf_counter()
    for k in range(K):
        step(k)
    torch.cuda.synchronize()
    ms = (time.perf_counter() - w0) * 1e3 / K
    barrier(world)
    return ms


def e2e_pipelined_entry(units_all, unit, ms, world, h2d, d2h):
    ms_max, _ = aggregate(ms, 0.0, world)
    return {"value": round(units_all / (ms_max * 1e-3), 2 if unit == "TFLOP/s" else 1), "unit": unit,
            "ms_per_step": round(ms_max, 4), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "note": "as e2e, with each step's input copy and result copy on their own streams, overlapping "
                    "the neighbouring steps' compute (two input and output buffer sets, one graph each)"}


def e2e_direct_entry(units_all, unit, ms, world, h2d, d2h):
    ms_max, _ = aggregate(ms, 0.0, world)
    return {"value": round(units_all / (ms_max * 1e-3), 2 if unit == "TFLOP/s" else 1), "unit": unit,
            "ms_per_step": round(ms_max, 4), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "note": "as e2e, but the step's C-ABI calls made through the Python binding every step "
                    "(argument checks, tensor-map encoding and launches on the host each time) instead of a "
                    "graph replay"}


def run_ours(args, world, rank, local):
    import numpy as np
    import torch

    import paged_kv_cache_140_gb300 as pa
    from paged_kv_cache_140_gb300 import workloads as W

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device for --impl ours")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist_init("nccl")
    pa._lib.load()  # fail loudly before any work if the library is missing

    cfg = W.CONFIGS[args.workload]
    seed = 140000 + cfg["number"] + 1000 * rank
    b = W.make_batch(args.workload, seed=seed)
    host, T = device_tensors(b, device)
    out = torch.empty(T["q"].shape, dtype=T["q"].dtype, device=device)
    P = pa.decode_partition_size(b.num_seqs, b.num_heads, b.num_kv_heads, b.head_dim, b.block_size,
                                 b.max_context_len, b.partition_size)
    ws = pa.DecodeWorkspace(device)
    has_pairs = len(b.block_mapping) > 0
    # pa_decode adds a merge launch when some sequence spans several partitions.
    split = pa.decode_workspace_size(b.num_seqs, b.num_heads, b.num_kv_heads, b.head_dim, b.block_size,
                                     b.max_context_len, b.partition_size) > 0
    stream = torch.cuda.current_stream(device)

    # The step as one pa_decode_append call where it applies (one new token
    # per sequence at position ctx - 1, no copy-on-write pairs first) and runs
    # on the cooperative kernel (append kernel + decode chained, measured
    # faster than the separate calls); --fused forces it on the per-warp kernel
    # too (in-kernel append, measured slower); else, or with --separate,
    # reshape_and_cache followed by decode.
    applicable = not has_pairs and len(b.slot_mapping) == int((b.context_lens > 0).sum())
    fused = applicable and not args.separate and (
        args.fused or decode_kernel_name(b) == "paged_decode_coop_kernel")
    if fused:
        has = torch.from_numpy(np.nonzero(b.context_lens > 0)[0]).to(device)
        T["key_rows"] = torch.zeros((b.num_seqs, b.num_kv_heads, b.head_dim), dtype=T["key"].dtype,
                                    device=device)
        T["value_rows"] = torch.zeros_like(T["key_rows"])
        T["key_rows"][has] = T["key"]
        T["value_rows"][has] = T["value"]

    def step(ev=None):
        if has_pairs:
            pa.copy_blocks(T["k_cache"], T["v_cache"], T["block_mapping"])
        if fused:
            # reshape_and_cache fused into the decode launch
            if ev is not None:
                ev[0].record(stream)
            pa.decode_append(out, T["q"], T["key_rows"], T["value_rows"], T["k_cache"], T["v_cache"],
                             T["block_tables"], T["context_lens"], float(b.scale),
                             max_context_len=b.max_context_len, partition_size=b.partition_size,
                             workspace=ws, k_scale=b.k_scale, v_scale=b.v_scale)
            if ev is not None:
                ev[1].record(stream)
            return
        pa.reshape_and_cache(T["key"], T["value"], T["k_cache"], T["v_cache"], T["slot_mapping"],
                             k_scale=b.k_scale, v_scale=b.v_scale)
        if ev is not None:
            ev[0].record(stream)
        pa.decode(out, T["q"], T["k_cache"], T["v_cache"], T["block_tables"], T["context_lens"],
                  float(b.scale), max_context_len=b.max_context_len, partition_size=b.partition_size,
                  workspace=ws, k_scale=b.k_scale, v_scale=b.v_scale)
        if ev is not None:
            ev[1].record(stream)

    err = pa.new_err_flag(device)
    pa.decode(out, T["q"], T["k_cache"], T["v_cache"], T["block_tables"], T["context_lens"],
              float(b.scale), max_context_len=b.max_context_len, partition_size=b.partition_size,
              workspace=ws, err_flag=err, k_scale=b.k_scale, v_scale=b.v_scale)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    flag = pa.read_err_flag(err)
    if flag:
        raise SystemExit(f"device error flag {flag:#x} during warm-up")

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(device).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    if args.clock_probe_s > 0:  # keep the GPU busy long enough for the sampler
        t_end = time.time() + args.clock_probe_s
        while time.time() < t_end:
            for _ in range(20):
                step()
            torch.cuda.synchronize()

    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    t0.record(stream)
    marks[0].record(stream)
    for k in range(K):
        step(evs[k])
        marks[k + 1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    ms_total = t0.elapsed_time(t1)
    ms_step = ms_total / K
    decode_ms = statistics.mean(a.elapsed_time(z) for a, z in evs)
    pct = step_percentiles(marks)

    # End to end: the step's inputs staged in one pinned host buffer and
    # copied in one transfer, the step's launches replayed as one CUDA graph
    # (pa.StepGraph), the result copied back to pinned host memory.
    used = {k: v for k, v in host.items() if k != "block_mapping" or has_pairs}
    if fused:
        # pa_decode_append takes one new row per sequence; no slot mapping
        used = {k: v for k, v in used.items() if k not in ("key", "value", "slot_mapping")}
        used["key_rows"] = T["key_rows"].cpu()
        used["value_rows"] = T["value_rows"].cpu()
    flat_h, flat_d, e2e_in = stage_inputs(used, device)
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in used.values())
    d2h = out_h.numel() * out_h.element_size()

    def e2e_kernels(e2e_in=e2e_in, out=out, ws=ws):
        if fused:
            pa.decode_append(out, e2e_in["q"], e2e_in["key_rows"], e2e_in["value_rows"], T["k_cache"],
                             T["v_cache"], e2e_in["block_tables"], e2e_in["context_lens"], float(b.scale),
                             max_context_len=b.max_context_len, partition_size=b.partition_size,
                             workspace=ws, k_scale=b.k_scale, v_scale=b.v_scale)
            return
        if has_pairs:
            pa.copy_blocks(T["k_cache"], T["v_cache"], e2e_in["block_mapping"])
        pa.reshape_and_cache(e2e_in["key"], e2e_in["value"], T["k_cache"], T["v_cache"], e2e_in["slot_mapping"],
                             k_scale=b.k_scale, v_scale=b.v_scale)
        pa.decode(out, e2e_in["q"], T["k_cache"], T["v_cache"], e2e_in["block_tables"], e2e_in["context_lens"],
                  float(b.scale), max_context_len=b.max_context_len, partition_size=b.partition_size,
                  workspace=ws, k_scale=b.k_scale, v_scale=b.v_scale)

    flat_d.copy_(flat_h, non_blocking=True)
    step_graph = pa.StepGraph(e2e_kernels)

    def e2e_step():
        flat_d.copy_(flat_h, non_blocking=True)
        step_graph.replay()
        out_h.copy_(out, non_blocking=True)
        stream.synchronize()

    for _ in range(max(3, args.warmup)):
        e2e_step()
    barrier(world)
    w0 = time.perf_counter()
    for _ in range(K):
        e2e_step()
    e2e_ms = (time.perf_counter() - w0) * 1e3 / K
    barrier(world)
    e2e_direct_ms = time_e2e_direct(e2e_kernels, flat_h, flat_d, out, out_h, stream, K, args.warmup, world)
    # the second buffer set of the overlapped loop (its own workspace: two
    # steps' decodes never overlap on the one compute stream, but each graph
    # keeps the addresses it was captured with)
    flat_h2, flat_d2, e2e_in2 = stage_inputs(used, device)
    out2 = torch.empty_like(out)
    out_h2 = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    ws2 = pa.DecodeWorkspace(device)
    flat_d2.copy_(flat_h2, non_blocking=True)
    step_graph2 = pa.StepGraph(lambda: e2e_kernels(e2e_in2, out2, ws2))
    e2e_pipe_ms = time_e2e_pipelined([step_graph, step_graph2], [(flat_h, flat_d), (flat_h2, flat_d2)],
                                     [out, out2], [out_h, out_h2], stream, K, args.warmup, world)

    kvb = kv_bytes(b)
    ms_max, kv_all = aggregate(ms_step, float(kvb), world)
    e2e_max, _ = aggregate(e2e_ms, float(kvb), world)
    dec_max, _ = aggregate(decode_ms, 0.0, world)
    peak, peak_kind = hbm_peak()
    value = kv_all / (ms_max * 1e-3) / 1e9
    dbytes = decode_bytes(b, P)
    achieved = dbytes / (decode_ms * 1e-3) / 1e9
    traffic = load_traffic(args.workload)

    line = {
        "metric": "paged decode attention: KV-read HBM GB/s (% of GB300 peak), us/step",
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 5),
        "us_per_step": round(ms_max * 1e3, 2),
        "us_per_step_pct": pct,
        "pct_of_hbm_peak": round(100 * value / world / peak, 1),
        "pct_of_nominal_8TBs": round(100 * value / world / NOMINAL_HBM_GBS, 1),
        "peak_kind": peak_kind,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": b.dtype if b.cache_dtype == b.dtype else f"{b.dtype} q, {b.cache_dtype} kv",
        "data": "synthetic (seeded N(0,1) K/V/Q, seeded block permutation, NaN in unused slots)",
        "impl": "ours",
        "config": decode_config(b, args.workload, world),
        "partition_size": P,
        "step_bytes": step_bytes(b, P),
        "seqs_tokens_per_s": round(float(b.context_lens.sum()) * world / (ms_max * 1e-3), 1),
        "roofline": {
            "kernel": decode_kernel_name(b),
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "algorithmic_bytes_per_launch": dbytes,
            "launch_us": round(decode_ms * 1e3, 2),
        },
        "e2e": {"value": round(kv_all / (e2e_max * 1e-3) / 1e9, 1), "unit": "GB/s",
                "ms_per_step": round(e2e_max, 4), "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "note": "per step: pinned host inputs (q, the new K/V rows, block_tables, context_lens; "
                        "slot_mapping too for the separate calls) staged in one pinned buffer -> device in one "
                        "copy, the step's launches replayed as one CUDA graph (pa.StepGraph), output -> pinned "
                        "host, stream sync; the KV cache stays resident"},
        "e2e_direct": e2e_direct_entry(kv_all / 1e9, "GB/s", e2e_direct_ms, world, h2d, d2h),
        "e2e_pipelined": e2e_pipelined_entry(kv_all / 1e9, "GB/s", e2e_pipe_ms, world, h2d, d2h),
        # fused on the cooperative kernel: an append kernel, then the decode
        "gpu_launches": K * ((2 if (not fused or decode_kernel_name(b) == "paged_decode_coop_kernel") else 1) +
                             (1 if has_pairs else 0) + (1 if split else 0)),
        "fused_append": bool(fused),
        "step": ("pa_decode_append (the new rows appended, then attended)" if fused else
                 ("pa_copy_blocks + " if has_pairs else "") + "pa_reshape_and_cache + pa_decode"),
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(b, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)


def _prefill_batch(args, rank=0):
    from paged_kv_cache_140_gb300 import workloads as W
    name = PREFILL_WORKLOADS[args.workload]
    if name == "prefix":
        seed = 140000 + W.CONFIGS["prefix"]["number"] + 1000 * rank
    else:
        seed = 140000 + W.PREFILL_CONFIGS[name]["number"] + 1000 * rank
    return W.make_prefill_batch(name, seed=seed)


def run_prefill(args, world, rank, local):
    """One prefill step: copy_blocks (if any), reshape_and_cache of the new
    tokens' K/V, causal prefill attention of their queries."""
    import numpy as np
    import torch

    import paged_kv_cache_140_gb300 as pa

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device for --impl ours")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist_init("nccl")
    pa._lib.load()
    b = _prefill_batch(args, rank)
    host, T = device_tensors(b, device)
    host["cu_seqlens_q"] = torch.from_numpy(b.cu_seqlens_q)
    T["cu_seqlens_q"] = host["cu_seqlens_q"].to(device)
    out = torch.empty(T["q"].shape, dtype=T["q"].dtype, device=device)
    has_pairs = len(b.block_mapping) > 0
    stream = torch.cuda.current_stream(device)

    def step(ev=None, src=T):
        if has_pairs:
            pa.copy_blocks(T["k_cache"], T["v_cache"], src["block_mapping"])
        pa.reshape_and_cache(src["key"], src["value"], T["k_cache"], T["v_cache"], src["slot_mapping"])
        if ev is not None:
            ev[0].record(stream)
        pa.prefill(out, src["q"], T["k_cache"], T["v_cache"], src["block_tables"], src["context_lens"],
                   src["cu_seqlens_q"], float(b.scale), max_q_len=b.max_q_len)
        if ev is not None:
            ev[1].record(stream)

    err = pa.new_err_flag(device)
    pa.prefill(out, T["q"], T["k_cache"], T["v_cache"], T["block_tables"], T["context_lens"], T["cu_seqlens_q"],
               float(b.scale), max_q_len=b.max_q_len, err_flag=err)
    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    flag = pa.read_err_flag(err)
    if flag:
        raise SystemExit(f"device error flag {flag:#x} during warm-up")

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(device).uuid)
        uuid = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
    except Exception:
        pass
    sampler = ClockSampler(uuid)
    sampler.start()
    if args.clock_probe_s > 0:
        t_end = time.time() + args.clock_probe_s
        while time.time() < t_end:
            for _ in range(10):
                step()
            torch.cuda.synchronize()
    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    t0.record(stream)
    marks[0].record(stream)
    for k in range(K):
        step(evs[k])
        marks[k + 1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    ms_step = t0.elapsed_time(t1) / K
    attn_ms = statistics.mean(a.elapsed_time(z) for a, z in evs)
    pct = step_percentiles(marks)

    # End to end as for decode: one staged copy in, the step as one graph
    # launch, the result back to pinned host memory.
    used = {k: v for k, v in host.items() if k != "block_mapping" or has_pairs}
    flat_h, flat_d, e2e_in = stage_inputs(used, device)
    out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(v.numel() * v.element_size() for v in used.values())
    d2h = out_h.numel() * out_h.element_size()
    flat_d.copy_(flat_h, non_blocking=True)
    step_graph = pa.StepGraph(lambda: step(src=e2e_in))

    def e2e_step():
        flat_d.copy_(flat_h, non_blocking=True)
        step_graph.replay()
        out_h.copy_(out, non_blocking=True)
        stream.synchronize()

    for _ in range(max(3, args.warmup)):
        e2e_step()
    barrier(world)
    w0 = time.perf_counter()
    for _ in range(K):
        e2e_step()
    e2e_ms = (time.perf_counter() - w0) * 1e3 / K
    barrier(world)
    e2e_direct_ms = time_e2e_direct(lambda: step(src=e2e_in), flat_h, flat_d, out, out_h, stream, K, args.warmup,
                                    world)

    flops = prefill_flops(b)
    ms_max, fl_all = aggregate(ms_step, float(flops), world)
    e2e_max, _ = aggregate(e2e_ms, float(flops), world)
    peak, peak_kind = tensor_peak()
    value = fl_all / (ms_max * 1e-3) / 1e12
    achieved = flops / (attn_ms * 1e-3) / 1e12
    kvb = kv_bytes(b)
    line = {
        "metric": "paged prefill attention: causal TFLOP/s (algorithmic), us/step",
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 5),
        "us_per_step": round(ms_max * 1e3, 2),
        "us_per_step_pct": pct,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": b.dtype,
        "data": "synthetic (seeded N(0,1) K/V/Q, seeded block permutation, NaN in unused slots)",
        "impl": "ours",
        "config": prefill_config(b, args.workload, world),
        "roofline": {
            "kernel": "paged_prefill_kernel",
            "bound": "tensor",
            "achieved": round(achieved, 2),
            "peak": peak,
            "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4),
            "traffic": load_traffic(args.workload, "prefill"),
            "algorithmic_flops_per_launch": flops,
            "launch_us": round(attn_ms * 1e3, 2),
            "peak_kind": peak_kind,
        },
        "e2e": {"value": round(fl_all / (e2e_max * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_max, 4), "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                "note": "per step: pinned host q/new K,V/slot_mapping/block_tables/context_lens/cu_seqlens_q "
                        "(staged in one pinned buffer) -> device in one copy, the step's launches replayed as one "
                        "CUDA graph (pa.StepGraph), output -> pinned host, stream sync; the KV cache stays resident"},
        "e2e_direct": e2e_direct_entry(fl_all / 1e12, "TFLOP/s", e2e_direct_ms, world, h2d, d2h),
        "gpu_launches": K * (2 + (1 if has_pairs else 0)),
        "step": ("pa_copy_blocks + " if has_pairs else "") + "pa_reshape_and_cache + pa_prefill",
        "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = prefill_cpu_baseline(b, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)


def _prefill_oracle_rows(b, kc, vc, rows):
    import numpy as np

    import oracle
    cu = b.cu_seqlens_q.astype(np.int64)
    seq = np.searchsorted(cu, rows, side="right") - 1
    pos = prefill_row_positions(b)[rows]
    return oracle.paged_attention(b.q[rows], kc, vc, b.dtype, b.block_tables[seq], (pos + 1).astype(np.int32),
                                  b.scale)


def _prefill_sample(b, kc, vc, target_s):
    """Evenly spaced query rows whose oracle attention takes about target_s."""
    import numpy as np
    n = b.num_tokens
    probe = np.linspace(0, n - 1, min(n, 32)).astype(np.int64)
    t = time.perf_counter()
    _prefill_oracle_rows(b, kc, vc, probe)
    per_flop = max(time.perf_counter() - t, 1e-4) / max(1, prefill_flops(b, probe))
    want = max(1, min(n, int(round(n * target_s / (per_flop * prefill_flops(b))))))
    return np.linspace(0, n - 1, want).astype(np.int64)


def prefill_cpu_baseline(b, target_s):
    threads = _oracle_threads()
    kc, vc = _post_step_caches(b)
    rows = _prefill_sample(b, kc, vc, target_s)
    t = time.perf_counter()
    _prefill_oracle_rows(b, kc, vc, rows)
    dt = time.perf_counter() - t
    fl = prefill_flops(b, rows)
    return {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": threads, "cpu_model": cpu_model(),
            "kind": "oracle",
            "seconds": round(dt, 2),
            "sample": f"{len(rows)} of {b.num_tokens} query rows (evenly spaced, all heads; {fl} FLOPs) over the "
                      f"post-step caches; fp64 C oracle, OpenMP over (row, head)"}


def run_prefill_reference(args, world, rank):
    if rank != 0:
        return
    threads = _oracle_threads()
    b = _prefill_batch(args)
    kc, vc = _post_step_caches(b)
    rows = _prefill_sample(b, kc, vc, min(2.0, 150.0 / max(1, args.steps + args.warmup)))
    for _ in range(args.warmup):
        _prefill_oracle_rows(b, kc, vc, rows)
    t = time.perf_counter()
    for _ in range(args.steps):
        _prefill_oracle_rows(b, kc, vc, rows)
    dt = (time.perf_counter() - t) / args.steps
    fl = prefill_flops(b, rows)
    value = fl / dt / 1e12
    print(json.dumps({
        "metric": "paged prefill attention: causal TFLOP/s (algorithmic), us/step",
        "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": b.dtype, "data": "synthetic", "impl": "reference",
        "config": prefill_config(b, args.workload, world),
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": threads, "cpu_model": cpu_model(),
                         "kind": "oracle",
                         "sample": f"{len(rows)} of {b.num_tokens} query rows per step ({fl} FLOPs)"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


KERNEL_SOURCES = {
    "decode": ("pa_decode.cu", "pa_decode_coop.cu", "pa_decode_common.cuh", "pa_device.cuh", "pa_internal.h"),
    "prefill": ("pa_prefill.cu", "pa_prefill.h", "pa_umma.cuh", "pa_device.cuh"),
}


def _code_only(text: str) -> str:
    """C++ source with comments and whitespace removed (string literals kept),
    so that editing a comment does not change a kernel's hash."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"' or c == "'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            if not c.isspace():
                out.append(c)
            i += 1
    return "".join(out)


def source_hash(kind: str = "decode") -> str:
    """Hash of a kernel's sources (code only, comments and whitespace
    ignored); a traffic figure taken from other kernel code is not reported."""
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "paged_kv_cache_140_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def decode_source_hash() -> str:
    return source_hash("decode")


def load_traffic(workload, kind: str = "decode"):
    """DRAM bytes per launch of the workload's main kernel (ncu
    dram__bytes_read.sum + write.sum) from the committed profile summary, or
    None when the summary was taken on a different kernel source."""
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}.json")
    try:
        with open(path) as f:
            d = json.load(f)
        if d.get("kernel_source_hash") != source_hash(kind):
            return None
        return d.get("dram_bytes_per_launch")
    except Exception:
        return None


# ------------------------------------------------------------- CPU oracle

def _oracle_threads() -> int:
    n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    os.environ.setdefault("OMP_NUM_THREADS", str(n))
    return int(os.environ["OMP_NUM_THREADS"])


def _post_step_caches(b):
    import oracle
    kc, vc = b.k_cache, b.v_cache
    fp8 = b.cache_dtype == "fp8"
    if len(b.block_mapping):
        kc, vc, _ = (oracle.copy_blocks_bytes if fp8 else oracle.copy_blocks)(kc, vc, b.block_mapping)
    if fp8:
        kc, vc, _ = oracle.reshape_and_cache_fp8(b.key, b.value, b.dtype, kc, vc, b.slot_mapping, b.k_scale,
                                                 b.v_scale)
    else:
        kc, vc, _ = oracle.reshape_and_cache(b.key, b.value, kc, vc, b.slot_mapping)
    return kc, vc


def _oracle_attention(b, sub, kc, vc):
    import oracle
    if b.cache_dtype == "fp8":
        return oracle.paged_attention_fp8(sub.q, b.dtype, kc, vc, b.k_scale, b.v_scale, sub.block_tables,
                                          sub.context_lens, b.scale)
    return oracle.paged_attention(sub.q, kc, vc, b.dtype, sub.block_tables, sub.context_lens, b.scale)


def _pick_sample(b, target_s, kc, vc):
    """Sequences (every k-th) whose oracle attention takes about target_s."""
    import numpy as np

    import oracle
    from paged_kv_cache_140_gb300 import workloads as W
    probe = list(range(0, b.num_seqs, max(1, b.num_seqs // 8)))[:8]
    sub = W.subset_batch(b, probe)
    t = time.perf_counter()
    _oracle_attention(b, sub, kc, vc)
    dt = max(time.perf_counter() - t, 1e-4)
    per_tok = dt / max(1, int(sub.context_lens.sum()))
    want_tok = target_s / per_tok
    order = np.arange(b.num_seqs)
    total = int(b.context_lens.sum())
    if want_tok >= total:
        return list(order)
    stride = max(1, int(round(total / want_tok)))
    return list(order[::stride])


def cpu_baseline(b, target_s):
    threads = _oracle_threads()
    import oracle
    from paged_kv_cache_140_gb300 import workloads as W
    kc, vc = _post_step_caches(b)
    pick = _pick_sample(b, target_s, kc, vc)
    sub = W.subset_batch(b, pick)
    runs = 0
    t = time.perf_counter()
    while True:  # repeat a sample that is the whole batch until ~target_s of CPU work
        _oracle_attention(b, sub, kc, vc)
        runs += 1
        if time.perf_counter() - t >= target_s or len(pick) < b.num_seqs:
            break
    dt = (time.perf_counter() - t) / runs
    sb = kv_bytes(sub)
    return {"value": round(sb / dt / 1e9, 4), "unit": "GB/s", "cores": threads, "cpu_model": cpu_model(),
            "kind": "oracle",
            "seconds": round(dt * runs, 2),
            "sample": f"attention of {len(pick)} of {b.num_seqs} sequences (every "
                      f"{max(1, b.num_seqs // max(1, len(pick)))}th; {int(sub.context_lens.sum())} tokens, "
                      f"{sb} KV bytes) over the post-step caches, run {runs}x; fp64 C oracle, "
                      f"OpenMP over (seq, head)"}


def run_reference(args, world, rank):
    """The CPU oracle as the reference arm (rank 0 only)."""
    if rank != 0:
        return
    threads = _oracle_threads()
    import oracle
    from paged_kv_cache_140_gb300 import workloads as W
    b = W.make_batch(args.workload)
    kc, vc = _post_step_caches(b)
    per_step_s = min(2.0, 150.0 / max(1, args.steps + args.warmup))
    pick = _pick_sample(b, per_step_s, kc, vc)
    sub = W.subset_batch(b, pick)

    def one():
        _oracle_attention(b, sub, kc, vc)

    for _ in range(args.warmup):
        one()
    t = time.perf_counter()
    for _ in range(args.steps):
        one()
    dt = (time.perf_counter() - t) / args.steps
    sb = kv_bytes(sub)
    value = sb / dt / 1e9
    line = {
        "metric": "paged decode attention: KV-read HBM GB/s (% of GB300 peak), us/step",
        "value": round(value, 4), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": b.dtype, "data": "synthetic", "impl": "reference",
        "config": decode_config(b, args.workload, world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads, "cpu_model": cpu_model(),
                         "kind": "oracle",
                         "sample": f"attention of {len(pick)} of {b.num_seqs} sequences per step "
                                   f"({int(sub.context_lens.sum())} tokens, {sb} KV bytes)"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_swap(args):
    """swap_blocks bandwidth between the GPU cache and pinned host memory
    (13B-shaped blocks: 16 tokens x 40 heads x 128 dims, bf16, K and V)."""
    import torch

    import paged_kv_cache_140_gb300 as pa
    if not torch.cuda.is_available():
        raise SystemExit("--swap needs a CUDA device")
    n_gpu, n_swap = 8192, 2048
    shape = (16, 40, 128)
    gk = torch.randn((n_gpu,) + shape, device="cuda").to(torch.bfloat16)
    gv = torch.randn((n_gpu,) + shape, device="cuda").to(torch.bfloat16)
    hk = torch.empty((n_swap,) + shape, dtype=torch.bfloat16).pin_memory()
    hv = torch.empty((n_swap,) + shape, dtype=torch.bfloat16).pin_memory()
    g = torch.Generator().manual_seed(140)
    src = torch.randperm(n_gpu, generator=g)[:n_swap]
    out_map = torch.stack([src, torch.arange(n_swap)], 1).to("cuda")
    in_map = torch.stack([torch.arange(n_swap), torch.randperm(n_gpu, generator=g)[:n_swap]], 1).to("cuda")
    nbytes = 2 * n_swap * 16 * 40 * 128 * 2
    res = {}
    for name, fn in (("swap_out", lambda: pa.swap_blocks(gk, gv, hk, hv, out_map)),
                     ("swap_in", lambda: pa.swap_blocks(hk, hv, gk, gv, in_map))):
        for _ in range(max(3, args.warmup)):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        res[name] = {"ms": round(ms, 4), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1)}
    print(json.dumps({"metric": "swap_blocks GPU<->pinned host GB/s", "blocks": n_swap,
                      "bytes_per_call": nbytes, "steps": args.steps, **res}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="13b", choices=sorted(WORKLOAD_TEXT))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--swap", action="store_true", help="measure swap_blocks bandwidth instead")
    ap.add_argument("--fused", action="store_true",
                    help="(the default where it applies) run the step as pa_decode_append: the new rows "
                         "appended and attended in one call")
    ap.add_argument("--separate", action="store_true",
                    help="run the step as pa_reshape_and_cache followed by pa_decode")
    ap.add_argument("--clock-probe-s", type=float, default=2.0,
                    help="seconds of steps run under the clock sampler before the timed region")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_env()
    if args.swap:
        return run_swap(args)
    if args.workload in PREFILL_WORKLOADS:
        if args.impl == "reference":
            run_prefill_reference(args, world, rank)
        else:
            run_prefill(args, world, rank, local)
    elif args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
