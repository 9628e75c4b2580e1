"""Seeded synthetic inputs for one paged decode-attention step.

This module builds everything one decode step over a paged KV cache consumes:
the query of every running sequence, the K/V cache (fixed-size physical blocks
scattered over a pool and reached through per-sequence block tables), the
context lengths, the step's new K/V rows with their slot mapping, and, for the
copy-on-write case, the block copy pairs.  It draws random numbers and hands
out physical blocks; it computes no part of attention, so the CPU oracle and
the CUDA path both take their inputs from here.

Sources of the shapes and structure:
  * KV layout ``[num_blocks, block_size, num_kv_heads, head_dim]`` per layer and
    the block table of logical -> physical block ids:
    "LLM推理优化：vLLM PagedAttention深度解析与工程实践", §3.1 and §4.1.
  * LLaMA-7B / LLaMA-13B shapes (32 x 128 and 40 x 128 heads):
    same page, §二, and the nano-vllm walkthrough (lqnn.cn/news/170268), §1.1.
  * GQA (H_kv < H_q) and copy-on-write of a shared 1000-token prompt for four
    samples: "优化大模型推理：PagedAttention 如何实现 GPU 显存高效管理",
    sections on the KV-cache size formula and on copy-on-write.
  * Slots past a sequence's length hold stale data that must never matter
    (nano-vllm walkthrough, §6): every unused slot and unused block is filled
    with NaN here.

Half-precision values travel as ``uint16`` bit patterns with a dtype tag
("f16" = IEEE binary16, "bf16" = bfloat16), so both consumers see the exact
same bits.  Values are drawn N(0, 1) in float32 and rounded to nearest-even.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

__all__ = ["CONFIGS", "PREFILL_CONFIGS", "Batch", "PrefillBatch", "make_batch", "make_prefill_batch",
           "make_context_lens", "subset_batch", "NAN_BITS", "BlockPool"]

# Quiet-NaN bit patterns used to poison unused cache slots (e4m3: 0x7F).
NAN_BITS = {"f16": 0x7E00, "bf16": 0x7FC0, "fp8": 0x7F}
# Scale of the e4m3 caches: a code c stands for c * FP8_SCALE, so N(0, 1)
# data uses codes of magnitude up to ~64 (well inside e4m3's +-448).
FP8_SCALE = 1.0 / 16.0

# The five decode workloads.  ``ctx`` describes the context-length law;
# ``ctx_max`` is the longest context the workload can produce and sizes the
# block tables.  Seeds are 140000 + the workload number.
CONFIGS = {
    # 4 sequences with fixed lengths {1, 17, 35, 100}, MHA, head_dim 64.
    "tiny": dict(number=1, num_seqs=4, num_heads=4, num_kv_heads=4, head_dim=64,
                 block_size=16, dtype="f16", ctx=("fixed", (1, 17, 35, 100)),
                 ctx_max=100, pool=("fixed", 64), partition_size=0),
    # LLaMA-7B-shaped layer: 64 sequences, 32 heads, lengths uniform on [32, 2048].
    "7b": dict(number=2, num_seqs=64, num_heads=32, num_kv_heads=32, head_dim=128,
               block_size=16, dtype="f16", ctx=("uniform", 32, 2048),
               ctx_max=2048, pool=("demand", 1.2), partition_size=0),
    # LLaMA-13B-shaped layer: 256 sequences, 40 heads, long-tailed lengths
    # (lognormal, median 300, sigma 1 in natural-log units, clipped to [1, 2048]).
    "13b": dict(number=3, num_seqs=256, num_heads=40, num_kv_heads=40, head_dim=128,
                block_size=16, dtype="bf16", ctx=("lognormal", 300.0, 1.0, 1, 2048),
                ctx_max=2048, pool=("demand", 1.2), partition_size=0),
    # The 13B-shaped step with an FP8 (e4m3) KV cache (per-tensor scales).
    "13b_fp8": dict(number=3, num_seqs=256, num_heads=40, num_kv_heads=40, head_dim=128,
                    block_size=16, dtype="bf16", cache_dtype="fp8", ctx=("lognormal", 300.0, 1.0, 1, 2048),
                    ctx_max=2048, pool=("demand", 1.2), partition_size=0),
    # GQA long context: 16 sequences, 32 query / 8 KV heads, 16k-32k tokens,
    # split into 512-token partitions; block_size 16 and 32 variants.
    "gqa": dict(number=4, num_seqs=16, num_heads=32, num_kv_heads=8, head_dim=128,
                block_size=16, dtype="bf16", ctx=("uniform", 16384, 32768),
                ctx_max=32768, pool=("demand", 1.2), partition_size=512),
    "gqa32": dict(number=4, num_seqs=16, num_heads=32, num_kv_heads=8, head_dim=128,
                  block_size=32, dtype="bf16", ctx=("uniform", 16384, 32768),
                  ctx_max=32768, pool=("demand", 1.2), partition_size=512),
    # Prefix sharing: 64 prompts x 4 samples; each group shares a 1000-token
    # prompt (refcount 4); each sample adds a private 0-256 token suffix plus
    # the step's new token; the shared, partly filled last prompt block is
    # copied before a sample first writes into it.
    "prefix": dict(number=5, groups=64, samples=4, prompt_len=1000, suffix_max=256,
                   num_heads=32, num_kv_heads=32, head_dim=128, block_size=16,
                   dtype="f16", ctx_max=1000 + 256 + 1, pool=("demand", 1.2),
                   partition_size=0),
}

# Prefill workloads: each sequence has ``prefix`` tokens already cached and
# ``q_len`` new tokens whose queries attend causally over prefix + new tokens
# (prefill of the uncached tail after a prefix-cache hit, or one chunk of a
# chunked prefill; nano-vllm walkthrough §3.4).  "prefix" reuses the prefix-
# sharing workload above: every sample's private tail is prefilled over the
# shared 1000-token prompt.
PREFILL_CONFIGS = {
    # LLaMA-13B-shaped layer, 16 sequences, a 512-token chunk over a cached
    # prefix of U{0..2048} tokens.
    "prefill": dict(number=6, num_seqs=16, num_heads=40, num_kv_heads=40, head_dim=128, block_size=16,
                    dtype="bf16", prefix=("uniform", 0, 2048), q_len=("fixed", 512), pool=("demand", 1.2)),
    # GQA (32 query / 8 KV heads), 8 sequences, 1024-token chunks over
    # U{0..8192} cached tokens.
    "prefill_gqa": dict(number=7, num_seqs=8, num_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                        dtype="bf16", prefix=("uniform", 0, 8192), q_len=("fixed", 1024), pool=("demand", 1.2)),
}


@dataclasses.dataclass
class Batch:
    """One decode step's inputs (host arrays).

    ``k_cache``/``v_cache`` hold the cache *before* the step: history tokens
    are filled, the step's new token slots and everything unused are NaN.
    The step is: copy_blocks(block_mapping), reshape_and_cache(key, value,
    slot_mapping), then decode over ``context_lens`` tokens (which include the
    tokens the step writes).
    """
    name: str
    dtype: str
    num_seqs: int
    num_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    max_blocks_per_seq: int
    max_context_len: int
    partition_size: int
    scale: np.float32
    q: np.ndarray             # uint16 [B, Hq, D]
    k_cache: np.ndarray       # uint16 [NB, bs, Hkv, D]
    v_cache: np.ndarray       # uint16 [NB, bs, Hkv, D]
    key: np.ndarray           # uint16 [T, Hkv, D]  rows written by this step
    value: np.ndarray         # uint16 [T, Hkv, D]
    slot_mapping: np.ndarray  # int64 [T]  flat slot = block * bs + offset
    block_tables: np.ndarray  # int32 [B, max_blocks_per_seq], padded with -1
    context_lens: np.ndarray  # int32 [B]
    block_mapping: np.ndarray  # int64 [P, 2] (src, dst) copy pairs, maybe empty
    seed: int = 0
    cache_dtype: str = ""     # "f16" / "bf16" (= dtype) or "fp8" (e4m3 codes, uint8 caches)
    k_scale: float = 1.0      # e4m3 caches: a code c stands for c * scale
    v_scale: float = 1.0

    def __post_init__(self):
        if not self.cache_dtype:
            self.cache_dtype = self.dtype

    @property
    def kv_token_count(self) -> int:
        return int(self.context_lens.astype(np.int64).sum())

    @property
    def elem_bytes(self) -> int:
        return 1 if self.cache_dtype == "fp8" else 2


class BlockPool:
    """Host-side free list of physical blocks with reference counts.

    A test fixture for building inputs, following the BlockManager sketch of
    "LLM推理优化：vLLM PagedAttention深度解析与工程实践", §3.2 (free list,
    allocate on demand, raise when the pool runs dry) and the reference counts
    of the copy-on-write section of "优化大模型推理：PagedAttention 如何实现
    GPU 显存高效管理".  The free list order is a seeded permutation, so the
    physical blocks of a sequence land scattered over the pool.
    """

    def __init__(self, num_blocks: int, rng: np.random.Generator):
        self.num_blocks = int(num_blocks)
        self.free = list(rng.permutation(self.num_blocks).tolist())
        self.refcount = np.zeros(self.num_blocks, dtype=np.int64)

    def allocate(self, n: int) -> list[int]:
        if n > len(self.free):
            raise MemoryError(f"block pool exhausted: need {n}, have {len(self.free)}")
        out = self.free[:n]
        del self.free[:n]
        for b in out:
            self.refcount[b] = 1
        return out

    def share(self, block: int) -> None:
        self.refcount[block] += 1

    def release(self, block: int) -> None:
        self.refcount[block] -= 1
        if self.refcount[block] == 0:
            self.free.append(block)


def _round_half(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to the half type (nearest-even) and return bits."""
    if dtype == "f16":
        return np.ascontiguousarray(x.astype(np.float16)).view(np.uint16)
    if dtype == "bf16":
        import torch
        t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
        return t.view(torch.int16).numpy().view(np.uint16)
    raise ValueError(dtype)


def _normal_bits(rng: np.random.Generator, shape, dtype: str, chunk: int = 1 << 24) -> np.ndarray:
    """Draw N(0,1) float32 values in a fixed order and return half bits
    (or, for "fp8", the e4m3 codes nearest to value / FP8_SCALE, via torch)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint8 if dtype == "fp8" else np.uint16)
    for lo in range(0, n, chunk):
        hi = min(n, lo + chunk)
        z = rng.standard_normal(hi - lo, dtype=np.float32)
        if dtype == "fp8":
            import torch
            out[lo:hi] = torch.from_numpy(z * np.float32(1.0 / FP8_SCALE)).to(torch.float8_e4m3fn) \
                .view(torch.uint8).numpy()
        else:
            out[lo:hi] = _round_half(z, dtype)
    return out.reshape(shape)


def _context_lens(spec, rng: np.random.Generator, num_seqs: int) -> np.ndarray:
    kind = spec[0]
    if kind == "fixed":
        vals = list(spec[1])
        if num_seqs > len(vals):
            raise ValueError("fixed context list is shorter than num_seqs")
        return np.array(vals[:num_seqs], dtype=np.int32)
    if kind == "uniform":
        return rng.integers(spec[1], spec[2], size=num_seqs, endpoint=True).astype(np.int32)
    if kind == "lognormal":
        median, sigma, lo, hi = spec[1:]
        x = rng.lognormal(mean=math.log(median), sigma=sigma, size=num_seqs)
        return np.clip(np.rint(x), lo, hi).astype(np.int32)
    raise ValueError(kind)


def _blocks_for(n: int, bs: int) -> int:
    return -(-int(n) // int(bs))


def _scatter_rows(cache: np.ndarray, slots: np.ndarray, rows: np.ndarray) -> None:
    nb, bs, hkv, d = cache.shape
    flat = cache.reshape(nb * bs, hkv * d)
    flat[slots] = rows.reshape(len(slots), hkv * d)


def make_context_lens(name: str, num_seqs: int | None = None, seed: int | None = None) -> np.ndarray:
    """The context lengths ``make_batch`` draws first for workload ``name``."""
    cfg = CONFIGS[name]
    rng = np.random.Generator(np.random.PCG64(140000 + cfg["number"] if seed is None else seed))
    if name == "prefix":
        suffix = rng.integers(0, cfg["suffix_max"], size=(num_seqs or cfg["groups"], cfg["samples"]),
                              endpoint=True)
        return (cfg["prompt_len"] + suffix + 1).reshape(-1).astype(np.int32)
    return _context_lens(cfg["ctx"], rng, int(num_seqs or cfg["num_seqs"]))


def make_batch(name: str, *, num_seqs: int | None = None, groups: int | None = None,
               seed: int | None = None, ctx_cap: int | None = None,
               block_size: int | None = None, context_lens=None, cache_dtype: str | None = None,
               **overrides) -> Batch:
    """Build the inputs of workload ``name`` (a key of :data:`CONFIGS`).

    ``num_seqs`` (or ``groups`` for "prefix") shrinks the batch while keeping
    every other property of the workload; ``ctx_cap`` clips the context law to
    a shorter maximum (for oracle-sized cases); ``context_lens`` replaces the
    drawn lengths outright (edge-case tests); other keywords (``num_heads``,
    ``num_kv_heads``, ``head_dim``, ``dtype``, ``partition_size``) override the
    workload's entries.
    """
    cfg = dict(CONFIGS[name])
    for k, v in overrides.items():
        if k not in ("num_heads", "num_kv_heads", "head_dim", "dtype", "partition_size"):
            raise TypeError(f"unknown override {k}")
        cfg[k] = v
    if cache_dtype is not None:
        cfg["cache_dtype"] = cache_dtype
    if seed is None:
        seed = 140000 + cfg["number"]
    rng = np.random.Generator(np.random.PCG64(seed))
    if block_size is not None:
        cfg["block_size"] = int(block_size)
    if name == "prefix":
        return _make_prefix(cfg, rng, groups or cfg["groups"], seed, ctx_cap)

    B = int(num_seqs or cfg["num_seqs"])
    Hq, Hkv, D, bs, dt = cfg["num_heads"], cfg["num_kv_heads"], cfg["head_dim"], cfg["block_size"], cfg["dtype"]
    if context_lens is not None:
        ctx = np.asarray(context_lens, dtype=np.int32).copy()
        B = len(ctx)
    else:
        ctx = _context_lens(cfg["ctx"], rng, B)
    ctx_max = cfg["ctx_max"]
    if ctx_cap is not None:
        ctx = np.minimum(ctx, ctx_cap).astype(np.int32)
        ctx_max = min(ctx_max, int(ctx_cap))
    ctx_max = max(ctx_max, int(ctx.max(initial=0)))
    nblk = np.array([_blocks_for(c, bs) for c in ctx], dtype=np.int64)
    demand = int(nblk.sum())
    if cfg["pool"][0] == "fixed":
        NB = max(int(cfg["pool"][1]), demand)
    else:
        NB = max(1, int(math.ceil(cfg["pool"][1] * demand)))
    maxNB = max(1, _blocks_for(ctx_max, bs))

    pool = BlockPool(NB, rng)
    tables = np.full((B, maxNB), -1, dtype=np.int32)
    for s in range(B):
        blocks = pool.allocate(int(nblk[s]))
        tables[s, : len(blocks)] = blocks

    cdt = cfg.get("cache_dtype", dt)
    q = _normal_bits(rng, (B, Hq, D), dt)
    nan = NAN_BITS[cdt]
    cnp = np.uint8 if cdt == "fp8" else np.uint16
    k_cache = np.full((NB, bs, Hkv, D), nan, dtype=cnp)
    v_cache = np.full((NB, bs, Hkv, D), nan, dtype=cnp)

    # History rows: positions 0 .. ctx-2 of every sequence (the last position
    # is this step's new token, written by reshape_and_cache).
    pos_slots = []
    for s in range(B):
        p = np.arange(max(int(ctx[s]) - 1, 0), dtype=np.int64)
        pos_slots.append(tables[s, p // bs].astype(np.int64) * bs + p % bs)
    hist = np.concatenate(pos_slots) if pos_slots else np.zeros(0, np.int64)
    _fill_history(rng, k_cache, v_cache, hist, cdt)

    T = int((ctx > 0).sum())
    seqs_with_token = np.nonzero(ctx > 0)[0]
    last = ctx[seqs_with_token].astype(np.int64) - 1
    slot_mapping = (tables[seqs_with_token, last // bs].astype(np.int64) * bs + last % bs).astype(np.int64)
    key = _normal_bits(rng, (T, Hkv, D), dt)
    value = _normal_bits(rng, (T, Hkv, D), dt)

    return Batch(name=name, dtype=dt, num_seqs=B, num_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                 block_size=bs, num_blocks=NB, max_blocks_per_seq=maxNB, max_context_len=int(ctx_max),
                 partition_size=int(cfg["partition_size"]), scale=np.float32(1.0 / math.sqrt(D)),
                 q=q, k_cache=k_cache, v_cache=v_cache, key=key, value=value,
                 slot_mapping=slot_mapping, block_tables=tables, context_lens=ctx,
                 block_mapping=np.zeros((0, 2), dtype=np.int64), seed=int(seed), cache_dtype=cdt,
                 k_scale=FP8_SCALE if cdt == "fp8" else 1.0, v_scale=FP8_SCALE if cdt == "fp8" else 1.0)


def _fill_history(rng, k_cache, v_cache, slots, dt, rows_per_chunk=1 << 14):
    """Fill K rows for ``slots`` then V rows, drawing values in slot order
    (``dt`` is the cache's element type)."""
    nb, bs, hkv, d = k_cache.shape
    for cache in (k_cache, v_cache):
        for lo in range(0, len(slots), rows_per_chunk):
            hi = min(len(slots), lo + rows_per_chunk)
            rows = _normal_bits(rng, (hi - lo, hkv, d), dt)
            _scatter_rows(cache, slots[lo:hi], rows)


def _make_prefix(cfg, rng, groups, seed, ctx_cap):
    """Prefix-sharing step with copy-on-write of the shared partial block.

    Every group of ``samples`` sequences shares the physical blocks of one
    ``prompt_len``-token prompt (reference count = samples).  Each sample
    then owns a private suffix of U{0..suffix_max} tokens plus the step's new
    token.  The first private token lands in the shared, partly filled last
    prompt block; samples are processed in order, and a sample that writes
    into a block still referenced by others first gets a private copy of it
    (one copy pair), while the last sample writes in place.
    """
    S = cfg["samples"]
    Hq, Hkv, D, bs, dt = cfg["num_heads"], cfg["num_kv_heads"], cfg["head_dim"], cfg["block_size"], cfg["dtype"]
    P = cfg["prompt_len"]
    smax = cfg["suffix_max"]
    if ctx_cap is not None:
        smax = max(0, min(smax, int(ctx_cap) - P - 1))
    suffix = rng.integers(0, smax, size=(groups, S), endpoint=True).astype(np.int64)
    ctx = (P + suffix + 1).reshape(-1).astype(np.int32)
    B = groups * S
    prompt_blocks = _blocks_for(P, bs)
    partial = (P % bs) != 0
    # Demand: shared prompt blocks, one copy per sample but the last when the
    # prompt's last block is partial, and each sample's private blocks.
    first_private_pos = prompt_blocks * bs
    priv = np.maximum(ctx.astype(np.int64) - first_private_pos, 0)
    priv_blocks = -(-priv // bs)
    demand = groups * prompt_blocks + int(priv_blocks.sum()) + (groups * (S - 1) if partial else 0)
    NB = int(math.ceil(cfg["pool"][1] * demand))
    ctx_max = max(cfg["ctx_max"] if ctx_cap is None else min(cfg["ctx_max"], int(ctx_cap)), int(ctx.max()))
    maxNB = _blocks_for(ctx_max, bs)

    pool = BlockPool(NB, rng)
    tables = np.full((B, maxNB), -1, dtype=np.int32)
    pairs = []
    shared_slots = []
    for g in range(groups):
        blocks = pool.allocate(prompt_blocks)
        for b in blocks:
            for _ in range(S - 1):
                pool.share(b)
        p = np.arange(P, dtype=np.int64)
        shared_slots.append(np.asarray(blocks, dtype=np.int64)[p // bs] * bs + p % bs)
        for i in range(S):
            s = g * S + i
            row = list(blocks)
            last = row[-1]
            if partial:
                if pool.refcount[last] > 1:
                    dst = pool.allocate(1)[0]
                    pairs.append((last, dst))
                    pool.release(last)
                    row[-1] = dst
            row += pool.allocate(int(priv_blocks[s]))
            tables[s, : len(row)] = row

    cdt = cfg.get("cache_dtype", dt)
    q = _normal_bits(rng, (B, Hq, D), dt)
    nan = NAN_BITS[cdt]
    cnp = np.uint8 if cdt == "fp8" else np.uint16
    k_cache = np.full((NB, bs, Hkv, D), nan, dtype=cnp)
    v_cache = np.full((NB, bs, Hkv, D), nan, dtype=cnp)
    _fill_history(rng, k_cache, v_cache, np.concatenate(shared_slots), cdt)

    # The step writes every private position P .. ctx-1 of every sample.
    slots = []
    for s in range(B):
        p = np.arange(P, int(ctx[s]), dtype=np.int64)
        slots.append(tables[s, p // bs].astype(np.int64) * bs + p % bs)
    slot_mapping = np.concatenate(slots).astype(np.int64)
    T = len(slot_mapping)
    key = _normal_bits(rng, (T, Hkv, D), dt)
    value = _normal_bits(rng, (T, Hkv, D), dt)
    bm = np.asarray(pairs, dtype=np.int64).reshape(-1, 2)
    return Batch(name="prefix", dtype=dt, num_seqs=B, num_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                 block_size=bs, num_blocks=NB, max_blocks_per_seq=maxNB, max_context_len=int(ctx_max),
                 partition_size=int(cfg["partition_size"]), scale=np.float32(1.0 / math.sqrt(D)),
                 q=q, k_cache=k_cache, v_cache=v_cache, key=key, value=value,
                 slot_mapping=slot_mapping, block_tables=tables, context_lens=ctx,
                 block_mapping=bm, seed=int(seed), cache_dtype=cdt,
                 k_scale=FP8_SCALE if cdt == "fp8" else 1.0, v_scale=FP8_SCALE if cdt == "fp8" else 1.0)


def subset_batch(b: Batch, seqs) -> Batch:
    """Restrict a batch to some sequences (same caches, same step writes).

    Used to check sampled outputs of a full-size step one sequence at a time.
    """
    seqs = np.asarray(seqs, dtype=np.int64)
    return dataclasses.replace(b, num_seqs=len(seqs), q=b.q[seqs].copy(),
                               block_tables=b.block_tables[seqs].copy(),
                               context_lens=b.context_lens[seqs].copy())


@dataclasses.dataclass
class PrefillBatch(Batch):
    """One prefill step's inputs: ``q`` is [T, Hq, D] for the T new tokens of
    all sequences, sequence s owning rows cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1
    (its newest tokens, positions ctx - q_len .. ctx - 1).  ``key``/``value``/
    ``slot_mapping`` are those tokens' K/V rows and slots; the caches hold the
    cached prefix (everything else NaN).  The step is copy_blocks, then
    reshape_and_cache, then the prefill attention."""
    cu_seqlens_q: np.ndarray = None   # int32 [B + 1]
    max_q_len: int = 0

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.cu_seqlens_q).astype(np.int64)

    @property
    def num_tokens(self) -> int:
        return int(self.cu_seqlens_q[-1])


def _law(spec, rng, n):
    if spec[0] == "fixed":
        return np.full(n, int(spec[1]), dtype=np.int64)
    if spec[0] == "uniform":
        return rng.integers(spec[1], spec[2], size=n, endpoint=True).astype(np.int64)
    raise ValueError(spec)


def make_prefill_batch(name: str, *, num_seqs: int | None = None, groups: int | None = None,
                       seed: int | None = None, prefix_cap: int | None = None, q_len_cap: int | None = None,
                       prefix_lens=None, q_lens=None, block_size: int | None = None,
                       **overrides) -> PrefillBatch:
    """Build prefill workload ``name`` (a key of :data:`PREFILL_CONFIGS`, or
    "prefix" for the tails of the prefix-sharing workload).

    ``num_seqs`` (``groups`` for "prefix") shrinks the batch; ``prefix_cap`` /
    ``q_len_cap`` clip the drawn lengths; ``prefix_lens`` / ``q_lens`` replace
    them outright (edge-case tests); ``num_heads``, ``num_kv_heads``,
    ``head_dim`` and ``dtype`` may be overridden.
    """
    if name == "prefix":
        b = make_batch("prefix", groups=groups, seed=seed, ctx_cap=None if prefix_cap is None
                       else CONFIGS["prefix"]["prompt_len"] + 1 + int(prefix_cap))
        P = CONFIGS["prefix"]["prompt_len"]
        ql = b.context_lens.astype(np.int64) - P
        rng = np.random.Generator(np.random.PCG64(b.seed + 1))
        q = _normal_bits(rng, (int(ql.sum()), b.num_heads, b.head_dim), b.dtype)
        cu = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
        fields = {f.name: getattr(b, f.name) for f in dataclasses.fields(Batch)}
        fields.update(name="prefill_prefix", q=q)
        return PrefillBatch(**fields, cu_seqlens_q=cu, max_q_len=int(ql.max(initial=0)))

    cfg = dict(PREFILL_CONFIGS[name])
    for k, v in overrides.items():
        if k not in ("num_heads", "num_kv_heads", "head_dim", "dtype"):
            raise TypeError(f"unknown override {k}")
        cfg[k] = v
    if block_size is not None:
        cfg["block_size"] = int(block_size)
    if seed is None:
        seed = 140000 + cfg["number"]
    rng = np.random.Generator(np.random.PCG64(seed))
    B = int(num_seqs or cfg["num_seqs"])
    if prefix_lens is not None:
        prefix = np.asarray(prefix_lens, dtype=np.int64).copy()
        B = len(prefix)
    else:
        prefix = _law(cfg["prefix"], rng, B)
    ql = np.asarray(q_lens, dtype=np.int64).copy() if q_lens is not None else _law(cfg["q_len"], rng, B)
    if len(ql) != B:
        raise ValueError("q_lens and prefix_lens differ in length")
    if prefix_cap is not None:
        prefix = np.minimum(prefix, prefix_cap)
    if q_len_cap is not None:
        ql = np.minimum(ql, q_len_cap)
    Hq, Hkv, D, bs, dt = cfg["num_heads"], cfg["num_kv_heads"], cfg["head_dim"], cfg["block_size"], cfg["dtype"]
    ctx = (prefix + ql).astype(np.int32)
    nblk = np.array([_blocks_for(c, bs) for c in ctx], dtype=np.int64)
    NB = max(1, int(math.ceil(cfg["pool"][1] * int(nblk.sum()))))
    maxNB = max(1, int(nblk.max(initial=1)))
    pool = BlockPool(NB, rng)
    tables = np.full((B, maxNB), -1, dtype=np.int32)
    for s in range(B):
        blocks = pool.allocate(int(nblk[s]))
        tables[s, : len(blocks)] = blocks

    k_cache = np.full((NB, bs, Hkv, D), NAN_BITS[dt], dtype=np.uint16)
    v_cache = np.full((NB, bs, Hkv, D), NAN_BITS[dt], dtype=np.uint16)
    hist, new = [], []
    for s in range(B):
        p = np.arange(int(ctx[s]), dtype=np.int64)
        slots = tables[s, p // bs].astype(np.int64) * bs + p % bs
        hist.append(slots[: int(prefix[s])])
        new.append(slots[int(prefix[s]):])
    _fill_history(rng, k_cache, v_cache, np.concatenate(hist) if hist else np.zeros(0, np.int64), dt)
    slot_mapping = np.concatenate(new).astype(np.int64) if new else np.zeros(0, np.int64)
    T = len(slot_mapping)
    key = _normal_bits(rng, (T, Hkv, D), dt)
    value = _normal_bits(rng, (T, Hkv, D), dt)
    q = _normal_bits(rng, (T, Hq, D), dt)
    cu = np.concatenate([[0], np.cumsum(ql)]).astype(np.int32)
    return PrefillBatch(name=name, dtype=dt, num_seqs=B, num_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                        block_size=bs, num_blocks=NB, max_blocks_per_seq=maxNB,
                        max_context_len=int(ctx.max(initial=0)), partition_size=0,
                        scale=np.float32(1.0 / math.sqrt(D)), q=q, k_cache=k_cache, v_cache=v_cache,
                        key=key, value=value, slot_mapping=slot_mapping, block_tables=tables,
                        context_lens=ctx, block_mapping=np.zeros((0, 2), dtype=np.int64), seed=int(seed),
                        cu_seqlens_q=cu, max_q_len=int(ql.max(initial=0)))
