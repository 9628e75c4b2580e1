"""Brute-force paged attention in NumPy, for tiny inputs -- TEST INFRASTRUCTURE ONLY.

An independent second route to the same definition as the C oracle: Python
loops walk each sequence's positions through its block table to build a
contiguous K and V, then NumPy evaluates softmax(q K^T * scale) V in float64
("LLM推理优化：vLLM PagedAttention深度解析与工程实践", §二 attention formula and
§4.1 cache layout).  Half values are widened by NumPy's own float16 type and,
for bfloat16, by placing the 16 bits in the top half of a float32.
"""
from __future__ import annotations

import numpy as np


def widen(bits: np.ndarray, dtype: str) -> np.ndarray:
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def gather_contiguous(cache_bits, block_table_row, n, kvh, dtype):
    """K (or V) rows of positions 0..n-1 of one KV head as a float64 [n, D]."""
    bs = cache_bits.shape[1]
    rows = []
    for p in range(n):
        rows.append(widen(cache_bits[block_table_row[p // bs], p % bs, kvh], dtype))
    return np.array(rows, dtype=np.float64).reshape(n, cache_bits.shape[3])


def attention_contiguous(q, K, V, scale):
    """softmax(q K^T * scale) V for one query vector over contiguous rows."""
    if K.shape[0] == 0:
        return np.zeros(q.shape[-1])
    x = (K @ q) * float(scale)
    w = np.exp(x - x.max())
    return (w[:, None] * V).sum(axis=0) / w.sum()


def paged_attention(q_bits, k_cache, v_cache, dtype, block_tables, context_lens, scale):
    B, Hq, D = q_bits.shape
    Hkv = k_cache.shape[2]
    G = Hq // Hkv
    out = np.zeros((B, Hq, D))
    for s in range(B):
        n = int(context_lens[s])
        for hq in range(Hq):
            if n <= 0:
                continue
            kvh = hq // G
            K = gather_contiguous(k_cache, block_tables[s], n, kvh, dtype)
            V = gather_contiguous(v_cache, block_tables[s], n, kvh, dtype)
            out[s, hq] = attention_contiguous(widen(q_bits[s, hq], dtype), K, V, scale)
    return out
