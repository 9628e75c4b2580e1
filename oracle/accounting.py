"""Block-count and KV-size formulas stated on the pages -- TEST INFRASTRUCTURE ONLY.

  * A sequence of n tokens needs ceil(n / block_size) blocks, and only its last
    block can hold unused slots (at most block_size - 1):
    "优化大模型推理：PagedAttention 如何实现 GPU 显存高效管理", section on
    on-demand allocation (35 tokens, block 16 -> 3 blocks, 13 empty slots);
    "vLLM 核心：PagedAttention 与 Continuous Batching", §3 (memory advantages).
  * KV bytes per token = 2 (K and V) x layers x d_model x bytes per value:
    "LLM推理优化：vLLM PagedAttention深度解析与工程实践", §二.  With grouped
    query attention d_model becomes H_kv x head_dim ("优化大模型推理…",
    KV-cache size formula with H_kv, D, T and B_dtype).
  * Contiguous worst-case reservation vs. actual use ("优化大模型推理…",
    section on why contiguous pre-allocation wastes memory).
"""
from __future__ import annotations


def blocks_needed(num_tokens: int, block_size: int) -> int:
    return -(-int(num_tokens) // int(block_size))


def empty_slots(num_tokens: int, block_size: int) -> int:
    return blocks_needed(num_tokens, block_size) * int(block_size) - int(num_tokens)


def last_block_fill(num_tokens: int, block_size: int) -> int:
    """Tokens held by the last block of a sequence (0 for an empty sequence)."""
    if num_tokens <= 0:
        return 0
    r = int(num_tokens) % int(block_size)
    return int(block_size) if r == 0 else r


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, dtype_bytes: int) -> int:
    return 2 * int(num_layers) * int(num_kv_heads) * int(head_dim) * int(dtype_bytes)


def kv_bytes(num_layers: int, num_kv_heads: int, head_dim: int, num_tokens: int,
             dtype_bytes: int, num_seqs: int = 1) -> int:
    return kv_bytes_per_token(num_layers, num_kv_heads, head_dim, dtype_bytes) * int(num_tokens) * int(num_seqs)


def contiguous_reservation(max_len: int, used_lengths) -> tuple[int, int, float]:
    """(reserved slots, used slots, used fraction) when every request reserves max_len."""
    reserved = int(max_len) * len(used_lengths)
    used = int(sum(int(u) for u in used_lengths))
    return reserved, used, used / reserved
