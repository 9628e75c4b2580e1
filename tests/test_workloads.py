"""The seeded input generators: determinism, shapes, block tables, poisoning."""
import numpy as np
import pytest

from oracle import accounting
from paged_kv_cache_140_gb300 import workloads as W


def _check_batch(b):
    B, Hq, Hkv, D, bs = b.num_seqs, b.num_heads, b.num_kv_heads, b.head_dim, b.block_size
    assert b.q.shape == (B, Hq, D) and b.q.dtype == np.uint16
    assert b.k_cache.shape == (b.num_blocks, bs, Hkv, D) == b.v_cache.shape
    assert b.block_tables.shape == (B, b.max_blocks_per_seq)
    assert b.context_lens.shape == (B,)
    assert b.key.shape == (len(b.slot_mapping), Hkv, D) == b.value.shape
    used = np.zeros(b.num_blocks, dtype=np.int64)
    for s in range(B):
        n = int(b.context_lens[s])
        nb = accounting.blocks_needed(n, bs)
        row = b.block_tables[s]
        assert np.all(row[:nb] >= 0) and np.all(row[:nb] < b.num_blocks)
        assert np.all(row[nb:] == -1)
        used[row[:nb]] += 1
    return used


@pytest.mark.parametrize("name,kw", [("tiny", {}), ("7b", dict(num_seqs=3)), ("13b", dict(num_seqs=5)),
                                     ("gqa", dict(num_seqs=2, ctx_cap=20000)),
                                     ("gqa32", dict(num_seqs=2, ctx_cap=20000)),
                                     ("prefix", dict(groups=2))])
def test_generator_is_deterministic_and_consistent(name, kw):
    a = W.make_batch(name, **kw)
    b = W.make_batch(name, **kw)
    for f in ("q", "k_cache", "v_cache", "key", "value", "slot_mapping", "block_tables", "context_lens",
              "block_mapping"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f
    used = _check_batch(a)
    if name != "prefix":
        assert used.max() <= 1          # no block shared between sequences
    nan = W.NAN_BITS[a.dtype]
    # the step's new-token slots and every unused slot are poisoned
    flat = a.k_cache.reshape(-1, a.num_kv_heads * a.head_dim)
    assert np.all(flat[a.slot_mapping] == nan)
    live = np.zeros(flat.shape[0], dtype=bool)
    for s in range(a.num_seqs):
        n = int(a.context_lens[s])
        p = np.arange(n)
        live[a.block_tables[s, p // a.block_size].astype(np.int64) * a.block_size + p % a.block_size] = True
    assert np.all(flat[~live] == nan)
    assert np.all(np.isfinite(a.q.view(np.float16 if a.dtype == "f16" else np.uint16).astype(np.float64))) \
        if a.dtype == "f16" else True


def test_new_token_slot_is_position_ctx_minus_one():
    b = W.make_batch("7b", num_seqs=6)
    for s in range(6):
        p = int(b.context_lens[s]) - 1
        want = int(b.block_tables[s, p // b.block_size]) * b.block_size + p % b.block_size
        assert int(b.slot_mapping[s]) == want


def test_context_laws():
    c13 = W.make_context_lens("13b")
    assert len(c13) == 256 and c13.min() >= 1 and c13.max() <= 2048
    assert 200 < np.median(c13) < 420
    assert np.array_equal(c13[:5], W.make_batch("13b", num_seqs=5).context_lens)
    c7 = W.make_context_lens("7b")
    assert len(c7) == 64 and c7.min() >= 32 and c7.max() <= 2048
    cg = W.make_context_lens("gqa")
    assert len(cg) == 16 and cg.min() >= 16384 and cg.max() <= 32768
    cp = W.make_context_lens("prefix")
    assert len(cp) == 256 and np.array_equal(cp[:8], W.make_batch("prefix", groups=2).context_lens)
    t = W.make_batch("tiny")
    assert list(t.context_lens) == [1, 17, 35, 100]
    assert t.num_blocks == 64 and t.max_blocks_per_seq == 7


def test_prefix_copy_on_write_structure():
    b = W.make_batch("prefix", groups=3)
    S, bs, P = 4, 16, 1000
    last = P // bs                        # index of the shared, partly filled block
    assert len(b.block_mapping) == 3 * (S - 1)
    for g in range(3):
        rows = b.block_tables[g * S:(g + 1) * S]
        assert np.all(rows[:, :last] == rows[0, :last])             # shared full blocks
        shared_last = rows[S - 1, last]                              # last sample writes in place
        pairs = b.block_mapping[g * (S - 1):(g + 1) * (S - 1)]
        assert np.all(pairs[:, 0] == shared_last)
        assert list(pairs[:, 1]) == list(rows[: S - 1, last])
    assert len(set(b.block_mapping[:, 1].tolist())) == len(b.block_mapping)
    assert not set(b.block_mapping[:, 1].tolist()) & set(b.block_mapping[:, 0].tolist())
    assert np.all(b.context_lens >= P + 1) and np.all(b.context_lens <= P + 256 + 1)
    assert len(b.slot_mapping) == int((b.context_lens - P).sum())


@pytest.mark.parametrize("name,kw", [("prefill", dict(num_seqs=3, prefix_cap=200, q_len_cap=70)),
                                     ("prefill_gqa", dict(num_seqs=2, prefix_cap=300, q_len_cap=50)),
                                     ("prefill", dict(prefix_lens=[0, 16, 5], q_lens=[3, 0, 17])),
                                     ("prefix", dict(groups=1))])
def test_prefill_batch_structure(name, kw):
    """Tails of q_len new tokens after `ctx - q_len` cached ones: the cache
    holds exactly the prefix, the step writes the tail's slots in sequence /
    position order, and query rows follow cu_seqlens_q."""
    b = W.make_prefill_batch(name, **kw)
    b2 = W.make_prefill_batch(name, **kw)
    assert np.array_equal(b.q, b2.q) and np.array_equal(b.k_cache, b2.k_cache)
    B, bs = b.num_seqs, b.block_size
    ql = b.q_lens
    assert b.cu_seqlens_q[0] == 0 and np.all(ql >= 0) and b.max_q_len == ql.max()
    assert b.q.shape == (b.num_tokens, b.num_heads, b.head_dim)
    assert b.key.shape == (b.num_tokens, b.num_kv_heads, b.head_dim) and len(b.slot_mapping) == b.num_tokens
    nan = W.NAN_BITS[b.dtype]
    flat = b.k_cache.reshape(-1, b.num_kv_heads * b.head_dim)
    expect = []
    for s in range(B):
        ctx, n = int(b.context_lens[s]), int(ql[s])
        assert n <= ctx
        p = np.arange(ctx)
        slots = b.block_tables[s, p // bs].astype(np.int64) * bs + p % bs
        prefix_slots, tail = slots[: ctx - n], slots[ctx - n:]
        if len(b.block_mapping) == 0 or name != "prefix":
            assert not np.any(flat[prefix_slots] == nan)
        assert np.all(flat[tail] == nan)
        expect.append(tail)
    assert np.array_equal(np.concatenate(expect), b.slot_mapping)
    assert len(np.unique(b.slot_mapping)) == len(b.slot_mapping)
