"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test ties the oracle to one of: exact library conversions, closed forms of
softmax attention, an independent brute force, invariants the pages state
(logical order, not physical placement, decides the result: "优化大模型推理：
PagedAttention 如何实现 GPU 显存高效管理", section on decoupling logical and
physical contiguity; stale slots must not matter: nano-vllm walkthrough
lqnn.cn/news/170268, §6), and the block tables the pages print.
"""
import math
import os
import re
import subprocess
import tempfile

import numpy as np
import pytest

from conftest import read_golden
from oracle import brute

NAN = {"f16": 0x7E00, "bf16": 0x7FC0}


def to_bits(x, dtype):
    x = np.asarray(x, dtype=np.float32)
    if dtype == "f16":
        return x.astype(np.float16).view(np.uint16)
    import torch
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def page(rows, table, bs, num_blocks, dtype, fill=None):
    """Place contiguous rows [n, Hkv, D] into a paged cache through `table`."""
    n, hkv, d = rows.shape
    cache = np.full((num_blocks, bs, hkv, d), NAN[dtype] if fill is None else fill, dtype=np.uint16)
    for p in range(n):
        cache[table[p // bs], p % bs] = rows[p]
    return cache


def random_case(rng, B=3, Hq=4, Hkv=2, D=8, bs=4, max_ctx=37, dtype="f16", ctx=None):
    if ctx is None:
        ctx = rng.integers(1, max_ctx + 1, size=B).astype(np.int32)
    ctx = np.asarray(ctx, dtype=np.int32)
    nblk = [-(-int(c) // bs) for c in ctx]
    NB = sum(nblk) + 5
    perm = rng.permutation(NB)
    maxnb = max(1, max(nblk))
    tables = np.full((len(ctx), maxnb), -1, dtype=np.int32)
    k = np.full((NB, bs, Hkv, D), NAN[dtype], dtype=np.uint16)
    v = np.full_like(k, NAN[dtype])
    i = 0
    for s, c in enumerate(ctx):
        tables[s, : nblk[s]] = perm[i:i + nblk[s]]
        i += nblk[s]
        for p in range(int(c)):
            k[tables[s, p // bs], p % bs] = to_bits(rng.standard_normal((Hkv, D)), dtype)
            v[tables[s, p // bs], p % bs] = to_bits(rng.standard_normal((Hkv, D)), dtype)
    q = to_bits(rng.standard_normal((len(ctx), Hq, D)), dtype)
    return q, k, v, tables, ctx


# ---------------------------------------------------------------- half decode

def test_binary16_decode_all_patterns(oracle_lib):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle_lib.half_to_double(bits, "f16")
    want = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


def test_bfloat16_decode_all_patterns(oracle_lib):
    import torch
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    got = oracle_lib.half_to_double(bits, "bf16")
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(want))
    ok = ~np.isnan(want)
    assert np.array_equal(got[ok], want[ok])


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_context_of_one_returns_v0_exactly(oracle_lib, dtype):
    rng = np.random.default_rng(1)
    q, k, v, t, ctx = random_case(rng, B=2, ctx=[1, 1], dtype=dtype)
    out = oracle_lib.paged_attention(q, k, v, dtype, t, ctx, 0.125)
    for s in range(2):
        for hq in range(4):
            want = brute.widen(v[t[s, 0], 0, hq // 2], dtype)
            assert np.array_equal(out[s, hq], want)


def test_constant_v_returns_v(oracle_lib):
    rng = np.random.default_rng(2)
    q, k, v, t, ctx = random_case(rng, B=3, ctx=[5, 16, 33])
    row = to_bits(rng.standard_normal((2, 8)), "f16")
    for s, c in enumerate(ctx):
        for p in range(c):
            v[t[s, p // 4], p % 4] = row
    out = oracle_lib.paged_attention(q, k, v, "f16", t, ctx, 0.3)
    want = brute.widen(row, "f16")
    for s in range(3):
        for hq in range(4):
            np.testing.assert_allclose(out[s, hq], want[hq // 2], rtol=1e-14, atol=1e-15)


def test_equal_keys_and_zero_scale_give_mean_of_v(oracle_lib):
    rng = np.random.default_rng(3)
    q, k, v, t, ctx = random_case(rng, B=3, ctx=[7, 12, 29])
    krow = to_bits(rng.standard_normal((2, 8)), "f16")
    k_eq = k.copy()
    for s, c in enumerate(ctx):
        for p in range(c):
            k_eq[t[s, p // 4], p % 4] = krow
    out_eq = oracle_lib.paged_attention(q, k_eq, v, "f16", t, ctx, 0.7)
    out_s0 = oracle_lib.paged_attention(q, k, v, "f16", t, ctx, 0.0)
    for s, c in enumerate(ctx):
        V = np.stack([brute.widen(v[t[s, p // 4], p % 4], "f16") for p in range(c)])
        for hq in range(4):
            np.testing.assert_allclose(out_eq[s, hq], V[:, hq // 2].mean(axis=0), rtol=1e-13, atol=1e-14)
            np.testing.assert_allclose(out_s0[s, hq], V[:, hq // 2].mean(axis=0), rtol=1e-13, atol=1e-14)


def test_two_tokens_logistic_weights(oracle_lib):
    rng = np.random.default_rng(4)
    q, k, v, t, ctx = random_case(rng, B=2, ctx=[2, 2], bs=1)
    scale = 0.41
    out = oracle_lib.paged_attention(q, k, v, "f16", t, ctx, scale)
    for s in range(2):
        for hq in range(4):
            qv = brute.widen(q[s, hq], "f16")
            k0, k1 = (brute.widen(k[t[s, p], 0, hq // 2], "f16") for p in (0, 1))
            v0, v1 = (brute.widen(v[t[s, p], 0, hq // 2], "f16") for p in (0, 1))
            x0, x1 = scale * qv.dot(k0), scale * qv.dot(k1)
            w0 = 1.0 / (1.0 + math.exp(x1 - x0))
            w1 = 1.0 / (1.0 + math.exp(x0 - x1))
            np.testing.assert_allclose(out[s, hq], w0 * v0 + w1 * v1, rtol=1e-13, atol=1e-14)


def test_zero_context_gives_zero_row(oracle_lib):
    rng = np.random.default_rng(5)
    q, k, v, t, ctx = random_case(rng, B=3, ctx=[3, 1, 9])
    ctx0 = ctx.copy()
    ctx0[1] = 0
    out = oracle_lib.paged_attention(q, k, v, "f16", t, ctx0, 0.5)
    assert np.array_equal(out[1], np.zeros_like(out[1]))
    assert np.all(np.isfinite(out))


# ------------------------------------------------------- brute force, contiguous

@pytest.mark.parametrize("bs", [1, 2, 4, 16])
@pytest.mark.parametrize("hq,hkv", [(4, 4), (4, 2), (8, 2)])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_matches_brute_force_on_tiny_inputs(oracle_lib, bs, hq, hkv, dtype):
    rng = np.random.default_rng(100 + bs * 10 + hq + hkv)
    q, k, v, t, ctx = random_case(rng, B=4, Hq=hq, Hkv=hkv, D=8, bs=bs, max_ctx=40, dtype=dtype)
    scale = 1.0 / math.sqrt(8)
    got = oracle_lib.paged_attention(q, k, v, dtype, t, ctx, scale)
    want = brute.paged_attention(q, k, v, dtype, t, ctx, scale)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


def test_equals_contiguous_attention(oracle_lib):
    """Rows built contiguously, then paged: paging must not change the result."""
    rng = np.random.default_rng(7)
    n, Hkv, G, D, bs = 53, 2, 3, 16, 4
    Kc = to_bits(rng.standard_normal((n, Hkv, D)), "bf16")
    Vc = to_bits(rng.standard_normal((n, Hkv, D)), "bf16")
    qc = to_bits(rng.standard_normal((1, Hkv * G, D)), "bf16")
    nblk = -(-n // bs)
    table = rng.permutation(40)[:nblk].astype(np.int32)
    kc, vc = page(Kc, table, bs, 40, "bf16"), page(Vc, table, bs, 40, "bf16")
    got = oracle_lib.paged_attention(qc, kc, vc, "bf16", table[None, :], np.array([n], np.int32), 0.25)
    for hq in range(Hkv * G):
        K = brute.widen(Kc[:, hq // G], "bf16")
        V = brute.widen(Vc[:, hq // G], "bf16")
        x = K @ brute.widen(qc[0, hq], "bf16") * 0.25
        w = np.exp(x - x.max())
        np.testing.assert_allclose(got[0, hq], (w @ V) / w.sum(), rtol=1e-12, atol=1e-13)


def test_gqa_equals_mha_with_repeated_kv_heads(oracle_lib):
    """Consecutive grouping: query head hq reads KV head hq // G.  Repeating each
    KV head G times and running MHA must give the same result."""
    rng = np.random.default_rng(8)
    q, k, v, t, ctx = random_case(rng, B=3, Hq=8, Hkv=2, D=8, bs=4, max_ctx=30)
    gqa = oracle_lib.paged_attention(q, k, v, "f16", t, ctx, 0.3)
    k_rep = np.repeat(k, 4, axis=2)
    v_rep = np.repeat(v, 4, axis=2)
    mha = oracle_lib.paged_attention(q, k_rep, v_rep, "f16", t, ctx, 0.3)
    assert np.array_equal(gqa, mha)


# ------------------------------------------------------------------- invariants

def test_block_permutation_invariance_is_bitwise(oracle_lib):
    rng = np.random.default_rng(9)
    q, k, v, t, ctx = random_case(rng, B=4, Hq=4, Hkv=2, D=8, bs=4, max_ctx=45)
    NB = k.shape[0]
    perm = rng.permutation(NB)
    k2 = np.empty_like(k)
    v2 = np.empty_like(v)
    k2[perm] = k
    v2[perm] = v
    t2 = np.where(t >= 0, perm[np.maximum(t, 0)], -1).astype(np.int32)
    a = oracle_lib.paged_attention(q, k, v, "f16", t, ctx, 0.35)
    b = oracle_lib.paged_attention(q, k2, v2, "f16", t2, ctx, 0.35)
    assert np.array_equal(a, b)


def test_stale_slots_do_not_matter(oracle_lib):
    rng = np.random.default_rng(10)
    q, k, v, t, ctx = random_case(rng, B=3, D=8, bs=16, ctx=[5, 17, 31])
    a = oracle_lib.paged_attention(q, k, v, "f16", t, ctx, 0.35)
    assert np.all(np.isfinite(a))
    used = np.zeros(k.shape[:2], dtype=bool)
    for s, c in enumerate(ctx):
        for p in range(c):
            used[t[s, p // 16], p % 16] = True
    junk = rng.integers(0, 1 << 16, size=k.shape, dtype=np.uint16)
    k2 = np.where(used[:, :, None, None], k, junk)
    v2 = np.where(used[:, :, None, None], v, junk[::-1])
    b = oracle_lib.paged_attention(q, k2, v2, "f16", t, ctx, 0.35)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("P", [4, 8, 16, 64])
def test_partition_merge_equals_single_pass(oracle_lib, P):
    rng = np.random.default_rng(11 + P)
    q, k, v, t, ctx = random_case(rng, B=4, Hq=4, Hkv=2, D=8, bs=4, max_ctx=61)
    ref = oracle_lib.paged_attention(q, k, v, "f16", t, ctx, 0.3)
    out, pm, ps, pa = oracle_lib.paged_attention_partitioned(q, k, v, "f16", t, ctx, 0.3, P)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)
    # Every live partition's sum of exp(x - m_j) holds exp(0) = 1 for its own
    # maximum and at most one per token.
    for s, c in enumerate(ctx):
        nparts = -(-int(c) // P)
        for j in range(nparts):
            n_j = min(P, int(c) - j * P)
            assert np.all(ps[s, :, j] >= 1.0) and np.all(ps[s, :, j] <= n_j + 1e-12)
        assert np.all(np.isneginf(pm[s, :, nparts:]))


def test_single_partition_is_bitwise_single_pass(oracle_lib):
    rng = np.random.default_rng(12)
    q, k, v, t, ctx = random_case(rng, B=4, bs=4, max_ctx=40)
    ref = oracle_lib.paged_attention(q, k, v, "f16", t, ctx, 0.3)
    out, *_ = oracle_lib.paged_attention_partitioned(q, k, v, "f16", t, ctx, 0.3, 64)
    assert np.array_equal(out, ref)


# ---------------------------------------------------------- the pages' tables

@pytest.mark.parametrize("row", read_golden("block_tables.txt"), ids=lambda r: r[0][0])
def test_printed_block_tables(oracle_lib, row):
    fields, cite = row
    name, bs, n = fields[0], int(fields[1]), int(fields[2])
    ids = [int(x) for x in fields[3].split(",")]
    assert -(-n // bs) == len(ids), cite
    rng = np.random.default_rng(13)
    D, Hkv = 8, 1
    K = to_bits(rng.standard_normal((n, Hkv, D)), "f16")
    V = to_bits(rng.standard_normal((n, Hkv, D)), "f16")
    qv = to_bits(rng.standard_normal((1, 1, D)), "f16")
    NB = max(ids) + 1
    table = np.array(ids, dtype=np.int32)
    kc, vc = page(K, table, bs, NB, "f16"), page(V, table, bs, NB, "f16")
    got = oracle_lib.paged_attention(qv, kc, vc, "f16", table[None, :], np.array([n], np.int32), 0.5)
    want = brute.attention_contiguous(brute.widen(qv[0, 0], "f16"), brute.widen(K[:, 0], "f16"),
                                      brute.widen(V[:, 0], "f16"), 0.5)
    np.testing.assert_allclose(got[0, 0], want, rtol=1e-12, atol=1e-13)


# ------------------------------------------------------ reshape and block copy

def test_reshape_and_cache_scatter(oracle_lib):
    rng = np.random.default_rng(14)
    NB, bs, Hkv, D, T = 6, 4, 2, 8, 9
    kc = rng.integers(0, 1 << 16, size=(NB, bs, Hkv, D), dtype=np.uint16)
    vc = rng.integers(0, 1 << 16, size=(NB, bs, Hkv, D), dtype=np.uint16)
    key = rng.integers(0, 1 << 16, size=(T, Hkv, D), dtype=np.uint16)
    val = rng.integers(0, 1 << 16, size=(T, Hkv, D), dtype=np.uint16)
    slots = rng.permutation(NB * bs)[:T].astype(np.int64)
    slots[3] = -1                      # padding token: no write
    slots[5] = NB * bs + 2             # out of range: skipped and counted
    k2, v2, bad = oracle_lib.reshape_and_cache(key, val, kc, vc, slots)
    assert bad == 1
    want_k = kc.reshape(NB * bs, Hkv, D).copy()
    want_v = vc.reshape(NB * bs, Hkv, D).copy()
    ok = (slots >= 0) & (slots < NB * bs)
    want_k[slots[ok]] = key[ok]
    want_v[slots[ok]] = val[ok]
    assert np.array_equal(k2.reshape(NB * bs, Hkv, D), want_k)
    assert np.array_equal(v2.reshape(NB * bs, Hkv, D), want_v)


def test_copy_blocks(oracle_lib):
    rng = np.random.default_rng(15)
    NB, bs, Hkv, D = 8, 4, 2, 8
    kc = rng.integers(0, 1 << 16, size=(NB, bs, Hkv, D), dtype=np.uint16)
    vc = rng.integers(0, 1 << 16, size=(NB, bs, Hkv, D), dtype=np.uint16)
    pairs = np.array([[1, 5], [1, 6], [2, 7], [3, 9]], dtype=np.int64)
    k2, v2, bad = oracle_lib.copy_blocks(kc, vc, pairs)
    assert bad == 1
    wk, wv = kc.copy(), vc.copy()
    for s, d in pairs[:3]:
        wk[d] = kc[s]
        wv[d] = vc[s]
    assert np.array_equal(k2, wk) and np.array_equal(v2, wv)


# ------------------------------------------- mutation check of the pins above

MUTANTS = {
    "gqa_mapping": ("int kvh = hq / group;", "int kvh = hq % num_kv_heads;"),
    "block_offset": ("int64_t offset = p % block_size;", "int64_t offset = (p + 1) % block_size;"),
    "v_from_k": ("const uint16_t *vr = v_cache +", "const uint16_t *vr = k_cache +"),
    "dropped_scale": ("x[p] = scale * dot;", "x[p] = dot;"),
}


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_pins_catch_planted_mistakes(mutant):
    """Compile a copy of the oracle with one plausible mistake and check that
    the brute-force pin rejects it (the mistake is planted on the CPU only)."""
    import ctypes
    src = open(os.path.join(os.path.dirname(__file__), "..", "oracle", "pa_oracle.c")).read()
    old, new = MUTANTS[mutant]
    assert src.count(old) >= 1
    src = src.replace(old, new)
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "m.c")
        so = os.path.join(d, "m.so")
        open(c, "w").write(src)
        subprocess.check_call(["gcc", "-O1", "-fPIC", "-shared", "-std=c11", c, "-o", so, "-lm"])
        lib = ctypes.CDLL(so)
        P, i32 = ctypes.c_void_p, ctypes.c_int
        lib.oracle_paged_attention.argtypes = [P, P, P, P, i32, P, i32, P, i32, i32, i32, i32, i32,
                                               ctypes.c_double]
        rng = np.random.default_rng(16)
        q, k, v, t, ctx = random_case(rng, B=3, Hq=4, Hkv=2, D=8, bs=4, max_ctx=30, ctx=[9, 22, 30])
        out = np.zeros(q.shape, dtype=np.float64)
        args = [np.ascontiguousarray(a) for a in (q, k, v, t, ctx)]
        lib.oracle_paged_attention(out.ctypes.data, args[0].ctypes.data, args[1].ctypes.data,
                                   args[2].ctypes.data, 0, args[3].ctypes.data, t.shape[1],
                                   args[4].ctypes.data, 3, 4, 2, 8, 4, 0.35)
        want = brute.paged_attention(q, k, v, "f16", t, ctx, 0.35)
        assert not np.allclose(out, want, rtol=1e-9, atol=1e-9, equal_nan=False)


def test_swap_blocks_between_two_caches(oracle_lib):
    rng = np.random.default_rng(17)
    gpu = rng.integers(0, 1 << 16, size=(9, 4, 2, 8), dtype=np.uint16)
    gpv = rng.integers(0, 1 << 16, size=(9, 4, 2, 8), dtype=np.uint16)
    host_k = np.zeros((5, 4, 2, 8), dtype=np.uint16)
    host_v = np.zeros_like(host_k)
    out_map = np.array([[3, 0], [7, 4], [1, 2], [8, 9]], dtype=np.int64)   # last pair out of range
    hk, hv, bad = oracle_lib.swap_blocks(gpu, gpv, host_k, host_v, out_map)
    assert bad == 1
    want_k, want_v = host_k.copy(), host_v.copy()
    for s, d in out_map[:3]:
        want_k[d], want_v[d] = gpu[s], gpv[s]
    assert np.array_equal(hk, want_k) and np.array_equal(hv, want_v)
    # ... and back in, to other physical blocks.
    in_map = np.array([[0, 5], [4, 6], [2, 0]], dtype=np.int64)
    gk2, gv2, bad = oracle_lib.swap_blocks(hk, hv, gpu, gpv, in_map)
    assert bad == 0
    assert np.array_equal(gk2[5], gpu[3]) and np.array_equal(gk2[6], gpu[7]) and np.array_equal(gk2[0], gpu[1])
    assert np.array_equal(gv2[5], gpv[3]) and np.array_equal(np.delete(gk2, [0, 5, 6], 0), np.delete(gpu, [0, 5, 6], 0))


def test_prefill_is_causal_attention_over_the_paged_context(oracle_lib):
    """Brute force: each query token attends exactly the positions up to its own,
    gathered through the block table; contiguous K/V built before paging."""
    rng = np.random.default_rng(19)
    Hq, Hkv, D, bs = 4, 2, 8, 4
    ctx = [9, 14, 5]
    qlen = [3, 6, 5]            # the last q_len tokens of each sequence are new
    nblk = [-(-c // bs) for c in ctx]
    NB = sum(nblk) + 2
    perm = rng.permutation(NB)
    tables = np.full((3, max(nblk)), -1, dtype=np.int32)
    Ks, Vs = [], []
    kc = np.full((NB, bs, Hkv, D), 0x7E00, dtype=np.uint16)
    vc = kc.copy()
    i = 0
    for s, c in enumerate(ctx):
        tables[s, :nblk[s]] = perm[i:i + nblk[s]]
        i += nblk[s]
        K = to_bits(rng.standard_normal((c, Hkv, D)), "f16")
        V = to_bits(rng.standard_normal((c, Hkv, D)), "f16")
        Ks.append(K)
        Vs.append(V)
        for p in range(c):
            kc[tables[s, p // bs], p % bs] = K[p]
            vc[tables[s, p // bs], p % bs] = V[p]
    cu = np.concatenate([[0], np.cumsum(qlen)]).astype(np.int32)
    q = to_bits(rng.standard_normal((int(cu[-1]), Hq, D)), "f16")
    got = oracle_lib.prefill_attention(q, kc, vc, "f16", tables, np.array(ctx, np.int32), cu, 0.4)
    for s in range(3):
        for j in range(qlen[s]):
            pos = ctx[s] - qlen[s] + j
            for hq in range(Hq):
                K = brute.widen(Ks[s][: pos + 1, hq // 2], "f16")
                V = brute.widen(Vs[s][: pos + 1, hq // 2], "f16")
                want = brute.attention_contiguous(brute.widen(q[cu[s] + j, hq], "f16"), K, V, 0.4)
                np.testing.assert_allclose(got[cu[s] + j, hq], want, rtol=1e-12, atol=1e-13)
    # The last new token of each sequence is exactly that sequence's decode query.
    last = cu[1:] - 1
    dec = oracle_lib.paged_attention(q[last], kc, vc, "f16", tables, np.array(ctx, np.int32), 0.4)
    assert np.array_equal(got[last], dec)


def test_copy_blocks_layers_is_per_layer_copy_blocks(oracle_lib):
    """[layers, 2, NB, bs, Hkv, D]: every layer's K and V get the same block copies;
    checked against NumPy assignment layer by layer, bad pairs counted per layer."""
    rng = np.random.default_rng(23)
    L, NB, bs, Hkv, D = 3, 10, 4, 2, 8
    kv = rng.integers(0, 2**16, size=(L, 2, NB, bs, Hkv, D), dtype=np.uint16)
    pairs = np.array([[1, 7], [3, 2], [9, 4], [12, 5], [0, -1]], dtype=np.int64)
    got, bad = oracle_lib.copy_blocks_layers(kv, pairs)
    want = kv.copy()
    for layer in range(L):
        for src, dst in pairs:
            if 0 <= src < NB and 0 <= dst < NB:
                want[layer, :, dst] = kv[layer, :, src]
    assert np.array_equal(got, want) and bad == 2 * L
    bytes_kv = rng.integers(0, 256, size=(2, 2, NB, bs, Hkv, 16), dtype=np.uint8)
    got8, _ = oracle_lib.copy_blocks_layers(bytes_kv, pairs[:3])
    want8 = bytes_kv.copy()
    for layer in range(2):
        for src, dst in pairs[:3]:
            want8[layer, :, dst] = bytes_kv[layer, :, src]
    assert np.array_equal(got8, want8)
