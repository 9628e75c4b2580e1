"""GPU parity of the FP8 (e4m3) KV-cache path against the CPU oracle.

The quantising reshape_and_cache must produce the oracle's codes bit for bit
(code = e4m3(fp32(x) / scale), nearest-even, saturating); attention over the
e4m3 cache must stay within 2e-3 of the oracle's fp64 result on the same codes.
"""
import numpy as np
import pytest

import oracle
from paged_kv_cache_140_gb300 import workloads as W

from pa_harness import assert_attention_close, cache_bits, run_step

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_140_gb300 import _build
    _build.build()
    oracle.build()


def check(b, out_dtype="f32", partition_size=None, caches=True):
    assert b.cache_dtype == "fp8"
    ref, kc, vc = oracle.decode_step(b)
    out, T, flag = run_step(b, out_dtype=out_dtype, partition_size=partition_size)
    assert flag == 0, f"err_flag {flag:#x}"
    assert_attention_close(out, ref, b.dtype if out_dtype == "native" else out_dtype, b.name + "/fp8")
    if caches:
        assert np.array_equal(cache_bits(T["k_cache"]), kc), "k_cache codes differ from oracle"
        assert np.array_equal(cache_bits(T["v_cache"]), vc), "v_cache codes differ from oracle"
    return out


CASES = [
    ("13b", dict(num_seqs=24)),
    ("7b", dict(num_seqs=6)),
    ("gqa", dict(num_seqs=2, ctx_cap=12000)),
    ("gqa32", dict(num_seqs=2, ctx_cap=12000)),
    ("prefix", dict(groups=2)),
]


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("out_dtype", ["f32", "native"])
def test_fp8_workloads(name, kw, out_dtype):
    check(W.make_batch(name, cache_dtype="fp8", **kw), out_dtype)


@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (16, 4), (16, 2)])
@pytest.mark.parametrize("qdt", ["f16", "bf16"])
def test_fp8_groups_and_query_types(hq, hkv, qdt):
    b = W.make_batch("7b", num_seqs=4, ctx_cap=700, num_heads=hq, num_kv_heads=hkv, dtype=qdt,
                     cache_dtype="fp8")
    check(b, "f32", partition_size=128)


@pytest.mark.parametrize("P", [0, 16, 48, 512])
def test_fp8_partition_sizes(P):
    check(W.make_batch("13b", num_seqs=6, cache_dtype="fp8"), "f32", partition_size=P, caches=False)


@pytest.mark.parametrize("bs", [8, 32])
def test_fp8_block_sizes(bs):
    check(W.make_batch("13b", num_seqs=8, block_size=bs, cache_dtype="fp8"), "f32",
          partition_size=128 if bs == 8 else 0)


def test_fp8_edge_lengths():
    b = W.make_batch("7b", context_lens=[0, 1, 16, 17, 0, 2048, 255, 257], cache_dtype="fp8")
    out = check(b, "f32")
    o = out.cpu().numpy()
    assert np.all(o[0] == 0) and np.all(o[4] == 0)


def test_fp8_full_size_every_row():
    """The 13B-shaped e4m3 workload at full size: every output element against
    the e4m3 oracle, both caches bit-exact after the quantising writes."""
    b = W.make_batch("13b_fp8")
    ref, kc, vc = oracle.decode_step(b)
    out, T, flag = run_step(b, out_dtype="native")
    assert flag == 0
    assert_attention_close(out, ref, b.dtype, "13b_fp8 full size")
    assert np.array_equal(cache_bits(T["k_cache"]), kc)
    assert np.array_equal(cache_bits(T["v_cache"]), vc)


def _spike_keys(b, every=64, step=9.0):
    """The e4m3 batch with a spike key every `every` positions: at the i-th
    one (position every * i) each KV head's cache row points along the first
    query of its group, with a length that puts that query's score at
    step * i in log2 units, so a row's running max jumps past the
    lazy-rescale margin (8) again and again."""
    import dataclasses
    G = b.num_heads // b.num_kv_heads
    sl = float(b.scale) * 1.4426950408889634
    bs = b.block_size
    q = b.q.astype(np.uint32)
    qf = (q << 16).view(np.float32) if b.dtype == "bf16" else b.q.view(np.float16).astype(np.float32)
    kc = b.k_cache.copy()
    seen = set()
    for s in range(b.num_seqs):
        ctx = int(b.context_lens[s])
        for i, pos in enumerate(range(every, ctx - 1, every), start=1):
            blk, off = int(b.block_tables[s, pos // bs]), pos % bs
            if (blk, off) in seen:
                continue
            seen.add((blk, off))
            for h in range(b.num_kv_heads):
                qm = qf[s, h * G].astype(np.float64)
                n2 = float(qm @ qm)
                k = qm * (step * i / sl) / n2
                kc[blk, off, h] = oracle.e4m3_encode((k / b.k_scale).astype(np.float32))
    return dataclasses.replace(b, k_cache=kc)


@pytest.mark.parametrize("hq,hkv,qdt,P", [(8, 8, "bf16", 0), (32, 8, "f16", 48), (16, 4, "bf16", 0)])
def test_fp8_rescales_as_the_max_grows(hq, hkv, qdt, P):
    """Spike keys whose scores climb by 9 (log2 units) every 64 positions make
    each row's running max overtake the lazy-rescale margin throughout the
    context, in the two-stages-per-slot e4m3 consumer (G = 1 and 4) and in
    the per-warp kernel (4 KV heads)."""
    b = W.make_batch("7b", num_seqs=4, ctx_cap=700, num_heads=hq, num_kv_heads=hkv, dtype=qdt,
                     cache_dtype="fp8")
    b = _spike_keys(b)
    codes = oracle.e4m3_decode(b.k_cache)
    assert np.nanmax(np.abs(codes)) < 448     # no spike saturated
    check(b, "f32", partition_size=P)
