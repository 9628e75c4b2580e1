"""GPU checks of the CTA-cooperative decode kernel (16-bit or e4m3 caches
whose KV heads come in groups of 8, head_dim 128, block size a multiple of
16): parity with the oracle for every group size, including G = 8 (shallower
ring), both query types over an e4m3 cache, sequences that share physical
blocks (served together from one copy of each shared stage), and, for 16-bit
caches, bit equality with the per-warp kernel, which a child process selects
with PA_DECODE_COOP=0."""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from paged_kv_cache_140_gb300 import workloads as W

from pa_harness import assert_attention_close, run_step

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_140_gb300 import _build
    _build.build()
    oracle.build()


CASES = [   # (workload, Hq, Hkv, dtype, block size)
    ("7b", 8, 8, "f16", 16),
    ("7b", 16, 8, "bf16", 16),
    ("7b", 32, 8, "bf16", 32),
    ("7b", 64, 8, "f16", 16),
    ("7b", 32, 16, "bf16", 64),
    ("7b", 48, 24, "f16", 16),
]


@pytest.mark.parametrize("name,hq,hkv,dtype,bs", CASES, ids=[f"{c[1]}x{c[2]}-{c[3]}-bs{c[4]}" for c in CASES])
def test_cooperative_kernel_matches_oracle(name, hq, hkv, dtype, bs):
    b = W.make_batch(name, num_seqs=6, ctx_cap=1500, num_heads=hq, num_kv_heads=hkv, dtype=dtype,
                     block_size=bs)
    ref, kc, vc = oracle.decode_step(b)
    out, T, flag = run_step(b)
    assert flag == 0
    assert_attention_close(out, ref, "f32", f"coop {hq}/{hkv} {dtype} bs {bs}")


BIT_CASES = [   # (workload, Hq, Hkv, dtype, partition size)
    ("7b", 40, 40, "bf16", None),
    ("7b", 32, 8, "bf16", None),
    ("7b", 64, 8, "f16", None),
    ("shared", 8, 8, "f16", None),       # runs of sequences sharing blocks, one member column each
    ("shared", 16, 8, "bf16", 48),       # G = 2: two members per run
    ("shared", 8, 8, "bf16", 16),        # every stage its own partition
    ("prefix", 32, 32, "f16", None),     # the prefix-sharing workload (three prompt groups)
]


@pytest.mark.parametrize("name,hq,hkv,dtype,P", BIT_CASES,
                         ids=[f"{c[0]}-{c[1]}x{c[2]}-{c[3]}-P{c[4]}" for c in BIT_CASES])
def test_cooperative_and_per_warp_kernels_agree_bit_for_bit(tmp_path, name, hq, hkv, dtype, P):
    """The per-warp kernel handles every sequence on its own; the cooperative
    kernel serves sequences that share a stage's block from one copy of it.
    Each sequence's arithmetic is the same, so the outputs agree bit for bit."""
    outs = {}
    for coop in ("1", "0"):
        path = str(tmp_path / f"out_{coop}.npy")
        env = dict(os.environ, PA_DECODE_COOP=coop)
        args = [sys.executable, os.path.join(HERE, "coop_child.py"), name, str(hq), str(hkv), dtype, path]
        if P is not None:
            args.append(str(P))
        r = subprocess.run(args, env=env, capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, r.stderr[-2000:]
        outs[coop] = np.load(path)
    assert np.array_equal(outs["1"], outs["0"])


SHARED_CASES = [   # (Hq, Hkv, dtype, block size, partition size)
    (8, 8, "f16", 16, 0),
    (8, 8, "bf16", 16, 16),
    (16, 8, "bf16", 32, 48),
    (8, 8, "f16", 64, 256),
    (32, 8, "bf16", 16, 0),     # G = 4: no runs, every sequence on its own
]


@pytest.mark.parametrize("hq,hkv,dtype,bs,P", SHARED_CASES,
                         ids=[f"{c[0]}x{c[1]}-{c[2]}-bs{c[3]}-P{c[4]}" for c in SHARED_CASES])
def test_sequences_sharing_blocks_match_oracle(hq, hkv, dtype, bs, P):
    """Chains of sequences reading the same leading physical blocks: longer
    than one run, with members ending before, inside and after the shared
    blocks, and two sequences equal but for their last block."""
    from pa_harness import cache_bits, shared_prefix_batch
    b = shared_prefix_batch(num_heads=hq, num_kv_heads=hkv, dtype=dtype, block_size=bs)
    ref, kc, vc = oracle.decode_step(b)
    out, T, flag = run_step(b, partition_size=P)
    assert flag == 0
    assert_attention_close(out, ref, "f32", f"shared blocks {hq}/{hkv} {dtype} bs {bs} P {P}")
    assert np.array_equal(cache_bits(T["k_cache"]), kc)


def test_shared_block_with_bad_id_is_flagged_and_isolated():
    """A bad block id inside a run's shared prefix: the run's members skip it
    and flag it; sequences outside the run are untouched."""
    import paged_kv_cache_140_gb300 as pa
    from pa_harness import shared_prefix_batch
    b = shared_prefix_batch(num_heads=8, num_kv_heads=8)
    b.block_tables[0:4, 3] = b.num_blocks + 9
    out, _, flag = run_step(b)
    assert flag & pa.FLAG_BAD_BLOCK_ID
    keep = list(range(4, b.num_seqs))
    ref, _, _ = oracle.decode_step(W.subset_batch(b, keep))
    assert_attention_close(out[keep], ref, "f32", "sequences outside the run")
    assert np.all(np.isfinite(out[:4].float().cpu().numpy()))


FP8_CASES = [   # (Hq, Hkv, query dtype, block size)
    (8, 8, "f16", 16),
    (16, 8, "bf16", 16),
    (32, 8, "f16", 32),
    (64, 8, "bf16", 16),
    (48, 24, "bf16", 64),
    (40, 40, "f16", 16),
]


@pytest.mark.parametrize("hq,hkv,qdt,bs", FP8_CASES, ids=[f"{c[0]}x{c[1]}-{c[2]}-bs{c[3]}" for c in FP8_CASES])
def test_cooperative_kernel_fp8_matches_oracle(hq, hkv, qdt, bs):
    """e4m3 cache: 8-head boxes of 128 codes per row, codes widened to f16 in
    registers; unused slots hold NaN codes."""
    b = W.make_batch("7b", num_seqs=6, ctx_cap=1500, num_heads=hq, num_kv_heads=hkv, dtype=qdt, block_size=bs,
                     cache_dtype="fp8")
    ref, _, _ = oracle.decode_step(b)
    out, _, flag = run_step(b)
    assert flag == 0
    assert_attention_close(out, ref, "f32", f"coop fp8 {hq}/{hkv} {qdt} bs {bs}")


@pytest.mark.parametrize("P", [16, 48, 0])
def test_cooperative_kernel_fp8_ragged_lengths(P):
    """Empty, one-token and stage-boundary contexts with small partitions
    (ragged last stages, many split sequences) over an e4m3 cache."""
    b = W.make_batch("13b", context_lens=[0, 1, 15, 16, 17, 31, 33, 2048, 0, 100], cache_dtype="fp8")
    ref, _, _ = oracle.decode_step(b)
    out, _, flag = run_step(b, partition_size=P)
    assert flag == 0
    assert_attention_close(out, ref, "f32", f"coop fp8 ragged P={P}")
    o = out.cpu().numpy()
    assert np.all(o[0] == 0) and np.all(o[8] == 0)


def test_cooperative_kernel_fp8_bad_block_id_is_flagged_and_isolated():
    """A block id outside the pool in an e4m3 cache is skipped and flagged;
    the other sequences are untouched and the affected row stays finite."""
    import paged_kv_cache_140_gb300 as pa
    b = W.make_batch("13b", num_seqs=8, cache_dtype="fp8")
    s_bad = int(np.argmax(b.context_lens))
    b.block_tables[s_bad, 0] = b.num_blocks + 5
    out, _, flag = run_step(b)
    assert flag & pa.FLAG_BAD_BLOCK_ID
    keep = [s for s in range(8) if s != s_bad]
    ref, _, _ = oracle.decode_step(W.subset_batch(b, keep))
    assert_attention_close(out[keep], ref, "f32", "unaffected sequences, fp8")
    assert np.all(np.isfinite(out[s_bad].float().cpu().numpy()))


def test_cooperative_kernel_fp8_is_bitwise_reproducible():
    b = W.make_batch("gqa", num_seqs=2, ctx_cap=9000, cache_dtype="fp8")
    a, _, fa = run_step(b)
    c, _, fc = run_step(b)
    assert fa == 0 and fc == 0
    assert np.array_equal(a.cpu().numpy().view(np.uint32), c.cpu().numpy().view(np.uint32))


def _ramp_keys(b, per_token):
    """The decode batch with every key row at position p scaled by
    1 + p * per_token (each physical cache row once, and the step's new rows
    at position ctx - 1), so that a row's running max keeps growing past the
    lazy-rescale margin from stage to stage."""
    import dataclasses

    def dec(bits):
        if b.dtype == "f16":
            return bits.view(np.float16).astype(np.float32)
        return (bits.astype(np.uint32) << 16).view(np.float32)

    def enc(x):
        if b.dtype == "f16":
            return x.astype(np.float16).view(np.uint16)
        u = x.astype(np.float32).view(np.uint32)
        return ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)

    bs = b.block_size
    kc = b.k_cache.copy()
    key = b.key.copy()
    seen = set()
    for s in range(b.num_seqs):
        ctx = int(b.context_lens[s])
        for pos in range(ctx - 1):
            blk, off = int(b.block_tables[s, pos // bs]), pos % bs
            if (blk, off) not in seen:
                seen.add((blk, off))
                kc[blk, off] = enc(dec(kc[blk, off]) * (1.0 + pos * per_token))
        if ctx > 0:
            key[s] = enc(dec(key[s]) * (1.0 + (ctx - 1) * per_token))
    return dataclasses.replace(b, k_cache=kc, key=key)


RAMP_CASES = [   # (batch, Hq, Hkv, dtype, head_dim, partition size)
    ("7b", 8, 8, "f16", 128, 0),        # cooperative kernel, one query row per KV head
    ("7b", 32, 8, "bf16", 128, 48),     # cooperative, G = 4, many partitions
    ("7b", 8, 4, "bf16", 128, 0),       # per-warp kernel (KV heads not a multiple of 8)
    ("7b", 8, 8, "f16", 64, 16),        # per-warp kernel, head_dim 64, a partition per stage
    ("shared", 8, 8, "f16", 128, 0),    # runs of sequences sharing blocks, one member column each
    ("shared", 16, 8, "bf16", 128, 48), # runs with G = 2
]


@pytest.mark.parametrize("name,hq,hkv,dtype,d,P", RAMP_CASES,
                         ids=[f"{c[0]}-{c[1]}x{c[2]}-{c[3]}-d{c[4]}-P{c[5]}" for c in RAMP_CASES])
def test_decode_rescales_as_the_max_grows(name, hq, hkv, dtype, d, P):
    """Keys that grow with their position raise each row's running max past
    the lazy-rescale margin every few stages, so the partial outputs are
    rescaled throughout the context (and the merge combines partitions whose
    maxima differ widely), on both kernels and in runs of shared blocks."""
    from pa_harness import shared_prefix_batch
    if name == "shared":
        b = shared_prefix_batch(num_heads=hq, num_kv_heads=hkv, dtype=dtype, block_size=16)
    else:
        b = W.make_batch(name, num_seqs=6, ctx_cap=1500, num_heads=hq, num_kv_heads=hkv, dtype=dtype,
                         head_dim=d)
    b = _ramp_keys(b, 1.0 / 16)
    ref, _, _ = oracle.decode_step(b)
    out, _, flag = run_step(b, partition_size=P)
    assert flag == 0
    assert_attention_close(out, ref, "f32", f"ramped keys {name} {hq}/{hkv} {dtype} D {d} P {P}")
